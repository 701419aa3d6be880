"""CPU oracle for the GDN verify step (test infrastructure, not the product path)."""
