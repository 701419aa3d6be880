"""The kernel digest that ties a committed ncu summary to the sources it was taken on ignores
commentary and nothing else."""
from speculative_decode_verify_gdn_gb300 import build


def test_code_only_drops_comments_and_keeps_literals():
    src = 'asm("mov.u32 %0, 1; // kept");  // dropped\nint a = 1; /* dropped\n too */ int b = \'/\';\n'
    assert build._code_only(src) == 'asm("mov.u32 %0, 1; // kept"); int a = 1; int b = \'/\';'


def test_code_only_sees_code_changes():
    assert build._code_only("x = a + b;") != build._code_only("x = a - b;")
    assert build._code_only("x = a + b; // one") == build._code_only("x  =  a + b;\n// two")


def test_digest_is_stable_and_short():
    d = build.kernel_source_digest()
    assert d == build.kernel_source_digest()
    assert len(d) == 16 and int(d, 16) >= 0


def test_verify_digest_covers_exactly_the_verify_translation_unit():
    """gdn_verify.cu includes gdn_common.cuh and gdn_kernels.h (which include gdn.h) and nothing
    else of this library, so those files are the ones its digest must cover."""
    import os
    import re
    src = open(os.path.join(build.CSRC_DIR, "gdn_verify.cu")).read()
    local = set(re.findall(r'#include "([^"]+)"', src))
    assert local == {"gdn_common.cuh", "gdn_kernels.h"}
    assert set(build.VERIFY_SOURCES) == {"gdn_verify.cu"} | local
    d = build.verify_kernel_digest()
    assert len(d) == 16 and d == build.verify_kernel_digest() and d != build.kernel_source_digest()
