"""GB300 (sm_103a) speculative-decoding verify step of one Gated DeltaNet layer.

* ``gdn``      - ctypes binding of the C ABI in include/gdn.h (libgdn_sm103a.so)
* ``runtime``  - device buffers of one layer and the verify -> rollback round
* ``synth``    - seeded synthetic inputs of the named workloads
* ``build``    - in-tree nvcc build of the library for sm_103a

Importing the package loads nothing; ``gdn.load_library()`` (called by every
binding function) raises if the library has not been built.
"""
