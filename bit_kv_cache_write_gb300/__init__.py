"""GB300-native OSCAR hot path: INT2 KV-cache write/demote and paged INT2 decode.

The compute lives in ``liboscar.so`` (hand-written CUDA for sm_103a behind a C
ABI declared in ``include/oscar.h``). ``bit_kv_cache_write_gb300.oscar`` is the
thin ctypes binding; ``synth`` draws the seeded synthetic inputs;
``calibration`` is the host-side offline calibration that produces the
rotations and thresholds the library consumes.

Importing this package does not load the CUDA library; the binding loads it on
first use and raises if it is missing.
"""
