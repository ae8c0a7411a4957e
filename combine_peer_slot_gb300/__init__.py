"""GB300 (sm_103a) library for the FFN side of Attention-FFN Disaggregation:
peer-slot fan-in, router, permutation, grouped SwiGLU experts, combine and
per-peer split.  `afd` is the ctypes binding of the C ABI in include/afd.h;
`workloads` draws the seeded synthetic inputs; `runtime` holds device-buffer
helpers built on torch (allocation and streams only)."""
