"""wgemm: dense C = A·Bᵀ (fp16 in, fp32 accumulate and out) on GB300 (sm_103a).

The compute path is the C-ABI library libwgemm.so (hand-written tcgen05 / TMA
kernels, declared in include/wgemm.h); `wgemm` is its ctypes binding and
`inputs` the seeded synthetic-input generator. Submodules load lazily, so
importing the package needs neither a GPU nor the built library.
"""
__all__ = ["wgemm", "inputs", "build"]
