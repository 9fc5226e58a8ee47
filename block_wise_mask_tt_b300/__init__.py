"""TwoTower block-wise mask-diffusion denoise step on B300 (sm_103a).

The compute lives in ``libtt.so`` (CUDA kernels behind a C ABI, declared in
``include/tt.h``); ``block_wise_mask_tt_b300.tt`` is the thin ctypes binding and is
imported lazily so that the seeded input generators (``synth``) stay usable on
machines without the library.
"""
__all__ = ["synth"]
