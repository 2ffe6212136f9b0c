"""GB300 (sm_103a) hot path of Looped Latent Attention: latent encode and
latent-store decode attention, as a C-ABI CUDA library (``lib/liblla.so``,
declared in ``include/lla.h``) with a thin ctypes binding (:mod:`.lla`).

Source: "Looped Latent Attention: Cross-Loop KV Compression for Looped
Transformers" (arXiv 2607.15456v2).
"""
__all__ = ["lla", "synth", "build"]
