"""GB300 (sm_103a) library for one denoising step of a chunked, flow-matching
Diffusion-Transformer avatar video generator.

The compute path is the C ABI of ``include/savgb.h``, implemented by the
hand-written CUDA kernels under ``csrc/`` and built in tree into
``libsavgb.so``; :mod:`streaming_avatar_video_gb300.savgb` is its Python
binding.  :mod:`streaming_avatar_video_gb300.inputs` holds the seeded
synthetic workloads.
"""

__all__ = ["savgb", "inputs", "build"]
