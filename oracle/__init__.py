"""Plain fp64 CPU oracle of one chunk denoising step (TEST INFRASTRUCTURE).

This package exists to check the CUDA library.  Only the tests, the smoke check
in ``__graft_entry__`` and the CPU-baseline legs of ``bench.py`` may import it;
the library's product path never does, and it shares no code with the library
(no headers, tables, constants or helpers).

What it computes follows HeyGen, "Avatar inference at scale":

* section "The underlying model architecture": the generator is a Diffusion
  Transformer trained with flow matching that attends to rich reference
  tokens; long videos are produced chunk by chunk, the first chunk relying on
  the static reference only and later chunks also on boundary data from the
  previous chunk.
* section "The streaming framework and pipeline loop": the reference identity
  is encoded once per request; the audio-to-video stage runs a multi-step
  diffusion pass per chunk, conditioned on the previous chunk's boundary
  frames.
* section "Boundary continuity and chunk consistency": interpolation (I)
  chunks between consecutive N chunks, generated after both, anchored on the
  previous chunk's last frame and the next chunk's first frame, anchor
  predictions discarded.
* section "Constant memory over duration": only the static reference
  conditioning and a minimal set of carried tensors survive from chunk to
  chunk.

The pages state the problem but no operator.  The operator-level readings
used here (3D RoPE split and frequencies, softmax scale, Euler rule, shifted
time grid, what the boundary holds) are the plainest ones consistent with the
pages and are listed with each function.  Everything is float64 computed from
the bfloat16-rounded inputs; no intermediate is rounded to bfloat16.

Parity pins (tests/test_oracle_pins.py) check every function here against
closed forms, invariants, complex-number rotations and brute-force loops
written separately; no function is "parity unpinned".
"""
from .step import (  # noqa: F401
    rope_axis_split,
    rope_frequencies,
    token_positions,
    rope3d,
    softmax_rows,
    attention,
    out_proj,
    euler_update,
    time_grid,
    boundary_from_chunk,
    chunk_step,
    run_stream,
    anchors_from_chunk,
    ichunk_step,
    run_stream_ni,
    qkv_project,
    block_step,
    run_stream_block,
)
