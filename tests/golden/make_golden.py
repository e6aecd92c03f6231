"""Writes tests/golden/tiny_step.json: the fp64 oracle's result of one
denoising step of the tiny chunk-0 workload (2 heads of 64, a 2x4x4 chunk, one
4x4 reference frame at t = -1, no boundary, dt = 0.25) on the seed-0 inputs.

The values come from oracle/ alone (HeyGen, "Avatar inference at scale", section
"The underlying model architecture": the first chunk relies on the static
reference only).  The GPU tests and the smoke check compare the library with
them.  Run from the repository root:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from streaming_avatar_video_gb300 import inputs as I  # noqa: E402


def main():
    w = I.WORKLOADS["tiny"]
    seed, dt = 0, 0.25
    st = I.step_inputs(w, seed, 0, 0)
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed)
    x0 = I.state_x(w, seed)
    f = lambda t: t.double().numpy()
    rk_rot = O.rope3d(f(rk), w.ref_frames, w.grid_h, w.grid_w, w.ref_t, w.rope_base)
    empty = np.zeros((w.B, 0, w.H, w.D))
    x1, o = O.chunk_step(f(st.q), f(st.k), f(st.v), rk_rot, f(rv), empty, empty, f(wo), f(x0), dt,
                         (w.F, w.grid_h, w.grid_w), w.rope_base)
    rng = np.random.default_rng(123)
    x_idx = sorted(rng.choice(x1.size, 96, replace=False).tolist())
    o_idx = sorted(rng.choice(o.size, 96, replace=False).tolist())
    digest = hashlib.sha256()
    for t in (st.q, st.k, st.v, rk, rv, wo):
        digest.update(t.view(dtype=__import__("torch").int16).numpy().tobytes())
    digest.update(x0.numpy().tobytes())
    out = {
        "inputs_sha256": digest.hexdigest(),
        "what": "fp64 oracle, tiny chunk-0 step (B1 H2 D64, 2x4x4 chunk, 16 reference tokens at t=-1, dt=0.25), seed 0",
        "written_by": "tests/golden/make_golden.py (calls oracle/ and the seeded input generator only)",
        "x_shape": list(x1.shape), "o_shape": list(o.shape),
        "x_index": x_idx, "x_value": [float(x1.reshape(-1)[i]) for i in x_idx],
        "o_index": o_idx, "o_value": [float(o.reshape(-1)[i]) for i in o_idx],
        "x_mean": float(x1.mean()), "x_std": float(x1.std()),
        "o_abs_mean": float(np.abs(o).mean()),
    }
    path = os.path.join(ROOT, "tests", "golden", "tiny_step.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
