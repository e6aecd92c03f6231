"""The stored tiny-step values (tests/golden/tiny_step.json, written by
tests/golden/make_golden.py from the oracle) against the oracle as it stands
(CPU) and against the library (GPU)."""
import hashlib
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
from streaming_avatar_video_gb300 import inputs as I
from tests._util import assert_close

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_step.json")))


def tiny_inputs():
    w = I.WORKLOADS["tiny"]
    st = I.step_inputs(w, 0, 0, 0)
    rk, rv = I.reference_kv(w, 0)
    wo = I.out_proj_weight(w, 0)
    x0 = I.state_x(w, 0)
    digest = hashlib.sha256()
    for t in (st.q, st.k, st.v, rk, rv, wo):
        digest.update(t.view(torch.int16).numpy().tobytes())
    digest.update(x0.numpy().tobytes())
    assert digest.hexdigest() == GOLDEN["inputs_sha256"], "the seeded generator no longer reproduces the stored inputs"
    return w, st, rk, rv, wo, x0


def test_oracle_reproduces_golden():
    w, st, rk, rv, wo, x0 = tiny_inputs()
    f = lambda t: t.double().numpy()
    rk_rot = O.rope3d(f(rk), 1, w.grid_h, w.grid_w, -1)
    empty = np.zeros((1, 0, w.H, w.D))
    x1, o = O.chunk_step(f(st.q), f(st.k), f(st.v), rk_rot, f(rv), empty, empty, f(wo), f(x0), 0.25,
                         (w.F, w.grid_h, w.grid_w))
    assert np.allclose(x1.reshape(-1)[GOLDEN["x_index"]], GOLDEN["x_value"], rtol=0, atol=1e-12)
    assert np.allclose(o.reshape(-1)[GOLDEN["o_index"]], GOLDEN["o_value"], rtol=0, atol=1e-12)


@pytest.mark.gpu
def test_library_matches_golden():
    import __graft_entry__ as g
    g.build()
    from streaming_avatar_video_gb300 import savgb as S
    w, st, rk, rv, wo, x0 = tiny_inputs()
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, 1, 0)
    cs.set_reference(rk.cuda(), rv.cuda())
    x = x0.cuda()
    cs.step(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo.cuda(), x, 0.25, True)
    cs.end_chunk()
    cs.sync()
    got = x.cpu().double().numpy().reshape(-1)[GOLDEN["x_index"]]
    assert_close(got, GOLDEN["x_value"], what="tiny step x vs golden")
    cs.close()
