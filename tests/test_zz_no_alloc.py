"""The allocation-free chunk step against the stream step.

chunk_step_noalloc exists for callers that cannot call cudaMalloc (a plugin in
a runtime that owns every device allocation, a real-time loop that may not
allocate once the session runs): its intermediates live in a fixed device
array inside the library.  Here it must give what chunk_stream_step gives on
the same inputs and state, on two calls in a row (the second reuses the
array the first filled), within the parity tolerance of the other tests.
This file is named so that pytest collects it last."""
import pytest
import torch

from streaming_avatar_video_gb300 import inputs as I
from tests._util import assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import __graft_entry__ as g
    g.build()
    from streaming_avatar_video_gb300 import savgb
    torch.cuda.set_device(0)
    return savgb


@pytest.mark.parametrize("w", [
    I.WORKLOADS["small"],
    I.Workload("d128", B=2, H=4, D=128, F=3, grid_h=8, grid_w=12, ref_frames=1, boundary_frames=1,
               steps=4, shift=3.0),
    # a 2 x 400 grid: the q RoPE table does not fit the attention kernel, so both take the unfused form
    I.Workload("wide", B=1, H=2, D=128, F=2, grid_h=2, grid_w=400, ref_frames=1, boundary_frames=1,
               steps=2, shift=1.0),
], ids=["small", "d128", "wide"])
def test_noalloc_step_matches_stream_step(S, w):
    seed = 17
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed).cuda()
    dts = S.flow_time_grid(w.steps, w.shift)
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base)
    cs.set_reference(rk.cuda(), rv.cuda())
    # chunk 0 through the stream, so that chunk 1 has a boundary
    x = I.state_x(w, seed).cuda()
    for s, dt in enumerate(dts):
        st = I.step_inputs(w, seed, 0, s)
        cs.step(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, x, dt, s == len(dts) - 1)
    cs.end_chunk()
    cs.sync()
    bk, bv = cs.boundary()
    ref_rot = torch.empty_like(rk).cuda()
    S.rope3d_apply(rk.cuda(), ref_rot, w.ref_frames, w.grid_h, w.grid_w, w.ref_t - w.ref_frames + 1,
                   w.rope_base)
    context = [(ref_rot, rv.cuda()), (bk.cuda(), bv.cuda())]

    x0 = torch.from_numpy(I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, 1)).cuda()
    x_stream, x_static = x0.clone(), x0.clone()
    for s in range(2):  # two calls in a row
        st = I.step_inputs(w, seed, 1, s)
        q, k, v = st.q.cuda(), st.k.cuda(), st.v.cuda()
        cs.step(q, k, v, wo, x_stream, dts[s], False)
        S.chunk_step_noalloc(q, k, v, context, wo, x_static, dts[s], (w.F, w.grid_h, w.grid_w),
                             rope_base=w.rope_base)
        torch.cuda.synchronize()
        S.savgb_device_check()
        assert_close(f64(x_static), f64(x_stream), what=f"{w.name} call {s}")
        assert not torch.equal(x_static, x0)
    cs.close()


def test_noalloc_rejects_steps_beyond_scratch(S):
    # a base-DiT-sized chunk needs 2 x 12480 x 3072 x 2 bytes and the RoPE table, beyond the fixed array
    w = I.WORKLOADS["base"]
    q = torch.zeros((1, 16, 24, 128), dtype=torch.bfloat16, device="cuda")  # pointers only
    wo = torch.zeros((w.hid, w.hid), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((16, w.hid), dtype=torch.float32, device="cuda")
    L = S.lib()
    rc = L.chunk_step_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), None, 0, wo.data_ptr(), None, x.data_ptr(),
                              0.1, 1, w.H, w.D, w.F, w.grid_h, w.grid_w, 1e4, 0.0, None)
    assert rc == -1
    msg = L.savgb_last_error().decode()
    assert "scratch" in msg and str(S.NOALLOC_SCRATCH_BYTES) in msg
