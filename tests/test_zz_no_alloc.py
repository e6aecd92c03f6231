"""The allocation-free chunk step against the fp64 oracle and the stream step.

chunk_step_noalloc exists for callers that cannot call cudaMalloc (a plugin in
a runtime that owns every device allocation, a real-time loop that may not
allocate once the session runs): its intermediates live in a fixed device
array inside the library.  Here it must give what the oracle's chunk step
gives on the same seeded inputs, and what chunk_stream_step gives on the same
inputs and state, on two calls in a row (the second reuses the array the
first filled), within the parity tolerance of the other tests.  This file is
named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import oracle as O
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


D128 = I.Workload("d128", B=2, H=4, D=128, F=3, grid_h=8, grid_w=12, ref_frames=1, boundary_frames=1,
                  steps=4, shift=3.0)
# a 2 x 400 grid: the q RoPE table does not fit the attention kernel, so the step takes the unfused form
WIDE = I.Workload("wide", B=1, H=2, D=128, F=2, grid_h=2, grid_w=400, ref_frames=1, boundary_frames=1,
                  steps=2, shift=1.0)


def _context_segments(w, seed, n_context):
    """Rotated context segments as the caller would hold them: the reference
    (frames ending at ref_t) and a boundary (t = -T_b..-1), rotated by the
    oracle in fp64 and rounded to bf16, the precision the entry point takes."""
    rk, rv = I.reference_kv(w, seed)
    bk, bv = I.boundary_kv(w, seed)
    ref_k = torch.from_numpy(O.rope3d(f64(rk), w.ref_frames, w.grid_h, w.grid_w, w.ref_t - w.ref_frames + 1,
                                      w.rope_base)).to(torch.bfloat16)
    bnd_k = torch.from_numpy(O.rope3d(f64(bk), w.boundary_frames, w.grid_h, w.grid_w, -w.boundary_frames,
                                      w.rope_base)).to(torch.bfloat16)
    return [(ref_k, rv), (bnd_k, bv)][:n_context]


@pytest.mark.parametrize("w,n_context,with_bias,fused", [
    (I.WORKLOADS["small"], 2, False, True),
    (D128, 2, True, True),
    (WIDE, 2, False, False),
    (I.WORKLOADS["small"], 0, True, True),   # chunk 0 with no context at all
    (D128, 1, True, True),                   # chunk 0: the reference alone
], ids=["small", "d128-bias", "wide-unfused", "small-no-context-bias", "d128-reference-only-bias"])
def test_noalloc_step_matches_oracle(S, w, n_context, with_bias, fused):
    seed = 23
    # which RoPE form the step takes: q rotated inside attention when its table fits
    assert S.chunk_attention_qrope_fits(w.D, (w.F, w.grid_h, w.grid_w)) is fused
    ctx = _context_segments(w, seed, n_context)
    wo = I.out_proj_weight(w, seed)
    bias = I.bias_vec(w, seed) if with_bias else None
    dts = O.time_grid(w.steps, w.shift)
    x0 = I.state_x(w, seed)
    x_dev = x0.cuda()
    want = f64(x0)
    empty = np.zeros((w.B, 0, w.H, w.D))
    ref = (f64(ctx[0][0]), f64(ctx[0][1])) if n_context >= 1 else (empty, empty)
    bnd = (f64(ctx[1][0]), f64(ctx[1][1])) if n_context >= 2 else (empty, empty)
    dctx = [(k.cuda(), v.cuda()) for k, v in ctx]
    for s in range(2):  # two calls in a row on one state
        st = I.step_inputs(w, seed, 1, s)
        S.chunk_step_noalloc(st.q.cuda(), st.k.cuda(), st.v.cuda(), dctx, wo.cuda(), x_dev, float(dts[s]),
                             (w.F, w.grid_h, w.grid_w), bias=None if bias is None else bias.cuda(),
                             rope_base=w.rope_base)
        S.savgb_device_check()
        want, _ = O.chunk_step(f64(st.q), f64(st.k), f64(st.v), ref[0], ref[1], bnd[0], bnd[1], f64(wo), want,
                               dts[s], (w.F, w.grid_h, w.grid_w), w.rope_base, None,
                               None if bias is None else f64(bias))
        mx, mn = assert_close(f64(x_dev), want, what=f"{w.name} call {s} x vs oracle")
        print(f"noalloc {w.name} ctx={n_context} bias={with_bias} call {s}: max-abs {mx:.2e} mean-abs {mn:.2e}")


@pytest.mark.parametrize("w", [I.WORKLOADS["small"], D128, WIDE], ids=["small", "d128", "wide"])
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
    assert cs.fused_q_rope == S.chunk_attention_qrope_fits(w.D, (w.F, w.grid_h, w.grid_w))

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


def test_noalloc_wrapper_rejects_bad_shapes(S):
    """The binding checks every shape against the grid and hid before the
    library sees a pointer (the library takes its sizes from the grid)."""
    w = I.WORKLOADS["small"]
    t = lambda *shp: torch.zeros(shp, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    q = t(w.B, w.n_q, w.H, w.D)
    wo = t(w.hid, w.hid)
    x = torch.zeros((w.B * w.n_q, w.hid), dtype=torch.float32, device="cuda")
    grid = (w.F, w.grid_h, w.grid_w)
    ok_ctx = [(t(w.B, 16, w.H, w.D), t(w.B, 16, w.H, w.D))]
    bad = [
        dict(grid=(w.F + 1, w.grid_h, w.grid_w)),
        dict(context=[(t(w.B, 16, w.H, w.D), t(w.B, 8, w.H, w.D))]),
        dict(context=[(t(w.B, 16, w.H + 1, w.D), t(w.B, 16, w.H + 1, w.D))]),
        dict(w_o=t(w.hid, w.hid // 2)),
        dict(x=torch.zeros((w.B * w.n_q - 1, w.hid), dtype=torch.float32, device="cuda")),
        dict(bias=torch.zeros(w.hid + 4, dtype=torch.float32, device="cuda")),
    ]
    for b in bad:
        args = dict(context=ok_ctx, w_o=wo, x=x, grid=grid, bias=None)
        args.update(b)
        with pytest.raises(ValueError):
            S.chunk_step_noalloc(q, q, q, args["context"], args["w_o"], args["x"], 0.1, args["grid"],
                                 bias=args["bias"])


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
