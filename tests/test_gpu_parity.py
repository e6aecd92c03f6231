"""GPU parity of each C-ABI call against the fp64 oracle (bf16 inputs, fp32
accumulation: max-abs 2e-2, mean-abs 2e-3 on every floating-point output).

Sizes the oracle finishes in seconds span several tiles and a ragged tail;
the full base-DiT and SR chunk shapes are checked on sampled query rows,
computed by the oracle one by one against the full key/value set."""
import math
import os

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


def bf16(shape, seed, kind=1, std=1.0, chunk=0, step=0):
    return I.normal_bf16(shape, std, seed, kind, chunk, step)


def rows_of(t, rows):
    return t[:, rows]


# ------------------------------------------------------------------- RoPE

@pytest.mark.parametrize("B,gt,gh,gw,H,D,t0", [
    (1, 2, 4, 4, 2, 64, 0),      # tiny chunk
    (1, 1, 4, 4, 2, 64, -1),     # reference frame at t = -1
    (2, 3, 5, 7, 3, 128, -2),    # ragged grid, B = 2, negative start
    (1, 4, 16, 16, 8, 64, 0),    # small chunk
    (1, 8, 30, 52, 24, 128, 0),  # base-DiT chunk, every element
    (2, 2, 3, 5, 2, 128, 0),     # 32 vectors a token: one per lane (lane-invariant path), B = 2
    (1, 2, 3, 4, 1, 256, 3),     # D = 256: a head is a whole warp-width of vectors
    (1, 1, 2, 3, 48, 128, 0),    # 768 vectors a token: general path, three batches a token
    (2, 2, 2, 2, 32, 40, -3),    # D/8 = 5 does not divide 32: general path
])
def test_rope3d_parity(S, B, gt, gh, gw, H, D, t0):
    N = gt * gh * gw
    x = bf16((B, N, H, D), 11 + D + gt)
    out = torch.empty((B, N, H, D), dtype=torch.bfloat16, device="cuda")
    S.rope3d_apply(x.cuda(), out, gt, gh, gw, t0)
    torch.cuda.synchronize()
    want = O.rope3d(f64(x), gt, gh, gw, t0, 10000.0)
    assert_close(f64(out), want, what="rope3d")


def test_rope3d_in_place_and_sr_grid(S):
    B, gt, gh, gw, H, D = 1, 2, 60, 104, 4, 128
    x = bf16((B, gt * gh * gw, H, D), 5)
    d = x.cuda()
    S.rope3d_apply(d, d, gt, gh, gw, -2)
    torch.cuda.synchronize()
    assert_close(f64(d), O.rope3d(f64(x), gt, gh, gw, -2, 10000.0), what="rope3d in place")


def test_rope3d_identity_at_origin(S):
    """All positions zero (a 1x1x1 grid at t0 = 0): output == input bit for bit."""
    x = bf16((3, 1, 5, 128), 9).cuda()
    out = torch.empty_like(x)
    S.rope3d_apply(x, out, 1, 1, 1, 0)
    torch.cuda.synchronize()
    assert torch.equal(out, x)


# -------------------------------------------------------------- attention

def attn_case(S, B, H, D, n_q, seg_lens, seed, scale=0.0, rows=None, lse=False, q_scale=1.0, margin=False):
    q = bf16((B, n_q, H, D), seed, I.KIND_Q, std=q_scale)
    segs = [(bf16((B, n, H, D), seed, I.KIND_K, chunk=i), bf16((B, n, H, D), seed, I.KIND_V, chunk=i))
            for i, n in enumerate(seg_lens)]
    dq = q.cuda()
    dsegs = [(k.cuda(), v.cuda()) for k, v in segs]
    lse_t = torch.empty((B, H, n_q), dtype=torch.float32, device="cuda") if lse else None
    o = S.chunk_attention(dq, dsegs, scale=scale, lse=lse_t)
    torch.cuda.synchronize()
    S.savgb_device_check()
    sc = scale if scale > 0 else 1.0 / math.sqrt(D)
    qq = f64(q) if rows is None else f64(q)[:, rows]
    want = O.attention(qq, [(f64(k), f64(v)) for k, v in segs], sc)
    got = f64(o) if rows is None else f64(o)[:, rows]
    assert_close(got, want, what=f"attention B{B} H{H} D{D} nq{n_q} segs{seg_lens}", margin=margin)
    if lse:
        kk = np.concatenate([f64(k) for k, _ in segs], axis=1)
        s = np.einsum("bnhd,bmhd->bhnm", qq, kk) * sc
        m = s.max(-1, keepdims=True)
        want_lse = (m[..., 0] + np.log(np.exp(s - m).sum(-1)))
        got_lse = f64(lse_t) if rows is None else f64(lse_t)[:, :, rows]
        assert_close(got_lse, want_lse, max_abs=1e-3, mean_abs=1e-4, what="lse")
    return o


@pytest.mark.parametrize("D", [64, 128])
def test_attention_tiny_and_ragged(S, D):
    attn_case(S, 1, 2, D, 32, [16, 0, 32], 1)                 # tiny chunk 0
    attn_case(S, 1, 3, D, 300, [100, 37, 300], 2, lse=True)   # ragged q and every segment tail
    attn_case(S, 2, 2, D, 129, [1, 255, 129], 3)              # B = 2: no cross-batch bleed


def test_attention_small_config(S):
    w = I.WORKLOADS["small"]
    attn_case(S, 1, w.H, w.D, w.n_q, [w.n_ref, w.n_b, w.n_q], 4, lse=True)


def test_attention_single_key_returns_v(S):
    """One key/value token in total: O = V exactly (p = 1)."""
    B, H, D, n_q = 1, 2, 128, 200
    q = bf16((B, n_q, H, D), 7).cuda()
    k = bf16((B, 1, H, D), 8).cuda()
    v = bf16((B, 1, H, D), 9).cuda()
    o = S.chunk_attention(q, [(k, v)])
    torch.cuda.synchronize()
    assert torch.equal(o, v.expand(B, n_q, H, D))


def test_attention_large_scores_stable(S):
    """Scores x50: the running max keeps every exponent in range."""
    attn_case(S, 1, 2, 128, 256, [64, 0, 384], 12, scale=50.0 / math.sqrt(128))


def test_attention_lazy_rescale_path(S):
    """Queries scaled x8 make later tiles raise the row max by far more than
    the lazy-rescale threshold, so O is rescaled in tensor memory."""
    attn_case(S, 1, 2, 128, 256, [512, 0, 768], 13, q_scale=8.0)


def test_attention_sharp_scale_takes_fp32_exponentials(S):
    """A softmax scale above 1.25 x 1/sqrt(D) selects the kernel with fp32
    exponentials (the one the log-sum-exp output selects): bit-identical
    outputs with and without lse there, different ones at the default scale
    (where the packed bf16x2 exponentials run)."""
    B, H, D, n_q = 2, 3, 128, 300
    q = bf16((B, n_q, H, D), 71, I.KIND_Q).cuda()
    segs = [(bf16((B, n, H, D), 71, I.KIND_K, chunk=j).cuda(), bf16((B, n, H, D), 71, I.KIND_V, chunk=j).cuda())
            for j, n in enumerate([100, 0, 300])]
    lse = torch.empty((B, H, n_q), dtype=torch.float32, device="cuda")
    sharp = 2.0 / math.sqrt(D)
    assert torch.equal(S.chunk_attention(q, segs, scale=sharp), S.chunk_attention(q, segs, scale=sharp, lse=lse))
    assert not torch.equal(S.chunk_attention(q, segs), S.chunk_attention(q, segs, lse=lse))
    S.savgb_device_check()


@pytest.mark.parametrize("name", ["base", "sr"])
def test_attention_full_size_sampled_rows(S, name):
    w = I.WORKLOADS[name]
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(w.n_q, 40, replace=False),
                                     [0, 127, 128, 255, w.n_q - 129, w.n_q - 65, w.n_q - 1]]))
    attn_case(S, w.B, w.H, w.D, w.n_q, [w.n_ref, w.n_b, w.n_q], 21, rows=rows, margin=True)


def test_attention_sr_every_element_by_invariants(S):
    """The SR-shaped attention on every output element, through properties
    that hold at any size (the oracle checks sampled rows above):
    - two sessions whose second is a copy of the first give two identical
      outputs, bit for bit (batch indexing);
    - reversing the heads of q, k and v reverses the output's heads, bit for
      bit (head indexing);
    - the same keys split as [reference | boundary | chunk] and as
      [reference + boundary | chunk] (other tile boundaries and tails) agree
      within twice the oracle bar, since each is within the bar of the exact
      result;
    - the fused-RoPE call on unrotated queries agrees with the plain call on
      queries rotated by rope3d_apply within the same bound."""
    w = I.WORKLOADS["sr"]
    seed = 22
    q = bf16((1, w.n_q, w.H, w.D), seed, I.KIND_Q).cuda()
    segs = [(bf16((1, n, w.H, w.D), seed, I.KIND_K, chunk=i).cuda(), bf16((1, n, w.H, w.D), seed, I.KIND_V,
                                                                          chunk=i).cuda())
            for i, n in enumerate([w.n_ref, w.n_b, w.n_q])]
    o = S.chunk_attention(q, segs)
    # batch: the session duplicated
    o2 = S.chunk_attention(torch.cat([q, q]), [(torch.cat([k, k]), torch.cat([v, v])) for k, v in segs])
    assert torch.equal(o2[0], o[0]) and torch.equal(o2[1], o[0])
    del o2
    # heads reversed
    flip = lambda t: t.flip(2).contiguous()  # noqa: E731
    of = S.chunk_attention(flip(q), [(flip(k), flip(v)) for k, v in segs])
    assert torch.equal(of.flip(2), o)
    del of
    # the keys re-split: reference and boundary in one segment
    joined = [(torch.cat([segs[0][0], segs[1][0]], 1), torch.cat([segs[0][1], segs[1][1]], 1)), segs[2]]
    oj = S.chunk_attention(q, joined)
    d = (oj.float() - o.float()).abs()
    resplit = (d.max().item(), d.mean().item())
    assert resplit[0] <= 4e-2 and resplit[1] <= 4e-3, resplit
    del oj
    # fused RoPE of q against rope3d_apply + the plain call
    qr = torch.empty_like(q)
    S.rope3d_apply(q, qr, w.F, w.grid_h, w.grid_w, 0)
    o_plain = S.chunk_attention(qr, segs)
    o_fused = S.chunk_attention_qrope(q, (w.F, w.grid_h, w.grid_w), segs, t0=0)
    S.savgb_device_check()
    d = (o_fused.float() - o_plain.float()).abs()
    fused = (d.max().item(), d.mean().item())
    assert fused[0] <= 4e-2 and fused[1] <= 4e-3, fused
    print(f"SR attention, every element: re-split max-abs {resplit[0]:.2e} mean-abs {resplit[1]:.2e}; "
          f"fused RoPE of q max-abs {fused[0]:.2e} mean-abs {fused[1]:.2e}")


# ------------------------------------------------------- W_o + Euler update

@pytest.mark.parametrize("with_v", [True, False])  # the velocity-out epilogue, and the staged one of the stream
@pytest.mark.parametrize("M,hid_in,hid_out,bias", [
    (32, 128, 128, False),      # tiny
    (1024, 512, 512, True),     # small
    (300, 384, 400, True),      # ragged M (whole 32-row groups past M), hid_out not a multiple of 32
    (1000, 3072, 3072, False),  # base width, ragged M
    # the CTA-pair kernel (x only, hid_out % 256 == 0):
    (300, 384, 512, True),      # the odd CTA's 128 rows of the second tile lie wholly past M
    (700, 200, 256, False),     # K tail: hid_in not a multiple of 64
    (32, 128, 256, True),       # a single tile: one cluster
    (2560, 1024, 768, False),   # several tiles per cluster, both accumulator buffers reused
])
def test_out_proj_euler_parity(S, M, hid_in, hid_out, bias, with_v):
    o = bf16((M, hid_in), 31, I.KIND_Q)
    w = bf16((hid_out, hid_in), 32, I.KIND_WO, std=1.0 / math.sqrt(hid_in))
    x0 = torch.from_numpy(I.normal_f32((M, hid_out), 1.0, 33, I.KIND_X))
    b = torch.from_numpy(I.normal_f32((hid_out,), 0.1, 34, I.KIND_BIAS)) if bias else None
    x = x0.cuda()
    v = torch.empty((M, hid_out), dtype=torch.float32, device="cuda") if with_v else None
    dt = 0.0113636
    S.out_proj_euler_step(o.cuda(), w.cuda(), x, dt, bias=None if b is None else b.cuda(), v_out=v)
    torch.cuda.synchronize()
    S.savgb_device_check()
    want_v = O.out_proj(f64(o), f64(w), None if b is None else f64(b))
    if with_v:
        assert_close(f64(v), want_v, what="velocity")
    assert_close(f64(x), O.euler_update(f64(x0), want_v, dt), max_abs=1e-4, mean_abs=1e-5, what="x")


def test_out_proj_euler_full_base(S):
    w = I.WORKLOADS["base"]
    M, hid = w.B * w.n_q, w.hid
    o = bf16((M, hid), 41, I.KIND_Q, std=0.05)
    wo = I.out_proj_weight(w, 41)
    x0 = I.state_x(w, 41)
    x = x0.cuda()
    dt = S.flow_time_grid(30, 3.0)[0]
    S.out_proj_euler_step(o.cuda(), wo.cuda(), x, dt)
    torch.cuda.synchronize()
    rows = np.r_[0:64, 6000:6064, M - 64:M]
    want = O.euler_update(f64(x0)[rows], O.out_proj(f64(o)[rows], f64(wo)), dt)
    assert_close(f64(x)[rows], want, max_abs=1e-5, mean_abs=1e-6, what="x base rows")


# ----------------------------------------------------------- chunk stream

def run_stream_gpu(S, w, seed, chunks, steps=None, bias=None):
    steps = w.steps if steps is None else steps
    dts = S.flow_time_grid(steps, w.shift)
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed).cuda()
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base)
    cs.set_reference(rk.cuda(), rv.cuda())
    xs, bnds = [], []
    for c in range(chunks):
        bnds.append(cs.boundary())
        x = torch.from_numpy(I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, c)).cuda()
        for s, dt in enumerate(dts):
            st = I.step_inputs(w, seed, c, s)
            cs.step(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, x, dt, s == len(dts) - 1, bias=bias)
        cs.end_chunk()
        cs.sync()
        xs.append(x.cpu())
    return cs, xs, bnds


def run_stream_oracle(w, seed, chunks, steps=None):
    steps = w.steps if steps is None else steps
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed)

    def step_in(c, s):
        st = I.step_inputs(w, seed, c, s)
        return f64(st.q), f64(st.k), f64(st.v)

    return O.run_stream(w, f64(rk), f64(rv), f64(wo),
                        lambda c: I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, c).astype(np.float64),
                        step_in, O.time_grid(steps, w.shift), chunks=chunks)


def test_stream_tiny(S):
    w = I.WORKLOADS["tiny"]
    cs, xs, _ = run_stream_gpu(S, w, 0, 1)
    assert cs.fused_q_rope  # the stream's RoPE table fits: q is rotated inside the attention kernel
    want, _ = run_stream_oracle(w, 0, 1)
    assert_close(f64(xs[0]), want[0], what="tiny x")
    cs.close()


def test_stream_wide_grid_unfused(S):
    """A 2 x 400 frame grid: the RoPE table of its w axis (67 KB) does not fit
    next to the attention operands, so the stream rotates q and k in one pass
    before the plain attention kernel, and the stand-alone fused call refuses
    the grid.  Two chunks x 2 steps against the oracle."""
    w = I.Workload("wide", B=1, H=2, D=128, F=2, grid_h=2, grid_w=400, ref_frames=1, boundary_frames=1,
                   ref_t=-1, steps=2, shift=1.0)
    cs, xs, _ = run_stream_gpu(S, w, 5, 2)
    assert not cs.fused_q_rope
    want, _ = run_stream_oracle(w, 5, 2)
    for c in range(2):
        assert_close(f64(xs[c]), want[c], what=f"wide-grid chunk {c} x")
    cs.close()
    q = torch.zeros(1, w.n_q, w.H, w.D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(S.SavgbError):
        S.chunk_attention_qrope(q, (w.F, w.grid_h, w.grid_w), [(q, q)])


def _cuda_dirs():
    """The CUDA toolkit's include and runtime-library directories."""
    import glob
    import shutil
    home = os.environ.get("CUDA_HOME") or os.path.dirname(os.path.dirname(shutil.which("nvcc") or
                                                                          "/usr/local/cuda/bin/nvcc"))
    incs = [os.path.join(home, "include")] + glob.glob(os.path.join(home, "targets", "*", "include"))
    libs = [os.path.join(home, "lib64")] + glob.glob(os.path.join(home, "targets", "*", "lib"))
    inc = next((d for d in incs if os.path.exists(os.path.join(d, "cuda_runtime_api.h"))), None)
    lib = next((d for d in libs if glob.glob(os.path.join(d, "libcudart.so*"))), None)
    return inc, lib


def test_c_program_runs_a_stream(S, tmp_path):
    """A plain C program (tests/abi_c_stream.c) runs a two-session stream of 3
    chunks x 3 shifted steps through the C ABI alone, with device buffers from
    its own CUDA runtime calls: each chunk's x equals, bit for bit, the same
    stream run through the Python binding, and matches the oracle."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    inc, cudalib = _cuda_dirs()
    if cc is None or inc is None or cudalib is None:
        pytest.skip("no C compiler or CUDA runtime headers")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(S.LIB_PATH)
    exe = str(tmp_path / "abi_c_stream")
    subprocess.run([cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(root, "include"),
                    "-I", inc, os.path.join(root, "tests", "abi_c_stream.c"), "-L", libdir, "-lsavgb",
                    "-L", cudalib, "-lcudart", f"-Wl,-rpath,{libdir}:{cudalib}", "-o", exe], check=True)
    w = I.Workload("cprog", B=2, H=2, D=64, F=3, grid_h=4, grid_w=6, ref_frames=1, boundary_frames=1, steps=3,
                   shift=3.0)
    seed, chunks = 15, 3
    raw = lambda t: t.contiguous().view(torch.int16).numpy().tobytes() if t.dtype == torch.bfloat16 \
        else t.contiguous().numpy().tobytes()  # noqa: E731
    rk, rv = I.reference_kv(w, seed)
    (tmp_path / "ref_k.bin").write_bytes(raw(rk))
    (tmp_path / "ref_v.bin").write_bytes(raw(rv))
    (tmp_path / "w_o.bin").write_bytes(raw(I.out_proj_weight(w, seed)))
    for c in range(chunks):
        (tmp_path / f"x_{c}.bin").write_bytes(I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, c).tobytes())
        for s_ in range(w.steps):
            st = I.step_inputs(w, seed, c, s_)
            for name, t in (("q", st.q), ("k", st.k), ("v", st.v)):
                (tmp_path / f"{name}_{c}_{s_}.bin").write_bytes(raw(t))
    r = subprocess.run([exe, str(tmp_path), *map(str, (w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames,
                                                          w.boundary_frames, w.ref_t, chunks, w.steps, w.shift))],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr
    got = [np.frombuffer((tmp_path / f"out_{c}.bin").read_bytes(), dtype=np.float32).reshape(w.B * w.n_q, w.hid)
           for c in range(chunks)]
    cs, xs, _ = run_stream_gpu(S, w, seed, chunks)
    cs.close()
    want, _ = run_stream_oracle(w, seed, chunks)
    for c in range(chunks):
        assert np.array_equal(got[c], xs[c].numpy()), f"chunk {c}: the C program and the binding differ"
        assert_close(got[c].astype(np.float64), want[c], what=f"C program chunk {c} x")


def test_stream_small_pair(S):
    """Two chunks x 4 steps; chunk 1 attends over the boundary rolled from chunk 0."""
    w = I.WORKLOADS["small"]
    cs, xs, bnds = run_stream_gpu(S, w, 0, 2)
    assert cs.fused_q_rope
    want, wbnds = run_stream_oracle(w, 0, 2)
    for c in range(2):
        assert_close(f64(xs[c]), want[c], what=f"small chunk {c} x")
    assert bnds[0] is None
    bk, bv = bnds[1]
    assert_close(f64(bk), wbnds[1][0], what="boundary k (rotated)")
    assert np.array_equal(f64(bv), wbnds[1][1]), "boundary v is a copy"
    inf = cs.info()
    assert inf["chunk_index"] == 2 and inf["boundary_tokens"] == w.n_b
    cs.close()


def test_stream_two_sessions_ragged_blocks(S):
    """B = 2 sessions of 1100 queries: the 256-row tiles of the W_o GEMM
    straddle the sessions and the last 256-query attention block of each
    session is ragged.  Two chunks x 3 steps against the oracle, and a second
    run that must reproduce the first bit for bit."""
    w = I.Workload("straddle", B=2, H=4, D=128, F=5, grid_h=10, grid_w=22, ref_frames=1,
                   boundary_frames=1, steps=3, shift=1.0)
    cs, xs, _ = run_stream_gpu(S, w, 3, 2)
    cs.close()
    want, _ = run_stream_oracle(w, 3, 2)
    for c in range(2):
        assert_close(f64(xs[c]), want[c], what=f"two-session chunk {c} x")
    cs2, xs2, _ = run_stream_gpu(S, w, 3, 2)
    cs2.close()
    for c in range(2):
        assert torch.equal(xs[c], xs2[c]), f"chunk {c}: rerun differs"


@pytest.mark.parametrize("slots", [1, 3], ids=["two-slots", "three-slots"])
def test_stream_host_io_matches_device_steps(S, slots):
    """chunk_stream_step_host (q, k, v from host memory, x read back every
    step) against chunk_stream_step on the same inputs: every step's read-back
    bit-identical to the device path's x after that step, the final state
    against the oracle.  One step in the middle runs through the device call:
    it updates x while the previous step's read-back, from its staging copy,
    may still be in flight.  Pageable input memory works too."""
    w = I.WORKLOADS["small"]
    seed = 9
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed).cuda()
    dts = S.flow_time_grid(w.steps, w.shift)
    plan = [(c, s_) for c in range(2) for s_ in range(w.steps)]
    device_call = (1, 2)                     # this step goes through chunk_stream_step
    pageable = (0, 1)                        # this step's inputs are not page-locked
    ins = {cs_: I.step_inputs(w, seed, *cs_) for cs_ in plan}

    def make(host_io):
        cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                           w.rope_base, host_io=int(host_io))
        cs.set_reference(rk.cuda(), rv.cuda())
        return cs

    ref = make(False)
    want = {}
    x = I.state_x(w, seed).cuda()
    for c, s_ in plan:
        st = ins[(c, s_)]
        ref.step(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, x, dts[s_], s_ == w.steps - 1)
        want[(c, s_)] = x.cpu()
        if s_ == w.steps - 1:
            ref.end_chunk()
    ref.sync()
    ref.close()

    hs = make(slots)
    x = I.state_x(w, seed).cuda()
    back = {cs_: torch.empty((w.B * w.n_q, w.hid), dtype=torch.float32).pin_memory() for cs_ in plan}
    # every host input stays alive until the sync below: the uploads read them asynchronously
    host_in = {cs_: ((ins[cs_].q, ins[cs_].k, ins[cs_].v) if cs_ == pageable else
                     tuple(t.pin_memory() for t in (ins[cs_].q, ins[cs_].k, ins[cs_].v))) for cs_ in plan}
    dev_in = tuple(t.cuda() for t in (ins[device_call].q, ins[device_call].k, ins[device_call].v))
    for c, s_ in plan:
        last = s_ == w.steps - 1
        if (c, s_) == device_call:
            hs.step(*dev_in, wo, x, dts[s_], last)
        else:
            hs.step_host(*host_in[(c, s_)], wo, x, dts[s_], last, x_host=back[(c, s_)])
        if last:
            hs.end_chunk()
    hs.sync()
    for cs_ in plan:
        if cs_ != device_call:
            assert torch.equal(back[cs_], want[cs_]), f"read-back after chunk {cs_[0]} step {cs_[1]}"
    assert torch.equal(x.cpu(), want[plan[-1]])
    hs.close()
    # the final state against the oracle
    f = lambda t: t.double().numpy()  # noqa: E731
    xs, _ = O.run_stream(w, f(rk), f(rv), f(wo.cpu()), lambda c: f(I.state_x(w, seed)) if c == 0 else None,
                         lambda c, s_: tuple(f(t) for t in (ins[(c, s_)].q, ins[(c, s_)].k, ins[(c, s_)].v)),
                         O.time_grid(w.steps, w.shift), chunks=1)
    assert_close(f64(want[(0, w.steps - 1)]), xs[0], what="host-io stream chunk 0 x")
    # without host_io the call is refused
    plain = make(False)
    st = ins[plan[0]]
    with pytest.raises(S.SavgbError) as e:
        plain.step_host(st.q, st.k, st.v, wo, x, 0.1, False)
    assert e.value.status == -7
    plain.close()


def test_stream_exact_softmax(S):
    """A stream created with exact_softmax runs its attention with fp32
    exponentials: its steps match the oracle, and differ (slightly) from the
    packed form's."""
    w = I.WORKLOADS["small"]
    seed = 19
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed).cuda()
    dts = S.flow_time_grid(w.steps, w.shift)
    xs = {}
    for exact in (False, True):
        cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                           w.rope_base, exact_softmax=exact)
        cs.set_reference(rk.cuda(), rv.cuda())
        x = I.state_x(w, seed).cuda()
        for s_, dt in enumerate(dts):
            st = I.step_inputs(w, seed, 0, s_)
            cs.step(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, x, dt, s_ == len(dts) - 1)
        cs.sync()
        xs[exact] = x.cpu()
        cs.close()
    f = lambda t: t.double().numpy()  # noqa: E731
    want, _ = O.run_stream(w, f(rk), f(rv), f(wo.cpu()), lambda c: f(I.state_x(w, seed)),
                           lambda c, s_: tuple(f(t) for t in (I.step_inputs(w, seed, c, s_).q,
                                                              I.step_inputs(w, seed, c, s_).k,
                                                              I.step_inputs(w, seed, c, s_).v)),
                           O.time_grid(w.steps, w.shift), chunks=1)
    assert_close(f64(xs[True]), want[0], what="exact-softmax stream chunk 0 x")
    assert not torch.equal(xs[True], xs[False])


def test_stream_export_import_resume(S):
    """Checkpoint after chunk 1, resume in a fresh handle: chunk 2 equals the
    uninterrupted run."""
    w = I.Workload("resume", B=2, H=2, D=128, F=3, grid_h=8, grid_w=8, ref_frames=1, boundary_frames=2,
                   steps=2, shift=3.0)
    seed = 3
    cs, xs, _ = run_stream_gpu(S, w, seed, 3)
    # rerun two chunks, export, import into a new handle, run chunk 2
    cs2, _, _ = run_stream_gpu(S, w, seed, 2)
    state = cs2.export_state()
    cs2.close()
    rk, rv = I.reference_kv(w, seed)
    cs3 = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                        w.rope_base)
    cs3.set_reference(rk.cuda(), rv.cuda())
    cs3.import_state(state)
    assert cs3.info()["chunk_index"] == 2
    wo = I.out_proj_weight(w, seed).cuda()
    x = torch.from_numpy(I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, 2)).cuda()
    dts = S.flow_time_grid(w.steps, w.shift)
    for s, dt in enumerate(dts):
        st = I.step_inputs(w, seed, 2, s)
        cs3.step(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, x, dt, s == len(dts) - 1)
    cs3.end_chunk()
    cs3.sync()
    assert torch.equal(x.cpu(), xs[2])
    cs3.close()
    cs.close()


def test_stream_memory_is_flat(S):
    """Device memory in use does not grow with the number of chunks."""
    w = I.Workload("flat", B=1, H=4, D=128, F=4, grid_h=8, grid_w=12, ref_frames=1, boundary_frames=2,
                   steps=2, shift=1.0)
    rk, rv = I.reference_kv(w, 1)
    wo = I.out_proj_weight(w, 1).cuda()
    st = I.step_inputs(w, 1, 0, 0)
    q, k, v = st.q.cuda(), st.k.cuda(), st.v.cuda()
    x = torch.zeros((w.n_q, w.hid), dtype=torch.float32, device="cuda")
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, 1, 2)
    cs.set_reference(rk.cuda(), rv.cuda())
    free = []
    for c in range(24):
        for s in range(2):
            cs.step(q, k, v, wo, x, 0.5, s == 1)
        cs.end_chunk()
        cs.sync()
        free.append(torch.cuda.mem_get_info()[0])
    assert max(free[1:]) == min(free[1:]), "device memory changed across chunks"
    assert cs.info()["chunk_index"] == 24
    cs.close()


def test_stream_state_errors(S):
    w = I.WORKLOADS["tiny"]
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, 1, 1)
    st = I.step_inputs(w, 0, 0, 0)
    wo = I.out_proj_weight(w, 0).cuda()
    x = torch.zeros((w.n_q, w.hid), dtype=torch.float32, device="cuda")
    with pytest.raises(S.SavgbError) as e:
        cs.step(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, x, 0.5, False)
    assert e.value.status == -7  # no reference yet
    rk, rv = I.reference_kv(w, 0)
    cs.set_reference(rk.cuda(), rv.cuda())
    cs.step(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, x, 0.5, False)
    with pytest.raises(S.SavgbError) as e:
        cs.end_chunk()  # no last step: no boundary captured
    assert e.value.status == -7
    cs.close()


def test_stream_arena_limit(S, monkeypatch):
    monkeypatch.setenv("SAVGB_ARENA_LIMIT_BYTES", "1024")
    with pytest.raises(S.SavgbError) as e:
        S.ChunkStream(1, 2, 64, 2, 4, 4)
    assert e.value.status == -4


def test_kernel_launch_counter(S):
    """savgb_kernel_launches counts the kernels each call enqueues: one per
    stand-alone kernel call; three per stream step (RoPE of k, attention with
    the RoPE of q inside, W_o + Euler), and one more, the boundary's RoPE, at a
    chunk's end; none for a call refused on the host.  The bench reports the
    same counter over its timed regions."""
    w = I.WORKLOADS["small"]
    seed = 14
    n = S.savgb_kernel_launches

    def delta(fn):
        before = n()
        fn()
        torch.cuda.synchronize()
        return n() - before

    q = bf16((1, 300, 2, 128), seed, I.KIND_Q).cuda()
    kv = (bf16((1, 200, 2, 128), seed, I.KIND_K).cuda(), bf16((1, 200, 2, 128), seed, I.KIND_V).cuda())
    assert delta(lambda: S.chunk_attention(q, [kv])) == 1
    assert delta(lambda: S.rope3d_apply(q, torch.empty_like(q), 3, 10, 10)) == 1
    o = bf16((300, 256), seed, I.KIND_Q).cuda()
    wt = bf16((256, 256), seed, I.KIND_WO, std=1 / 16).cuda()
    x = torch.zeros((300, 256), dtype=torch.float32, device="cuda")
    assert delta(lambda: S.out_proj_euler_step(o, wt, x, 0.1)) == 1
    before = n()
    with pytest.raises(S.SavgbError):
        S._check(S.lib().rope3d_apply(None, None, 1, 16, 2, 64, 1, 4, 4, 0, 1e4, None))
    assert n() == before

    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed).cuda()
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base)
    cs.set_reference(rk.cuda(), rv.cuda())
    assert cs.fused_q_rope
    xs = torch.from_numpy(I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, 0)).cuda()
    dts = S.flow_time_grid(w.steps, w.shift)
    ins = [tuple(t.cuda() for t in (st.q, st.k, st.v)) for st in (I.step_inputs(w, seed, 0, s_) for s_ in range(2))]
    assert delta(lambda: cs.step(*ins[0], wo, xs, dts[0], False)) == 3

    def last_step():
        cs.step(*ins[1], wo, xs, dts[1], True)
        cs.end_chunk()
    assert delta(last_step) == 4
    cs.sync()
    cs.close()


# ------------------------------------------------------------- watchdog

def test_watchdog_timeout_is_reported(S):
    """A wait on a barrier that nothing arrives on gives up after its limit;
    the host reads SAVGB_ERR_TIMEOUT and the context stays usable."""
    S.savgb_device_check()
    S.savgb_watchdog_selftest(50_000_000)  # 50 ms
    with pytest.raises(S.SavgbError) as e:
        S.savgb_device_check()
    assert e.value.status == -6 and "watchdog" in str(e.value)
    S.savgb_device_check()  # cleared
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0


@pytest.mark.parametrize("fused", [False, True], ids=["plain", "rope-q-fused"])
def test_attention_give_up_path(S, fused):
    """The real attention kernel's give-up path: block (0, 0, 0)'s key
    producer skips the copy of key tile 1, so the block's waits for it run
    out after 20 ms.  The block records the timeout, drains its copies and
    MMAs, frees its tensor memory and returns; the host reads
    SAVGB_ERR_TIMEOUT, and the next launch, with no fault, passes parity."""
    B, H, D, gt, gh, gw = 1, 2, 128, 3, 10, 10   # 300 queries: two query blocks per head
    segs = [100, 37]                              # with the chunk: 1 + 1 + 3 key tiles
    n_q = gt * gh * gw
    q = bf16((B, n_q, H, D), 61, I.KIND_Q)
    kc, vc = bf16((B, n_q, H, D), 61, I.KIND_K), bf16((B, n_q, H, D), 61, I.KIND_V)
    ctx = [(bf16((B, n, H, D), 61, I.KIND_K, chunk=i + 1), bf16((B, n, H, D), 61, I.KIND_V, chunk=i + 1))
           for i, n in enumerate(segs)]
    dsegs = [(k.cuda(), v.cuda()) for k, v in ctx] + [(kc.cuda(), vc.cuda())]

    def run():
        if fused:
            return S.chunk_attention_qrope(q.cuda(), (gt, gh, gw), dsegs)
        return S.chunk_attention(q.cuda(), dsegs)

    S.savgb_device_check()
    S.savgb_arm_wait_fault(S.FAULT_ATTENTION_K_TILE, 1, 20_000_000)
    run()
    with pytest.raises(S.SavgbError) as e:
        S.savgb_device_check()
    assert e.value.status == -6 and "chunk_attention" in str(e.value)
    S.savgb_device_check()  # cleared
    o = run()               # the arm was taken: a normal launch
    S.savgb_device_check()
    q_ref = O.rope3d(f64(q), gt, gh, gw, 0) if fused else f64(q)
    want = O.attention(q_ref, [(f64(k), f64(v)) for k, v in ctx] + [(f64(kc), f64(vc))])
    assert_close(f64(o), want, what=f"attention after a give-up ({'fused' if fused else 'plain'})")


def test_out_proj_pair_give_up_path(S):
    """The W_o CTA-pair kernel's give-up path: the odd CTA of the first
    cluster skips its relay of k-block iteration 3, so the even CTA's MMA
    issuer gives up after 20 ms; both CTAs drain, reach the cluster barriers
    and free their tensor memory.  SAVGB_ERR_TIMEOUT on the host, then a
    normal launch passes parity."""
    M, hid = 1024, 512   # 8 tiles of 256 x 256, 8 k-blocks each
    o = bf16((M, hid), 62, I.KIND_Q, std=0.05)
    wo = bf16((hid, hid), 62, I.KIND_WO, std=1.0 / math.sqrt(hid))
    x0 = torch.from_numpy(I.normal_f32((M, hid), 1.0, 62, I.KIND_X))
    dt = 0.125
    S.savgb_device_check()
    S.savgb_arm_wait_fault(S.FAULT_WO_PAIR_RELAY, 3, 20_000_000)
    x = x0.cuda()
    S.out_proj_euler_step(o.cuda(), wo.cuda(), x, dt)
    with pytest.raises(S.SavgbError) as e:
        S.savgb_device_check()
    assert e.value.status == -6 and "out_proj_euler_step" in str(e.value)
    S.savgb_device_check()  # cleared
    x = x0.cuda()
    S.out_proj_euler_step(o.cuda(), wo.cuda(), x, dt)
    S.savgb_device_check()
    want = O.euler_update(f64(x0), O.out_proj(f64(o), f64(wo)), dt)
    assert_close(f64(x), want, max_abs=1e-4, mean_abs=1e-5, what="x after a give-up")


@pytest.mark.parametrize("name", ["base", "sr1"])
def test_stream_step_full_size_sampled_rows(S, name):
    """Two one-step chunks of a full-size workload through chunk_stream_step:
    chunk 1 attends over the boundary rolled from chunk 0.  Sampled rows of
    chunk 1's x against the oracle (every key, every head)."""
    w = I.WORKLOADS[name]
    seed = 5
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed)
    dt = 1.0 if w.steps == 1 else S.flow_time_grid(w.steps, w.shift)[0]
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base)
    cs.set_reference(rk.cuda(), rv.cuda())
    st0 = I.step_inputs(w, seed, 0, 0)
    x_scratch = torch.zeros((w.B * w.n_q, w.hid), dtype=torch.float32, device="cuda")
    cs.step(st0.q.cuda(), st0.k.cuda(), st0.v.cuda(), wo.cuda(), x_scratch, dt, True)
    cs.end_chunk()
    del x_scratch
    st1 = I.step_inputs(w, seed, 1, 0)
    x0 = torch.from_numpy(I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, 1))
    x = x0.cuda()
    cs.step(st1.q.cuda(), st1.k.cuda(), st1.v.cuda(), wo.cuda(), x, dt, False)
    cs.sync()
    got = x.cpu()
    cs.close()
    # oracle on sampled rows: rotations of the full chunk, attention for the sampled queries only
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([rng.choice(w.n_q, 24, replace=False), [0, 255, 256, w.n_q - 1]]))
    rk_rot = O.rope3d(f64(rk), w.ref_frames, w.grid_h, w.grid_w, w.ref_t, w.rope_base)
    bk_rot, bv = O.boundary_from_chunk(f64(st0.k), f64(st0.v), w.frame_tokens, w.boundary_frames, w.grid_h,
                                       w.grid_w, w.rope_base)
    q_rot = O.rope3d(f64(st1.q), w.F, w.grid_h, w.grid_w, 0, w.rope_base)[:, rows]
    k_rot = O.rope3d(f64(st1.k), w.F, w.grid_h, w.grid_w, 0, w.rope_base)
    o = O.attention(q_rot, [(rk_rot, f64(rv)), (bk_rot, bv), (k_rot, f64(st1.v))])
    want = O.euler_update(f64(x0)[rows], O.out_proj(o.reshape(len(rows), w.hid), f64(wo)), dt)
    assert_close(f64(got)[rows], want, what=f"{name} step x (sampled rows)", margin=True)


def _stream_sampled_rows(S, w, seed, chunk_dts, rows, check_chunks):
    """Runs the chunks through chunk_stream_step (chunk c takes the steps
    chunk_dts[c]; the last step of every chunk rolls the boundary) and replays
    them on the oracle for the sampled query rows of every session, over every
    key and head.  Compares x after each chunk in check_chunks."""
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed)
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base)
    cs.set_reference(rk.cuda(), rv.cuda())
    dwo = wo.cuda()
    rk_rot = O.rope3d(f64(rk), w.ref_frames, w.grid_h, w.grid_w, w.ref_t, w.rope_base)
    segs_ref = (rk_rot, f64(rv))
    bnd = None
    x_rows_of = [b * w.n_q + rows for b in range(w.B)]
    for c, dts in enumerate(chunk_dts):
        x0 = I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, c)
        x = torch.from_numpy(x0).cuda()
        want = np.concatenate([x0[r] for r in x_rows_of]).astype(np.float64).reshape(w.B, len(rows), w.hid)
        last_kv = None
        for s_, dt in enumerate(dts):
            st = I.step_inputs(w, seed, c, s_)
            cs.step(st.q.cuda(), st.k.cuda(), st.v.cuda(), dwo, x, dt, s_ == len(dts) - 1)
            q_rot = O.rope3d(f64(st.q), w.F, w.grid_h, w.grid_w, 0, w.rope_base)[:, rows]
            k_rot = O.rope3d(f64(st.k), w.F, w.grid_h, w.grid_w, 0, w.rope_base)
            segs = [segs_ref] + ([bnd] if bnd is not None else []) + [(k_rot, f64(st.v))]
            o = O.attention(q_rot, segs)
            for b in range(w.B):
                want[b] = O.euler_update(want[b], O.out_proj(o[b].reshape(len(rows), w.hid), f64(wo)), dt)
            last_kv = (st.k, st.v)
        cs.end_chunk()
        cs.sync()
        if c in check_chunks:
            got = x.cpu()
            for b in range(w.B):
                assert_close(f64(got)[x_rows_of[b]], want[b], what=f"{w.name} chunk {c} session {b} x (sampled rows)",
                             margin=True)
        bnd = O.boundary_from_chunk(f64(last_kv[0]), f64(last_kv[1]), w.frame_tokens, w.boundary_frames,
                                    w.grid_h, w.grid_w, w.rope_base)
    cs.close()


def test_stream_sr_chunk_all_steps_sampled_rows(S):
    """The SR-shaped workload as configured: a chunk of 8 uniform Euler steps
    (after a one-step chunk that supplies the boundary), sampled rows of x
    after all 8 steps."""
    w = I.WORKLOADS["sr"]
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.choice(w.n_q, 12, replace=False), [0, 256, w.n_q - 1]]))
    _stream_sampled_rows(S, w, 7, [[1.0], list(S.flow_time_grid(w.steps, w.shift))], rows, {1})


def test_stream_long_sessions_sampled_rows(S):
    """The long-session workload's shape: 4 batched sessions of base-DiT
    chunks, 3 consecutive chunks (2 shifted steps each here) so that the
    boundary rolls twice; sampled rows of every session's x."""
    w = I.WORKLOADS["long"]
    assert w.B == 4
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([rng.choice(w.n_q, 10, replace=False), [0, w.n_q - 1]]))
    dts = list(S.flow_time_grid(2, w.shift))
    _stream_sampled_rows(S, w, 8, [dts, dts, dts], rows, {1, 2})


# ---------------------------------------------------- interpolation chunks

def _ni_workload(D):
    if D == 64:
        return I.Workload("ni64", B=1, H=4, D=64, F=4, grid_h=8, grid_w=12, ref_frames=1, boundary_frames=1,
                          steps=2, shift=1.0)
    return I.Workload("ni128", B=2, H=2, D=128, F=5, grid_h=6, grid_w=10, ref_frames=1, boundary_frames=2,
                      steps=2, shift=3.0)


def _run_ni_gpu(S, w, seed, n_chunks, stop_after=None, cs=None):
    """N0, N1, I0, N2, I1, ... through the driver; returns the x of every chunk."""
    dts = S.flow_time_grid(w.steps, w.shift)
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed).cuda()
    if cs is None:
        cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                           w.rope_base, interp_chunks=True)
        cs.set_reference(rk.cuda(), rv.cuda())
    xs_n, xs_i = [], []
    n_int = (w.F - 2) * w.frame_tokens
    for c in range(n_chunks):
        x = torch.from_numpy(I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, c)).cuda()
        for s, dt in enumerate(dts):
            st = I.step_inputs(w, seed, c, s)
            cs.step(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, x, dt, s == len(dts) - 1)
        cs.end_chunk()
        xs_n.append(x.cpu())
        if stop_after is not None and c == stop_after:
            return cs, xs_n, xs_i
        if c >= 1:
            assert cs.ichunk_index() == c - 1
            xi = torch.from_numpy(I.normal_f32((w.B * n_int, w.hid), 1.0, seed, I.KIND_X, 0x4000 + c - 1)).cuda()
            for s, dt in enumerate(dts):
                st = I.istep_inputs(w, seed, c - 1, s)
                cs.istep(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, xi, dt)
            cs.end_ichunk()
            xs_i.append(xi.cpu())
    cs.sync()
    return cs, xs_n, xs_i


@pytest.mark.parametrize("D", [64, 128])
def test_stream_interp_chunks(S, D):
    """N0, N1, I0, N2, I1: every N and I chunk's x against the oracle."""
    w = _ni_workload(D)
    seed = 8
    cs, xs_n, xs_i = _run_ni_gpu(S, w, seed, 3)
    cs.close()
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed)
    n_int = (w.F - 2) * w.frame_tokens

    def n_in(c, s):
        st = I.step_inputs(w, seed, c, s)
        return f64(st.q), f64(st.k), f64(st.v)

    def i_in(c, s):
        st = I.istep_inputs(w, seed, c, s)
        return f64(st.q), f64(st.k), f64(st.v)

    want_n, want_i, _ = O.run_stream_ni(
        w, f64(rk), f64(rv), f64(wo),
        lambda c: I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, c).astype(np.float64),
        lambda c: I.normal_f32((w.B * n_int, w.hid), 1.0, seed, I.KIND_X, 0x4000 + c).astype(np.float64),
        n_in, i_in, O.time_grid(w.steps, w.shift), O.time_grid(w.steps, w.shift), 3)
    for c in range(3):
        assert_close(f64(xs_n[c]), want_n[c], what=f"N{c} x")
    for c in range(2):
        assert_close(f64(xs_i[c]), want_i[c], what=f"I{c} x")


def test_interp_state_and_resume(S):
    w = _ni_workload(128)
    seed = 4
    wo = I.out_proj_weight(w, seed).cuda()
    n_int = (w.F - 2) * w.frame_tokens
    st = I.istep_inputs(w, seed, 0, 0)
    xi = torch.zeros((w.B * n_int, w.hid), dtype=torch.float32, device="cuda")
    # an I step needs two finished N chunks
    cs, _, _ = _run_ni_gpu(S, w, seed, 1, stop_after=0)
    with pytest.raises(S.SavgbError) as e:
        cs.istep(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, xi, 0.5)
    assert e.value.status == -7
    cs.close()
    # without interp_chunks there is no I step
    plain = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, 1, 2)
    with pytest.raises(S.SavgbError):
        plain.istep(st.q.cuda(), st.k.cuda(), st.v.cuda(), wo, xi, 0.5)
    plain.close()
    # checkpoint between N1 and I0, resume in a fresh handle: I0 and N2 equal the uninterrupted run
    cs_full, xs_n, xs_i = _run_ni_gpu(S, w, seed, 3)
    cs_full.close()
    cs_a, _, _ = _run_ni_gpu(S, w, seed, 2, stop_after=1)
    state = cs_a.export_state()
    cs_a.close()
    rk, rv = I.reference_kv(w, seed)
    cs_b = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                         w.rope_base, interp_chunks=True)
    cs_b.set_reference(rk.cuda(), rv.cuda())
    cs_b.import_state(state)
    assert cs_b.info()["chunk_index"] == 2 and cs_b.ichunk_index() == 0
    dts = S.flow_time_grid(w.steps, w.shift)
    xi = torch.from_numpy(I.normal_f32((w.B * n_int, w.hid), 1.0, seed, I.KIND_X, 0x4000)).cuda()
    for s, dt in enumerate(dts):
        sti = I.istep_inputs(w, seed, 0, s)
        cs_b.istep(sti.q.cuda(), sti.k.cuda(), sti.v.cuda(), wo, xi, dt)
    cs_b.end_ichunk()
    cs_b.sync()
    assert torch.equal(xi.cpu(), xs_i[0])
    cs_b.close()


# ------------------------------------------------- RoPE of Q inside attention

@pytest.mark.parametrize("D,B,gt,gh,gw,t0,segs", [
    (64, 1, 2, 4, 4, 0, [16, 0]),            # tiny chunk
    (128, 2, 3, 7, 9, 1, [63, 200, 0]),      # ragged: 189 queries, B = 2, t0 = 1
    (128, 1, 8, 30, 52, 0, [1560, 3120]),    # base-DiT chunk (sampled rows)
    (128, 1, 2, 4, 150, -3, [600, 0]),       # t0 < 0; a 26 KB table, near the shared-memory limit
])
def test_attention_qrope_parity(S, D, B, gt, gh, gw, t0, segs):
    """Unrotated queries, rotated inside the kernel, against the oracle's
    RoPE followed by attention (chunk keys rotated by the oracle)."""
    H = 4 if D == 128 else 2
    n_q = gt * gh * gw
    seed = 40 + D
    q = bf16((B, n_q, H, D), seed, I.KIND_Q)
    kc = bf16((B, n_q, H, D), seed, I.KIND_K)
    vc = bf16((B, n_q, H, D), seed, I.KIND_V)
    ctx = [(bf16((B, n, H, D), seed, I.KIND_K, chunk=i + 1), bf16((B, n, H, D), seed, I.KIND_V, chunk=i + 1))
           for i, n in enumerate(segs)]
    kc_rot = torch.empty_like(kc).cuda()
    S.rope3d_apply(kc.cuda(), kc_rot, gt, gh, gw, t0)
    dsegs = [(k.cuda(), v.cuda()) for k, v in ctx] + [(kc_rot, vc.cuda())]
    dsegs = [sg for sg in dsegs if sg[0].shape[1] > 0][:3]
    o = S.chunk_attention_qrope(q.cuda(), (gt, gh, gw), dsegs, t0=t0)
    torch.cuda.synchronize()
    S.savgb_device_check()
    rows = None if n_q <= 512 else np.unique(np.r_[np.random.default_rng(2).choice(n_q, 32, replace=False),
                                                   [0, 127, 255, 256, n_q - 1]])
    q_rot = O.rope3d(f64(q), gt, gh, gw, t0)
    k_rot = O.rope3d(f64(kc), gt, gh, gw, t0)
    osegs = [(f64(k), f64(v)) for k, v in ctx if k.shape[1] > 0] + [(k_rot, f64(vc))]
    qq = q_rot if rows is None else q_rot[:, rows]
    want = O.attention(qq, osegs)
    got = f64(o) if rows is None else f64(o)[:, rows]
    assert_close(got, want, what=f"attention with RoPE of q inside (D={D}, grid {gt}x{gh}x{gw})", margin=n_q > 512)
    # the same kernel reading a table the caller built once: bit-identical output
    tab = S.chunk_attention_qrope_table(D, (gt, gh, gw), t0)
    o_tab = S.chunk_attention_qrope_with_table(q.cuda(), (gt, gh, gw), tab, dsegs, t0=t0)
    torch.cuda.synchronize()
    S.savgb_device_check()
    assert torch.equal(o_tab, o)
    # with the log-sum-exp output the kernel takes fp32 exponentials and exact row sums
    lse = torch.empty(B, H, n_q, dtype=torch.float32, device="cuda")
    o2 = S.chunk_attention_qrope(q.cuda(), (gt, gh, gw), dsegs, t0=t0, lse=lse)
    torch.cuda.synchronize()
    S.savgb_device_check()
    got2 = f64(o2) if rows is None else f64(o2)[:, rows]
    assert_close(got2, want, what=f"attention with RoPE of q inside and lse (D={D})")
    kk = np.concatenate([k for k, _ in osegs], axis=1)
    sc = 1.0 / math.sqrt(D)
    sco = np.einsum("bnhd,bmhd->bhnm", qq, kk) * sc
    mx = sco.max(-1, keepdims=True)
    want_lse = mx[..., 0] + np.log(np.exp(sco - mx).sum(-1))
    got_lse = f64(lse) if rows is None else f64(lse)[:, :, rows]
    # The kernel rounds the rotated queries to bf16 (its MMA operand) and the
    # oracle does not.  A score then moves by at most 2^-9 * sum_d |q_d k_d| *
    # scale (~0.014 at D = 128 for unit normals, ~1e-3 rms), and lse by a
    # p-weighted mean of those moves: bars 5e-3 / 1e-3 instead of the 1e-3 /
    # 1e-4 of the test whose queries arrive as bf16.
    assert_close(got_lse, want_lse, max_abs=5e-3, mean_abs=1e-3, what=f"lse with RoPE of q inside (D={D})")


# ------------------------------------------------------- DiT attention block

@pytest.mark.parametrize("B,H,D,gt,gh,gw,t0", [
    (1, 2, 64, 2, 4, 4, 0),     # tiny: 32 rows, 3*hid = 384 (single-CTA kernel, 128-column tiles)
    (2, 2, 128, 3, 5, 7, 1),    # ragged: 210 rows over two batches, t0 = 1 (CTA-pair kernel, one tile per cluster)
    (2, 8, 128, 3, 10, 30, 0),  # CTA pair: 96 tiles of 256 x 256 over 76 clusters, both accumulator buffers
    (1, 8, 64, 2, 7, 9, -1),    # CTA pair at D = 64: 126 rows (one partial row block), t0 = -1
])
def test_qkv_rope_project_parity(S, B, H, D, gt, gh, gw, t0):
    N, hid = gt * gh * gw, H * D
    x = torch.from_numpy(I.normal_f32((B, N, hid), 1.0, 50 + D, I.KIND_X))
    xb = x.to(torch.bfloat16)
    w = bf16((3 * hid, hid), 51, I.KIND_WQKV, std=1.0 / math.sqrt(hid))
    q, k, v = S.qkv_rope_project(xb.cuda(), w.cuda(), (gt, gh, gw), H, D, t0=t0)
    torch.cuda.synchronize()
    S.savgb_device_check()
    oq, ok_, ov = O.qkv_project(f64(xb).reshape(B * N, hid), f64(w), B, H, D)
    assert_close(f64(q), O.rope3d(oq, gt, gh, gw, t0), what="q (rotated)")
    assert_close(f64(k), O.rope3d(ok_, gt, gh, gw, t0), what="k (rotated)")
    assert_close(f64(v), ov, what="v")


_HOST_IO_WORKLOADS = {
    # two sessions of 1100 queries: W_o tiles straddle the sessions, ragged last attention blocks; the deepest
    # ring (8 slots: more than the 9 steps of the run can fill ahead of the compute)
    "two-sessions": (I.Workload("straddle", B=2, H=4, D=128, F=5, grid_h=10, grid_w=22, ref_frames=1,
                                boundary_frames=1, steps=3, shift=1.0), 8),
    # hid = 192: the single-CTA W_o kernel writes the staging copy
    "narrow": (I.Workload("narrow", B=1, H=3, D=64, F=3, grid_h=6, grid_w=10, ref_frames=1,
                          boundary_frames=1, steps=3, shift=1.0), 4),
}


@pytest.mark.parametrize("wname", list(_HOST_IO_WORKLOADS))
def test_stream_host_io_deep_rings(S, wname):
    """chunk_stream_step_host with deep input rings (4 and 8 device slots),
    three chunks: every step's read-back (from the staging copy the W_o update
    writes) bit-identical to chunk_stream_step's x after that step, each
    chunk's final x against the oracle.  Each chunk's x is a new device
    tensor; all of them stay alive until the sync, since the read-backs run
    after the call returns."""
    w, slots = _HOST_IO_WORKLOADS[wname]
    seed, chunks = 4, 3
    dts = S.flow_time_grid(w.steps, w.shift)
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed).cuda()
    plan = [(c, s_) for c in range(chunks) for s_ in range(w.steps)]
    ins = {p: I.step_inputs(w, seed, *p) for p in plan}
    x0 = [torch.from_numpy(I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, c)) for c in range(chunks)]

    def run(host_io):
        cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                           w.rope_base, host_io=host_io)
        cs.set_reference(rk.cuda(), rv.cuda())
        host_in = {p: tuple(t.pin_memory() for t in (ins[p].q, ins[p].k, ins[p].v)) for p in plan}
        out = {p: torch.empty((w.B * w.n_q, w.hid), dtype=torch.float32).pin_memory() for p in plan}
        xs = []
        for c in range(chunks):
            xs.append(x0[c].cuda())
            for s_ in range(w.steps):
                p, last = (c, s_), s_ == w.steps - 1
                if host_io:
                    cs.step_host(*host_in[p], wo, xs[c], dts[s_], last, x_host=out[p])
                else:
                    cs.step(*(t.cuda() for t in host_in[p]), wo, xs[c], dts[s_], last)
                    out[p].copy_(xs[c])
                if last:
                    cs.end_chunk()
        cs.sync()
        torch.cuda.synchronize()
        cs.close()
        return out, [x.cpu() for x in xs]

    want, _ = run(0)
    got, finals = run(slots)
    for p in plan:
        assert torch.equal(got[p], want[p]), f"read-back after chunk {p[0]} step {p[1]}"
    oracle_x, _ = run_stream_oracle(w, seed, chunks)
    for c in range(chunks):
        assert torch.equal(finals[c], want[(c, w.steps - 1)])
        assert_close(f64(finals[c]), oracle_x[c], what=f"host-io {wname} chunk {c} x")


_BLOCK_WORKLOADS = {
    "d64": I.Workload("blk", B=1, H=4, D=64, F=3, grid_h=8, grid_w=8, ref_frames=1, boundary_frames=1, steps=2,
                      shift=1.0),
    # two sessions of 189 tokens: projection and W_o tiles straddle the sessions, ragged attention blocks
    "d128-two-sessions": I.Workload("blk2", B=2, H=4, D=128, F=3, grid_h=7, grid_w=9, ref_frames=1,
                                    boundary_frames=1, steps=2, shift=1.0),
}


@pytest.mark.parametrize("wname", list(_BLOCK_WORKLOADS))
def test_stream_block_steps(S, wname):
    """Two chunks x two steps through one DiT attention block (q, k, v
    projected from x): every chunk's x against the oracle."""
    w = _BLOCK_WORKLOADS[wname]
    seed = 12
    rk, rv = I.reference_kv(w, seed)
    wqkv, wo = I.qkv_weight(w, seed), I.out_proj_weight(w, seed)
    dts = S.flow_time_grid(w.steps, w.shift)
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base, qkv_block=True)
    cs.set_reference(rk.cuda(), rv.cuda())
    xs = []
    for c in range(2):
        x = torch.from_numpy(I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, c)).cuda()
        for s, dt in enumerate(dts):
            cs.block_step(wqkv.cuda(), wo.cuda(), x, dt, s == len(dts) - 1)
        cs.end_chunk()
        xs.append(x.cpu())
    cs.sync()
    cs.close()
    want, _ = O.run_stream_block(w, f64(rk), f64(rv), f64(wqkv), f64(wo),
                              lambda c: I.normal_f32((w.B * w.n_q, w.hid), 1.0, seed, I.KIND_X, c).astype(np.float64),
                              O.time_grid(w.steps, w.shift), 2)
    for c in range(2):
        assert_close(f64(xs[c]), want[c], what=f"block chunk {c} x")


def test_stream_block_full_base_sampled_rows(S):
    """One base-shaped block step: sampled rows of x against the oracle
    (projection of every token, attention for the sampled queries)."""
    w = I.WORKLOADS["base"]
    seed = 13
    rk, rv = I.reference_kv(w, seed)
    wqkv, wo = I.qkv_weight(w, seed), I.out_proj_weight(w, seed)
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base, qkv_block=True)
    cs.set_reference(rk.cuda(), rv.cuda())
    x0 = I.state_x(w, seed)
    x = x0.cuda()
    dt = S.flow_time_grid(w.steps, w.shift)[0]
    cs.block_step(wqkv.cuda(), wo.cuda(), x, dt, False)
    cs.sync()
    got = x.cpu()
    cs.close()
    rows = np.unique(np.r_[np.random.default_rng(3).choice(w.n_q, 16, replace=False), [0, w.n_q - 1]])
    q, k, v = O.qkv_project(f64(x0), f64(wqkv), w.B, w.H, w.D)
    q_rot = O.rope3d(q, w.F, w.grid_h, w.grid_w, 0)[:, rows]
    k_rot = O.rope3d(k, w.F, w.grid_h, w.grid_w, 0)
    rk_rot = O.rope3d(f64(rk), 1, w.grid_h, w.grid_w, -1)
    o = O.attention(q_rot, [(rk_rot, f64(rv)), (k_rot, v)])
    want = O.euler_update(f64(x0)[rows], O.out_proj(o.reshape(len(rows), w.hid), f64(wo)), dt)
    assert_close(f64(got)[rows], want, what="base block step x (sampled rows)")
