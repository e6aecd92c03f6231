"""Python binding of the C ABI in include/savgb.h (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks tensor dtypes, devices, shapes and
contiguity, passes raw pointers, sizes and the current CUDA stream, and turns
a non-zero status into :class:`SavgbError`.  PyTorch supplies device memory and
streams.  If ``libsavgb.so`` has not been built the first call raises; nothing
falls back to another implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsavgb.so")

SAVGB_OK = 0
STATUS = {
    0: "SAVGB_OK", -1: "SAVGB_ERR_INVALID_ARG", -2: "SAVGB_ERR_UNSUPPORTED", -3: "SAVGB_ERR_ALIGNMENT",
    -4: "SAVGB_ERR_OOM", -5: "SAVGB_ERR_CUDA", -6: "SAVGB_ERR_TIMEOUT", -7: "SAVGB_ERR_STATE",
}

# every entry point of include/savgb.h
EXPORTS = (
    "savgb_status_string", "savgb_last_error", "savgb_version", "savgb_kernel_launches", "savgb_device_check",
    "savgb_watchdog_selftest", "savgb_arm_wait_fault", "rope3d_apply", "chunk_attention", "out_proj_euler_step",
    "flow_time_grid", "chunk_stream_create", "chunk_stream_set_reference", "chunk_stream_step",
    "chunk_stream_end_chunk", "chunk_stream_set_step_events", "chunk_stream_sync", "chunk_stream_info", "chunk_stream_export_state",
    "chunk_stream_import_state", "chunk_stream_destroy", "chunk_step_noalloc",
    "chunk_stream_istep", "chunk_stream_end_ichunk", "chunk_stream_ichunk_index", "chunk_attention_qrope",
    "qkv_rope_project", "chunk_stream_block_step", "chunk_stream_fused_q_rope", "chunk_attention_qrope_fits",
    "chunk_attention_qrope_table_bytes", "chunk_attention_qrope_build_table", "chunk_attention_qrope_with_table",
    "chunk_stream_step_host", "chunk_stream_join_copies",
)


class SavgbError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class KVSegment(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("n_tokens", ctypes.c_int64)]


class ChunkStreamConfig(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("D", ctypes.c_int), ("F", ctypes.c_int),
                ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int), ("ref_frames", ctypes.c_int),
                ("boundary_frames", ctypes.c_int), ("ref_t", ctypes.c_int),
                ("rope_base", ctypes.c_double), ("softmax_scale", ctypes.c_float),
                ("interp_chunks", ctypes.c_int), ("qkv_block", ctypes.c_int), ("host_io", ctypes.c_int),
                ("exact_softmax", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libsavgb.so (once) and declares the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    c_int, c_i64, c_vp, c_f, c_d = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_double
    sig = {
        "savgb_status_string": (ctypes.c_char_p, [c_int]),
        "savgb_last_error": (ctypes.c_char_p, []),
        "savgb_version": (c_int, []),
        "savgb_kernel_launches": (ctypes.c_uint64, []),
        "savgb_device_check": (c_int, [c_vp]),
        "savgb_watchdog_selftest": (c_int, [ctypes.c_uint64, c_vp]),
        "savgb_arm_wait_fault": (c_int, [c_int, c_int, ctypes.c_uint64]),
        "rope3d_apply": (c_int, [c_vp, c_vp, c_int, c_i64, c_int, c_int, c_int, c_int, c_int, c_int, c_d, c_vp]),
        "chunk_attention": (c_int, [c_vp, c_int, c_i64, c_int, c_int, ctypes.POINTER(KVSegment), c_int, c_f,
                                    c_vp, c_vp, c_vp]),
        "out_proj_euler_step": (c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_int, c_int, c_f, c_vp, c_vp]),
        "chunk_attention_qrope": (c_int, [c_vp, c_int, c_i64, c_int, c_int, c_int, c_int, c_int, c_int, c_d,
                                          ctypes.POINTER(KVSegment), c_int, c_f, c_vp, c_vp, c_vp]),
        "flow_time_grid": (c_int, [c_int, c_d, ctypes.POINTER(c_d)]),
        "chunk_stream_create": (c_int, [ctypes.POINTER(ChunkStreamConfig), c_vp, ctypes.POINTER(c_vp)]),
        "chunk_stream_set_reference": (c_int, [c_vp, c_vp, c_vp]),
        "chunk_stream_step": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f, c_int]),
        "chunk_stream_end_chunk": (c_int, [c_vp]),
        "chunk_stream_step_host": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f, c_int, c_vp]),
        "chunk_stream_join_copies": (c_int, [c_vp]),
        "chunk_stream_istep": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f]),
        "chunk_stream_block_step": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_f, c_int]),
        "qkv_rope_project": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_i64, c_int, c_int, c_int, c_int, c_int,
                                     c_int, c_d, c_vp]),
        "chunk_stream_end_ichunk": (c_int, [c_vp]),
        "chunk_stream_ichunk_index": (c_int, [c_vp, ctypes.POINTER(c_i64)]),
        "chunk_stream_set_step_events": (c_int, [c_vp, ctypes.POINTER(c_vp)]),
        "chunk_stream_sync": (c_int, [c_vp]),
        "chunk_stream_fused_q_rope": (c_int, [c_vp, ctypes.POINTER(c_int)]),
        "chunk_attention_qrope_fits": (c_int, [c_int, c_int, c_int, c_int, ctypes.POINTER(c_int)]),
        "chunk_attention_qrope_table_bytes": (c_int, [c_int, c_int, c_int, c_int, ctypes.POINTER(c_i64)]),
        "chunk_attention_qrope_build_table": (c_int, [c_vp, c_int, c_int, c_int, c_int, c_int, c_d, c_vp]),
        "chunk_attention_qrope_with_table": (c_int, [c_vp, c_int, c_i64, c_int, c_int, c_int, c_int, c_int, c_int,
                                                     c_vp, ctypes.POINTER(KVSegment), c_int, c_f, c_vp, c_vp, c_vp]),
        "chunk_stream_info": (c_int, [c_vp, ctypes.POINTER(c_i64), ctypes.POINTER(c_i64), ctypes.POINTER(c_i64),
                                      ctypes.POINTER(c_vp), ctypes.POINTER(c_vp)]),
        "chunk_stream_export_state": (c_int, [c_vp, c_vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]),
        "chunk_stream_import_state": (c_int, [c_vp, c_vp, ctypes.c_size_t]),
        "chunk_stream_destroy": (c_int, [c_vp]),
        "chunk_step_noalloc": (c_int, [c_vp, c_vp, c_vp, ctypes.POINTER(KVSegment), c_int, c_vp, c_vp, c_vp, c_f,
                                       c_int, c_int, c_int, c_int, c_int, c_int, c_d, c_f, c_vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(status: int) -> None:
    if status != SAVGB_OK:
        raise SavgbError(status, lib().savgb_last_error().decode(errors="replace"))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: Optional[int] = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _need_host(t: torch.Tensor, name: str, dtype: torch.dtype, numel: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {t.numel()}")


# ------------------------------------------------------------------ status

def savgb_version() -> int:
    return lib().savgb_version()


def savgb_kernel_launches() -> int:
    """Kernels this process has enqueued through the library so far (a host
    counter); the difference of two readings counts the calls' launches."""
    return int(lib().savgb_kernel_launches())


def savgb_device_check(stream=None) -> None:
    """Synchronises the stream and raises if a kernel's bounded wait ran out."""
    _check(lib().savgb_device_check(_stream(stream)))


def savgb_watchdog_selftest(limit_ns: int, stream=None) -> None:
    _check(lib().savgb_watchdog_selftest(int(limit_ns), _stream(stream)))


FAULT_ATTENTION_K_TILE = 1
FAULT_WO_PAIR_RELAY = 2


def savgb_arm_wait_fault(kind: int, index: int, limit_ns: int = 20_000_000) -> None:
    """Failure-path test hook: the next launch of the kernel of ``kind``
    skips one arrival at ``index`` and gives up its waits after ``limit_ns``
    (index < 0 disarms)."""
    _check(lib().savgb_arm_wait_fault(int(kind), int(index), int(limit_ns)))


# ------------------------------------------------------------------ kernels

def rope3d_apply(inp: torch.Tensor, out: torch.Tensor, grid_t: int, grid_h: int, grid_w: int,
                 t0: int = 0, base: float = 10000.0, stream=None) -> torch.Tensor:
    """out[B][N][H][D] <- 3D RoPE of inp (bf16; out may be inp)."""
    _need(inp, "inp", torch.bfloat16, 4)
    _need(out, "out", torch.bfloat16, 4)
    if out.shape != inp.shape:
        raise ValueError("out must have the shape of inp")
    B, N, H, D = inp.shape
    _check(lib().rope3d_apply(inp.data_ptr(), out.data_ptr(), B, N, H, D, grid_t, grid_h, grid_w, t0,
                              float(base), _stream(stream)))
    return out


def chunk_attention(q: torch.Tensor, segments: Sequence[Tuple[torch.Tensor, torch.Tensor]],
                    out: Optional[torch.Tensor] = None, scale: float = 0.0,
                    lse: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """O = softmax(scale q K^T) V over the concatenated (k, v) segments."""
    _need(q, "q", torch.bfloat16, 4)
    B, Nq, H, D = q.shape
    if not 1 <= len(segments) <= 3:
        raise ValueError("1 to 3 segments")
    segs = (KVSegment * 3)()
    for i, (k, v) in enumerate(segments):
        n = k.shape[1] if k.dim() == 4 else 0
        if n > 0:
            _need(k, f"segments[{i}].k", torch.bfloat16, 4)
            _need(v, f"segments[{i}].v", torch.bfloat16, 4)
            if k.shape != (B, n, H, D) or v.shape != k.shape:
                raise ValueError(f"segment {i} must be [B][n][H][D] like q")
            segs[i] = KVSegment(k.data_ptr(), v.data_ptr(), n)
        else:
            segs[i] = KVSegment(None, None, 0)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 4)
    if out.shape != q.shape:
        raise ValueError("out must have the shape of q")
    if lse is not None:
        _need(lse, "lse", torch.float32)
        if lse.numel() != B * H * Nq:
            raise ValueError("lse must hold B*H*n_q floats")
    _check(lib().chunk_attention(q.data_ptr(), B, Nq, H, D, segs, len(segments), float(scale),
                                 out.data_ptr(), _ptr(lse), _stream(stream)))
    return out


def chunk_attention_qrope(q: torch.Tensor, grid, segments: Sequence[Tuple[torch.Tensor, torch.Tensor]],
                          t0: int = 0, base: float = 10000.0, out: Optional[torch.Tensor] = None,
                          scale: float = 0.0, lse: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """chunk_attention with the 3D RoPE of the (unrotated) queries applied in
    the kernel; grid = (grid_t, grid_h, grid_w) of the queries."""
    _need(q, "q", torch.bfloat16, 4)
    B, Nq, H, D = q.shape
    gt, gh, gw = (int(g) for g in grid)
    if min(gt, gh, gw) < 1 or Nq != gt * gh * gw:
        raise ValueError(f"q has {Nq} tokens, the grid {gt}x{gh}x{gw} holds {gt * gh * gw}")
    if not 1 <= len(segments) <= 3:
        raise ValueError("1 to 3 segments")
    segs = (KVSegment * 3)()
    for i, (k, v) in enumerate(segments):
        n = k.shape[1] if k.dim() == 4 else 0
        if n > 0:
            _need(k, f"segments[{i}].k", torch.bfloat16, 4)
            _need(v, f"segments[{i}].v", torch.bfloat16, 4)
            if k.shape != (B, n, H, D) or v.shape != k.shape:
                raise ValueError(f"segment {i} must be [B][n][H][D] like q")
            segs[i] = KVSegment(k.data_ptr(), v.data_ptr(), n)
        else:
            segs[i] = KVSegment(None, None, 0)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 4)
    if out.shape != q.shape:
        raise ValueError("out must have the shape of q")
    if lse is not None:
        _need(lse, "lse", torch.float32)
        if lse.numel() != B * H * Nq:
            raise ValueError("lse must hold B*H*n_q floats")
    _check(lib().chunk_attention_qrope(q.data_ptr(), B, Nq, H, D, gt, gh, gw, t0, float(base), segs, len(segments),
                                       float(scale), out.data_ptr(), _ptr(lse), _stream(stream)))
    return out


def chunk_attention_qrope_table(D: int, grid, t0: int = 0, base: float = 10000.0, stream=None) -> torch.Tensor:
    """A cos/sin table for chunk_attention_qrope_with_table, built on the
    device for the query grid (grid_t, grid_h, grid_w) starting at time t0
    (the tensor is allocated here, by torch, once; the library allocates
    nothing)."""
    gt, gh, gw = (int(g) for g in grid)
    n = ctypes.c_int64()
    _check(lib().chunk_attention_qrope_table_bytes(int(D), gt, gh, gw, ctypes.byref(n)))
    tab = torch.empty(n.value, dtype=torch.uint8, device="cuda")
    _check(lib().chunk_attention_qrope_build_table(tab.data_ptr(), int(D), gt, gh, gw, int(t0), float(base),
                                                   _stream(stream)))
    return tab


def chunk_attention_qrope_with_table(q: torch.Tensor, grid, table: torch.Tensor,
                                     segments: Sequence[Tuple[torch.Tensor, torch.Tensor]], t0: int = 0,
                                     out: Optional[torch.Tensor] = None, scale: float = 0.0,
                                     lse: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """chunk_attention_qrope reading a table from chunk_attention_qrope_table
    (same D, grid and t0) instead of building one per call."""
    _need(q, "q", torch.bfloat16, 4)
    _need(table, "table", torch.uint8, 1)
    B, Nq, H, D = q.shape
    gt, gh, gw = (int(g) for g in grid)
    if min(gt, gh, gw) < 1 or Nq != gt * gh * gw:
        raise ValueError(f"q has {Nq} tokens, the grid {gt}x{gh}x{gw} holds {gt * gh * gw}")
    n = ctypes.c_int64()
    _check(lib().chunk_attention_qrope_table_bytes(D, gt, gh, gw, ctypes.byref(n)))
    if table.numel() < n.value:
        raise ValueError(f"table holds {table.numel()} bytes, the grid needs {n.value}")
    if not 1 <= len(segments) <= 3:
        raise ValueError("1 to 3 segments")
    segs = (KVSegment * 3)()
    for i, (k, v) in enumerate(segments):
        nk = k.shape[1] if k.dim() == 4 else 0
        if nk > 0:
            _need(k, f"segments[{i}].k", torch.bfloat16, 4)
            _need(v, f"segments[{i}].v", torch.bfloat16, 4)
            if k.shape != (B, nk, H, D) or v.shape != k.shape:
                raise ValueError(f"segment {i} must be [B][n][H][D] like q")
            segs[i] = KVSegment(k.data_ptr(), v.data_ptr(), nk)
        else:
            segs[i] = KVSegment(None, None, 0)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 4)
    if out.shape != q.shape:
        raise ValueError("out must have the shape of q")
    if lse is not None:
        _need(lse, "lse", torch.float32)
        if lse.numel() != B * H * Nq:
            raise ValueError("lse must hold B*H*n_q floats")
    _check(lib().chunk_attention_qrope_with_table(q.data_ptr(), B, Nq, H, D, gt, gh, gw, int(t0), table.data_ptr(),
                                                  segs, len(segments), float(scale), out.data_ptr(), _ptr(lse),
                                                  _stream(stream)))
    return out


def chunk_attention_qrope_fits(D: int, grid) -> bool:
    """Host query: whether the RoPE of q can run inside the attention kernel
    for this query grid (grid_t, grid_h, grid_w), the test that picks the
    RoPE form of the stream steps and of chunk_step_noalloc."""
    f = ctypes.c_int()
    gt, gh, gw = grid
    _check(lib().chunk_attention_qrope_fits(int(D), int(gt), int(gh), int(gw), ctypes.byref(f)))
    return bool(f.value)


def qkv_rope_project(x_bf16: torch.Tensor, w_qkv: torch.Tensor, grid, H: int, D: int, t0: int = 0,
                     base: float = 10000.0, stream=None):
    """q, k, v bf16 [B][N][H][D] = x W_qkv^T, q and k rotated (3D RoPE) in the
    GEMM epilogue; x_bf16 [B][N][H*D], grid = (grid_t, grid_h, grid_w)."""
    _need(x_bf16, "x_bf16", torch.bfloat16, 3)
    _need(w_qkv, "w_qkv", torch.bfloat16, 2)
    B, N, hid = x_bf16.shape
    if hid != H * D or tuple(w_qkv.shape) != (3 * hid, hid):
        raise ValueError("x must be [B][N][H*D] and w_qkv [3*H*D][H*D]")
    q, k, v = (torch.empty((B, N, H, D), dtype=torch.bfloat16, device=x_bf16.device) for _ in range(3))
    gt, gh, gw = grid
    _check(lib().qkv_rope_project(x_bf16.data_ptr(), w_qkv.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), B, N,
                                  H, D, gt, gh, gw, t0, float(base), _stream(stream)))
    return q, k, v


def out_proj_euler_step(o: torch.Tensor, w_o: torch.Tensor, x: torch.Tensor, dt: float,
                        bias: Optional[torch.Tensor] = None, v_out: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """x <- x + dt * (o W_o^T + bias); o bf16 [M][hid_in] (or [B][N][H][D]), x fp32 [M][hid_out]."""
    _need(o, "o", torch.bfloat16)
    _need(w_o, "w_o", torch.bfloat16, 2)
    _need(x, "x", torch.float32)
    hid_out, hid_in = w_o.shape
    M = o.numel() // hid_in
    if M * hid_in != o.numel() or x.numel() != M * hid_out:
        raise ValueError("o must hold M*hid_in and x M*hid_out elements")
    if bias is not None:
        _need(bias, "bias", torch.float32, 1)
        if bias.numel() != hid_out:
            raise ValueError("bias must have hid_out elements")
    if v_out is not None:
        _need(v_out, "v_out", torch.float32)
        if v_out.numel() != M * hid_out:
            raise ValueError("v_out must hold M*hid_out floats")
    _check(lib().out_proj_euler_step(o.data_ptr(), w_o.data_ptr(), _ptr(bias), x.data_ptr(), M, hid_in,
                                     hid_out, float(dt), _ptr(v_out), _stream(stream)))
    return x


def flow_time_grid(steps: int, shift: float = 1.0):
    """Host: step sizes dt_0..dt_{steps-1} of the (shifted) sampling grid."""
    buf = (ctypes.c_double * max(int(steps), 1))()
    _check(lib().flow_time_grid(int(steps), float(shift), buf))
    return [buf[i] for i in range(int(steps))]


# -------------------------------------------------------------- chunk stream

class ChunkStream:
    """Handle of chunk_stream_* (one fixed device arena per handle)."""

    def __init__(self, B: int, H: int, D: int, F: int, grid_h: int, grid_w: int, ref_frames: int = 1,
                 boundary_frames: int = 0, ref_t: int = -1, rope_base: float = 10000.0,
                 softmax_scale: float = 0.0, stream=None, interp_chunks: bool = False, qkv_block: bool = False,
                 host_io: int = 0, exact_softmax: bool = False):
        self.cfg = ChunkStreamConfig(B, H, D, F, grid_h, grid_w, ref_frames, boundary_frames, ref_t,
                                     float(rope_base), float(softmax_scale), int(bool(interp_chunks)),
                                     int(bool(qkv_block)), int(host_io), int(bool(exact_softmax)))
        self.stream = _stream(stream)
        h = ctypes.c_void_p()
        _check(lib().chunk_stream_create(ctypes.byref(self.cfg), self.stream, ctypes.byref(h)))
        self.handle = h

    def set_reference(self, k_ref: torch.Tensor, v_ref: torch.Tensor) -> None:
        _need(k_ref, "k_ref", torch.bfloat16, 4)
        _need(v_ref, "v_ref", torch.bfloat16, 4)
        c = self.cfg
        shp = (c.B, c.ref_frames * c.grid_h * c.grid_w, c.H, c.D)
        if tuple(k_ref.shape) != shp or tuple(v_ref.shape) != shp:
            raise ValueError(f"reference must be {shp}")
        _check(lib().chunk_stream_set_reference(self.handle, k_ref.data_ptr(), v_ref.data_ptr()))

    def step(self, q, k, v, w_o, x, dt: float, is_last_step: bool, bias=None) -> None:
        c = self.cfg
        shp = (c.B, c.F * c.grid_h * c.grid_w, c.H, c.D)
        for name, t in (("q", q), ("k", k), ("v", v)):
            _need(t, name, torch.bfloat16, 4)
            if tuple(t.shape) != shp:
                raise ValueError(f"{name} must be {shp}")
        _need(w_o, "w_o", torch.bfloat16, 2)
        _need(x, "x", torch.float32)
        hid = c.H * c.D
        if tuple(w_o.shape) != (hid, hid) or x.numel() != shp[0] * shp[1] * hid:
            raise ValueError("w_o must be [hid][hid] and x [B*N][hid]")
        if bias is not None:
            _need(bias, "bias", torch.float32, 1)
            if bias.numel() != hid:
                raise ValueError("bias must hold hid floats")
        _check(lib().chunk_stream_step(self.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), w_o.data_ptr(),
                                       _ptr(bias), x.data_ptr(), float(dt), int(bool(is_last_step))))

    def end_chunk(self) -> None:
        _check(lib().chunk_stream_end_chunk(self.handle))

    def step_host(self, q_host, k_host, v_host, w_o, x, dt: float, is_last_step: bool, bias=None,
                  x_host=None) -> None:
        """chunk_stream_step with q, k, v in host memory (bf16 CPU tensors,
        pinned for overlap) and, with x_host (fp32 CPU tensor), the updated
        state read back; x stays on the device.  Needs host_io.  The host
        tensors must stay untouched until sync() or a join_copies() that the
        stream has passed."""
        c = self.cfg
        n = c.B * c.F * c.grid_h * c.grid_w * c.H * c.D
        for name, t in (("q_host", q_host), ("k_host", k_host), ("v_host", v_host)):
            _need_host(t, name, torch.bfloat16, n)
        _need(w_o, "w_o", torch.bfloat16, 2)
        _need(x, "x", torch.float32)
        hid = c.H * c.D
        if tuple(w_o.shape) != (hid, hid) or x.numel() != n:
            raise ValueError("w_o must be [hid][hid] and x [B*N][hid]")
        if bias is not None:
            _need(bias, "bias", torch.float32, 1)
            if bias.numel() != hid:
                raise ValueError("bias must hold hid floats")
        if x_host is not None:
            _need_host(x_host, "x_host", torch.float32, n)
        _check(lib().chunk_stream_step_host(self.handle, q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(),
                                            w_o.data_ptr(), _ptr(bias), x.data_ptr(), float(dt),
                                            int(bool(is_last_step)), _ptr(x_host)))

    def join_copies(self) -> None:
        """The stream waits for every upload and read-back enqueued so far."""
        _check(lib().chunk_stream_join_copies(self.handle))

    def istep(self, q, k, v, w_o, x, dt: float, bias=None) -> None:
        """One step of the pending interpolation chunk (interior frames only)."""
        c = self.cfg
        shp = (c.B, (c.F - 2) * c.grid_h * c.grid_w, c.H, c.D)
        for name, t in (("q", q), ("k", k), ("v", v)):
            _need(t, name, torch.bfloat16, 4)
            if tuple(t.shape) != shp:
                raise ValueError(f"{name} must be {shp}")
        _need(w_o, "w_o", torch.bfloat16, 2)
        _need(x, "x", torch.float32)
        hid = c.H * c.D
        if tuple(w_o.shape) != (hid, hid) or x.numel() != shp[0] * shp[1] * hid:
            raise ValueError("w_o must be [hid][hid] and x [B*(F-2)*h*w][hid]")
        if bias is not None:
            _need(bias, "bias", torch.float32, 1)
            if bias.numel() != hid:
                raise ValueError("bias must hold hid floats")
        _check(lib().chunk_stream_istep(self.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), w_o.data_ptr(),
                                        _ptr(bias), x.data_ptr(), float(dt)))

    def block_step(self, w_qkv, w_o, x, dt: float, is_last_step: bool, bias=None) -> None:
        """One denoising step through one DiT attention block: q, k, v are
        projected from x itself (needs qkv_block)."""
        c = self.cfg
        hid = c.H * c.D
        _need(w_qkv, "w_qkv", torch.bfloat16, 2)
        _need(w_o, "w_o", torch.bfloat16, 2)
        _need(x, "x", torch.float32)
        if tuple(w_qkv.shape) != (3 * hid, hid) or tuple(w_o.shape) != (hid, hid):
            raise ValueError("w_qkv must be [3*hid][hid] and w_o [hid][hid]")
        if x.numel() != c.B * c.F * c.grid_h * c.grid_w * hid:
            raise ValueError("x must be [B*N][hid]")
        if bias is not None:
            _need(bias, "bias", torch.float32, 1)
            if bias.numel() != hid:
                raise ValueError("bias must hold hid floats")
        _check(lib().chunk_stream_block_step(self.handle, w_qkv.data_ptr(), w_o.data_ptr(), _ptr(bias), x.data_ptr(),
                                             float(dt), int(bool(is_last_step))))

    def end_ichunk(self) -> None:
        _check(lib().chunk_stream_end_ichunk(self.handle))

    def ichunk_index(self) -> int:
        i = ctypes.c_int64()
        _check(lib().chunk_stream_ichunk_index(self.handle, ctypes.byref(i)))
        return i.value

    def set_step_events(self, events) -> None:
        """events: 4 torch.cuda.Event (created with enable_timing) recorded by
        the next step at its start, after RoPE, after attention and after
        the W_o/Euler GEMM; None clears them."""
        if events is None:
            _check(lib().chunk_stream_set_step_events(self.handle, None))
            return
        if len(events) != 4:
            raise ValueError("4 events")
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event on its first record
                e.record()
        arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
        _check(lib().chunk_stream_set_step_events(self.handle, arr))

    def sync(self) -> None:
        _check(lib().chunk_stream_sync(self.handle))

    @property
    def fused_q_rope(self) -> bool:
        """True when the steps rotate q inside the attention kernel (the RoPE
        pass then rotates k only)."""
        f = ctypes.c_int()
        _check(lib().chunk_stream_fused_q_rope(self.handle, ctypes.byref(f)))
        return bool(f.value)

    def info(self) -> dict:
        ci, bt, ab = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        bk, bv = ctypes.c_void_p(), ctypes.c_void_p()
        _check(lib().chunk_stream_info(self.handle, ctypes.byref(ci), ctypes.byref(bt), ctypes.byref(ab),
                                       ctypes.byref(bk), ctypes.byref(bv)))
        return {"chunk_index": ci.value, "boundary_tokens": bt.value, "arena_bytes": ab.value,
                "boundary_k": bk.value, "boundary_v": bv.value}

    # magic u64, 8 x int32, chunk index, boundary tokens, payload bytes, I-chunk index, reserved (int64)
    STATE_HEADER_BYTES = 80

    def boundary(self):
        """Host copies of the boundary K (rotated) and V in use, bf16 [B][n_b][H][D]
        (None on chunk 0), read back through export_state."""
        raw = self.export_state()
        n = int.from_bytes(raw[48:56], "little", signed=True)
        if n == 0:
            return None
        c = self.cfg
        shp = (c.B, n, c.H, c.D)
        count = c.B * n * c.H * c.D
        body = torch.frombuffer(bytearray(raw[self.STATE_HEADER_BYTES:]), dtype=torch.bfloat16)
        return body[:count].reshape(shp).clone(), body[count:2 * count].reshape(shp).clone()

    def export_state(self) -> bytes:
        n = ctypes.c_size_t()
        _check(lib().chunk_stream_export_state(self.handle, None, 0, ctypes.byref(n)))
        buf = ctypes.create_string_buffer(n.value)
        _check(lib().chunk_stream_export_state(self.handle, buf, n.value, ctypes.byref(n)))
        return buf.raw[: n.value]

    def import_state(self, state: bytes) -> None:
        buf = ctypes.create_string_buffer(state, len(state))
        _check(lib().chunk_stream_import_state(self.handle, buf, len(state)))

    def close(self) -> None:
        if getattr(self, "handle", None):
            _check(lib().chunk_stream_destroy(self.handle))
            self.handle = None

    def __enter__(self) -> "ChunkStream":
        return self

    def __exit__(self, *exc) -> None:
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------ allocation-free step

NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def chunk_step_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       context: Sequence[Tuple[torch.Tensor, torch.Tensor]], w_o: torch.Tensor,
                       x: torch.Tensor, dt: float, grid: Tuple[int, int, int], bias: Optional[torch.Tensor] = None,
                       rope_base: float = 10000.0, softmax_scale: float = 0.0, stream=None) -> torch.Tensor:
    """One chunk step whose intermediates live in the library's fixed device
    scratch array (no allocation by the library).  For callers that cannot
    allocate device memory while a session runs; the caller passes the
    already-rotated reference / boundary segments in ``context``.
    grid = (F, grid_h, grid_w)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 4)
    B, N, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have one shape")
    F, gh, gw = (int(g) for g in grid)
    if min(F, gh, gw) < 1 or N != F * gh * gw:
        raise ValueError(f"q has {N} tokens, the grid {F}x{gh}x{gw} holds {F * gh * gw}")
    hid = H * D
    if len(context) > 2:
        raise ValueError("0 to 2 context segments")
    segs = (KVSegment * 2)()
    for i, (ck, cv) in enumerate(context):
        _need(ck, f"context[{i}].k", torch.bfloat16, 4)
        _need(cv, f"context[{i}].v", torch.bfloat16, 4)
        if ck.shape[0] != B or tuple(ck.shape[2:]) != (H, D) or cv.shape != ck.shape:
            raise ValueError(f"context[{i}] k and v must both be [B][n][H][D] = [{B}][n][{H}][{D}]")
        segs[i] = KVSegment(ck.data_ptr(), cv.data_ptr(), ck.shape[1])
    _need(w_o, "w_o", torch.bfloat16, 2)
    if tuple(w_o.shape) != (hid, hid):
        raise ValueError(f"w_o must be [{hid}][{hid}]")
    _need(x, "x", torch.float32)
    if x.numel() != B * N * hid:
        raise ValueError(f"x must hold B*N*H*D = {B * N * hid} floats")
    if bias is not None:
        _need(bias, "bias", torch.float32, 1)
        if bias.numel() != hid:
            raise ValueError(f"bias must hold {hid} floats")
    _check(lib().chunk_step_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), segs, len(context), w_o.data_ptr(),
                                    _ptr(bias), x.data_ptr(), float(dt), B, H, D, F, gh, gw, float(rope_base),
                                    float(softmax_scale), _stream(stream)))
    return x
