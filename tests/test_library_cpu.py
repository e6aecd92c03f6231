"""CPU-side checks of the built library: it loads, exports every symbol that
include/savgb.h declares, and its host-only logic (time grid, argument
validation before any launch) behaves."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def S():
    import __graft_entry__ as g
    g.build()
    from streaming_avatar_video_gb300 import savgb
    return savgb


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "savgb.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(S):
    names = declared_symbols()
    assert "chunk_attention" in names and "rope3d_apply" in names and "chunk_stream_step" in names
    lib = ctypes.CDLL(S.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"libsavgb.so does not export {n}"
    assert sorted(S.EXPORTS) == names, "binding and header disagree"


def test_status_strings(S):
    L = S.lib()
    for code, name in S.STATUS.items():
        assert L.savgb_status_string(code).decode() == name
    assert S.savgb_version() >= 100


@pytest.mark.parametrize("steps,shift", [(1, 1.0), (4, 1.0), (8, 1.0), (30, 3.0), (30, 5.0), (7, 0.5)])
def test_time_grid_matches_oracle(S, steps, shift):
    got = np.array(S.flow_time_grid(steps, shift))
    assert np.allclose(got, O.time_grid(steps, shift), rtol=1e-14, atol=1e-16)
    assert abs(got.sum() - 1.0) < 1e-13


def test_time_grid_rejects_bad_args(S):
    with pytest.raises(S.SavgbError) as e:
        S.flow_time_grid(0, 1.0)
    assert e.value.status == -1
    buf = (ctypes.c_double * 4)()
    assert S.lib().flow_time_grid(4, -1.0, buf) == -1
    assert S.lib().flow_time_grid(4, float("nan"), buf) == -1
    assert b"shift" in S.lib().savgb_last_error()


def test_entry_points_validate_before_launch(S):
    """Invalid sizes and pointers are refused on the host, with no device call."""
    L = S.lib()
    c_vp = ctypes.c_void_p
    # rope: null, misaligned, grid mismatch, odd D
    assert L.rope3d_apply(None, None, 1, 8, 1, 64, 2, 2, 2, 0, 1e4, None) == -1
    assert L.rope3d_apply(c_vp(17), c_vp(32), 1, 8, 1, 64, 2, 2, 2, 0, 1e4, None) == -3
    assert L.rope3d_apply(c_vp(16), c_vp(32), 1, 9, 1, 64, 2, 2, 2, 0, 1e4, None) == -1
    assert L.rope3d_apply(c_vp(16), c_vp(32), 1, 8, 1, 60, 2, 2, 2, 0, 1e4, None) == -1
    assert L.rope3d_apply(c_vp(16), c_vp(32), 1, 8, 1, 64, 2, 2, 2, 0, -1.0, None) == -1
    # attention: bad head_dim, no segments, zero tokens, misaligned
    segs = (S.KVSegment * 3)()
    segs[0] = S.KVSegment(16, 32, 4)
    assert L.chunk_attention(c_vp(16), 1, 8, 2, 96, segs, 1, 0.0, c_vp(16), None, None) == -2
    assert L.chunk_attention(c_vp(16), 1, 8, 2, 64, segs, 0, 0.0, c_vp(16), None, None) == -1
    segs[0] = S.KVSegment(16, 32, 0)
    assert L.chunk_attention(c_vp(16), 1, 8, 2, 64, segs, 1, 0.0, c_vp(16), None, None) == -1
    segs[0] = S.KVSegment(24, 32, 4)
    assert L.chunk_attention(c_vp(16), 1, 8, 2, 64, segs, 1, 0.0, c_vp(16), None, None) == -3
    # projection: bad sizes
    assert L.out_proj_euler_step(c_vp(16), c_vp(16), None, c_vp(16), 4, 12, 16, 0.1, None, None) == -1
    assert L.out_proj_euler_step(c_vp(16), c_vp(16), None, c_vp(16), 4, 16, 24, 0.1, None, None) == -1
    assert L.out_proj_euler_step(c_vp(16), c_vp(16), None, c_vp(16), 0, 16, 16, 0.1, None, None) == -1
    # stream: bad config
    cfg = S.ChunkStreamConfig(1, 2, 96, 2, 4, 4, 1, 0, -1, 1e4, 0.0)
    h = ctypes.c_void_p()
    assert L.chunk_stream_create(ctypes.byref(cfg), None, ctypes.byref(h)) == -2
    cfg = S.ChunkStreamConfig(1, 2, 64, 2, 4, 4, 1, 3, -1, 1e4, 0.0)  # boundary_frames > F
    assert L.chunk_stream_create(ctypes.byref(cfg), None, ctypes.byref(h)) == -1
    for bad in (-1, 9):  # host_io: 0 (off), else 1 to 8 input slots
        cfg = S.ChunkStreamConfig(1, 2, 64, 2, 4, 4, 1, 1, -1, 1e4, 0.0, 0, 0, bad)
        assert L.chunk_stream_create(ctypes.byref(cfg), None, ctypes.byref(h)) == -1
    assert L.chunk_stream_end_chunk(None) == -1
    assert L.chunk_stream_destroy(None) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from streaming_avatar_video_gb300 import savgb
    monkeypatch.setattr(savgb, "_lib", None)
    monkeypatch.setattr(savgb, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        savgb.lib()


def test_qrope_fits_query(S):
    """The host query that picks the RoPE form: every configured grid fits,
    a 2 x 400 grid (table past the shared-memory limit) does not, another
    head_dim never does, and a grid size below 1 is refused."""
    for D, grid in [(64, (2, 4, 4)), (64, (4, 16, 16)), (128, (8, 30, 52)), (128, (8, 60, 104)), (128, (3, 8, 12))]:
        assert S.chunk_attention_qrope_fits(D, grid), (D, grid)
    assert not S.chunk_attention_qrope_fits(128, (2, 2, 400))
    assert not S.chunk_attention_qrope_fits(96, (2, 4, 4))
    with pytest.raises(S.SavgbError):
        S.chunk_attention_qrope_fits(128, (0, 4, 4))
    assert S.lib().chunk_attention_qrope_fits(128, 1, 1, 1, None) == -1


def test_noalloc_validates_before_any_device_call(S):
    """chunk_step_noalloc refuses, on the host, a step beyond its fixed
    scratch array (naming the array's size, also for sizes whose product
    would overflow), out-of-range counts, an unsupported head_dim and a
    non-finite dt."""
    L = S.lib()
    c_vp = ctypes.c_void_p
    p = c_vp(256)
    # base-DiT chunk: 2 x 12480 x 3072 x 2 bytes alone exceed the array
    assert L.chunk_step_noalloc(p, p, p, None, 0, p, None, p, 0.1, 1, 24, 128, 8, 30, 52, 1e4, 0.0, None) == -1
    msg = L.savgb_last_error().decode()
    assert "scratch" in msg and str(S.NOALLOC_SCRATCH_BYTES) in msg
    # sizes whose product would overflow 64-bit arithmetic are refused the same way
    assert L.chunk_step_noalloc(p, p, p, None, 0, p, None, p, 0.1, 65535, 65535, 128, 4096, 4096, 4096, 1e4, 0.0,
                                None) == -1
    # heads beyond the launch grid's limit
    assert L.chunk_step_noalloc(p, p, p, None, 0, p, None, p, 0.1, 1, 65536, 128, 1, 1, 1, 1e4, 0.0, None) == -1
    assert L.chunk_step_noalloc(p, p, p, None, 0, p, None, p, 0.1, 1, 2, 96, 1, 4, 4, 1e4, 0.0, None) == -2
    assert L.chunk_step_noalloc(p, p, p, None, 3, p, None, p, 0.1, 1, 2, 64, 1, 4, 4, 1e4, 0.0, None) == -1
    assert L.chunk_step_noalloc(p, p, p, None, 0, p, None, p, float("nan"), 1, 2, 64, 1, 4, 4, 1e4, 0.0, None) == -1


def test_arm_wait_fault_validates(S):
    """The failure-path hook refuses unknown kinds and out-of-range limits;
    a negative index disarms (no device work either way)."""
    L = S.lib()
    assert L.savgb_arm_wait_fault(0, 1, 1000) == -1
    assert L.savgb_arm_wait_fault(3, 1, 1000) == -1
    assert L.savgb_arm_wait_fault(S.FAULT_ATTENTION_K_TILE, 1, 0) == -1
    assert L.savgb_arm_wait_fault(S.FAULT_ATTENTION_K_TILE, 1, 10_000_000_001) == -1
    assert L.savgb_arm_wait_fault(S.FAULT_WO_PAIR_RELAY, 2, 5_000_000) == 0
    assert L.savgb_arm_wait_fault(S.FAULT_WO_PAIR_RELAY, -1, 0) == 0  # disarmed


def test_qrope_table_calls_validate(S):
    """The caller-built table path: size query, null / misaligned tables,
    and a grid the table does not cover are refused on the host."""
    L = S.lib()
    c_vp = ctypes.c_void_p
    n = ctypes.c_int64()
    assert L.chunk_attention_qrope_table_bytes(128, 8, 30, 52, ctypes.byref(n)) == 0
    assert n.value == 8 * (8 * 22 + 30 * 21 + 52 * 21 + (30 * 21) % 2 + (52 * 21) % 2)  # [t | h | w], sections even
    assert L.chunk_attention_qrope_table_bytes(96, 8, 30, 52, ctypes.byref(n)) == -2
    assert L.chunk_attention_qrope_table_bytes(128, 0, 30, 52, ctypes.byref(n)) == -1
    assert L.chunk_attention_qrope_build_table(None, 128, 2, 4, 4, 0, 1e4, None) == -1
    assert L.chunk_attention_qrope_build_table(c_vp(24), 128, 2, 4, 4, 0, 1e4, None) == -3
    assert L.chunk_attention_qrope_build_table(c_vp(32), 128, 2, 4, 4, 0, -1.0, None) == -1
    segs = (S.KVSegment * 3)()
    segs[0] = S.KVSegment(16, 32, 4)
    assert L.chunk_attention_qrope_with_table(c_vp(16), 1, 32, 2, 128, 2, 4, 4, 0, None, segs, 1, 0.0, c_vp(16),
                                              None, None) == -1
    assert L.chunk_attention_qrope_with_table(c_vp(16), 1, 33, 2, 128, 2, 4, 4, 0, c_vp(64), segs, 1, 0.0,
                                              c_vp(16), None, None) == -1  # n_q != grid


def test_c_abi_from_plain_c(S, tmp_path):
    """The header compiles as C99 and as C++17 with every warning an error, and
    a plain C program linked against libsavgb.so runs the host-only calls as
    the header states (tests/abi_c_check.c)."""
    import shutil
    import subprocess
    cc, cxx = shutil.which("gcc") or shutil.which("cc"), shutil.which("g++") or shutil.which("c++")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(S.LIB_PATH)
    exe = str(tmp_path / "abi_c_check")
    flags = ["-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include")]
    subprocess.run([cc, "-std=c99", "-pedantic", *flags, os.path.join(ROOT, "tests", "abi_c_check.c"),
                    "-L", lib_dir, "-lsavgb", f"-Wl,-rpath,{lib_dir}", "-lm", "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr
    if cxx is not None:
        src = tmp_path / "header.cpp"
        src.write_text('#include "savgb.h"\nint main() { return savgb_version() > 0 ? 0 : 1; }\n')
        subprocess.run([cxx, "-std=c++17", *flags, "-fsyntax-only", str(src)], check=True)
