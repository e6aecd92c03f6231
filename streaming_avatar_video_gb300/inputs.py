"""Seeded synthetic inputs for the chunk denoising step.

This module is shared by the tests, the benchmark and the oracle's callers. It
holds the workload shapes and a seeded Gaussian generator, and nothing of the
step's arithmetic (no RoPE, attention, projection or time grid).

The workloads are shaped like the two DiT stages described in HeyGen,
"Avatar inference at scale", section "The underlying model architecture": a
base audio-to-video DiT producing low-resolution video latents chunk by chunk
and an identity-aware super-resolution DiT on the same chunks at higher
resolution.  The pages give no token counts; the shapes below are the
synthetic stand-ins used throughout this library.

Every tensor is drawn from NumPy's PCG64 stream keyed by
``(seed, kind, chunk, step)``, as float32 standard normals, scaled by a float32
constant and rounded to bfloat16 with round-to-nearest-even (torch's
conversion).  The state ``x`` stays float32.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

# tensor kinds: part of each stream key
KIND_Q, KIND_K, KIND_V, KIND_REF_K, KIND_REF_V, KIND_WO, KIND_X, KIND_BIAS, KIND_WQKV = range(1, 10)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One chunk-step workload: B sessions of H heads of size D on a
    F x grid_h x grid_w latent chunk, with ``ref_frames`` reference frames
    and ``boundary_frames`` frames carried from the previous chunk."""

    name: str
    B: int
    H: int
    D: int
    F: int
    grid_h: int
    grid_w: int
    ref_frames: int
    boundary_frames: int
    steps: int
    shift: float  # 1.0 = uniform time grid
    chunks: int = 1
    ref_t: int = -1
    rope_base: float = 10000.0

    @property
    def hid(self) -> int:
        return self.H * self.D

    @property
    def frame_tokens(self) -> int:
        return self.grid_h * self.grid_w

    @property
    def n_q(self) -> int:
        return self.F * self.frame_tokens

    @property
    def n_ref(self) -> int:
        return self.ref_frames * self.frame_tokens

    @property
    def n_b(self) -> int:
        return self.boundary_frames * self.frame_tokens

    @property
    def n_kv(self) -> int:
        return self.n_ref + self.n_b + self.n_q

    def attn_flops(self, with_boundary: bool = True) -> float:
        """Dense attention flops of one step: 2 GEMMs of 2*Nq*Nkv*D per head."""
        n_kv = self.n_kv if with_boundary else self.n_ref + self.n_q
        return 4.0 * self.B * self.H * self.n_q * n_kv * self.D

    def wo_flops(self) -> float:
        return 2.0 * self.B * self.n_q * self.hid * self.hid


WORKLOADS = {
    # tiny chunk 0: 2 heads of 64, a 2x4x4 chunk, one 4x4 reference frame, no boundary
    "tiny": Workload("tiny", B=1, H=2, D=64, F=2, grid_h=4, grid_w=4, ref_frames=1,
                     boundary_frames=0, steps=1, shift=1.0),
    # small streamed pair: 8 heads of 64, 4x16x16 chunks, 1-frame boundary, 2 chunks x 4 steps
    "small": Workload("small", B=1, H=8, D=64, F=4, grid_h=16, grid_w=16, ref_frames=1,
                      boundary_frames=1, steps=4, shift=1.0, chunks=2),
    # base-DiT-shaped chunk: 24 heads of 128, 8x30x52 chunk, 2-frame boundary, 30 shifted steps
    "base": Workload("base", B=1, H=24, D=128, F=8, grid_h=30, grid_w=52, ref_frames=1,
                     boundary_frames=2, steps=30, shift=3.0),
    # SR-shaped chunk: 24 heads of 128, 8x60x104 chunk, 2-frame boundary, 8 uniform steps
    "sr": Workload("sr", B=1, H=24, D=128, F=8, grid_h=60, grid_w=104, ref_frames=1,
                   boundary_frames=2, steps=8, shift=1.0),
    # SR-shaped chunk refined in a single step (dt = 1)
    "sr1": Workload("sr1", B=1, H=24, D=128, F=8, grid_h=60, grid_w=104, ref_frames=1,
                    boundary_frames=2, steps=1, shift=1.0),
    # long session: 4 sessions batched, 64 base-shaped chunks each
    "long": Workload("long", B=4, H=24, D=128, F=8, grid_h=30, grid_w=52, ref_frames=1,
                     boundary_frames=2, steps=30, shift=3.0, chunks=64),
}


def _rng(seed: int, kind: int, chunk: int = 0, step: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, kind, chunk, step])))


def normal_f32(shape, std: float, seed: int, kind: int, chunk: int = 0, step: int = 0) -> np.ndarray:
    """float32 N(0, std^2) samples of ``shape`` from the keyed stream."""
    a = _rng(seed, kind, chunk, step).standard_normal(size=int(np.prod(shape)), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a.reshape(shape)


def normal_bf16(shape, std: float, seed: int, kind: int, chunk: int = 0, step: int = 0) -> torch.Tensor:
    """bfloat16 (CPU) N(0, std^2) tensor, rounded to nearest even from float32."""
    return torch.from_numpy(normal_f32(shape, std, seed, kind, chunk, step)).to(torch.bfloat16)


@dataclasses.dataclass
class StepInputs:
    """Host tensors of one chunk step (CPU, contiguous).

    q, k, v: bf16 [B][n_q][H][D] (the chunk's projected tokens, before RoPE)
    """

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor


def step_inputs(w: Workload, seed: int, chunk: int, step: int) -> StepInputs:
    shp = (w.B, w.n_q, w.H, w.D)
    return StepInputs(
        q=normal_bf16(shp, 1.0, seed, KIND_Q, chunk, step),
        k=normal_bf16(shp, 1.0, seed, KIND_K, chunk, step),
        v=normal_bf16(shp, 1.0, seed, KIND_V, chunk, step),
    )


def istep_inputs(w: Workload, seed: int, ichunk: int, step: int) -> StepInputs:
    """Interior tokens of an interpolation chunk: bf16 [B][(F-2)*h*w][H][D]."""
    shp = (w.B, (w.F - 2) * w.frame_tokens, w.H, w.D)
    key = 0x4000 + ichunk
    return StepInputs(
        q=normal_bf16(shp, 1.0, seed, KIND_Q, key, step),
        k=normal_bf16(shp, 1.0, seed, KIND_K, key, step),
        v=normal_bf16(shp, 1.0, seed, KIND_V, key, step),
    )


def reference_kv(w: Workload, seed: int):
    """Static reference tokens' K and V, bf16 [B][n_ref][H][D], before RoPE."""
    shp = (w.B, w.n_ref, w.H, w.D)
    return (normal_bf16(shp, 1.0, seed, KIND_REF_K), normal_bf16(shp, 1.0, seed, KIND_REF_V))


def boundary_kv(w: Workload, seed: int):
    """Stand-alone boundary K and V, bf16 [B][n_b][H][D], before RoPE.

    Used when one step is run on its own rather than inside a stream, where the
    boundary is the previous chunk's last frames instead."""
    shp = (w.B, w.n_b, w.H, w.D)
    return (normal_bf16(shp, 1.0, seed, KIND_K, chunk=-1 & 0xFFFF, step=0xB0),
            normal_bf16(shp, 1.0, seed, KIND_V, chunk=-1 & 0xFFFF, step=0xB0))


def out_proj_weight(w: Workload, seed: int) -> torch.Tensor:
    """W_o, bf16 [hid_out][hid_in] ~ N(0, 1/hid)."""
    return normal_bf16((w.hid, w.hid), 1.0 / math.sqrt(w.hid), seed, KIND_WO)


def qkv_weight(w: Workload, seed: int) -> torch.Tensor:
    """W_qkv = [W_q; W_k; W_v], bf16 [3*hid][hid] ~ N(0, 1/hid)."""
    return normal_bf16((3 * w.hid, w.hid), 1.0 / math.sqrt(w.hid), seed, KIND_WQKV)


def state_x(w: Workload, seed: int) -> torch.Tensor:
    """Flow state x, float32 [B*n_q][hid] ~ N(0, 1)."""
    return torch.from_numpy(normal_f32((w.B * w.n_q, w.hid), 1.0, seed, KIND_X))


def bias_vec(w: Workload, seed: int) -> torch.Tensor:
    """Optional projection bias, float32 [hid_out] ~ N(0, 1/hid)."""
    return torch.from_numpy(normal_f32((w.hid,), 1.0 / math.sqrt(w.hid), seed, KIND_BIAS))
