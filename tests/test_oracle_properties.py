"""Property-based checks of the oracle on random small shapes (hypothesis):
the same facts as the fixed pins in test_oracle_pins.py, drawn over many
shapes, sizes, scales and positions instead of a few hand-picked ones.

- attention equals the literal loops of tests/_brute.py, for any split of
  the keys into 1 to 3 segments (empty ones included) and any scale;
- attention does not change when the key/value rows are permuted jointly,
  and returns the mean of V when every key is the same vector;
- RoPE equals the per-token loops of tests/_brute.py, keeps each channel
  pair's norm, and leaves every q.k score unchanged when q's and k's times
  move by the same offset (the rotation is relative);
- the shifted time grid is positive and sums to one; a shift of 1 is the
  uniform grid.
"""
import math

import numpy as np
import pytest

import oracle as O
from tests import _brute as brute

try:
    from hypothesis import given, settings
    from hypothesis import strategies as st
except ImportError:  # an image without hypothesis: the module defines no tests
    given = None

SETTINGS = dict(max_examples=60, deadline=None, derandomize=True)  # the same examples every run


if given is not None:
    def _normal(rng, *shape):
        return rng.standard_normal(shape)


    @st.composite
    def attention_cases(draw):
        B = draw(st.integers(1, 2))
        H = draw(st.integers(1, 3))
        D = draw(st.sampled_from([2, 4, 6, 8]))
        n_q = draw(st.integers(1, 5))
        lens = draw(st.lists(st.integers(0, 4), min_size=1, max_size=3).filter(lambda v: sum(v) > 0))
        scale = draw(st.one_of(st.none(), st.floats(0.05, 3.0)))
        seed = draw(st.integers(0, 2**31 - 1))
        return B, H, D, n_q, lens, scale, seed


    @settings(**SETTINGS)
    @given(attention_cases())
    def test_attention_equals_loops(case):
        B, H, D, n_q, lens, scale, seed = case
        rng = np.random.default_rng(seed)
        q = _normal(rng, B, n_q, H, D)
        segs = [(_normal(rng, B, n, H, D), _normal(rng, B, n, H, D)) for n in lens]
        got = O.attention(q, segs, scale)
        sc = scale if scale is not None else 1.0 / math.sqrt(D)
        for b in range(B):
            keys = [row for k, _ in segs for row in k[b]]
            values = [row for _, v in segs for row in v[b]]
            want = np.array(brute.attend(q[b], keys, values, sc))
            np.testing.assert_allclose(got[b], want, rtol=0, atol=1e-12)


    @settings(**SETTINGS)
    @given(attention_cases())
    def test_attention_permutation_and_identical_keys(case):
        B, H, D, n_q, lens, scale, seed = case
        rng = np.random.default_rng(seed)
        q = _normal(rng, B, n_q, H, D)
        n = sum(lens)
        k = _normal(rng, B, n, H, D)
        v = _normal(rng, B, n, H, D)
        base = O.attention(q, [(k, v)], scale)
        perm = rng.permutation(n)
        # permuted rows, re-split into the drawn segment lengths
        kp, vp = k[:, perm], v[:, perm]
        cuts = np.cumsum([0] + lens)
        segs = [(kp[:, cuts[i]:cuts[i + 1]], vp[:, cuts[i]:cuts[i + 1]]) for i in range(len(lens))]
        np.testing.assert_allclose(O.attention(q, segs, scale), base, rtol=0, atol=1e-12)
        # every key the same vector: uniform weights, O = mean of V
        same = np.broadcast_to(k[:, :1], k.shape).copy()
        mean_v = np.broadcast_to(v.mean(axis=1, keepdims=True), (B, n_q, H, D))
        np.testing.assert_allclose(O.attention(q, [(same, v)], scale), mean_v, rtol=0, atol=1e-12)


    @st.composite
    def rope_cases(draw):
        B = draw(st.integers(1, 2))
        H = draw(st.integers(1, 2))
        D = draw(st.sampled_from([6, 8, 12, 16, 64]))
        gt, gh, gw = draw(st.integers(1, 3)), draw(st.integers(1, 3)), draw(st.integers(1, 4))
        t0 = draw(st.integers(-6, 6))
        base = draw(st.sampled_from([100.0, 10000.0, 1e6]))
        seed = draw(st.integers(0, 2**31 - 1))
        return B, H, D, gt, gh, gw, t0, base, seed


    @settings(**SETTINGS)
    @given(rope_cases())
    def test_rope_equals_loops_and_keeps_norms(case):
        B, H, D, gt, gh, gw, t0, base, seed = case
        rng = np.random.default_rng(seed)
        x = _normal(rng, B, gt * gh * gw, H, D)
        got = O.rope3d(x, gt, gh, gw, t0, base)
        want = np.array(brute.rope_block(x, gt, gh, gw, t0, base))
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
        # every channel pair keeps its length
        pr_in = np.hypot(x[..., 0::2], x[..., 1::2])
        pr_out = np.hypot(got[..., 0::2], got[..., 1::2])
        np.testing.assert_allclose(pr_out, pr_in, rtol=1e-12, atol=1e-12)


    @settings(**SETTINGS)
    @given(rope_cases(), st.integers(-20, 20))
    def test_rope_scores_depend_on_time_differences_only(case, shift):
        B, H, D, gt, gh, gw, t0, base, seed = case
        rng = np.random.default_rng(seed)
        n = gt * gh * gw
        q = _normal(rng, B, n, H, D)
        k = _normal(rng, B, n, H, D)
        s0 = np.einsum("bnhd,bmhd->bhnm", O.rope3d(q, gt, gh, gw, t0, base), O.rope3d(k, gt, gh, gw, t0, base))
        s1 = np.einsum("bnhd,bmhd->bhnm", O.rope3d(q, gt, gh, gw, t0 + shift, base),
                       O.rope3d(k, gt, gh, gw, t0 + shift, base))
        np.testing.assert_allclose(s1, s0, rtol=0, atol=1e-9 * max(1.0, np.abs(s0).max()))


    @settings(**SETTINGS)
    @given(st.integers(1, 64), st.floats(0.1, 10.0))
    def test_time_grid_positive_and_sums_to_one(steps, shift):
        dt = O.time_grid(steps, shift)
        assert dt.shape == (steps,)
        assert np.all(dt > 0)
        assert abs(dt.sum() - 1.0) < 1e-12
        np.testing.assert_allclose(O.time_grid(steps, 1.0), np.full(steps, 1.0 / steps), rtol=0, atol=1e-15)
