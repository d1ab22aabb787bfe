"""Pins of the oracle's compressor front end (CPU only): the exp it uses, the softmax-gated
overlap pooling, RMSNorm and the composed store, each against something other than itself.

vllm PR 60834 "Changes / K write": the DeepSeek-V4 indexer K is pooled by its compressor
(softmax-gated overlap pooling), RMSNorm'd, RoPE'd, quantised and stored, one entry per
compress-ratio boundary token. The window, gate softmax and norm formulas are readings of
that description (R13-R16 at the oracle function); the pins fix the oracle to them.
"""
import math

import numpy as np
import pytest

import oracle as O
from sparse_attention_indexer_mqa_gb300 import workloads as W

F32 = np.float32


def test_exp_neg_against_math_exp():
    """Within 1 ulp of the exact exp over [-87, 0] (dense grid plus the ends)."""
    # the method measures <= 0.86 ulp here; one Taylor term fewer reaches over 2 ulp
    grid = np.concatenate([np.linspace(-86.99, 0, 200_001, dtype=np.float64),
                           -np.logspace(-8, 0, 2000), [0.0, -1e-30, -86.999]]).astype(F32)
    got = np.array([O.exp_neg(float(a)) for a in grid[::7]], dtype=np.float64)
    ref = np.exp(grid[::7].astype(np.float64))
    ulp = np.spacing(ref.astype(F32)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1.0 * ulp), np.max(np.abs(got - ref) / ulp)
    assert O.exp_neg(0.0) == 1.0
    assert O.exp_neg(-87.0) == 0.0 and O.exp_neg(-88.0) == 0.0 and O.exp_neg(-1e6) == 0.0


def _rows(vals):
    return W.bf16_bits(np.asarray(vals, F32))


def test_pool_equal_gates_is_the_window_mean():
    rng = np.random.default_rng(70)
    x = rng.standard_normal((8, 128)).astype(F32)
    k = _rows(x)
    g = _rows(np.zeros((8, 128)))
    got = O.compress_pool128(k, g, 0, 7)
    np.testing.assert_allclose(got, W.bf16_to_f32(k).astype(np.float64).mean(0), rtol=0, atol=2e-6)
    got4 = O.compress_pool128(k, g, 4, 7)
    np.testing.assert_allclose(got4, W.bf16_to_f32(k[4:]).astype(np.float64).mean(0), rtol=0, atol=2e-6)


def test_pool_dominant_gate_selects_its_row():
    rng = np.random.default_rng(71)
    k = _rows(rng.standard_normal((8, 128)))
    gv = np.zeros((8, 128), F32)
    gv[5] = 60.0  # e^-60 of the others underflows against it
    got = O.compress_pool128(k, _rows(gv), 0, 7)
    np.testing.assert_array_equal(got, W.bf16_to_f32(k[5]))


def test_pool_softmax_weights_against_fp64():
    """Random gates: the pooled row matches an fp64 softmax-weighted sum (per dimension)."""
    rng = np.random.default_rng(72)
    for _ in range(20):
        n = int(rng.integers(1, 17))
        k = _rows(rng.standard_normal((n, 128)) * 3)
        g = _rows(rng.standard_normal((n, 128)) * 2)
        xf = W.bf16_to_f32(k).astype(np.float64)
        gf = W.bf16_to_f32(g).astype(np.float64)
        wts = np.exp(gf - gf.max(0))
        wts /= wts.sum(0)
        ref = (wts * xf).sum(0)
        got = O.compress_pool128(k, g, 0, n - 1)
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-5 * np.abs(xf).max())


def test_rmsnorm_closed_form_and_fp64():
    for c in (0.5, 3.0, 100.0):
        y = O.rmsnorm128(np.array([c, -c] * 64, F32))
        np.testing.assert_allclose(y[0::2], c / math.sqrt(c * c + 1e-6), rtol=3e-7)
    rng = np.random.default_rng(73)
    gam = rng.standard_normal(128).astype(F32)
    for _ in range(50):
        x = (rng.standard_normal(128) * rng.uniform(0.1, 30) + rng.uniform(-3, 3)).astype(F32)
        xd = x.astype(np.float64)
        ref = xd / np.sqrt((xd * xd).mean() + 1e-6) * gam
        np.testing.assert_allclose(O.rmsnorm128(x, gam), ref, rtol=2e-6, atol=2e-6 * np.abs(ref).max())
        # it is not a LayerNorm (the mean is kept)
        assert not np.allclose(O.rmsnorm128(x, gam), O.layernorm128(x, gam, np.zeros(128)), atol=1e-3)


def _compress_case(seed, n_raw, ratio, dtype, rope, gamma=None):
    rng = np.random.default_rng(seed)
    k = _rows(rng.standard_normal((n_raw, 128)) * rng.uniform(0.5, 3) + rng.uniform(-4, 4))
    g = _rows(rng.standard_normal((n_raw, 128)) * 1.5)
    n_e = n_raw // ratio
    boundary = ratio * np.arange(n_e, dtype=np.int64) + ratio - 1
    first = np.zeros(n_e, np.int64)
    P = 64
    stride = O.page_bytes(dtype, P)
    pages = (n_e + P - 1) // P + 1
    slots = rng.permutation(pages * P)[:n_e].astype(np.int64)
    pos = boundary.astype(np.int32)
    cs = W.rope_table(n_raw)
    pool = np.zeros(pages * stride, np.uint8)
    assert O.compress_k_store(pool, k, g, boundary, first, ratio, slots, pos, cs, rope, 2, dtype,
                              pages, P, stride, gamma=gamma) == 0
    return k, g, boundary, first, slots, pos, pool, P, stride


def test_compress_windows_are_the_readings():
    """Index-coded rows with equal gates: the pooled value of entry j is the mean of its
    window's row indices, [max(0, r*j - r), r*j + r - 1]."""
    for ratio in (2, 4, 8):
        n = 9 * ratio
        x = np.repeat(np.arange(n, dtype=F32)[:, None], 128, 1)
        k, g = _rows(x), _rows(np.zeros((n, 128)))
        for j in range(9):
            hi = ratio * j + ratio - 1
            lo = max(0, hi - 2 * ratio + 1)
            got = O.compress_pool128(k, g, lo, hi)
            assert np.allclose(got, (lo + hi) / 2, atol=1e-5), (ratio, j)


@pytest.mark.parametrize("dtype", [O.MXFP4, O.FP8])
@pytest.mark.parametrize("rope", [O.ROPE_NEOX, O.ROPE_INTERLEAVED])
def test_compress_store_composition(dtype, rope):
    """Each stored entry, dequantised, lies within half a quantisation step of an fp64
    softmax pool -> RMSNorm (gamma) -> RoPE at the boundary position; the plausible slips
    (LayerNorm, a window shifted by one token, RoPE before the norm, which a non-uniform
    gamma makes visible) fall outside that bound for most entries."""
    from test_oracle_pins import _deq_stored_row, _np64_rope, _within_quant_bound
    ratio = 4
    gam = np.random.default_rng(5).uniform(0.3, 3.0, 128).astype(F32)
    k, g, boundary, first, slots, pos, pool, P, stride = _compress_case(80 + dtype + 3 * rope, 256, ratio,
                                                                        dtype, rope, gamma=gam)
    kf, gf = W.bf16_to_f32(k).astype(np.float64), W.bf16_to_f32(g).astype(np.float64)

    def pool64(lo, hi):
        w = np.exp(gf[lo:hi + 1] - gf[lo:hi + 1].max(0))
        w /= w.sum(0)
        return (w * kf[lo:hi + 1]).sum(0)

    def rms64(p):
        return p / np.sqrt((p * p).mean() + 1e-6) * gam

    def ln64(p):
        return (p - p.mean()) / np.sqrt(((p - p.mean()) ** 2).mean() + 1e-6) * gam

    slips = {"layernorm": 0, "shifted window": 0, "rope before norm": 0}
    n_e = boundary.size
    for e in range(n_e):
        hi = int(boundary[e])
        lo = max(0, hi - 2 * ratio + 1)
        deq, es = _deq_stored_row(pool, dtype, P, stride, int(slots[e]))
        ref = _np64_rope(rms64(pool64(lo, hi)), float(pos[e]), rope)
        assert _within_quant_bound(deq, ref, dtype, es), e
        slips["layernorm"] += not _within_quant_bound(deq, _np64_rope(ln64(pool64(lo, hi)), float(pos[e]), rope),
                                                      dtype, es)
        if hi + 1 < k.shape[0]:
            slips["shifted window"] += not _within_quant_bound(
                deq, _np64_rope(rms64(pool64(lo + 1, hi + 1)), float(pos[e]), rope), dtype, es)
        slips["rope before norm"] += not _within_quant_bound(
            deq, rms64(_np64_rope(pool64(lo, hi), float(pos[e]), rope)), dtype, es)
    assert all(v >= n_e // 2 for v in slips.values()), slips


def test_compress_shifted_window_changes_the_bytes():
    """A window shifted by one raw token changes most stored bytes (the pages' own check of
    a wrong pooling window)."""
    k, g, boundary, first, slots, pos, pool, P, stride = _compress_case(90, 512, 4, O.MXFP4, O.ROPE_NEOX)
    pool2 = np.zeros_like(pool)
    O.compress_k_store(pool2, k, g, boundary + 1, first, 4, slots, pos, W.rope_table(513), O.ROPE_NEOX, 2,
                       O.MXFP4, pool.size // stride, P, stride)
    used = np.zeros(pool.size, bool)
    for sl in slots:
        pg, r = divmod(int(sl), P)
        for j in range(64):
            used[pg * stride + O.code_offset(O.MXFP4, P, r, j)] = True
    frac = np.mean(pool[used] != pool2[used])
    assert frac > 0.5, frac


def test_compress_window_clips_at_the_sequence_start():
    """Two sequences share the raw buffer: the entries of the second (first = n1) pool no
    row of the first. Index-coded rows, equal gates, no norm/RoPE, FP8 (a constant row
    stores exactly): entry j of the second sequence holds the mean of its clipped window."""
    from test_oracle_pins import _deq_stored_row
    ratio, n1, n2 = 4, 10, 16
    n = n1 + n2
    x = np.repeat(np.arange(n, dtype=F32)[:, None], 128, 1)
    k, g = _rows(x), _rows(np.zeros((n, 128)))
    boundary = n1 + ratio * np.arange(n2 // ratio, dtype=np.int64) + ratio - 1
    first = np.full(boundary.shape, n1, np.int64)
    P, dt = 64, O.FP8
    stride = O.page_bytes(dt, P)
    slots = np.arange(boundary.size, dtype=np.int64)
    pool = np.zeros(stride, np.uint8)
    assert O.compress_k_store(pool, k, g, boundary, first, ratio, slots, None, None, O.ROPE_NONE, 0,
                              dt, 1, P, stride) == 0
    for j, hi in enumerate(boundary):
        lo = max(n1, hi - 2 * ratio + 1)
        v, _ = _deq_stored_row(pool, dt, P, stride, j)
        np.testing.assert_allclose(v, (lo + hi) / 2, rtol=1e-6)


def test_compress_rejects_windows_outside_the_rows():
    """first > boundary, first < 0 or boundary >= n_raw: the entry is rejected and its slot
    left untouched; a negative slot is skipped without counting."""
    rng = np.random.default_rng(74)
    n, P, dt = 12, 64, O.MXFP4
    k, g = _rows(rng.standard_normal((n, 128))), _rows(rng.standard_normal((n, 128)))
    stride = O.page_bytes(dt, P)
    boundary = np.array([5, 3, 12, 4, 7], np.int64)
    first = np.array([6, -1, 0, 0, 0], np.int64)
    slots = np.array([0, 1, 2, 3, -1], np.int64)
    pool = np.full(stride, 0xA5, np.uint8)
    assert O.compress_k_store(pool, k, g, boundary, first, 4, slots, None, None, O.ROPE_NONE, 2, dt,
                              1, P, stride) == 3
    untouched = np.full(stride, 0xA5, np.uint8)
    for s in (0, 1, 2):
        for j in range(64):
            assert pool[O.code_offset(dt, P, s, j)] == 0xA5
    changed = np.nonzero(pool != untouched)[0]
    assert changed.size > 0 and all(
        any(off == O.code_offset(dt, P, 3, j) for j in range(64)) or
        any(off == O.scale_offset(dt, P, 3, b) for b in range(4)) for off in changed)
