"""Pins of the CPU oracle to facts fixed outside it (CPU only).

Each test checks the oracle against something other than itself: hand-worked encodings
(tests/golden/encodings.json), a library routine that implements the same rounding
(torch's float8_e4m3fn cast, numpy's round-half-even, math.frexp, numpy matmul), closed
forms, invariants, or brute force written a different way. A plausible slip in the oracle
(wrong tie rule, dropped term, swapped operand, wrong pairing, off-by-one page) fails at
least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
from sparse_attention_indexer_mqa_gb300 import workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "encodings.json")))


# --------------------------------------------------------------------------------------
# element encoders
# --------------------------------------------------------------------------------------

def test_e2m1_hand_worked():
    for v, code in GOLD["e2m1_relative_to_scale"]:
        assert O.e2m1_encode(v) == code, (v, code)


def _e2m1_by_rounding(v):
    """Round-half-even onto the e2m1 grid by scaling each binade to integers (numpy's
    np.round is round-half-even): [0,2) step 0.5, [2,4) step 1, [4,inf) step 2, cap 6."""
    a = np.abs(v).astype(np.float64)
    q = np.where(a < 2, np.round(a * 2) / 2, np.where(a < 4, np.round(a), np.round(a / 2) * 2))
    q = np.minimum(q, 6.0)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    code = np.searchsorted(grid, q)
    return (code | (np.signbit(v) * 8)).astype(np.uint8)


def test_e2m1_sweep_against_half_even_rounding():
    # every bf16 pattern whose magnitude is below 8 (the encoder's input range), plus
    # random fp32 values and exact midpoints
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = W.bf16_to_f32(b)
    v = v[np.isfinite(v) & (np.abs(v) < 8)]
    rng = np.random.default_rng(1)
    r = (rng.random(200_000, dtype=np.float32) * 16 - 8).astype(np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    allv = np.concatenate([v, r, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 9)])
    np.testing.assert_array_equal(O.e2m1_encode_n(allv), _e2m1_by_rounding(allv))


def test_e2m1_decode_matches_bit_fields():
    # value = (-1)^s * (e ? (1 + m/2) * 2^(e-1) : m/2), the FP4 E2M1 bit-field definition
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        val = (1 + m / 2) * 2.0 ** (e - 1) if e else m / 2
        assert O.e2m1_decode(code) == (-val if s else val)


def test_e4m3_hand_worked():
    for v, code in GOLD["e4m3"]:
        assert O.e4m3_encode(v) == code, (v, code)


def test_e4m3_sweep_against_torch_cast():
    torch = pytest.importorskip("torch")
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = W.bf16_to_f32(b)
    v = v[np.isfinite(v) & (np.abs(v) <= 448)]
    rng = np.random.default_rng(2)
    r = np.concatenate([(rng.standard_normal(300_000) * 100).astype(np.float32),
                        (rng.random(100_000) * 0.03).astype(np.float32)])
    r = r[np.abs(r) <= 448]
    allv = np.concatenate([v, r])
    ref = torch.from_numpy(allv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_encode_n(allv), ref)
    # saturation above 448 (torch's cast does not saturate, so check it by hand)
    big = np.array([448.1, 463.9, 464.0, 1e6, -1e6], np.float32)
    assert list(O.e4m3_encode_n(big)) == [126, 126, 126, 126, 254]


def test_e4m3_decode_matches_torch():
    torch = pytest.importorskip("torch")
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = np.array([O.e4m3_decode(int(c)) for c in codes])
    np.testing.assert_array_equal(got, ref)


def test_mx_shared_exponent():
    for amax, e in GOLD["mx_shared_exponent"]:
        assert O.mx_shared_exponent(amax) == e
    rng = np.random.default_rng(3)
    vals = np.concatenate([np.exp(rng.uniform(-100, 80, 5000)).astype(np.float32),
                           np.array([1e-40, 1e-45, 3e-39, 1.17549435e-38], np.float32)])
    for a in vals:
        a = float(a)
        m, e = math.frexp(a)  # a = m * 2^e, m in [0.5, 1) -> floor(log2 a) = e - 1
        assert O.mx_shared_exponent(a) == max(-127, min(127, e - 1 - 2)), a


def test_mx_block_examples():
    for key in ("mx_block_A", "mx_block_B"):
        ex = GOLD[key]
        x = np.zeros(128, np.float32)
        x[:len(ex["x"])] = ex["x"]
        codes, sc = O.mxfp4_quant128(x)
        assert sc[0] == ex["scale_byte"]
        got = [(codes[i // 2] >> (4 * (i % 2))) & 15 for i in range(len(ex["x"]))]
        assert got == ex["codes"], key
        # the zero blocks: scale byte 0, codes 0
        assert list(sc[1:]) == [0, 0, 0]
        assert not codes[16:].any()


def _dequant_mx(codes, sc):
    vals = np.array([O.e2m1_decode(c) for c in range(16)])
    lo, hi = vals[codes & 15], vals[codes >> 4]
    e = np.empty(128)
    e[0::2], e[1::2] = lo, hi
    return e * np.repeat(2.0 ** (sc.astype(np.int64) - 127), 32)


def test_mxfp4_error_bound_and_equivariance():
    rng = np.random.default_rng(4)
    for _ in range(300):
        x = (rng.standard_normal(128) * np.exp(rng.uniform(-8, 8))).astype(np.float32)
        codes, sc = O.mxfp4_quant128(x)
        deq = _dequant_mx(codes, sc)
        # relative to the block scale 2^E: error <= half the local grid step (0.25 below 2,
        # 0.5 in [2,4), 1 in [4,6]); values above 6 saturate to exactly +-6
        E = sc.astype(np.int64) - 127
        scale = np.repeat(2.0 ** E, 32)
        v = x / scale
        a = np.abs(v)
        half = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))
        ok_in = np.abs(deq / scale - v) <= half
        sat = a > 6
        assert np.all(ok_in[~sat])
        assert np.all(deq[sat] / scale[sat] == np.sign(v[sat]) * 6)
        assert np.all(a < 8) and np.all(a.reshape(4, 32).max(axis=1) >= 4)
        # quantise(2^n x): same codes, scale bytes + n (away from the clamps)
        n = int(rng.integers(-20, 20))
        c2, s2 = O.mxfp4_quant128((x * np.float32(2.0 ** n)).astype(np.float32))
        assert np.array_equal(c2, codes) and np.array_equal(s2.astype(int), sc.astype(int) + n)


def test_fp8_quant_row():
    rng = np.random.default_rng(5)
    for _ in range(100):
        x = (rng.standard_normal(128) * np.exp(rng.uniform(-5, 5))).astype(np.float32)
        codes, s = O.fp8_quant128(x)
        amax = np.abs(x).max()
        assert s == np.float32(np.float32(amax) / np.float32(448.0))
        deq = np.array([O.e4m3_decode(int(c)) for c in codes]) * s
        # e4m3 has 3 mantissa bits: relative error <= 2^-4 for normal values
        big = np.abs(x) > 2.0 ** -6 * s
        assert np.all(np.abs(deq - x)[big] <= np.abs(x)[big] * 2.0 ** -4 * 1.0001)
        assert O.e4m3_encode(amax / s) == 126  # the largest element maps to 448
    codes, s = O.fp8_quant128(np.zeros(128, np.float32))
    assert s == np.float32(np.float32(1e-10) / np.float32(448.0)) and not codes.any()


# --------------------------------------------------------------------------------------
# LayerNorm / RoPE
# --------------------------------------------------------------------------------------

def test_layernorm_closed_form():
    # +c/-c alternating row: mean 0, biased variance c^2 -> y = +-c / sqrt(c^2 + eps)
    for c in [0.5, 1.0, 3.0, 100.0, 1e-3]:
        x = np.array([c, -c] * 64, np.float32)
        y = O.layernorm128(x)
        expect = c / math.sqrt(c * c + 1e-6)
        np.testing.assert_allclose(y[0::2], expect, rtol=3e-7)
        np.testing.assert_allclose(y[1::2], -expect, rtol=3e-7)


def test_layernorm_against_fp64():
    rng = np.random.default_rng(6)
    g = rng.standard_normal(128).astype(np.float32)
    b = rng.standard_normal(128).astype(np.float32)
    for _ in range(200):
        x = (rng.standard_normal(128) * rng.uniform(0.01, 50) + rng.uniform(-5, 5)).astype(np.float32)
        xd = x.astype(np.float64)
        mu = xd.mean()
        var = ((xd - mu) ** 2).mean()  # biased
        ref = (xd - mu) / np.sqrt(var + 1e-6) * g + b
        y = O.layernorm128(x, g, b, 1e-6)
        np.testing.assert_allclose(y, ref, rtol=2e-5, atol=2e-5 * np.abs(ref).max())


def _table_row(pos):
    return W.rope_table(pos + 1)[pos]


def test_rope_pairing_and_identity():
    cs = _table_row(7)
    for i in range(32):
        # NeoX: dims (i, i+32); (1, 0) rotates to (cos, sin) of frequency i
        x = np.zeros(128, np.float32); x[i] = 1
        y = O.rope128(x, cs, O.ROPE_NEOX)
        assert y[i] == cs[i] and y[i + 32] == cs[32 + i]
        # interleaved: dims (2i, 2i+1)
        x = np.zeros(128, np.float32); x[2 * i] = 1
        y = O.rope128(x, cs, O.ROPE_INTERLEAVED)
        assert y[2 * i] == cs[i] and y[2 * i + 1] == cs[32 + i]
        # (0, 1) rotates to (-sin, cos)
        x = np.zeros(128, np.float32); x[i + 32] = 1
        y = O.rope128(x, cs, O.ROPE_NEOX)
        assert y[i] == -cs[32 + i] and y[i + 32] == cs[i]
    rng = np.random.default_rng(7)
    x = rng.standard_normal(128).astype(np.float32)
    assert np.array_equal(O.rope128(x, _table_row(0), O.ROPE_NEOX), x)  # position 0
    assert np.array_equal(O.rope128(x, cs, O.ROPE_NONE), x)
    y = O.rope128(x, cs, O.ROPE_NEOX)
    assert np.array_equal(y[64:], x[64:])  # dims 64..127 pass through


def test_rope_inverse_and_norm():
    rng = np.random.default_rng(8)
    for mode in (O.ROPE_NEOX, O.ROPE_INTERLEAVED):
        for pos in [1, 17, 1000, 9000]:
            cs = _table_row(pos)
            inv = cs.copy(); inv[32:] = -inv[32:]  # cos(-a) = cos a, sin(-a) = -sin a
            x = rng.standard_normal(128).astype(np.float32)
            y = O.rope128(x, cs, mode)
            z = O.rope128(y, inv, mode)
            np.testing.assert_allclose(z, x, rtol=0, atol=4e-7 * np.abs(x).max() * 4)
            if mode == O.ROPE_NEOX:
                n0 = x[:32].astype(np.float64) ** 2 + x[32:64].astype(np.float64) ** 2
                n1 = y[:32].astype(np.float64) ** 2 + y[32:64].astype(np.float64) ** 2
                np.testing.assert_allclose(n1, n0, rtol=2e-6)


# --------------------------------------------------------------------------------------
# layout
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,P", [(O.MXFP4, 64), (O.MXFP4, 128), (O.FP8, 64), (O.FP8, 128)])
def test_layout_is_a_bijection(dtype, P):
    per_tok = 68 if dtype == O.MXFP4 else 132
    assert O.page_bytes(dtype, P) == per_tok * P
    offs = []
    ncode = 64 if dtype == O.MXFP4 else 128
    for s in range(P):
        offs += [O.code_offset(dtype, P, s, j) for j in range(ncode)]
        if dtype == O.MXFP4:
            offs += [O.scale_offset(dtype, P, s, b) for b in range(4)]
        else:
            offs += [O.scale_offset(dtype, P, s, 0) + i for i in range(4)]
    assert sorted(offs) == list(range(per_tok * P))


@pytest.mark.parametrize("dtype", [O.MXFP4, O.FP8])
def test_k_store_write_footprint(dtype):
    """One stored row changes exactly its 68/132 bytes, whatever the canary."""
    P = 64
    stride = O.page_bytes(dtype, P)
    rng = np.random.default_rng(9)
    k = W.bf16_bits(rng.standard_normal((1, 128)).astype(np.float32))
    for canary in (0x00, 0xA5):
        pool = np.full(stride * 4, canary, np.uint8)
        slot = 2 * P + 37
        O.k_store(pool, k, np.array([slot]), np.array([5]), W.rope_table(8), O.ROPE_NEOX, 1,
                  dtype, 4, P, stride)
        changed = np.nonzero(pool != canary)[0]
        per_tok = 68 if dtype == O.MXFP4 else 132
        assert len(changed) <= per_tok
        assert changed.min() >= 2 * stride and changed.max() < 3 * stride
        ncode = 64 if dtype == O.MXFP4 else 128
        allowed = {2 * stride + O.code_offset(dtype, P, 37, j) for j in range(ncode)}
        if dtype == O.MXFP4:
            allowed |= {2 * stride + O.scale_offset(dtype, P, 37, b) for b in range(4)}
        else:
            allowed |= {2 * stride + O.scale_offset(dtype, P, 37) + i for i in range(4)}
        assert set(changed.tolist()) <= allowed
    # a negative slot writes nothing
    pool = np.zeros(stride * 4, np.uint8)
    O.k_store(pool, k, np.array([-1]), np.array([0]), W.rope_table(8), O.ROPE_NEOX, 1, dtype, 4,
              P, stride)
    assert not pool.any()


# --------------------------------------------------------------------------------------
# scorer and top-k
# --------------------------------------------------------------------------------------

def _deq_pool_rows(wl, pool, b, n):
    """Dequantised keys 0..n-1 of sequence b, read with the oracle's layout functions and
    numpy (a second reader, written apart from the oracle's scorer)."""
    P, dt = wl.page_size, wl.dtype
    e2 = np.array([O.e2m1_decode(c) for c in range(16)])
    e4 = np.array([O.e4m3_decode(c) if (c & 0x7F) != 0x7F else np.nan for c in range(256)])
    base = wl.base_offset_pages * wl.page_stride
    rows = np.zeros((n, 128))
    for s in range(n):
        pg = int(wl.page_table[b, s // P])
        off = base + pg * wl.page_stride
        r = s % P
        if dt == O.MXFP4:
            cb = np.array([pool[off + O.code_offset(dt, P, r, j)] for j in range(64)])
            sc = np.array([pool[off + O.scale_offset(dt, P, r, bb)] for bb in range(4)])
            vals = np.empty(128)
            vals[0::2], vals[1::2] = e2[cb & 15], e2[cb >> 4]
            rows[s] = vals * np.repeat(2.0 ** (sc.astype(np.int64) - 127), 32)
        else:
            cb = np.array([pool[off + O.code_offset(dt, P, r, j)] for j in range(128)])
            ks = np.frombuffer(bytes(pool[off + O.scale_offset(dt, P, r):][:4]), np.float32)[0]
            rows[s] = e4[cb] * ks
    return rows


def _prepare_tiny(wl):
    pool = np.zeros(wl.pool_nbytes(), np.uint8)
    view = pool[wl.base_offset_pages * wl.page_stride:]
    O.k_store(view, wl.k, wl.slot_mapping, wl.k_positions, wl.cos_sin, wl.k_rope, wl.k_norm,
              wl.dtype, wl.pool_pages, wl.page_size, wl.page_stride)
    qc, qs, w = O.q_quant(wl.q, wl.q_positions, wl.cos_sin, wl.q_rope, wl.w_in,
                          wl.softmax_scale, wl.head_scale, wl.dtype)
    return pool, view, qc, qs, w


def _score(wl, view, qc, qs, w, page_table=None):
    return O.mqa_logits(qc, qs, w, wl.dtype, view, wl.pool_pages, wl.page_size, wl.page_stride,
                        wl.page_table if page_table is None else page_table, wl.seq_lens_k,
                        wl.cu_seqlens_q, wl.causal, wl.ld_logits)


def test_scorer_brute_force_tiny():
    wl = W.make("tiny_decode")
    pool, view, qc, qs, w = _prepare_tiny(wl)
    got = _score(wl, view, qc, qs, w)
    e2 = np.array([O.e2m1_decode(c) for c in range(16)])
    for t in range(wl.T):
        b = t
        n = int(wl.seq_lens_k[b])
        K = _deq_pool_rows(wl, pool, b, n)
        Q = np.empty((wl.H, 128))
        Q[:, 0::2], Q[:, 1::2] = e2[qc[t] & 15], e2[qc[t] >> 4]
        Q *= np.repeat(2.0 ** (qs[t].astype(np.int64) - 127), 32, axis=1)
        ref = np.maximum(Q @ K.T, 0).T @ w[t].astype(np.float64)
        np.testing.assert_allclose(got[t, :n], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
        assert np.isnan(got[t, n:]).all()  # entries past visible(t) untouched


def test_scorer_fp8_brute_force_causal():
    wl = W.make("prefill_fp8", B=2, cached=100, new=37, H=8)
    pool, view, qc, qs, w = _prepare_tiny(wl)
    got = _score(wl, view, qc, qs, w)
    vis = wl.visible()
    e4 = np.array([O.e4m3_decode(c) if (c & 0x7F) != 0x7F else np.nan for c in range(256)])
    for b in range(wl.B):
        K = _deq_pool_rows(wl, pool, b, int(wl.seq_lens_k[b]))
        for t in range(int(wl.cu_seqlens_q[b]), int(wl.cu_seqlens_q[b + 1]), 5):
            Q = e4[qc[t]]
            ref = np.maximum(Q @ K[:vis[t]].T, 0).T @ w[t].astype(np.float64)
            # w carries the q scale; K rows are already multiplied by their scale
            np.testing.assert_allclose(got[t, :vis[t]], ref, rtol=1e-12,
                                       atol=1e-12 * np.abs(ref).max())
            assert np.isnan(got[t, vis[t]:]).all()


def test_scorer_closed_form_and_invariants():
    wl = W.make("tiny_decode")
    pool, view, qc, qs, w = _prepare_tiny(wl)
    base = _score(wl, view, qc, qs, w)
    # w -> 2w doubles every logit exactly; |w| gives non-negative logits
    assert np.array_equal(_score(wl, view, qc, qs, 2 * w), 2 * base, equal_nan=True)
    pos = _score(wl, view, qc, qs, np.abs(w))
    assert np.nanmin(pos) >= 0
    # shuffled physical pages with a rewritten page table: identical logits
    rng = np.random.default_rng(10)
    perm = rng.permutation(wl.pool_pages)
    view2 = np.zeros_like(view)
    for p in range(wl.pool_pages):
        view2[perm[p] * wl.page_stride:(perm[p] + 1) * wl.page_stride] = \
            view[p * wl.page_stride:(p + 1) * wl.page_stride]
    pt2 = np.where(wl.page_table >= 0, perm[np.maximum(wl.page_table, 0)], -1).astype(np.int32)
    got = O.mqa_logits(qc, qs, w, wl.dtype, view2, wl.pool_pages, wl.page_size, wl.page_stride,
                       pt2, wl.seq_lens_k, wl.cu_seqlens_q, wl.causal, wl.ld_logits)
    assert np.array_equal(got, base, equal_nan=True)


def test_scorer_constant_rows_closed_form():
    """Constant q = a and k = b rows: every dot is 128*a*b, so logit = sum_h w_h max(128ab, 0)."""
    P, H = 64, 3
    stride = O.page_bytes(O.MXFP4, P)
    pool = np.zeros(stride * 2, np.uint8)
    for kval in (1.5, -2.0):
        k = np.full((5, 128), W.bf16_bits(np.array([kval], np.float32))[0], np.uint16)
        O.k_store(pool, k, np.arange(5) + P, np.zeros(5), None, O.ROPE_NONE, 0, O.MXFP4, 2, P,
                  stride)
        q = np.full((1, H, 128), W.bf16_bits(np.array([3.0], np.float32))[0], np.uint16)
        w = np.array([[0.5, -0.25, 2.0]], np.float32)
        qc, qs, wo = O.q_quant(q, None, None, O.ROPE_NONE, w, 1.0, 1.0, O.MXFP4)
        got = O.mqa_logits(qc, qs, wo, O.MXFP4, pool, 2, P, stride, np.array([[1]], np.int32),
                           np.array([5], np.int32), np.array([0, 1], np.int32), 0, 5)
        expect = sum(float(x) * max(128 * 3.0 * kval, 0) for x in w[0])
        assert np.all(got[0] == expect)


def test_mutations_change_the_scores():
    """A page table shifted by one, one flipped scale byte and swapped nibbles must each
    change the oracle's logits (the oracle really reads what it should)."""
    wl = W.make("tiny_decode")
    pool, view, qc, qs, w = _prepare_tiny(wl)
    base = _score(wl, view, qc, qs, w)
    pt = np.roll(wl.page_table, 1, axis=1)
    assert not np.allclose(_score(wl, view, qc, qs, w, pt), base, equal_nan=True)
    v2 = view.copy()
    pg = int(wl.page_table[0, 0])
    v2[pg * wl.page_stride + O.scale_offset(O.MXFP4, wl.page_size, 3, 1)] += 1
    assert not np.allclose(_score(wl, v2, qc, qs, w), base, equal_nan=True)
    qc2 = ((qc >> 4) | (qc << 4)).astype(np.uint8)
    assert not np.allclose(_score(wl, view, qc2, qs, w), base, equal_nan=True)


def test_visible_rule():
    sl = np.array([10, 7], np.int32)
    cu = np.array([0, 3, 7], np.int32)
    assert [O.visible(t, sl, cu, 1) for t in range(7)] == [8, 9, 10, 4, 5, 6, 7]
    assert [O.visible(t, sl, cu, 0) for t in range(7)] == [10] * 3 + [7] * 4


def test_topk_against_argsort():
    rng = np.random.default_rng(11)
    T, L, k = 6, 300, 32
    lg = rng.standard_normal((T, L))
    sl = np.array([L], np.int32)
    cu = np.array([0, T], np.int32)
    got = O.topk(lg, sl, cu, 1, k)
    for t in range(T):
        vis = L - T + t + 1
        ref = np.argsort(-lg[t, :vis], kind="stable")[:k]
        assert set(got[t]) == set(ref.tolist())
    # fewer visible keys than k: all of them, then -1 padding
    sl2 = np.array([20], np.int32)
    got = O.topk(lg[:1], sl2, np.array([0, 1], np.int32), 0, k)
    assert sorted(got[0][:20].tolist()) == list(range(20)) and (got[0][20:] == -1).all()


# --------------------------------------------------------------------------------------
# composition pins: the weight fold, the RoPE position of every head, and the order
# LayerNorm -> RoPE -> quantisation of the K store, each against an independent numpy
# restatement (fp32 numpy arithmetic is one correctly rounded operation per ufunc, so the
# restatement reproduces the stated rounding order without sharing any code with oracle.c)
# --------------------------------------------------------------------------------------

F32 = np.float32


def _np_rope(x, cs_row, mode):
    """RoPE of one fp32 row (dims 0..63; NeoX pairs (i, i+32), interleaved (2i, 2i+1)):
    a' = a*c - b*s, b' = b*c + a*s, every product and sum rounded to fp32."""
    y = x.astype(F32).copy()
    c, s = cs_row[:32].astype(F32), cs_row[32:].astype(F32)
    ia = np.arange(32) if mode == O.ROPE_NEOX else 2 * np.arange(32)
    ib = ia + 32 if mode == O.ROPE_NEOX else ia + 1
    a, b = y[ia].copy(), y[ib].copy()
    y[ia] = (a * c) - (b * s)
    y[ib] = (b * c) + (a * s)
    return y


def _np_mx_quant(x):
    """OCP MX quantisation of a 128-value fp32 row: per 32-block E = floor(log2 amax) - 2
    (frexp), clamped to [-127, 127] (amax 0 -> -127), elements x * 2^-E in fp32, then
    round-half-even onto the e2m1 grid with saturation (`_e2m1_by_rounding`). Returns the
    64 packed code bytes and the 4 scale bytes."""
    codes = np.empty(128, np.uint8)
    scales = np.empty(4, np.uint8)
    for b in range(4):
        blk = x[32 * b:32 * b + 32].astype(F32)
        amax = float(np.abs(blk).max())
        if amax == 0.0:
            E = -127
        else:
            _, e = math.frexp(amax)
            E = max(-127, min(127, e - 1 - 2))
        scales[b] = E + 127
        v = blk * F32(2.0 ** -E)
        codes[32 * b:32 * b + 32] = _e2m1_by_rounding(v)
    return (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8), scales


def _fold_case(dtype, seed):
    rng = np.random.default_rng(seed)
    T, H = 7, 4
    q = W.bf16_bits((rng.standard_normal((T, H, 128)) * 2).astype(F32))
    pos = rng.permutation(np.arange(40, 40 + T)).astype(np.int32)   # distinct, not t
    cs = W.rope_table(64)
    w_in = rng.standard_normal((T, H)).astype(F32)
    return q, pos, cs, w_in


@pytest.mark.parametrize("dtype", [O.MXFP4, O.FP8])
def test_q_weight_fold_against_restatement(dtype):
    """w_out = fp32(w_in * fp32(softmax_scale * head_scale)) for MXFP4, and
    fp32(fp32(w_in * c) * q_scale) with q_scale = fp32(max(amax, 1e-10) / 448) of the RoPE'd
    row for FP8 (vllm PR 60834 "Changes / Q quant": fp32 weights with the softmax and head
    scales folded in; vllm PR 53094 "Purpose" step 4: the q scale folded into the weights).
    Scales away from 1 so that a dropped factor, or the q scale left out, is visible."""
    q, pos, cs, w_in = _fold_case(dtype, 40 + dtype)
    ss, hs = 0.08838834764831845, 0.125
    _, qs, w_out = O.q_quant(q, pos, cs, O.ROPE_NEOX, w_in, ss, hs, dtype)
    c = F32(np.float64(F32(ss)) * np.float64(F32(hs)))
    wc = w_in * c
    if dtype == O.MXFP4:
        expect = wc
    else:
        T, H = w_in.shape
        expect = np.empty_like(w_in)
        for t in range(T):
            for h in range(H):
                y = _np_rope(W.bf16_to_f32(q[t, h]), cs[pos[t]], O.ROPE_NEOX)
                scale = F32(max(F32(np.abs(y).max()), F32(1e-10))) / F32(448.0)
                assert qs[t, h].view(np.uint32) == F32(scale).view(np.uint32)
                expect[t, h] = wc[t, h] * F32(scale)
    np.testing.assert_array_equal(w_out.view(np.uint32), expect.astype(F32).view(np.uint32))
    # the pin separates the plausible slips
    assert not np.array_equal(w_out, w_in * F32(hs))        # softmax scale dropped
    assert not np.array_equal(w_out, w_in * F32(ss))        # head scale dropped
    if dtype == O.FP8:
        assert not np.array_equal(w_out, wc)                 # q scale not folded


@pytest.mark.parametrize("mode", [O.ROPE_NEOX, O.ROPE_INTERLEAVED])
def test_q_quant_rope_position_of_every_head(mode):
    """Every head of query t is rotated at positions[t] (vllm PR 53094 "Purpose" step 2:
    RoPE on the leading rope dims of q): the oracle's MXFP4 codes and scales equal an
    independent numpy RoPE + MX quantisation at positions[t], and differ from the same at
    the plausible wrong positions (t itself, or a per-row index t*H + h)."""
    q, pos, cs, w_in = _fold_case(O.MXFP4, 50 + mode)
    T, H = w_in.shape
    qc, qs, _ = O.q_quant(q, pos, cs, mode, w_in, 1.0, 1.0, O.MXFP4)
    wrong_t = wrong_row = 0
    for t in range(T):
        for h in range(H):
            x = W.bf16_to_f32(q[t, h])
            c, s = _np_mx_quant(_np_rope(x, cs[pos[t]], mode))
            np.testing.assert_array_equal(qc[t, h], c)
            np.testing.assert_array_equal(qs[t, h], s)
            c1, _ = _np_mx_quant(_np_rope(x, cs[t], mode))
            c2, _ = _np_mx_quant(_np_rope(x, cs[(t * H + h) % cs.shape[0]], mode))
            wrong_t += not np.array_equal(c1, c)
            wrong_row += not np.array_equal(c2, c)
    assert wrong_t > 0 and wrong_row > 0


def _deq_stored_row(pool, dtype, P, stride, slot):
    """Dequantised 128 values of the token at `slot`, read through the layout functions."""
    page, r = slot // P, slot % P
    off = page * stride
    if dtype == O.MXFP4:
        cb = np.array([pool[off + O.code_offset(dtype, P, r, j)] for j in range(64)])
        sc = np.array([pool[off + O.scale_offset(dtype, P, r, b)] for b in range(4)])
        e2 = np.array([O.e2m1_decode(c) for c in range(16)])
        v = np.empty(128)
        v[0::2], v[1::2] = e2[cb & 15], e2[cb >> 4]
        return v * np.repeat(2.0 ** (sc.astype(np.int64) - 127), 32), sc.astype(np.int64) - 127
    cb = np.array([pool[off + O.code_offset(dtype, P, r, j)] for j in range(128)])
    ks = np.frombuffer(bytes(pool[off + O.scale_offset(dtype, P, r):][:4]), np.float32)[0]
    return np.array([O.e4m3_decode(int(c)) for c in cb]) * float(ks), float(ks)


def _np64_layernorm(x, eps=1e-6):
    xd = x.astype(np.float64)
    mu = xd.mean()
    return (xd - mu) / np.sqrt(((xd - mu) ** 2).mean() + eps)


def _np64_rope(x, pos, mode):
    y = x.copy()
    ang = pos * 10000.0 ** (-np.arange(32) / 32.0)
    c, s = np.cos(ang), np.sin(ang)
    ia = np.arange(32) if mode == O.ROPE_NEOX else 2 * np.arange(32)
    ib = ia + 32 if mode == O.ROPE_NEOX else ia + 1
    a, b = x[ia], x[ib]
    y[ia], y[ib] = a * c - b * s, b * c + a * s
    return y


def _within_quant_bound(deq, ref, dtype, E_or_scale):
    """|dequantised - ref| within half a quantisation step (plus fp32 slack)."""
    if dtype == O.MXFP4:
        scale = np.repeat(2.0 ** E_or_scale, 32)
        v = ref / scale
        a = np.abs(v)
        half = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))
        err = np.abs(deq / scale - v)
        sat = a > 6
        ok = np.where(sat, np.abs(deq / scale) == 6, err <= half + 1e-4 * np.maximum(a, 1))
        return bool(ok.all())
    s = E_or_scale
    err = np.abs(deq - ref)
    bound = np.maximum(np.abs(ref) * 2.0 ** -4, 2.0 ** -10 * s) * 1.0001 + 1e-6 * np.abs(ref)
    return bool((err <= bound).all())


@pytest.mark.parametrize("dtype", [O.MXFP4, O.FP8])
@pytest.mark.parametrize("mode", [O.ROPE_NEOX, O.ROPE_INTERLEAVED])
def test_k_store_norm_then_rope_then_quant(dtype, mode):
    """The K store applies LayerNorm, then RoPE at positions[row], then quantisation
    (vllm PR 53094 "Purpose" steps 1, 2, 5; vllm PR 60834 "Changes / K write": norm ->
    RoPE -> MXFP4 -> store). Each stored row, dequantised, lies within half a quantisation
    step of an fp64 RoPE(LayerNorm(x)) at positions[row]; rows with a large common offset
    make the other orders (RoPE before the norm, no norm) and a wrong position (the row
    index) fall far outside that bound."""
    rng = np.random.default_rng(60 + 2 * dtype + mode)
    P, n = 64, 24
    stride = O.page_bytes(dtype, P)
    x = (rng.standard_normal((n, 128)) * rng.uniform(0.5, 3, (n, 1))
         + rng.uniform(4, 12, (n, 1)) * rng.choice([-1, 1], (n, 1))).astype(F32)
    k = W.bf16_bits(x)
    xf = W.bf16_to_f32(k)
    slots = rng.permutation(2 * P)[:n].astype(np.int64)
    pos = rng.integers(100, 3000, n).astype(np.int32)
    pool = np.zeros(2 * stride, np.uint8)
    assert O.k_store(pool, k, slots, pos, W.rope_table(3000), mode, 1, dtype, 2, P, stride) == 0
    slips = {"rope before norm": 0, "no norm": 0, "position = row": 0}
    for r in range(n):
        deq, es = _deq_stored_row(pool, dtype, P, stride, int(slots[r]))
        ref = _np64_rope(_np64_layernorm(xf[r]), float(pos[r]), mode)
        assert _within_quant_bound(deq, ref, dtype, es), f"row {r}"
        slips["rope before norm"] += not _within_quant_bound(
            deq, _np64_layernorm(_np64_rope(xf[r].astype(np.float64), float(pos[r]), mode)), dtype, es)
        slips["no norm"] += not _within_quant_bound(
            deq, _np64_rope(xf[r].astype(np.float64), float(pos[r]), mode), dtype, es)
        slips["position = row"] += not _within_quant_bound(
            deq, _np64_rope(_np64_layernorm(xf[r]), float(r), mode), dtype, es)
    assert all(v >= n // 2 for v in slips.values()), slips
