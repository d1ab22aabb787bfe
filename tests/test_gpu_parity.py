"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Bit-exact: packed cache bytes (codes and scales), quantised Q, folded weights, element
encoders. Tolerance: logits within 1e-4 * max |exact logit| of the row with cosine >=
0.999999; top-k sets equal up to ties within that tolerance of the k-th value.
"""
import numpy as np
import pytest

import oracle as O
from sparse_attention_indexer_mqa_gb300 import workloads as W

from helpers import (Dev, assert_logits_close, assert_topk_valid, oracle_logits, oracle_q,
                     oracle_store, oracle_topk, q_image_to_plain)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as T
    from sparse_attention_indexer_mqa_gb300 import binding
    binding.load()
    return T


# ------------------------------------------------------------------ element encoders

def _sweep_values():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = W.bf16_to_f32(b)
    v = v[np.isfinite(v)]
    rng = np.random.default_rng(20)
    r = np.concatenate([(rng.standard_normal(2_000_000) * 3).astype(np.float32),
                        (rng.random(1_000_000) * 16 - 8).astype(np.float32),
                        (rng.standard_normal(1_000_000) * 200).astype(np.float32)])
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 448.0, 464.0], np.float32)
    near = np.concatenate([np.nextafter(mids, 0), np.nextafter(mids, 1e9), mids])
    return np.concatenate([v, r, near, -near, np.array([0.0, -0.0], np.float32)])


def test_e2m1_encoder_matches_oracle(torch):
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    v = _sweep_values()
    v = v[np.abs(v) < 8]
    x = torch.from_numpy(v).cuda()
    out = torch.empty(v.shape[0], dtype=torch.uint8, device="cuda")
    Bn.idx_debug_encode(0, x, out)
    np.testing.assert_array_equal(out.cpu().numpy(), O.e2m1_encode_n(v))


def test_e4m3_encoder_matches_oracle(torch):
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    v = _sweep_values()
    x = torch.from_numpy(v).cuda()
    out = torch.empty(v.shape[0], dtype=torch.uint8, device="cuda")
    Bn.idx_debug_encode(1, x, out)
    np.testing.assert_array_equal(out.cpu().numpy(), O.e4m3_encode_n(v))


# ------------------------------------------------------------------ K store / Q quant

def _check_store_and_quant(wl, label, fused=False):
    d = Dev(wl)
    if fused:  # one launch (idx_qk_prep) must give the same bytes as the two entry points
        d.prep()
    else:
        d.store()
        d.quant()
    pool_gpu = d.host("pool_buf")
    pool_ref = oracle_store(wl)
    assert d.host("status")[0] == 0
    diff = np.nonzero(pool_gpu != pool_ref)[0]
    assert diff.size == 0, f"{label}: {diff.size} cache bytes differ, first at {diff[:8]}"
    qc, qs, w = oracle_q(wl)
    gc, gs = q_image_to_plain(d.host("q_codes"), d.host("q_scales"), wl.H, wl.dtype)
    np.testing.assert_array_equal(gc, qc, err_msg=label)
    if wl.dtype == W.MXFP4:
        np.testing.assert_array_equal(gs, qs, err_msg=label)
    else:
        np.testing.assert_array_equal(d.host("q_scales").view(np.uint32), qs.view(np.uint32), err_msg=label)
    np.testing.assert_array_equal(d.host("w").view(np.uint32), w.view(np.uint32), err_msg=label)
    return d, pool_ref, (qc, qs, w)


def test_store_quant_tiny_decode(torch):
    wl = W.make("tiny_decode")
    d, pool_ref, _ = _check_store_and_quant(wl, "tiny")
    # the page of slack in front of the pool view stays untouched
    assert not d.host("pool_buf")[:wl.page_stride].any()


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("n", [1, 7, 32, 257, 1023])
@pytest.mark.parametrize("P", [64, 128])
@pytest.mark.parametrize("rope", [W.ROPE_NEOX, W.ROPE_INTERLEAVED])
@pytest.mark.parametrize("dtype", [W.MXFP4, W.FP8])
def test_store_quant_grid(torch, n, P, rope, dtype, fused):
    """Token-count x page-size x RoPE-layout grid of the fused pre-processing op test
    (vllm PR 53094 "Test Plan / Op test"), here bit-exact against the oracle."""
    rng = np.random.default_rng(1000 + n)
    pages = (n + P - 1) // P + 3
    perm = rng.permutation(pages).astype(np.int32)
    slots = (perm[np.arange(n) // P].astype(np.int64) * P + np.arange(n) % P)
    slots[rng.random(n) < 0.1] = -1  # padded rows are skipped
    H = 4
    wl = W.Workload(
        name="grid", dtype=dtype, B=1, H=H, page_size=P, pool_pages=pages, base_offset_pages=1,
        page_stride=W.page_bytes(dtype, P) + 16 * int(rng.integers(0, 3)),
        seq_lens_k=np.array([n], np.int32), cu_seqlens_q=np.array([0, n], np.int32),
        page_table=perm[None, :], causal=1, topk=8,
        k=W.bf16_bits((rng.standard_normal((n, 128)) * rng.uniform(0.1, 30)).astype(np.float32)),
        slot_mapping=slots, k_positions=rng.integers(0, 4000, n).astype(np.int32), k_rope=rope,
        k_norm=1, step_rows=np.arange(n), q=W.bf16_bits(rng.standard_normal((n, H, 128)).astype(np.float32)),
        q_positions=rng.integers(0, 4000, n).astype(np.int32), q_rope=rope,
        w_in=rng.standard_normal((n, H)).astype(np.float32), softmax_scale=0.088388,
        head_scale=0.5, cos_sin=W.rope_table(4000), ld_logits=n)
    _check_store_and_quant(wl, f"grid n={n} P={P} rope={rope} dtype={dtype} fused={fused}", fused)


def test_store_quant_only_mode_outliers(torch):
    wl = W.make("decode_b64", B=4, ctx=1000)
    _check_store_and_quant(wl, "quant-only")


@pytest.mark.parametrize("fused", [False, True])
def test_store_quant_compressed_full(torch, fused):
    _check_store_and_quant(W.make("decode_compressed"), "compressed decode, full size", fused)


@pytest.mark.parametrize("fused", [False, True])
def test_store_quant_fp8_full(torch, fused):
    _check_store_and_quant(W.make("prefill_fp8"), "fp8 prefill, full size", fused)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("dtype", [W.MXFP4, W.FP8])
def test_store_quant_many_tokens(torch, dtype, fused):
    """Enough tokens for the Q quant's several-tokens-per-CTA launch (2501 tokens x 2 head
    blocks; the last CTA's group is ragged), bit-exact against the oracle."""
    rng = np.random.default_rng(77)
    n, H, P = 2501, 32, 128
    pages = (n + P - 1) // P + 1
    perm = rng.permutation(pages).astype(np.int32)
    slots = perm[np.arange(n) // P].astype(np.int64) * P + np.arange(n) % P
    wl = W.Workload(
        name="many", dtype=dtype, B=1, H=H, page_size=P, pool_pages=pages, base_offset_pages=0,
        page_stride=W.page_bytes(dtype, P), seq_lens_k=np.array([n], np.int32),
        cu_seqlens_q=np.array([0, n], np.int32), page_table=perm[None, :], causal=1, topk=8,
        k=W.bf16_bits(rng.standard_normal((n, 128)).astype(np.float32)), slot_mapping=slots,
        k_positions=np.arange(n, dtype=np.int32), k_rope=W.ROPE_NEOX, k_norm=1, step_rows=np.arange(n),
        q=W.bf16_bits((rng.standard_normal((n, H, 128)) * 4).astype(np.float32)),
        q_positions=np.arange(n, dtype=np.int32), q_rope=W.ROPE_NEOX,
        w_in=rng.standard_normal((n, H)).astype(np.float32), softmax_scale=0.088388, head_scale=1.0,
        cos_sin=W.rope_table(n), ld_logits=n)
    _check_store_and_quant(wl, f"many tokens dtype={dtype} fused={fused}", fused)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("H", [20, 64])
@pytest.mark.parametrize("rope", [W.ROPE_NEOX, W.ROPE_INTERLEAVED])
@pytest.mark.parametrize("dtype", [W.MXFP4, W.FP8])
def test_store_quant_two_q_rows_per_lanes(torch, dtype, rope, H, fused):
    """Enough tokens for the Q launch that gives each 16 lanes two heads (h, h + 16) sharing one
    position: padded head counts (20 -> 24, the second rows partly padding) and 64 heads (two
    head blocks per token), both RoPE layouts, bit-exact against the oracle."""
    rng = np.random.default_rng(78 + H)
    n, P = 700, 64
    pages = (n + P - 1) // P + 1
    perm = rng.permutation(pages).astype(np.int32)
    slots = perm[np.arange(n) // P].astype(np.int64) * P + np.arange(n) % P
    wl = W.Workload(
        name="two_rows", dtype=dtype, B=1, H=H, page_size=P, pool_pages=pages, base_offset_pages=0,
        page_stride=W.page_bytes(dtype, P), seq_lens_k=np.array([n], np.int32),
        cu_seqlens_q=np.array([0, n], np.int32), page_table=perm[None, :], causal=1, topk=8,
        k=W.bf16_bits(rng.standard_normal((n, 128)).astype(np.float32)), slot_mapping=slots,
        k_positions=rng.integers(0, 3000, n).astype(np.int32), k_rope=rope, k_norm=1, step_rows=np.arange(n),
        q=W.bf16_bits((rng.standard_normal((n, H, 128)) * 3).astype(np.float32)),
        q_positions=rng.integers(0, 3000, n).astype(np.int32), q_rope=rope,
        w_in=rng.standard_normal((n, H)).astype(np.float32), softmax_scale=0.088388, head_scale=0.75,
        cos_sin=W.rope_table(3000), ld_logits=n)
    _check_store_and_quant(wl, f"two rows H={H} rope={rope} dtype={dtype} fused={fused}", fused)


@pytest.mark.parametrize("n", [8, 700])
@pytest.mark.parametrize("dtype", [W.MXFP4, W.FP8])
def test_q_bad_position_sets_status(torch, dtype, n):
    """A query token whose position lies beyond the RoPE table: IDX_STATUS_BAD_POS, its real
    head rows and weights left untouched, its padding rows written; every other token
    bit-exact. Few tokens (one Q row per 16 lanes) and many (two per 16 lanes)."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    rng = np.random.default_rng(90 + n)
    H, P, bad = 20, 64, 3
    pages = (n + P - 1) // P + 1
    perm = rng.permutation(pages).astype(np.int32)
    slots = perm[np.arange(n) // P].astype(np.int64) * P + np.arange(n) % P
    wl = W.Workload(
        name="badq", dtype=dtype, B=1, H=H, page_size=P, pool_pages=pages, base_offset_pages=0,
        page_stride=W.page_bytes(dtype, P), seq_lens_k=np.array([n], np.int32),
        cu_seqlens_q=np.array([0, n], np.int32), page_table=perm[None, :], causal=1, topk=8,
        k=W.bf16_bits(rng.standard_normal((n, 128)).astype(np.float32)), slot_mapping=slots,
        k_positions=np.arange(n, dtype=np.int32), k_rope=W.ROPE_NEOX, k_norm=1, step_rows=np.arange(n),
        q=W.bf16_bits(rng.standard_normal((n, H, 128)).astype(np.float32)),
        q_positions=rng.integers(0, 1000, n).astype(np.int32), q_rope=W.ROPE_NEOX,
        w_in=rng.standard_normal((n, H)).astype(np.float32), softmax_scale=0.088388, head_scale=1.0,
        cos_sin=W.rope_table(1000), ld_logits=n)
    qc, qs, w = oracle_q(wl)
    d = Dev(wl)
    d.qpos[bad] = 10 ** 6
    d.w.fill_(-3.0)
    d.quant()
    assert int(d.host("status")[0]) & Bn.IDX_STATUS_BAD_POS
    codes = d.host("q_codes")
    Hq = (H + 7) // 8 * 8
    kc = 4 if dtype == W.MXFP4 else 8
    plain = codes.reshape(n, Hq // 8, kc, 8, 16).transpose(0, 1, 3, 2, 4).reshape(n, Hq, kc * 16)
    assert (plain[bad, :H] == 0xEE).all(), "the rejected token's rows were written"
    assert not plain[bad, H:].any(), "the rejected token's padding rows must be zero"
    assert (d.host("w")[bad] == -3.0).all(), "the rejected token's weights were written"
    ok = np.setdiff1d(np.arange(n), [bad])
    codes[bad] = 0  # the rejected token is checked above; the rest through the plain layout
    gc, gs = q_image_to_plain(codes, d.host("q_scales"), H, dtype)
    np.testing.assert_array_equal(gc[ok], qc[ok])
    if dtype == W.MXFP4:
        np.testing.assert_array_equal(gs[ok], qs[ok])
    else:
        np.testing.assert_array_equal(d.host("q_scales").view(np.uint32)[ok], qs.view(np.uint32)[ok])
    np.testing.assert_array_equal(d.host("w").view(np.uint32)[ok], w.view(np.uint32)[ok])


def test_qk_prep_one_side_empty(torch):
    """idx_qk_prep with no K rows only quantises Q; with no queries only stores K."""
    import torch as T
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    wl = W.make("tiny_decode")
    d = Dev(wl)
    Bn.idx_qk_prep(None, None, None, wl.k_rope, wl.k_norm, d.pool, wl.pool_pages, wl.page_size,
                   wl.page_stride, d.q, d.qpos, wl.q_rope, d.w_in, wl.softmax_scale, wl.head_scale,
                   d.q_codes, d.q_scales, d.w, d.cos_sin, wl.dtype, dev_status=d.status)
    assert not d.host("pool_buf").any()
    qc, qs, w = oracle_q(wl)
    gc, _ = q_image_to_plain(d.host("q_codes"), d.host("q_scales"), wl.H, wl.dtype)
    np.testing.assert_array_equal(gc, qc)
    d2 = Dev(wl)
    empty_q = d2.q[:0]
    Bn.idx_qk_prep(d2.k, d2.slot, d2.kpos, wl.k_rope, wl.k_norm, d2.pool, wl.pool_pages,
                   wl.page_size, wl.page_stride, empty_q, d2.qpos, wl.q_rope, d2.w_in,
                   wl.softmax_scale, wl.head_scale, d2.q_codes, d2.q_scales, d2.w, d2.cos_sin,
                   wl.dtype, dev_status=d2.status)
    np.testing.assert_array_equal(d2.host("pool_buf"), oracle_store(wl))
    assert (d2.host("q_codes") == 0xEE).all()  # untouched


def test_store_bad_rows_set_status(torch):
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    wl = W.make("tiny_decode")
    d = Dev(wl)
    slot = d.slot.clone()
    slot[3] = wl.pool_pages * wl.page_size + 5  # beyond the pool
    pos = d.kpos.clone()
    pos[5] = 10 ** 6                            # beyond the RoPE table
    Bn.idx_k_store(d.k, slot, pos, d.cos_sin, wl.k_rope, 1, wl.dtype, d.pool, wl.pool_pages,
                   wl.page_size, wl.page_stride, dev_status=d.status)
    st = int(d.host("status")[0])
    assert st & Bn.IDX_STATUS_BAD_SLOT and st & Bn.IDX_STATUS_BAD_POS
    ref = oracle_store(wl, rows=np.setdiff1d(np.arange(wl.n_k_rows), [3, 5]))
    np.testing.assert_array_equal(d.host("pool_buf"), ref)


# ------------------------------------------------------------------ scorer + top-k

def torch_rows(rows):
    import torch as T
    return T.from_numpy(np.asarray(rows, np.int64)).cuda()


def _full_path(wl, rows=None, label=""):
    d = Dev(wl)
    d.run_all()
    assert d.host("status")[0] == 0
    pool_ref = oracle_store(wl)
    np.testing.assert_array_equal(d.host("pool_buf"), pool_ref)
    qc, qs, w = oracle_q(wl)
    exact = oracle_logits(wl, pool_ref, qc, qs, w, rows=rows)
    vis = wl.visible()
    if rows is not None:
        r = torch_rows(rows)
        got, tk, vis = d.logits[r].cpu().numpy(), d.topk[r].cpu().numpy(), vis[rows]
    else:
        got, tk = d.host("logits"), d.host("topk")
    worst = assert_logits_close(got, exact, vis, label=label)
    assert_topk_valid(tk, exact, got, vis, wl.topk, label=label)
    # entries past visible(t) are not written
    for r in range(got.shape[0]):
        assert np.isnan(got[r, vis[r]:]).all(), f"{label}: wrote past visible in row {r}"
    return d, worst


def test_path_tiny_decode(torch):
    _full_path(W.make("tiny_decode"), label="tiny")


def test_path_decode_b64_full(torch):
    _full_path(W.make("decode_b64"), label="decode B64/H32/8K")


def test_path_decode_compressed_full(torch):
    _full_path(W.make("decode_compressed"), label="decode compressed B256/H64")


def test_path_fp8_decode(torch):
    # one new query per sequence: the FP8 decode kernel, page 64, ragged lengths
    _full_path(W.make("prefill_fp8", B=5, cached=3001, new=1), label="fp8 decode")


def test_path_decode_h64_p128_ragged(torch):
    wl = W.make("decode_b64", B=9, ctx=1000, H=64)
    _full_path(wl, label="decode H64 P128 ragged")


def test_path_prefill_small_ragged(torch):
    # several tiles, a ragged tail, causal
    _full_path(W.make("prefill_8k", T=700), label="prefill 700")


def test_path_prefill_8k_sampled(torch):
    """At least 512 rows: 8 from every 128-row band of queries (the band's first rows, which sit
    on the diagonal key tile, its middle and its last row), plus the k-boundary rows."""
    wl = W.make("prefill_8k")
    bands = np.arange(0, 8192, 128)
    rows = np.unique(np.concatenate([bands[:, None] + np.array([0, 1, 2, 31, 63, 64, 100, 127])[None, :],
                                     [[1022, 1023, 1024, 1025]]], axis=None))
    assert rows.size >= 512
    _full_path(wl, rows=rows, label="prefill 8192 (sampled rows)")


def test_path_fp8_small(torch):
    _full_path(W.make("prefill_fp8", B=2, cached=300, new=200), label="fp8 small")


def test_path_fp8_full_sampled(torch):
    """256 rows per sequence: its first and last 16 queries, the first and last rows of 64-query
    bands (block edges of the scorer's query blocks and of the 64-key pages), spread middles."""
    wl = W.make("prefill_fp8")
    per = np.unique(np.concatenate([np.arange(16), np.arange(4080, 4096), np.arange(0, 4096, 64),
                                    np.arange(63, 4096, 64), np.linspace(0, 4095, 120).astype(int)]))
    assert per.size >= 256
    rows = np.concatenate([b * 4096 + per for b in range(8)])
    _full_path(wl, rows=rows, label="fp8 32K (sampled rows)")


def test_shuffled_pages_bitwise(torch):
    wl = W.make("tiny_decode")
    d = Dev(wl)
    d.run_all()
    base = d.host("logits").copy()
    rng = np.random.default_rng(30)
    perm = rng.permutation(wl.pool_pages)
    pool = d.host("pool").copy()
    new = np.zeros_like(pool)
    ps = wl.page_stride
    for p in range(wl.pool_pages):
        new[perm[p] * ps:(perm[p] + 1) * ps] = pool[p * ps:(p + 1) * ps]
    d.pool.copy_(torch.from_numpy(new).cuda())
    pt = torch.from_numpy(perm[wl.page_table].astype(np.int32)).cuda()
    d.logits.fill_(float("nan"))
    d.score(page_table=pt)
    assert np.array_equal(d.host("logits"), base, equal_nan=True)


def test_mutations_break_parity(torch):
    """Shifted page table, one flipped scale byte: the comparison must fail."""
    wl = W.make("tiny_decode")
    d = Dev(wl)
    d.run_all()
    pool_ref = oracle_store(wl)
    qc, qs, w = oracle_q(wl)
    exact = oracle_logits(wl, pool_ref, qc, qs, w)
    vis = wl.visible()
    d.logits.fill_(float("nan"))
    d.score(page_table=torch.roll(d.page_table, 1, dims=1).contiguous())
    with pytest.raises(AssertionError):
        assert_logits_close(d.host("logits"), exact, vis)
    pg = int(wl.page_table[0, 0])
    d.pool[pg * wl.page_stride + O.scale_offset(0, wl.page_size, 2, 0)] += 3
    d.logits.fill_(float("nan"))
    d.score()
    with pytest.raises(AssertionError):
        assert_logits_close(d.host("logits"), exact, vis)


def test_bad_page_sets_status(torch):
    wl = W.make("tiny_decode")
    d = Dev(wl)
    d.store(); d.quant()
    pt = d.page_table.clone()
    pt[1, 0] = wl.pool_pages + 3
    d.score(page_table=pt)
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    assert int(d.host("status")[0]) & Bn.IDX_STATUS_BAD_PAGE


def test_large_pool_addresses(torch):
    """Pages placed across the 2^31, 2^32 and 4.608e9-byte offsets of a 4.7 GB pool
    (the 64-bit page rebasing cases of vllm PR 57517 "Test plan")."""
    wl = W.make("tiny_decode")
    ps = wl.page_stride
    targets = [2 ** 31, 2 ** 32, 4_608_000_000]
    n_pages = 4_700_000_000 // ps
    # choose physical page ids whose byte range straddles or follows each target
    ids = []
    for tgt in targets:
        p = tgt // ps
        ids += [p - 1, p, p + 1]
    ids = np.array(ids[:8], np.int32)
    pt = np.full_like(wl.page_table, 0)
    need0 = (int(wl.seq_lens_k[0]) + wl.page_size - 1) // wl.page_size
    need1 = (int(wl.seq_lens_k[1]) + wl.page_size - 1) // wl.page_size
    pt[0, :need0] = ids[:need0]
    pt[1, :need1] = ids[need0:need0 + need1]
    slots = []
    for b, L in enumerate(wl.seq_lens_k):
        s = np.arange(int(L))
        slots.append(pt[b, s // wl.page_size].astype(np.int64) * wl.page_size + s % wl.page_size)
    slots = np.concatenate(slots)
    big = W.Workload(**{**wl.__dict__, "page_table": pt, "slot_mapping": slots,
                        "pool_pages": int(n_pages), "base_offset_pages": 0})
    d = Dev(big)
    d.run_all()
    assert d.host("status")[0] == 0
    # oracle on a compact pool holding only the used pages (same bytes, remapped ids)
    remap = {int(p): i for i, p in enumerate(sorted(set(ids.tolist())))}
    pt_c = np.vectorize(lambda p: remap.get(int(p), 0))(pt).astype(np.int32)
    small = W.Workload(**{**wl.__dict__, "page_table": pt_c, "pool_pages": len(remap),
                          "base_offset_pages": 0,
                          "slot_mapping": np.concatenate([pt_c[b, np.arange(int(L)) // wl.page_size].astype(np.int64) * wl.page_size + np.arange(int(L)) % wl.page_size for b, L in enumerate(wl.seq_lens_k)])})
    pool_ref = oracle_store(small)
    torch.cuda.synchronize()
    for p, i in remap.items():
        np.testing.assert_array_equal(d.pool[p * ps:(p + 1) * ps].cpu().numpy(),
                                      pool_ref[i * ps:(i + 1) * ps])
    qc, qs, w = oracle_q(small)
    exact = oracle_logits(small, pool_ref, qc, qs, w)
    assert_logits_close(d.host("logits"), exact, wl.visible(), label="large pool")


def _chunked_prefill(dtype, H, P, causal, lens, nqs, seed):
    """Several sequences, each scoring its last nq tokens (chunked prefill) against all of
    its keys, K stored by the full LayerNorm + RoPE path."""
    rng = np.random.default_rng(seed)
    lens = np.array(lens, np.int32)
    nqs = np.array(nqs, np.int32)
    B = len(lens)
    need = [(int(L) + P - 1) // P for L in lens]
    pool = sum(need) + 5
    perm = rng.permutation(pool).astype(np.int32)
    pt = np.full((B, max(need)), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[o:o + n]
        o += n
    slots = np.concatenate([pt[b, np.arange(L) // P].astype(np.int64) * P + np.arange(L) % P
                            for b, L in enumerate(lens)])
    kpos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    qpos = np.concatenate([np.arange(L - n, L, dtype=np.int32).clip(0) for L, n in zip(lens, nqs)])
    T = int(nqs.sum())
    rope = W.ROPE_INTERLEAVED if dtype == W.FP8 else W.ROPE_NEOX
    return W.Workload(
        name="chunked", dtype=dtype, B=B, H=H, page_size=P, pool_pages=pool, base_offset_pages=1,
        page_stride=W.page_bytes(dtype, P), seq_lens_k=lens,
        cu_seqlens_q=np.concatenate([[0], np.cumsum(nqs)]).astype(np.int32), page_table=pt,
        causal=causal, topk=64, k=W.bf16_bits(rng.standard_normal((int(lens.sum()), 128)).astype(np.float32)),
        slot_mapping=slots, k_positions=kpos, k_rope=rope, k_norm=1, step_rows=np.arange(1),
        q=W.bf16_bits(rng.standard_normal((T, H, 128)).astype(np.float32)), q_positions=qpos,
        q_rope=rope, w_in=(rng.standard_normal((T, H)) / np.sqrt(H)).astype(np.float32),
        softmax_scale=float(128 ** -0.5), head_scale=1.0, cos_sin=W.rope_table(int(lens.max())),
        ld_logits=(int(lens.max()) + 3) // 4 * 4)


@pytest.mark.parametrize("dtype,H,P,causal", [
    (W.MXFP4, 4, 64, 1), (W.MXFP4, 24, 128, 0), (W.MXFP4, 64, 64, 1), (W.MXFP4, 32, 64, 0),
    (W.FP8, 64, 64, 1), (W.FP8, 8, 128, 0), (W.FP8, 32, 128, 1)])
def test_path_chunked_prefill(torch, dtype, H, P, causal):
    wl = _chunked_prefill(dtype, H, P, causal, [300, 517, 129, 1], [37, 200, 129, 1], seed=H * 7 + P)
    _full_path(wl, label=f"chunked prefill dtype={dtype} H={H} P={P} causal={causal}")


@pytest.mark.parametrize("dtype,H,P,B", [(W.MXFP4, 32, 64, 20000), (W.FP8, 16, 128, 3000)])
def test_path_decode_many_short_sequences(torch, dtype, H, P, B):
    """Thousands of short decode sequences (1..300 keys, some empty of queries' keys): a
    scorer CTA's slice then spans more sequences than its shared-memory window describes,
    and the prologue scans past its first 256 sequences."""
    rng = np.random.default_rng(B)
    lens = rng.integers(1, 301, B)
    wl = _chunked_prefill(dtype, H, P, 0, lens.tolist(), [1] * B, seed=B + H)
    _full_path(wl, rows=np.sort(rng.choice(B, 400, replace=False)),
               label=f"many short decode dtype={dtype} B={B}")


# ------------------------------------------------------------------ injected length faults

def _status_bad_len(d):
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    return bool(int(d.host("status")[0]) & Bn.IDX_STATUS_BAD_LEN)


@pytest.mark.parametrize("fault", ["over_max", "negative"])
def test_decode_bad_key_length_is_skipped_and_reported(torch, fault):
    """A decode sequence whose key count is above max_seq_len_k (or negative) is skipped:
    its logits row stays untouched, the status word gets IDX_STATUS_BAD_LEN, and the other
    sequences are scored exactly as before."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    wl = W.make("tiny_decode")
    d = Dev(wl)
    d.store(); d.quant()
    sl = d.seq_lens_k.clone()
    sl[1] = int(wl.seq_lens_k.max()) + 64 if fault == "over_max" else -5
    Bn.idx_mqa_logits_paged(d.q_codes, d.q_scales, d.w, wl.dtype, d.pool, wl.pool_pages,
                            wl.page_size, wl.page_stride, d.page_table, sl, d.cu, wl.causal, 1,
                            int(wl.seq_lens_k.max()), d.logits, dev_status=d.status)
    assert _status_bad_len(d)
    got = d.host("logits")
    assert np.isnan(got[1]).all()
    pool_ref = oracle_store(wl)
    qc, qs, w = oracle_q(wl)
    exact = oracle_logits(wl, pool_ref, qc, qs, w, rows=np.array([0]))
    assert_logits_close(got[:1], exact, wl.visible()[:1], label="good sequence")


def test_decode_kernel_rejects_multi_query_sequence(torch):
    """max_q_len = 1 selects the decode scorer; a sequence that nevertheless owns two
    queries is skipped and reported instead of being scored with the wrong window."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    wl = _chunked_prefill(W.MXFP4, 8, 64, 1, [300, 200], [2, 1], seed=3)
    d = Dev(wl)
    d.store(); d.quant()
    Bn.idx_mqa_logits_paged(d.q_codes, d.q_scales, d.w, wl.dtype, d.pool, wl.pool_pages,
                            wl.page_size, wl.page_stride, d.page_table, d.seq_lens_k, d.cu,
                            wl.causal, 1, int(wl.seq_lens_k.max()), d.logits, dev_status=d.status)
    assert _status_bad_len(d)
    got = d.host("logits")
    assert np.isnan(got[:2]).all()          # both queries of sequence 0 untouched
    pool_ref = oracle_store(wl)
    qc, qs, w = oracle_q(wl)
    exact = oracle_logits(wl, pool_ref, qc, qs, w, rows=np.array([2]))
    assert_logits_close(got[2:3], exact, wl.visible()[2:3], label="single-query sequence")


@pytest.mark.parametrize("fault", ["too_many_queries", "over_max", "negative"])
def test_prefill_bad_lengths_are_skipped_and_reported(torch, fault):
    """Prefill scorer: a sequence with more queries than max_q_len, or a key count above
    max_seq_len_k or negative, is skipped and reported; the other sequences are exact."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    wl = _chunked_prefill(W.MXFP4, 32, 128, 1, [400, 300], [150, 40], seed=4)
    d = Dev(wl)
    d.store(); d.quant()
    sl = d.seq_lens_k.clone()
    max_q, max_k = 150, int(wl.seq_lens_k.max())
    if fault == "too_many_queries":
        max_q = 100
    elif fault == "over_max":
        sl[0] = max_k + 1
    else:
        sl[0] = -1
    Bn.idx_mqa_logits_paged(d.q_codes, d.q_scales, d.w, wl.dtype, d.pool, wl.pool_pages,
                            wl.page_size, wl.page_stride, d.page_table, sl, d.cu, wl.causal,
                            max_q, max_k, d.logits, dev_status=d.status)
    assert _status_bad_len(d)
    got = d.host("logits")
    assert np.isnan(got[:150]).all()        # sequence 0 untouched
    rows = np.arange(150, 190)
    pool_ref = oracle_store(wl)
    qc, qs, w = oracle_q(wl)
    exact = oracle_logits(wl, pool_ref, qc, qs, w, rows=rows)
    assert_logits_close(got[rows], exact, wl.visible()[rows], label="good sequence")


def test_topk_bad_lengths_give_padding_and_status(torch):
    """Top-k rows of a sequence whose key count is above max_seq_len_k (here also above the
    row stride) or negative are all -1 and set IDX_STATUS_BAD_LEN; the rows of consistent
    sequences are unaffected."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    rng = np.random.default_rng(9)
    ld, k = 3000, 256
    logits = torch.from_numpy(rng.standard_normal((3, ld)).astype(np.float32)).cuda()
    sl = torch.tensor([ld + 500, -3, 2500], dtype=torch.int32, device="cuda")
    cu = torch.arange(4, dtype=torch.int32, device="cuda")
    out = torch.full((3, k), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Bn.idx_topk(logits, sl, cu, 0, ld, k, out, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & Bn.IDX_STATUS_BAD_LEN
    o = out.cpu().numpy()
    assert (o[0] == -1).all() and (o[1] == -1).all()
    row = logits[2, :2500].cpu().numpy()
    assert set(o[2].tolist()) == set(np.argsort(-row, kind="stable")[:k].tolist())
    # a bound below the true length: the row is reported, not ranked past the bound
    status.zero_()
    sl2 = torch.tensor([2000, 2000, 2500], dtype=torch.int32, device="cuda")
    Bn.idx_topk(logits, sl2, cu, 0, 2400, k, out, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & Bn.IDX_STATUS_BAD_LEN
    assert (out[2].cpu().numpy() == -1).all()
