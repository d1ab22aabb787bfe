"""GPU parity of the compressed K store (idx_compress_k_store) against the oracle's
compress_k_store, through the C ABI: the packed cache bytes must be identical.

vllm PR 60834 "Changes / K write": pool (softmax-gated overlap pooling) -> RMSNorm -> RoPE ->
MXFP4 -> store, one entry per compress-ratio boundary token. Cases: every dtype, RoPE mode
and norm; ratios 1..128; ragged sequences whose tails form no entry; several CTAs plus a
partial one; padded row strides; both page sizes; a pool view at a nonzero offset; the
rejection paths; and sampled entries of the full 256-sequence workload.
"""
import numpy as np
import pytest

import oracle as O
from sparse_attention_indexer_mqa_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as T
    from sparse_attention_indexer_mqa_gb300 import binding
    binding.load()
    return T


def _dev(torch, a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def _run_gpu(torch, cw, offset_pages=0, boundary=None, first=None, slots=None, positions=None,
             expect_status=0):
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    nbytes = (cw.pool_pages + offset_pages) * cw.page_stride
    buf = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    view = buf[offset_pages * cw.page_stride:]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bnd = cw.boundary if boundary is None else boundary
    Bn.idx_compress_k_store(
        _dev(torch, cw.k_raw), _dev(torch, cw.gate), _dev(torch, bnd),
        _dev(torch, cw.first if first is None else first), cw.ratio,
        _dev(torch, cw.slot_mapping if slots is None else slots),
        _dev(torch, cw.positions if positions is None else positions),
        _dev(torch, cw.cos_sin), cw.rope, cw.norm, cw.dtype, view, cw.pool_pages, cw.page_size,
        cw.page_stride, gamma=_dev(torch, cw.gamma), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == expect_status
    return buf.cpu().numpy(), offset_pages * cw.page_stride


def _run_oracle(cw, offset_bytes=0, boundary=None, first=None, slots=None, positions=None):
    buf = np.zeros(cw.pool_pages * cw.page_stride + offset_bytes, np.uint8)
    view = buf[offset_bytes:]
    bad = O.compress_k_store(view, cw.k_raw, cw.gate, cw.boundary if boundary is None else boundary,
                             cw.first if first is None else first, cw.ratio,
                             cw.slot_mapping if slots is None else slots,
                             cw.positions if positions is None else positions, cw.cos_sin, cw.rope,
                             cw.norm, cw.dtype, cw.pool_pages, cw.page_size, cw.page_stride,
                             gamma=cw.gamma)
    buf[offset_bytes:] = view
    return buf, bad


@pytest.mark.parametrize("dtype", [W.MXFP4, W.FP8])
@pytest.mark.parametrize("rope", [W.ROPE_NONE, W.ROPE_NEOX, W.ROPE_INTERLEAVED])
@pytest.mark.parametrize("norm", [0, 1, 2])
def test_compress_store_bit_exact(torch, dtype, rope, norm):
    cw = W.compress_work(seed=10 + 9 * dtype + 3 * rope + norm, raw_lens=(37, 64, 130, 3, 261),
                         dtype=dtype, rope=rope, norm=norm)
    assert cw.n_entries > 4 * 16  # several CTAs and a partial one
    got, off = _run_gpu(torch, cw, offset_pages=1)
    ref, bad = _run_oracle(cw, offset_bytes=off)
    assert bad == 0
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("ratio", [1, 2, 3, 8, 128])
def test_compress_ratios(torch, ratio):
    cw = W.compress_work(seed=30 + ratio, raw_lens=(5, 300, 129, 1100), ratio=ratio,
                         page_size=128, row_stride=136)
    got, off = _run_gpu(torch, cw)
    ref, bad = _run_oracle(cw, offset_bytes=off)
    assert bad == 0
    np.testing.assert_array_equal(got, ref)


def test_compress_large_gates_and_outlier_rows(torch):
    """Gates spread over +-40 (exp of the differences reaches the cut-off at -87 and the
    underflow range) and K rows scaled x20 (E8M0 scales far from the rest)."""
    cw = W.compress_work(seed=41, raw_lens=(400, 77), ratio=4, dtype=W.MXFP4, norm=0)
    rng = np.random.default_rng(42)
    g = W.bf16_to_f32(cw.gate[:, :128]) * np.float32(20.0)
    cw.gate[:, :128] = W.bf16_bits(g)
    rows = rng.choice(cw.k_raw.shape[0], 40, replace=False)
    cw.k_raw[rows, :128] = W.bf16_bits(W.bf16_to_f32(cw.k_raw[rows, :128]) * np.float32(20.0))
    got, off = _run_gpu(torch, cw)
    ref, bad = _run_oracle(cw, offset_bytes=off)
    assert bad == 0
    np.testing.assert_array_equal(got, ref)


def test_compress_rejections(torch):
    """A negative slot is skipped; a slot past the pool, a window outside the raw rows and a
    position outside the table each set their status bit and leave the slot unwritten; the
    other entries are stored exactly."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    cw = W.compress_work(seed=50, raw_lens=(64, 64), ratio=4, dtype=W.FP8, spare_pages=2)
    slots = cw.slot_mapping.copy()
    bnd, fst, pos = cw.boundary.copy(), cw.first.copy(), cw.positions.copy()
    slots[1] = -1
    slots[2] = cw.pool_pages * cw.page_size          # past the pool
    fst[5] = bnd[5] + 1                              # first after the boundary
    bnd[7] = cw.k_raw.shape[0]                       # boundary past the raw rows
    pos[9] = cw.cos_sin.shape[0]                     # position outside the table
    want = Bn.IDX_STATUS_BAD_SLOT | Bn.IDX_STATUS_BAD_LEN | Bn.IDX_STATUS_BAD_POS
    got, off = _run_gpu(torch, cw, boundary=bnd, first=fst, slots=slots, positions=pos,
                        expect_status=want)
    ref, bad = _run_oracle(cw, offset_bytes=off, boundary=bnd, first=fst, slots=slots, positions=pos)
    assert bad == 4
    np.testing.assert_array_equal(got, ref)


def test_compress_empty_and_argument_errors(torch):
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    cw = W.compress_work(seed=60, raw_lens=(16,), ratio=4)
    k, g = _dev(torch, cw.k_raw), _dev(torch, cw.gate)
    pool = torch.zeros(cw.pool_pages * cw.page_stride, dtype=torch.uint8, device="cuda")
    e = torch.zeros(0, dtype=torch.int64, device="cuda")
    p = torch.zeros(0, dtype=torch.int32, device="cuda")
    cs = _dev(torch, cw.cos_sin)
    Bn.idx_compress_k_store(k, g, e, e, 4, e, p, cs, cw.rope, 2, cw.dtype, pool, cw.pool_pages,
                            cw.page_size, cw.page_stride)
    torch.cuda.synchronize()
    assert int(pool.count_nonzero().item()) == 0
    b = _dev(torch, cw.boundary)
    for ratio, norm, err in ((0, 2, "unsupported"), (129, 2, "unsupported"), (4, 3, "invalid")):
        with pytest.raises(RuntimeError, match=err):
            Bn.idx_compress_k_store(k, g, b, _dev(torch, cw.first), ratio, _dev(torch, cw.slot_mapping),
                                    _dev(torch, cw.positions), cs, cw.rope, norm, cw.dtype, pool,
                                    cw.pool_pages, cw.page_size, cw.page_stride)


def test_compress_full_workload_sampled(torch):
    """All entries of the 256-sequence workload in one launch; 4096 sampled entries are
    recomputed by the oracle over the GPU's pool, which must not change a byte."""
    cw = W.compress_b256(seed=0)
    got, off = _run_gpu(torch, cw)
    rng = np.random.default_rng(61)
    sample = np.sort(rng.choice(cw.n_entries, 4096, replace=False))
    sample = np.union1d(sample, [0, cw.n_entries - 1])
    view = got.copy()
    bad = O.compress_k_store(view, cw.k_raw, cw.gate, cw.boundary[sample], cw.first[sample], cw.ratio,
                             cw.slot_mapping[sample], cw.positions[sample], cw.cos_sin, cw.rope,
                             cw.norm, cw.dtype, cw.pool_pages, cw.page_size, cw.page_stride,
                             gamma=cw.gamma)
    assert bad == 0
    np.testing.assert_array_equal(view, got)
    # and every entry's slot was written (no code byte block left all zero is not a proof,
    # but scales are never 0 for N(0, 1) inputs after RMSNorm)
    P = cw.page_size
    for s in rng.choice(cw.slot_mapping, 256, replace=False):
        page, r = int(s) // P, int(s) % P
        assert any(got[page * cw.page_stride + O.scale_offset(cw.dtype, P, r, b)] != 0 for b in range(4))
