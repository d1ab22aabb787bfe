"""GPU top-k against the oracle on the same fp32 logits, index for index.

Both sides decide on the same fp32 values, so the selected set must be identical (ties at
the k-th value resolved towards the lowest indices on both sides). The library's documented
order is also checked: indices above the k-th value in increasing order, then the indices
equal to it in increasing order. The cases reach every branch of the kernel: rows shorter
than k, rows staged in shared memory and rows too long for it, the narrow (many short rows)
and wide CTA shapes, candidate lists that fit and ones that overflow (heavy ties), unaligned
row starts, signed zeros, and causal prefill rows of growing length.
"""
import numpy as np
import pytest

import oracle as O
from sparse_attention_indexer_mqa_gb300 import binding as Bn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as T
    Bn.load()
    return T


def expected_order(logits32, vis, k):
    """The documented order, built from the oracle's selection."""
    if vis <= k:
        return np.concatenate([np.arange(vis), np.full(k - vis, -1)]).astype(np.int32)
    sel = O.topk(logits32.astype(np.float64)[None, :], np.array([vis], np.int32),
                 np.array([0, 1], np.int32), 0, k)[0]
    chosen = sel[:k]
    kth = logits32[chosen].min()
    above = np.sort(chosen[logits32[chosen] > kth])
    equal = np.sort(chosen[logits32[chosen] == kth])
    return np.concatenate([above, equal]).astype(np.int32)


def run_rows(torch, rows, k, ld=None, causal=0, cu=None, seq_lens=None):
    """rows: list of fp32 arrays (one query row each, decode layout) or an explicit
    (T, ld) matrix with cu/seq_lens for causal prefill."""
    if isinstance(rows, np.ndarray) and rows.ndim == 2:
        mat = rows
    else:
        L = max(len(r) for r in rows)
        ld = ld or L
        mat = np.full((len(rows), ld), np.nan, np.float32)
        for i, r in enumerate(rows):
            mat[i, :len(r)] = r
        seq_lens = np.array([len(r) for r in rows], np.int32)
        cu = np.arange(len(rows) + 1, dtype=np.int32)
    T = mat.shape[0]
    dl = torch.from_numpy(mat).cuda()
    dsl = torch.from_numpy(seq_lens).cuda()
    dcu = torch.from_numpy(cu).cuda()
    out = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    Bn.idx_topk(dl, dsl, dcu, causal, int(seq_lens.max()), k, out)
    torch.cuda.synchronize()
    return mat, out.cpu().numpy()


def check(mat, got, seq_lens, cu, causal, k):
    B = len(seq_lens)
    for b in range(B):
        q0, q1 = int(cu[b]), int(cu[b + 1])
        for t in range(q0, q1):
            L = int(seq_lens[b])
            vis = L - (q1 - q0) + (t - q0) + 1 if causal else L
            vis = max(0, min(L, vis))
            exp = expected_order(mat[t, :vis], vis, k)
            np.testing.assert_array_equal(got[t], exp, err_msg=f"row {t} (visible {vis})")


def _decode(torch, rows, k, ld=None):
    """Each case runs in both kernel forms: a 16-byte aligned leading dimension (four keys
    per shared-memory access) and an odd one (the generic form)."""
    L = max(len(r) for r in rows)
    lds = [ld] if ld is not None else [(L + 3) // 4 * 4, (L + 3) // 4 * 4 + 1]
    seq = np.array([len(r) for r in rows], np.int32)
    for d in lds:
        mat, got = run_rows(torch, rows, k, ld=d)
        check(mat, got, seq, np.arange(len(rows) + 1), 0, k)


def test_topk_lengths_around_k(torch):
    rng = np.random.default_rng(1)
    k = 1024
    rows = [rng.standard_normal(n).astype(np.float32) for n in
            (0, 1, 5, 1023, 1024, 1025, 1100, 2047, 4096, 8192, 8191, 12289)]
    _decode(torch, rows, k)


def test_topk_wide_uncached_rows(torch):
    """Rows longer than the shared-memory staging capacity (48K keys) are re-read; a row just below it stays staged."""
    rng = np.random.default_rng(2)
    rows = [rng.standard_normal(n).astype(np.float32) * 3 for n in (48 * 1024 - 3, 49153, 65536, 70001)]
    _decode(torch, rows, 2048)


def test_topk_narrow_ctas_many_rows(torch):
    """More rows than SMs with rows of up to 9000 keys: the 512-thread CTA shape."""
    rng = np.random.default_rng(3)
    rows = [rng.standard_normal(int(n)).astype(np.float32) for n in rng.integers(1, 9000, 400)]
    _decode(torch, rows, 512)


@pytest.mark.parametrize("n_rows", [8, 400])
def test_topk_heavy_ties_overflow_candidates(torch, n_rows):
    """Few distinct values: the candidate list overflows and the k-th value is tied."""
    rng = np.random.default_rng(4)
    rows = [rng.integers(0, 3, 9000).astype(np.float32) for _ in range(n_rows)]
    rows[0][:] = 1.5  # one all-equal row
    _decode(torch, rows, 1024)


def test_topk_unaligned_rows_and_signed_zero(torch):
    """Odd leading dimension (row starts off 16-byte boundaries); -0.0 equals +0.0."""
    rng = np.random.default_rng(5)
    rows = []
    for n in (3001, 3000, 2999, 5003):
        r = rng.standard_normal(n).astype(np.float32)
        z = rng.random(n) < 0.3
        r[z] = np.where(rng.random(z.sum()) < 0.5, np.float32(0.0), np.float32(-0.0))
        r[r < 0] = np.abs(r[r < 0]) * 0  # many zeros of both signs at the boundary
        rows.append(r)
    _decode(torch, rows, 1500, ld=5007)
    _decode(torch, rows, 1500, ld=5008)


@pytest.mark.parametrize("k", [1, 7, 4096])
def test_topk_extreme_k(torch, k):
    rng = np.random.default_rng(6)
    rows = [rng.standard_normal(n).astype(np.float32) for n in (10000, 4097, 300)]
    _decode(torch, rows, k)


def test_topk_causal_prefill_rows(torch):
    """Causal chunked prefill: each query sees a longer prefix; two sequences."""
    rng = np.random.default_rng(7)
    lens = np.array([3000, 2200], np.int32)
    nq = np.array([700, 300], np.int32)
    cu = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    for ld in (3004, 3005):
        mat = rng.standard_normal((int(nq.sum()), ld)).astype(np.float32)
        _, got = run_rows(torch, mat, 512, causal=1, cu=cu, seq_lens=lens)
        check(mat, got, lens, cu, 1, 512)


@pytest.mark.parametrize("lens,n_rows", [((8191, 8192, 100), 8), ((8193, 16384, 9000), 8),
                                         ((16385, 20000), 4), ((8192, 3000, 5000), 300)])
def test_topk_form_boundaries(torch, lens, n_rows):
    """Each launch shape on aligned rows: up to 8192 keys with few rows (registers: 1024
    threads, 8 keys each) or many rows (shared memory, 256 threads), up to 16384 keys (1024 x
    16), and longer rows (shared memory, 1024 threads); the many-row case mixes in tied rows
    whose candidates overflow."""
    rng = np.random.default_rng(8)
    rows = []
    for i in range(n_rows):
        n = lens[i % len(lens)]
        r = rng.standard_normal(n).astype(np.float32) * rng.uniform(0.1, 50)
        if i % 7 == 3:
            r = rng.integers(0, 4, n).astype(np.float32)
        rows.append(r)
    L = max(len(r) for r in rows)
    _decode(torch, rows, 1024, ld=(L + 3) // 4 * 4)


@pytest.mark.parametrize("ld_pad", [0, 1])
def test_topk_many_rows_narrowing_fallback(torch, ld_pad):
    """Many rows (the shared-memory form): rows where an outlier spreads the key range, rows
    half tied at one value, rows of two values only; both the aligned and the unaligned
    row layout."""
    rng = np.random.default_rng(9)
    rows = []
    for i in range(320):
        n = int(rng.integers(1100, 6000))
        r = (rng.standard_normal(n) * 3).astype(np.float32)
        if i % 3 == 0:
            r[rng.integers(0, n)] = np.float32(1e30)
        if i % 5 == 0:
            r[rng.random(n) < 0.5] = np.float32(0.75)
        if i % 7 == 0:
            r[:] = np.float32(-2.0)
            r[rng.integers(0, n, 50)] = np.float32(-1.0)
        rows.append(r)
    L = max(len(r) for r in rows)
    _decode(torch, rows, 1024, ld=(L + 3) // 4 * 4 + ld_pad)


@pytest.mark.parametrize("ld_pad", [0, 1])
def test_topk_many_long_rows(torch, ld_pad):
    """More rows than SMs, rows longer than 12K keys: aligned rows take the form that stages
    nothing and re-reads the row on each pass (several rows per SM), unaligned ones the generic
    form; rows with an outlier, rows of few distinct values (overflowing candidates)."""
    rng = np.random.default_rng(10)
    rows = []
    for i in range(200):
        n = int(rng.integers(12289, 20000))
        r = (rng.standard_normal(n) * 2).astype(np.float32)
        if i % 4 == 1:
            r[rng.integers(0, n)] = np.float32(-1e30)
        if i % 6 == 2:
            r = rng.integers(0, 5, n).astype(np.float32)
        rows.append(r)
    L = max(len(r) for r in rows)
    _decode(torch, rows, 2048, ld=(L + 3) // 4 * 4 + ld_pad)


@pytest.mark.parametrize("n_rows", [64, 300])
def test_topk_kth_value_repeated(torch, n_rows):
    """The k-th value has several copies and k cuts through them (few enough for the direct
    ranking): the lowest-indexed copies are taken, placed after the keys above it. Few rows
    (the register form) and many (the shared-memory linear form)."""
    rng = np.random.default_rng(11)
    k = 1024
    rows = []
    for i in range(n_rows):
        n = int(rng.integers(3000, 8000))
        r = rng.standard_normal(n).astype(np.float32)
        order = np.argsort(-r, kind="stable")
        v = r[order[k - 3]]                       # 3rd value from the cut
        lower = order[k + 10:]                    # positions holding smaller values
        r[rng.choice(lower, size=2 + i % 5, replace=False)] = v  # extra copies of v
        rows.append(r)
    L = max(len(r) for r in rows)
    _decode(torch, rows, k, ld=(L + 3) // 4 * 4)
