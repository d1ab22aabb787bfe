"""Test helpers: run a workload through the CUDA library and through the oracle, and the
comparison rules (bit-exact bytes; logits within 1e-4 * row max with cosine >= 0.999999;
top-k sets equal up to ties within that tolerance of the k-th value)."""
from __future__ import annotations

import numpy as np

import oracle as O
from sparse_attention_indexer_mqa_gb300 import workloads as W

LOGIT_RTOL = 1e-4        # |gpu - exact| <= 1e-4 * max_s |exact[t, s]| per row
COSINE_MIN = 0.999999


# ------------------------------------------------------------------------------ oracle side

def oracle_store(wl, rows=None, pool=None):
    """Oracle K store of all rows (or `rows`) into a fresh zeroed pool (with the slack
    pages in front); returns the whole pool buffer (uint8)."""
    if pool is None:
        pool = np.zeros(wl.pool_nbytes(), np.uint8)
    view = pool[wl.base_offset_pages * wl.page_stride:]
    sel = slice(None) if rows is None else rows
    bad = O.k_store(view, wl.k[sel], wl.slot_mapping[sel], wl.k_positions[sel], wl.cos_sin,
                    wl.k_rope, wl.k_norm, wl.dtype, wl.pool_pages, wl.page_size, wl.page_stride)
    assert bad == 0
    return pool


def oracle_q(wl):
    return O.q_quant(wl.q, wl.q_positions, wl.cos_sin, wl.q_rope, wl.w_in, wl.softmax_scale,
                     wl.head_scale, wl.dtype)


def oracle_logits(wl, pool, qc, qs, w, rows=None):
    view = pool[wl.base_offset_pages * wl.page_stride:]
    return O.mqa_logits(qc, qs, w, wl.dtype, view, wl.pool_pages, wl.page_size, wl.page_stride,
                        wl.page_table, wl.seq_lens_k, wl.cu_seqlens_q, wl.causal, wl.ld_logits,
                        rows=rows)


def oracle_topk(wl, logits, rows=None):
    return O.topk(np.nan_to_num(logits, nan=-np.inf), wl.seq_lens_k, wl.cu_seqlens_q,
                  wl.causal, wl.topk, rows=rows)


# ------------------------------------------------------------------------------ GPU side

class Dev:
    """Device copies of a workload's inputs and the outputs of each step."""

    def __init__(self, wl, device="cuda"):
        import torch
        self.wl = wl
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.k = t(wl.k.view(np.int16))
        self.slot = t(wl.slot_mapping)
        self.kpos = t(wl.k_positions)
        self.cos_sin = t(wl.cos_sin)
        self.q = t(wl.q.view(np.int16))
        self.qpos = t(wl.q_positions)
        self.w_in = t(wl.w_in)
        self.page_table = t(wl.page_table)
        self.seq_lens_k = t(wl.seq_lens_k)
        self.cu = t(wl.cu_seqlens_q)
        self.pool_buf = torch.zeros(wl.pool_nbytes(), dtype=torch.uint8, device=device)
        off = wl.base_offset_pages * wl.page_stride
        self.pool = self.pool_buf[off:]
        T, H = wl.T, wl.H
        Hq = (H + 7) // 8 * 8
        if wl.dtype == W.MXFP4:
            self.q_codes = torch.full((T, Hq, 64), 0xEE, dtype=torch.uint8, device=device)
            self.q_scales = torch.full((T, 512), 0xEE, dtype=torch.uint8, device=device)
        else:
            self.q_codes = torch.full((T, Hq, 128), 0xEE, dtype=torch.uint8, device=device)
            self.q_scales = torch.zeros((T, H), dtype=torch.float32, device=device)
        self.w = torch.zeros((T, H), dtype=torch.float32, device=device)
        self.logits = torch.full((T, wl.ld_logits), float("nan"), dtype=torch.float32,
                                 device=device)
        self.topk = torch.full((T, wl.topk), -7, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def store(self, rows=None):
        from sparse_attention_indexer_mqa_gb300 import binding as Bn
        import torch
        wl = self.wl
        if rows is None:
            k, slot, pos = self.k, self.slot, self.kpos
        else:
            r = torch.from_numpy(np.asarray(rows, np.int64)).to(self.k.device)
            k, slot, pos = self.k[r].contiguous(), self.slot[r].contiguous(), self.kpos[r].contiguous()
        Bn.idx_k_store(k, slot, pos if wl.k_rope else None, self.cos_sin if wl.k_rope else None,
                       wl.k_rope, wl.k_norm, wl.dtype, self.pool, wl.pool_pages, wl.page_size,
                       wl.page_stride, dev_status=self.status)

    def prep(self):
        """K store and Q quant in one launch (idx_qk_prep)."""
        from sparse_attention_indexer_mqa_gb300 import binding as Bn
        wl = self.wl
        Bn.idx_qk_prep(self.k, self.slot, self.kpos if wl.k_rope else None, wl.k_rope, wl.k_norm,
                       self.pool, wl.pool_pages, wl.page_size, wl.page_stride, self.q,
                       self.qpos if wl.q_rope else None, wl.q_rope, self.w_in, wl.softmax_scale,
                       wl.head_scale, self.q_codes, self.q_scales, self.w,
                       self.cos_sin if (wl.k_rope or wl.q_rope) else None, wl.dtype,
                       dev_status=self.status)

    def quant(self):
        from sparse_attention_indexer_mqa_gb300 import binding as Bn
        wl = self.wl
        Bn.idx_q_quant(self.q, self.qpos if wl.q_rope else None,
                       self.cos_sin if wl.q_rope else None, wl.q_rope, self.w_in,
                       wl.softmax_scale, wl.head_scale, wl.dtype, self.q_codes, self.q_scales,
                       self.w, dev_status=self.status)

    def score(self, page_table=None, workspace=None):
        from sparse_attention_indexer_mqa_gb300 import binding as Bn
        wl = self.wl
        nq = np.diff(wl.cu_seqlens_q)
        Bn.idx_mqa_logits_paged(self.q_codes, self.q_scales, self.w, wl.dtype, self.pool,
                                wl.pool_pages, wl.page_size, wl.page_stride,
                                self.page_table if page_table is None else page_table,
                                self.seq_lens_k, self.cu, wl.causal, int(nq.max()),
                                int(wl.seq_lens_k.max()), self.logits, dev_status=self.status,
                                workspace=workspace)

    def select(self):
        from sparse_attention_indexer_mqa_gb300 import binding as Bn
        wl = self.wl
        Bn.idx_topk(self.logits, self.seq_lens_k, self.cu, wl.causal, int(wl.seq_lens_k.max()),
                    wl.topk, self.topk, dev_status=self.status)

    def select_fused(self, out=None, workspace=None):
        """Scorer and top-k in one launch (idx_mqa_topk_paged) into `out` (default: a fresh
        buffer); returns (out, workspace)."""
        from sparse_attention_indexer_mqa_gb300 import binding as Bn
        import torch
        wl = self.wl
        nq = np.diff(wl.cu_seqlens_q)
        max_q, max_k = int(nq.max()), int(wl.seq_lens_k.max())
        if workspace is None:
            n = Bn.idx_mqa_topk_workspace_bytes(wl.T, wl.H, wl.B, max_q, max_k)
            workspace = torch.zeros(max(n, 256), dtype=torch.uint8, device=self.k.device)
        if out is None:
            out = torch.full((wl.T, wl.topk), -7, dtype=torch.int32, device=self.k.device)
        Bn.idx_mqa_topk_paged(self.q_codes, self.q_scales, self.w, wl.dtype, self.pool, wl.pool_pages,
                              wl.page_size, wl.page_stride, self.page_table, self.seq_lens_k, self.cu,
                              wl.causal, max_q, max_k, wl.topk, out, workspace, dev_status=self.status)
        return out, workspace

    def run_all(self):
        self.store()
        self.quant()
        self.score()
        self.select()

    def host(self, name):
        import torch
        torch.cuda.synchronize()
        return getattr(self, name).cpu().numpy()


# ------------------------------------------------------------------------------ Q layout

def q_image_to_plain(codes, scales, H, dtype):
    """The library's Q output (tensor-core image per query, see include/idx.h) mapped to
    the oracle's plain layout: MXFP4 codes [T][H][64] + scales [T][H][4]; FP8 codes
    [T][H][128]. Also checks the documented padding (heads H..Hq-1: zero codes, scale
    bytes 127)."""
    T = codes.shape[0]
    Hq = (H + 7) // 8 * 8
    kc = 4 if dtype == W.MXFP4 else 8          # 16-byte chunks per head row
    img = codes.reshape(T, Hq // 8, kc, 8, 16)  # [t][group][chunk][head in group][byte]
    plain = img.transpose(0, 1, 3, 2, 4).reshape(T, Hq, kc * 16)
    assert not plain[:, H:].any(), "padding heads must be zero"
    if dtype != W.MXFP4:
        return plain[:, :H], None
    h = np.arange(Hq)
    atom = scales.reshape(T, 512)
    idx = (h % 32)[:, None] * 16 + (h // 32)[:, None] * 4 + np.arange(4)[None, :]
    sc = atom[:, idx]                            # [T][Hq][4]
    assert (sc[:, H:] == 127).all(), "padding heads must have scale byte 127"
    return plain[:, :H], sc[:, :H]


# ------------------------------------------------------------------------------ comparisons

def assert_logits_close(got, exact, vis, rows=None, label=""):
    """got: fp32 [n, ld] (rows already selected), exact: fp64 [n, ld]."""
    n = got.shape[0]
    worst = 0.0
    for r in range(n):
        v = int(vis[r])
        if v == 0:
            continue
        e = exact[r, :v]
        g = got[r, :v].astype(np.float64)
        assert np.isfinite(g).all(), f"{label} row {r}: non-finite logits"
        scale = np.abs(e).max()
        err = np.abs(g - e).max()
        worst = max(worst, err / scale if scale > 0 else err)
        assert err <= LOGIT_RTOL * scale + 1e-30, \
            f"{label} row {r}: max err {err:.3e} > {LOGIT_RTOL} * {scale:.3e}"
        den = np.linalg.norm(g) * np.linalg.norm(e)
        if den > 0:
            cos = float(g @ e / den)
            assert cos >= COSINE_MIN, f"{label} row {r}: cosine {cos:.9f}"
    return worst


def assert_topk_valid(got_idx, exact_logits, gpu_logits, vis, k, label=""):
    """GPU top-k set vs the exact scores: same size, no duplicates, in range, padding only at
    the tail, and every index in the symmetric difference with the exact set within
    tolerance of the exact k-th value. Also: the set is an exact top-k of the GPU's own
    fp32 logits."""
    for r in range(got_idx.shape[0]):
        v = int(vis[r])
        g = got_idx[r]
        n = min(k, v)
        assert (g[n:] == -1).all(), f"{label} row {r}: bad padding"
        sel = g[:n]
        assert (sel >= 0).all() and (sel < v).all(), f"{label} row {r}: index out of range"
        assert len(np.unique(sel)) == n, f"{label} row {r}: duplicates"
        if v <= k:
            assert set(sel.tolist()) == set(range(v))
            continue
        e = exact_logits[r, :v]
        order = np.argsort(-e, kind="stable")
        exact_set = set(order[:k].tolist())
        kth = e[order[k - 1]]
        tol = LOGIT_RTOL * np.abs(e).max()
        for i in exact_set.symmetric_difference(sel.tolist()):
            assert abs(e[i] - kth) <= tol, f"{label} row {r}: index {i} off by {e[i] - kth:.3e}"
        # exactness on the GPU's own values: min selected >= max unselected
        gl = gpu_logits[r, :v]
        mask = np.zeros(v, bool)
        mask[sel] = True
        assert gl[mask].min() >= gl[~mask].max(), f"{label} row {r}: not a top-k of its input"
