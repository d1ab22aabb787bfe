"""Seeded synthetic inputs for the indexer hot path.

This module only draws numbers: it holds none of the method's arithmetic (no norm, RoPE,
quantisation or scoring). The tests feed the same arrays to the CUDA library and to the
CPU oracle; the benchmark feeds them to the CUDA library.

Recipe (numpy PCG64, ``SeedSequence(seed).spawn``, one sub-stream per tensor):
  * bf16 tensors: float32 N(0, 1) draws rounded to bf16 (round to nearest even) and kept
    as uint16 bit patterns;
  * head weights: float32 N(0, 1/H);
  * physical pages: ``rng.permutation(pool_pages)``; each sequence takes the next
    ceil(len / page_size) pages of that permutation, in order;
  * RoPE table (an input of both sides): cos/sin of pos * 10000^(-i/32), i = 0..31,
    evaluated in float64 and rounded to float32, laid out [max_pos][cos 0..31, sin 0..31].

The shapes follow the pages' isolated-scorer and pre-processing workloads (see the config
builders below); no public dataset is involved.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

MXFP4, FP8 = 0, 1
ROPE_NONE, ROPE_NEOX, ROPE_INTERLEAVED = 0, 1, 2


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even. Inputs are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def rope_table(max_pos: int, base: float = 10000.0) -> np.ndarray:
    i = np.arange(32, dtype=np.float64)
    inv_freq = base ** (-i / 32.0)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def page_bytes(dtype: int, page_size: int) -> int:
    """Bytes of one page: 68 B/token for MXFP4, 132 B/token for FP8 (format sizes only)."""
    return (68 if dtype == MXFP4 else 132) * page_size


@dataclasses.dataclass
class Workload:
    name: str
    dtype: int
    B: int
    H: int
    page_size: int
    pool_pages: int             # physical pages in the pool view
    base_offset_pages: int      # pages of slack in front of the pool view (nonzero offset)
    page_stride: int            # bytes between physical pages
    seq_lens_k: np.ndarray      # int32 [B], keys per sequence
    cu_seqlens_q: np.ndarray    # int32 [B+1]
    page_table: np.ndarray      # int32 [B, max_pages]
    causal: int
    topk: int
    # K store inputs
    k: np.ndarray               # uint16 [N, 128]
    slot_mapping: np.ndarray    # int64 [N]
    k_positions: np.ndarray     # int32 [N]
    k_rope: int
    k_norm: int
    step_rows: np.ndarray       # int64: K rows stored inside a timed step (rest = setup)
    # Q quant inputs
    q: np.ndarray               # uint16 [T, H, 128]
    q_positions: np.ndarray     # int32 [T]
    q_rope: int
    w_in: np.ndarray            # float32 [T, H]
    softmax_scale: float
    head_scale: float
    cos_sin: np.ndarray         # float32 [max_pos, 64]
    ld_logits: int
    note: str = ""

    @property
    def T(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def n_k_rows(self) -> int:
        return int(self.k.shape[0])

    def visible(self) -> np.ndarray:
        """Keys visible to each query (int64 [T]); same rule as the library's."""
        out = np.empty(self.T, np.int64)
        for b in range(self.B):
            lo, hi = int(self.cu_seqlens_q[b]), int(self.cu_seqlens_q[b + 1])
            nq = hi - lo
            for i in range(nq):
                v = int(self.seq_lens_k[b]) - nq + i + 1 if self.causal else int(self.seq_lens_k[b])
                out[lo + i] = min(max(v, 0), int(self.seq_lens_k[b]))
        return out

    def pairs(self) -> int:
        return int(self.visible().sum())

    def pool_nbytes(self) -> int:
        return (self.pool_pages + self.base_offset_pages) * self.page_stride


def _streams(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def _assign_pages(rng, pool_pages, lens, P):
    perm = rng.permutation(pool_pages).astype(np.int32)
    need = [(int(L) + P - 1) // P for L in lens]
    assert sum(need) <= pool_pages, "pool too small"
    max_pages = max(need)
    pt = np.full((len(lens), max_pages), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[o:o + n]
        o += n
    return pt


def _slots(pt, lens, P):
    """slot of token s of sequence b = page_table[b, s // P] * P + s % P (int64)."""
    out = []
    for b, L in enumerate(lens):
        s = np.arange(int(L), dtype=np.int64)
        out.append(pt[b, s // P].astype(np.int64) * P + s % P)
    return np.concatenate(out)


def _ld(n):
    """Logits row stride: the longest row rounded up to 4 floats (16-byte aligned rows)."""
    return (int(n) + 3) // 4 * 4


def _normal_bf16(rng, shape):
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def make(name: str, seed: int = 0, **over) -> Workload:
    return BUILDERS[name](seed, **over)


def tiny_decode(seed=0, **over) -> Workload:
    """Tiny MXFP4 decode: 2 sequences (256 and 193 keys), H=4, page 64, a shuffled pool
    of 16 physical pages placed one page after the start of the buffer; full K store
    (LayerNorm + NeoX RoPE); top-k 32."""
    rk, rq, rw, rp = _streams(seed, 4)
    B, H, P, pool = 2, 4, 64, 16
    lens = np.array(over.get("lens", [256, 193]), np.int32)
    pt = _assign_pages(rp, pool, lens, P)
    slots = _slots(pt, lens, P)
    kpos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    max_pos = int(lens.max())
    return Workload(
        name="tiny_decode_mxfp4", dtype=MXFP4, B=B, H=H, page_size=P, pool_pages=pool,
        base_offset_pages=1, page_stride=page_bytes(MXFP4, P), seq_lens_k=lens,
        cu_seqlens_q=np.arange(B + 1, dtype=np.int32), page_table=pt, causal=0, topk=32,
        k=_normal_bf16(rk, (int(lens.sum()), 128)), slot_mapping=slots, k_positions=kpos,
        k_rope=ROPE_NEOX, k_norm=1, step_rows=np.cumsum(lens).astype(np.int64) - 1,
        q=_normal_bf16(rq, (B, H, 128)), q_positions=(lens - 1).astype(np.int32),
        q_rope=ROPE_NEOX, w_in=(rw.standard_normal((B, H), dtype=np.float32)
                                 / np.float32(math.sqrt(H))).astype(np.float32),
        softmax_scale=1.0, head_scale=1.0, cos_sin=rope_table(max_pos), ld_logits=_ld(lens.max()),
    )


def decode_b64(seed=0, B=64, ctx=8192, H=32, **over) -> Workload:
    """MXFP4 decode: B sequences x 1 query, H=32, 8192 keys each, page 128 from a
    permuted pool of 4608 pages; 1% of the K rows scaled x20 (outlier blocks); K stored
    with NeoX RoPE at position s but without LayerNorm (the norm would undo the x20 rows
    that exercise the E8M0 scales); Q RoPE'd at the last position; top-k 1024."""
    rk, rq, rw, rp, ro = _streams(seed, 5)
    P = 128
    pool = max(4608, B * ((ctx + P - 1) // P))
    lens = np.full(B, ctx, np.int32)
    pt = _assign_pages(rp, pool, lens, P)
    slots = _slots(pt, lens, P)
    N = int(lens.sum())
    kf = rk.standard_normal((N, 128), dtype=np.float32)
    n_out = max(1, N // 100)
    rows = ro.choice(N, size=n_out, replace=False)
    kf[rows] *= np.float32(20.0)
    return Workload(
        name=f"decode_mxfp4_b{B}_h{H}_{ctx}", dtype=MXFP4, B=B, H=H, page_size=P,
        pool_pages=pool, base_offset_pages=0, page_stride=page_bytes(MXFP4, P),
        seq_lens_k=lens, cu_seqlens_q=np.arange(B + 1, dtype=np.int32), page_table=pt,
        causal=0, topk=1024, k=bf16_bits(kf), slot_mapping=slots,
        k_positions=np.concatenate([np.arange(L, dtype=np.int32) for L in lens]),
        k_rope=ROPE_NEOX, k_norm=0, step_rows=np.cumsum(lens).astype(np.int64) - 1,
        q=_normal_bf16(rq, (B, H, 128)), q_positions=(lens - 1).astype(np.int32),
        q_rope=ROPE_NEOX,
        w_in=(rw.standard_normal((B, H), dtype=np.float32) / np.float32(math.sqrt(H))),
        softmax_scale=1.0, head_scale=1.0, cos_sin=rope_table(ctx), ld_logits=_ld(ctx),
    )


def prefill_8k(seed=0, T=8192, H=32, **over) -> Workload:
    """MXFP4 causal prefill: one sequence of T queries against its own T paged keys
    (page 128, shuffled), H=32; K through the full store (LayerNorm + NeoX RoPE at
    position s), query i RoPE'd at position i; top-k 1024."""
    rk, rq, rw, rp = _streams(seed, 4)
    P = 128
    lens = np.array([T], np.int32)
    pool = (T + P - 1) // P
    pt = _assign_pages(rp, pool, lens, P)
    slots = _slots(pt, lens, P)
    return Workload(
        name=f"prefill_mxfp4_{T}q_h{H}", dtype=MXFP4, B=1, H=H, page_size=P, pool_pages=pool,
        base_offset_pages=0, page_stride=page_bytes(MXFP4, P), seq_lens_k=lens,
        cu_seqlens_q=np.array([0, T], np.int32), page_table=pt, causal=1, topk=1024,
        k=_normal_bf16(rk, (T, 128)), slot_mapping=slots,
        k_positions=np.arange(T, dtype=np.int32), k_rope=ROPE_NEOX, k_norm=1,
        step_rows=np.arange(T, dtype=np.int64),
        q=_normal_bf16(rq, (T, H, 128)), q_positions=np.arange(T, dtype=np.int32),
        q_rope=ROPE_NEOX,
        w_in=(rw.standard_normal((T, H), dtype=np.float32) / np.float32(math.sqrt(H))),
        softmax_scale=1.0, head_scale=1.0, cos_sin=rope_table(T), ld_logits=_ld(T),
    )


def decode_compressed(seed=0, B=256, H=64, **over) -> Workload:
    """MXFP4 decode over a compressed indexer (compress ratio 4): raw contexts uniform in
    [1024, 9472] give raw//4 entries (256..2368) in 64-entry pages from a shuffled pool of
    B*37 pages; K rows go through the full store (LayerNorm + NeoX RoPE) at position 4j+3;
    Q is RoPE'd at position raw-1; softmax scale 128^-0.5 folded; top-k 1024."""
    rk, rq, rw, rp, rl = _streams(seed, 5)
    P, ratio = 64, 4
    raw = rl.integers(over.get("raw_lo", 1024), over.get("raw_hi", 9472) + 1, size=B)
    lens = (raw // ratio).astype(np.int32)
    pool = B * 37
    pt = _assign_pages(rp, pool, lens, P)
    slots = _slots(pt, lens, P)
    kpos = np.concatenate([ratio * np.arange(L, dtype=np.int32) + (ratio - 1) for L in lens])
    max_pos = int(max(raw.max(), kpos.max() + 1))
    return Workload(
        name=f"decode_mxfp4_compressed_b{B}_h{H}", dtype=MXFP4, B=B, H=H, page_size=P,
        pool_pages=pool, base_offset_pages=0, page_stride=page_bytes(MXFP4, P),
        seq_lens_k=lens, cu_seqlens_q=np.arange(B + 1, dtype=np.int32), page_table=pt,
        causal=0, topk=1024, k=_normal_bf16(rk, (int(lens.sum()), 128)), slot_mapping=slots,
        k_positions=kpos, k_rope=ROPE_NEOX, k_norm=1,
        step_rows=np.cumsum(lens).astype(np.int64) - 1,
        q=_normal_bf16(rq, (B, H, 128)), q_positions=(raw - 1).astype(np.int32),
        q_rope=ROPE_NEOX,
        w_in=(rw.standard_normal((B, H), dtype=np.float32) / np.float32(math.sqrt(H))),
        softmax_scale=float(128 ** -0.5), head_scale=1.0, cos_sin=rope_table(max_pos),
        ld_logits=_ld(lens.max()),
    )


def prefill_fp8(seed=0, B=8, cached=28672, new=4096, H=32, **over) -> Workload:
    """FP8 batched causal prefill: B sequences of `new` tokens on top of `cached` keys,
    e4m3 K cache with per-token fp32 scale, page 64, interleaved RoPE, LayerNorm on K,
    per-token-group (128) FP8 Q with the scale folded into the weights; top-k 2048.
    Cached keys are stored during set-up; the new keys are stored inside the step."""
    rk, rq, rw, rp = _streams(seed, 4)
    P = 64
    L = cached + new
    lens = np.full(B, L, np.int32)
    pool = B * ((L + P - 1) // P)
    pt = _assign_pages(rp, pool, lens, P)
    slots = _slots(pt, lens, P)
    kpos = np.concatenate([np.arange(L, dtype=np.int32) for _ in range(B)])
    step_rows = np.concatenate([b * L + cached + np.arange(new, dtype=np.int64) for b in range(B)])
    qpos = np.concatenate([cached + np.arange(new, dtype=np.int32) for _ in range(B)])
    return Workload(
        name=f"prefill_fp8_b{B}_{new}on{cached}", dtype=FP8, B=B, H=H, page_size=P,
        pool_pages=pool, base_offset_pages=0, page_stride=page_bytes(FP8, P), seq_lens_k=lens,
        cu_seqlens_q=(np.arange(B + 1) * new).astype(np.int32), page_table=pt, causal=1,
        topk=2048, k=_normal_bf16(rk, (B * L, 128)), slot_mapping=slots, k_positions=kpos,
        k_rope=ROPE_INTERLEAVED, k_norm=1, step_rows=step_rows,
        q=_normal_bf16(rq, (B * new, H, 128)), q_positions=qpos, q_rope=ROPE_INTERLEAVED,
        w_in=(rw.standard_normal((B * new, H), dtype=np.float32) / np.float32(math.sqrt(H))),
        softmax_scale=1.0, head_scale=1.0, cos_sin=rope_table(L), ld_logits=_ld(L),
    )


@dataclasses.dataclass
class CompressWork:
    """Inputs of the compressed K store: raw rows of several sequences back to back, one
    entry per compress-ratio boundary token of each sequence."""
    name: str
    dtype: int
    ratio: int
    page_size: int
    pool_pages: int
    page_stride: int
    raw_lens: np.ndarray        # int64 [B], raw rows per sequence
    k_raw: np.ndarray           # uint16 [N_raw, row_stride] (bf16; columns past 128 unused)
    gate: np.ndarray            # uint16 [N_raw, row_stride]
    boundary: np.ndarray        # int64 [E], raw row of each entry's boundary token
    first: np.ndarray           # int64 [E], first raw row of the entry's sequence
    slot_mapping: np.ndarray    # int64 [E]
    positions: np.ndarray       # int32 [E], boundary position within its sequence
    rope: int
    norm: int                   # 0 none, 1 LayerNorm, 2 RMSNorm
    gamma: np.ndarray           # float32 [128]
    cos_sin: np.ndarray

    @property
    def n_entries(self) -> int:
        return int(self.boundary.shape[0])


def compress_work(seed=0, raw_lens=(37, 64, 130), ratio=4, page_size=64, dtype=MXFP4,
                  rope=ROPE_NEOX, norm=2, row_stride=128, name=None, spare_pages=1) -> CompressWork:
    """Raw K and gate rows bf16 N(0, 1); per sequence the entries are its tokens
    r*j + r - 1 (j = 0 .. len//r - 1; a ragged tail of fewer than r tokens has none), stored
    in pages of a shuffled pool in entry order, RoPE'd at that in-sequence position; RMSNorm
    weight uniform in [0.5, 1.5]."""
    rk, rg, rp, rw = _streams(seed, 4)
    lens = np.asarray(raw_lens, np.int64)
    n = int(lens.sum())
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    ents = (lens // ratio).astype(np.int32)
    P = page_size
    pool = int(sum((int(e) + P - 1) // P for e in ents)) + spare_pages
    pt = _assign_pages(rp, pool, ents, P) if ents.sum() > 0 else np.zeros((len(lens), 1), np.int32)
    slots = _slots(pt, ents, P) if ents.sum() > 0 else np.zeros(0, np.int64)
    j = [np.arange(int(e), dtype=np.int64) for e in ents]
    boundary = np.concatenate([starts[b] + ratio * j[b] + ratio - 1 for b in range(len(lens))])
    first = np.concatenate([np.full(int(ents[b]), starts[b], np.int64) for b in range(len(lens))])
    positions = np.concatenate([(ratio * j[b] + ratio - 1) for b in range(len(lens))]).astype(np.int32)
    k_raw = np.zeros((n, row_stride), np.uint16)
    gate = np.zeros((n, row_stride), np.uint16)
    k_raw[:, :128] = _normal_bf16(rk, (n, 128))
    gate[:, :128] = _normal_bf16(rg, (n, 128))
    max_pos = int(max(lens.max(), 1))
    return CompressWork(
        name=name or f"compress_r{ratio}_{len(lens)}seq_{n}raw", dtype=dtype, ratio=ratio,
        page_size=P, pool_pages=pool, page_stride=page_bytes(dtype, P), raw_lens=lens,
        k_raw=k_raw, gate=gate, boundary=boundary.astype(np.int64), first=first,
        slot_mapping=slots.astype(np.int64), positions=positions, rope=rope, norm=norm,
        gamma=rw.uniform(0.5, 1.5, 128).astype(np.float32), cos_sin=rope_table(max_pos))


def compress_b256(seed=0, B=256, **over) -> CompressWork:
    """The compressed-indexer decode workload's contexts through the compressor: B raw
    contexts uniform in [1024, 9472] tokens, ratio 4, 64-entry MXFP4 pages, NeoX RoPE,
    RMSNorm (the whole context compressed, as a prefill of those sequences does)."""
    rl = _streams(seed, 5)[4]
    raw = rl.integers(over.pop("raw_lo", 1024), over.pop("raw_hi", 9472) + 1, size=B)
    return compress_work(seed, raw_lens=raw, ratio=4, page_size=64, dtype=MXFP4, rope=ROPE_NEOX,
                         norm=2, name=f"compress_mxfp4_r4_b{B}_raw1024-9472", **over)


def candidate_blocks(wl, seed=0, n_blocks=16, messy=False):
    """A stand-in for the two-level indexer's first level: per query, n_blocks distinct block
    ids (blocks of page_size keys) drawn uniformly from its visible blocks, always including
    the last one (the local window); all visible blocks when there are fewer. messy: the
    lists also carry repeats and ids naming no visible block (negative, past the visible
    blocks, past the sequence) in shuffled order. Returns (cand int32 [T, stride], n_cand
    int32 [T], max_cand)."""
    rng = _streams(seed + 7919, 1)[0]
    vis = wl.visible()
    P = wl.page_size
    rows = []
    for t in range(wl.T):
        nb = int((vis[t] + P - 1) // P)
        if nb == 0:
            ids = np.zeros(0, np.int64)
        elif nb <= n_blocks:
            ids = np.arange(nb)
        else:
            ids = np.concatenate([rng.choice(nb - 1, n_blocks - 1, replace=False), [nb - 1]])
        if messy and nb > 0:
            junk = np.array([-1, nb, nb + 5, -(1 << 20), 1 << 28])
            ids = np.concatenate([ids, rng.choice(ids, 3), rng.choice(junk, 3)])
        rows.append(rng.permutation(ids).astype(np.int32))
    max_cand = max(1, max(len(r) for r in rows))
    cand = np.full((wl.T, max_cand + 3), -1, np.int32)
    n_cand = np.zeros(wl.T, np.int32)
    for t, r in enumerate(rows):
        cand[t, :len(r)] = r
        n_cand[t] = len(r)
    return cand, n_cand, max_cand


BUILDERS = {
    "tiny_decode": tiny_decode,
    "decode_b64": decode_b64,
    "prefill_8k": prefill_8k,
    "decode_compressed": decode_compressed,
    "prefill_fp8": prefill_fp8,
}
