"""Oracle: plain fp64 CPU paged GQA attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import or call this module. The product path (the CUDA library and
its Python binding) never touches it, and this module imports nothing from the product.

What it computes (sources, by page and section):

* "Optimizing ASR Models to Transcribe 90-Minute Multi-Speaker Audio", *ASR Model Primer*
  (component table: Qwen3 text decoder, 28 layers, hidden 1024, GQA 16/8) and *Chunked
  Prefill for Long Audio* (the prompt is prefilled in 4096-token pieces, one per scheduling
  step, each building on the KV cache of the earlier pieces).
* "MOSS-Transcribe-Diarize" (SGLang-Omni cookbook), *Inference Pipeline* items 2-3 (prefill
  builds the KV cache; decode produces one token at a time against it) and *Optimization
  Strategies* (KV-cache management shared with the TTS stack).
* "MOSS-Transcribe-Diarize" README, *Quickstart* (attention must not be the quadratic-memory
  eager path on long recordings: nothing here depends on that, the oracle is allowed to be
  slow; only the kernels must be O(L) in memory).

The pages give no formula; attention itself is the textbook scaled-dot-product softmax
attention, and the paged layout, GQA grouping and log-sum-exp output are the plainest
readings of the problem statement (query tensor, per-layer K/V page pools, block tables,
ragged sequence lengths, softmax scale):

    s_t   = scale * <q, k_t>                         for every visible key t
    m     = max_t s_t
    l     = sum_t exp(s_t - m)
    o     = sum_t exp(s_t - m) * v_t / l
    lse   = m + ln(l)                                (natural log)

with key t of sequence b and KV head g stored at pool[block_table[b, t // P], t % P, g, :],
and query head h reading KV head h // (Hq / Hkv). A chunk of q_len queries whose sequence
holds seq_len keys (the chunk's own keys included) is aligned bottom-right: query i sees keys
0 .. seq_len - q_len + i. An empty key set gives o = 0 and lse = -inf.

Every function works in float64 on arrays widened from the exact input bytes (bf16 bit
patterns are widened exactly). There is no online softmax, no split of the key range and no
reordering of a row's reduction: a library matmul evaluates the score vectors of a group of
independent query rows of one (sequence, head) at once, then the definition above is applied
to each row as written.

The audio-text bridge that feeds those embeddings to the decoder ("Optimizing ASR Models to
Transcribe 90-Minute Multi-Speaker Audio", "ASR Model Primer", encoder bullet and component
table; "MOSS-Transcribe-Diarize 0.9B", "Model Architecture": 4x temporal merge + MLP adaptor)
concatenates every 4 consecutive encoder frames (d_model 1024 -> 4096) and applies
Linear -> SiLU -> Linear -> LayerNorm down to 1024. The hidden width is not stated; the plainest
reading, taken here, is Linear(4096 -> 1024), SiLU, Linear(1024 -> 1024), LayerNorm(1024) with
a learned scale and shift.

Parity pins: every function here is pinned by tests in ``tests/test_oracle_pins.py`` and
``tests/test_oracle_adaptor_pins.py`` against hand-worked fixtures (``tests/golden/``), closed
forms, invariants, brute force and an independent library.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "as_f64",
    "kv_head_of",
    "gather_keys",
    "visible_key_count",
    "attend_rows",
    "decode",
    "prefill",
    "kv_append",
    "merge_lse",
    "temporal_merge",
    "adaptor",
]


# ----------------------------------------------------------------------------------------------
# Small named steps (kept separate so each can be read, and tested, on its own).
# ----------------------------------------------------------------------------------------------
def as_f64(x) -> np.ndarray:
    """Widen an input array to float64 exactly.

    ``uint16`` / ``int16`` arrays are read as bf16 bit patterns (a bf16 value is the upper half
    of the fp32 with the same sign, exponent and leading mantissa bits), everything else is cast.
    """
    x = np.asarray(x)
    if x.dtype in (np.uint16, np.int16):
        bits = x.view(np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def kv_head_of(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    """GQA grouping: consecutive groups of Hq/Hkv query heads share one KV head."""
    group = num_q_heads // num_kv_heads
    return h // group


def gather_keys(pool, block_table_row, length: int, kv_head: int) -> np.ndarray:
    """Logical tokens 0..length-1 of one KV head of one sequence, as float64 [length, D].

    Token t lives in physical page ``block_table_row[t // P]`` at slot ``t % P`` (P = the
    pool's page size, its second axis). Block-table entries past ceil(length / P) are never
    read.
    """
    page_size = pool.shape[1]
    n_pages = -(-length // page_size)
    pages = np.asarray(block_table_row[:n_pages], dtype=np.int64)
    rows = pool[pages, :, kv_head, :]                      # [n_pages, P, D]
    return as_f64(rows).reshape(n_pages * page_size, pool.shape[3])[:length]


def visible_key_count(i: int, q_len: int, seq_len: int) -> int:
    """Keys seen by query i of a chunk of q_len queries in a sequence of seq_len keys.

    Bottom-right causal alignment: the chunk's tokens are the last q_len positions of the
    sequence, so query i sits at absolute position seq_len - q_len + i and sees keys
    0 .. seq_len - q_len + i.
    """
    return seq_len - q_len + i + 1


def attend_rows(Q, K, V, counts, scale: float):
    """Softmax attention of R query rows Q [R, D] over keys K [L, D] and values V [L, D].

    Row r sees only keys 0 .. counts[r]-1 (its causal prefix). The rows are independent: the
    matmul merely evaluates the R score vectors together. Returns (o [R, D], lse [R]) in
    float64; a row with counts[r] = 0 gives (zeros, -inf).
    """
    Q = as_f64(Q)
    counts = np.asarray(counts, dtype=np.int64)
    R, D = Q.shape
    n = int(counts.max()) if R else 0
    o = np.zeros((R, V.shape[1]), dtype=np.float64)
    lse = np.full(R, -math.inf)
    if n == 0:
        return o, lse
    s = scale * (Q @ K[:n].T)                                   # [R, n]
    s[np.arange(n)[None, :] >= counts[:, None]] = -math.inf     # keys outside the prefix
    live = counts > 0
    m = np.where(live, s.max(axis=1), 0.0)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    o[live] = (e[live] @ V[:n]) / l[live, None]
    lse[live] = m[live] + np.log(l[live])
    return o, lse


# ----------------------------------------------------------------------------------------------
# The four operations of the path.
# ----------------------------------------------------------------------------------------------
def _pool_map(fn, items, threads):
    if threads is None or threads <= 1 or len(items) <= 1:
        return [fn(it) for it in items]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))


def decode(q, k_pool, v_pool, block_table, seq_lens, scale: float, *, seqs=None, threads=None):
    """One decode step: each sequence's single query row against its whole cached KV.

    q [B, Hq, D]; pools [NP, P, Hkv, D]; block_table [B, stride]; seq_lens [B].
    Returns (o [B, Hq, D] float64, lse [B, Hq] float64). ``seqs`` limits the work to a subset
    of sequences (rows of the others are left as NaN). ``threads`` runs (sequence, head) items
    on a thread pool (numpy releases the GIL inside matmul and exp).
    """
    B, Hq, D = q.shape
    Hkv = k_pool.shape[2]
    o = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    seqs = range(B) if seqs is None else seqs

    def one(item):
        b, g = item
        L = int(seq_lens[b])
        K = gather_keys(k_pool, block_table[b], L, g)
        V = gather_keys(v_pool, block_table[b], L, g)
        res = []
        for h in range(Hq):
            if kv_head_of(h, Hq, Hkv) == g:
                oh, lh = attend_rows(q[b, h][None, :], K, V, [L], scale)
                res.append((h, (oh[0], lh[0])))
        return b, res

    for b, res in _pool_map(one, [(b, g) for b in seqs for g in range(Hkv)], threads):
        for h, (oh, lh) in res:
            o[b, h] = oh
            lse[b, h] = lh
    return o, lse


def prefill(q, cu_q_lens, k_pool, v_pool, block_table, seq_lens, scale: float, *,
            rows=None, threads=None, row_block=128):
    """Chunked prefill: every query row of every chunk against its causal prefix.

    q [Tq, Hq, D] packs the chunks of all sequences; chunk b holds rows
    cu_q_lens[b] .. cu_q_lens[b+1]-1 and its sequence holds seq_lens[b] keys, the chunk's own
    keys included (they are appended before attention). Returns (o [Tq, Hq, D], lse [Tq, Hq])
    in float64; ``rows`` restricts the work to a list of packed row indices (other rows NaN).
    """
    Tq, Hq, D = q.shape
    Hkv = k_pool.shape[2]
    cu = [int(c) for c in cu_q_lens]
    o = np.full((Tq, Hq, D), np.nan)
    lse = np.full((Tq, Hq), np.nan)
    want = None if rows is None else set(int(r) for r in rows)

    items = []
    for b in range(len(cu) - 1):
        chunk_rows = [r for r in range(cu[b], cu[b + 1]) if want is None or r in want]
        if chunk_rows:
            for g in range(Hkv):
                items.append((b, g, chunk_rows))

    def one(item):
        b, g, chunk_rows = item
        q_len = cu[b + 1] - cu[b]
        L = int(seq_lens[b])
        K = gather_keys(k_pool, block_table[b], L, g)
        V = gather_keys(v_pool, block_table[b], L, g)
        res = []
        for h in range(Hq):
            if kv_head_of(h, Hq, Hkv) != g:
                continue
            for i0 in range(0, len(chunk_rows), row_block):
                blk = chunk_rows[i0:i0 + row_block]
                counts = [visible_key_count(r - cu[b], q_len, L) for r in blk]
                ob, lb = attend_rows(q[blk, h], K, V, counts, scale)
                res.extend((r, h, (ob[k], lb[k])) for k, r in enumerate(blk))
        return res

    for res in _pool_map(one, items, threads):
        for r, h, (oh, lh) in res:
            o[r, h] = oh
            lse[r, h] = lh
    return o, lse


def kv_append(k_new, v_new, cu_new_lens, start_pos, block_table, k_pool, v_pool):
    """Write new tokens' K/V rows into the page pools; returns the updated (copied) pools.

    New token j of sequence b (packed row cu_new_lens[b] + j of k_new/v_new [T, Hkv, D]) has
    logical position start_pos[b] + j and goes to page block_table[b, pos // P], slot pos % P.
    The copy is bit-for-bit (the pools keep their dtype); nothing else in the pools changes.
    """
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    P = k_pool.shape[1]
    cu = [int(c) for c in cu_new_lens]
    for b in range(len(cu) - 1):
        for j in range(cu[b + 1] - cu[b]):
            pos = int(start_pos[b]) + j
            page = int(block_table[b, pos // P])
            k_out[page, pos % P] = k_new[cu[b] + j]
            v_out[page, pos % P] = v_new[cu[b] + j]
    return k_out, v_out


def merge_lse(o_parts, lse_parts):
    """Combine partial attention results over disjoint key sets.

    o_parts [S, ..., D] (each part normalised by its own softmax denominator) and lse_parts
    [S, ...]. Returns (o [..., D], lse [...]) in float64:

        lse = ln sum_s exp(lse_s),   o = sum_s exp(lse_s - lse) * o_s

    Parts with lse = -inf (empty key sets) carry weight 0; if every part is empty the result
    is o = 0, lse = -inf.
    """
    o_parts = as_f64(o_parts)
    lse_parts = as_f64(lse_parts)
    present = np.isfinite(lse_parts)
    m = np.where(present, lse_parts, -np.inf).max(axis=0)
    any_part = np.isfinite(m)
    m_safe = np.where(any_part, m, 0.0)
    w = np.where(present, np.exp(np.where(present, lse_parts, 0.0) - m_safe), 0.0)
    total = w.sum(axis=0)
    contrib = np.where(present[..., None], w[..., None] * np.where(present[..., None], o_parts, 0.0), 0.0)
    safe_total = np.where(any_part, total, 1.0)
    o = np.where(any_part[..., None], contrib.sum(axis=0) / safe_total[..., None], 0.0)
    lse = np.where(any_part, m_safe + np.log(safe_total), -np.inf)
    return o, lse


# ----------------------------------------------------------------------------------------------
# Audio-text bridge: 4x temporal merge + adaptor MLP.
# ----------------------------------------------------------------------------------------------
def temporal_merge(frames, factor: int = 4):
    """[T_enc, d] encoder frames -> [T_enc / factor, factor * d]: row t is frames
    factor*t .. factor*t + factor - 1 laid side by side."""
    frames = as_f64(frames)
    T_enc, d = frames.shape
    assert T_enc % factor == 0, "the frame count must be a multiple of the merge factor"
    return np.concatenate([frames[k::factor] for k in range(factor)], axis=1)


def adaptor(frames, w1, b1, w2, b2, gamma, beta, eps: float = 1e-5):
    """Audio embeddings for the decoder: LayerNorm(SiLU(x W1^T + b1) W2^T + b2), x the
    4x-merged frames. w1 [H, 4d], w2 [E, H] as (out, in); returns float64 [T, E]."""
    x = temporal_merge(frames)
    h = x @ as_f64(w1).T + as_f64(b1)
    h = h / (1.0 + np.exp(-h))                       # SiLU(h) = h * sigmoid(h)
    y = h @ as_f64(w2).T + as_f64(b2)
    mu = y.mean(axis=1, keepdims=True)
    var = ((y - mu) ** 2).mean(axis=1, keepdims=True)  # biased variance
    return (y - mu) / np.sqrt(var + eps) * as_f64(gamma) + as_f64(beta)
