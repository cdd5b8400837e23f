"""Seeded synthetic inputs for paged GQA attention and the audio-text adaptor.

This module is shared by the parity tests, the smoke check and the bench. It holds none of the
method's arithmetic: only shapes, sequence lengths, page placement and random values. The
oracle and the CUDA path both consume what it produces; neither is imported here.

Workloads (sizes of the long-audio transcription setting: 12.5 encoder tokens per second of
audio after Whisper framing and the 4x temporal merge, so 30 s = 375 tokens, a 38-minute
meeting is about 28.5K tokens and 90 minutes is 67.5K tokens; Qwen3 decoder with GQA 16/8,
head_dim 128; pages of 16 tokens):

=====================  =============================================================
name                   what it is
=====================  =============================================================
decode_b1_l1000        1 sequence of 1,000 cached tokens (80 s of audio), pages placed by
                       a seeded random permutation of a 128-page pool
decode_b16_l27k        16 sequences (16 concurrent 38-minute meetings), lengths uniform in
                       [27,000, 30,000], pages scattered in one shared pool
decode_ragged_b64      64 sequences, lengths log-uniform in [375, 70,000] (30 s .. 90 min
                       plus transcript), Q scaled by 4 (peaked softmax)
prefill_4096_at_61440  one 4,096-query chunk at offset 61,440 (the last chunk of a 67,500-
                       token recording) over 61,440 cached tokens plus itself
mixed_28l              28 layers, each with its own K/V pools: one 4,096-query chunk at
                       offset 32,768 plus 31 decode sequences with lengths uniform in
                       [5,000, 90,000]; the new tokens are appended before attention
prefill_4096_at_32768  the prefill launch of one mixed_28l layer on its own (a 4,096-query
                       chunk at offset 32,768): a small case for memory-traffic counters
prefill_ragged_mix     one prefill call over six requests (RAGGED_PREFILL_MIX): chunks of
                       4,096 / 2,048 / 1,024 / 512 queries at offsets 28,672 / 61,440 /
                       10,000 / 0 and extends of 1 and 2 tokens after 5,000 and 20,000
decode_graph_buckets   batches of 1, 2, 4, 8, 16 and 32 sequences of 1,000 tokens, 28
                       layers with their own pools (CUDA-graph replay latency)
adaptor_90min          270,000 encoder frames (90 minutes) through the 4x merge and the
                       adaptor MLP (make_adaptor)
=====================  =============================================================

Recipe: sequence lengths and page permutations come from numpy ``PCG64(seed)``; tensor
values come from ``torch.randn`` with a ``torch.Generator`` seeded with the same seed and
are rounded to bf16. Unused page slots, unused pages and block-table entries past a
sequence's last page can be poisoned (NaN values; table entries pointing at a NaN page) so
that any read outside the defined key set shows up in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

HQ = 16          # query heads
HKV = 8          # KV heads
HEAD_DIM = 128
PAGE = 16        # tokens per page
SCALE = 1.0 / math.sqrt(HEAD_DIM)

CONFIG_SEED = {
    "decode_b1_l1000": 1001,
    "decode_b16_l27k": 1002,
    "decode_ragged_b64": 1003,
    "prefill_4096_at_61440": 1004,
    "mixed_28l": 1005,
    "prefill_4096_at_32768": 1008,
}


@dataclass
class PagedInputs:
    """One batch of paged-attention inputs (all tensors on ``device``).

    q            bf16 [Tq, Hq, D]   packed query rows (decode: one row per sequence)
    cu_q_lens    int32 [B+1]        row offsets of each sequence's queries in q
    k_pools      list of bf16 [NP, PAGE, Hkv, D], one per layer (v_pools likewise)
    block_table  int32 [B, stride]  logical page -> physical page, shared by all layers
    seq_lens     int32 [B]          keys per sequence after this step's tokens are appended
    start_pos    int32 [B]          position of each sequence's first new token
    k_new/v_new  list of bf16 [Tq, Hkv, D] per layer: the K/V rows of the new tokens
    """
    q: list
    cu_q_lens: torch.Tensor
    k_pools: list
    v_pools: list
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    start_pos: torch.Tensor
    k_new: list = field(default_factory=list)
    v_new: list = field(default_factory=list)
    scale: float = SCALE
    num_pages: int = 0
    poison_page: int = -1
    host_seq_lens: np.ndarray = None
    host_q_lens: np.ndarray = None
    host_block_table: np.ndarray = None

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def layers(self) -> int:
        return len(self.k_pools)


def _randn_bf16(shape, gen, device, scale=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def _randn_bf16_chunked(shape, gen, device, chunk_elems=1 << 28):
    """randn straight to bf16 without a full-size fp32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(flat.numel(), s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device,
                                dtype=torch.float32).to(torch.bfloat16)
    return out


def make_paged(seed: int, seq_lens, q_lens, *, layers: int = 1, pool_factor: float = 1.25,
               extra_pages: int = 1, pool_pages: int | None = None, q_scale: float = 1.0,
               poison: bool = False, device="cpu", distinct_layers: bool = True,
               with_new_kv: bool = True) -> PagedInputs:
    """Build a paged batch.

    seq_lens[b] keys per sequence (the step's new tokens included), q_lens[b] query rows (and
    new tokens) per sequence; the new tokens are the last q_lens[b] positions. Pages of every
    sequence are drawn from one random permutation of a shared pool of ``pool_pages`` pages
    (default ceil(pool_factor * needed) + extra_pages).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    B = len(seq_lens)
    n_pages = -(-seq_lens // PAGE)
    needed = int(n_pages.sum())
    if pool_pages is None:
        pool_pages = int(math.ceil(pool_factor * needed)) + extra_pages
    assert pool_pages >= needed + (1 if poison else 0)
    perm = rng.permutation(pool_pages)
    stride = max(1, int(n_pages.max()) if B else 1)
    used = perm[:needed]
    spare = perm[needed:]
    poison_page = int(spare[0]) if len(spare) else -1
    bt = np.full((B, stride), poison_page if poison else 0, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :n_pages[b]] = used[off:off + n_pages[b]]
        off += n_pages[b]

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (pool_pages, PAGE, HKV, HEAD_DIM)
    k0 = _randn_bf16_chunked(shape, gen, device)
    v0 = _randn_bf16_chunked(shape, gen, device)
    k_pools, v_pools = [k0], [v0]
    for layer in range(1, layers):
        if distinct_layers:
            # a cheap, distinct copy per layer: rotate the pages of layer 0's pools
            k_pools.append(torch.roll(k0, shifts=7919 * layer, dims=0))
            v_pools.append(torch.roll(v0, shifts=104729 * layer, dims=0))
        else:
            k_pools.append(k0)
            v_pools.append(v0)
    if poison:
        nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device=device)
        mask = torch.ones(pool_pages, PAGE, dtype=torch.bool)
        for b in range(B):
            for p in range(n_pages[b]):
                page = bt[b, p]
                valid = min(PAGE, seq_lens[b] - p * PAGE)
                mask[page, :valid] = False
        mask = mask.to(device)
        for pools in (k_pools, v_pools):
            for t in pools:
                t[mask] = nan

    Tq = int(q_lens.sum())
    q = [_randn_bf16((Tq, HQ, HEAD_DIM), gen, device, q_scale) for _ in range(layers)]
    k_new, v_new = [], []
    if with_new_kv:
        for _ in range(layers):
            k_new.append(_randn_bf16((Tq, HKV, HEAD_DIM), gen, device))
            v_new.append(_randn_bf16((Tq, HKV, HEAD_DIM), gen, device))
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    start = (seq_lens - q_lens).astype(np.int32)
    as_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return PagedInputs(q=q, cu_q_lens=as_dev(cu), k_pools=k_pools, v_pools=v_pools,
                       block_table=as_dev(bt), seq_lens=as_dev(seq_lens.astype(np.int32)),
                       start_pos=as_dev(start), k_new=k_new, v_new=v_new, num_pages=pool_pages,
                       poison_page=poison_page, host_seq_lens=seq_lens.astype(np.int32),
                       host_q_lens=q_lens.astype(np.int32), host_block_table=bt)


# ----------------------------------------------------------------------------------------------
# Sequence-length recipes of the five workloads.
# ----------------------------------------------------------------------------------------------
def lengths_for(name: str, seed: int | None = None):
    """(seq_lens, q_lens) of a named workload; decode rows have q_len 1."""
    seed = CONFIG_SEED[name] if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    if name == "decode_b1_l1000":
        return np.array([1000]), np.array([1])
    if name == "decode_b16_l27k":
        L = rng.integers(27_000, 30_000, size=16, endpoint=True)
        return L, np.ones(16, dtype=np.int64)
    if name == "decode_ragged_b64":
        L = np.round(np.exp(rng.uniform(math.log(375), math.log(70_000), size=64))).astype(np.int64)
        return L, np.ones(64, dtype=np.int64)
    if name == "prefill_4096_at_61440":
        return np.array([61_440 + 4096]), np.array([4096])
    if name == "prefill_4096_at_32768":
        return np.array([32_768 + 4096]), np.array([4096])
    if name == "mixed_28l":
        L = rng.integers(5_000, 90_000, size=31, endpoint=True)
        return np.concatenate([[32_768 + 4096], L]), np.concatenate([[4096], np.ones(31, np.int64)])
    raise KeyError(name)


def make_workload(name: str, *, device="cpu", poison=False, seed=None, **kw) -> PagedInputs:
    """The named workload at full size."""
    seed = CONFIG_SEED[name] if seed is None else seed
    L, ql = lengths_for(name, seed)
    if name == "decode_b1_l1000":
        return make_paged(seed, L, ql, pool_pages=128, poison=poison, device=device, **kw)
    if name == "decode_ragged_b64":
        return make_paged(seed, L, ql, q_scale=4.0, poison=poison, device=device, **kw)
    if name == "mixed_28l":
        kw.setdefault("layers", 28)
        return make_paged(seed, L, ql, pool_factor=1.0, extra_pages=16, poison=poison,
                          device=device, **kw)
    return make_paged(seed, L, ql, poison=poison, device=device, **kw)


# Coalesced prefill step of several requests (q_len, offset): prompt chunks at different depths,
# a new request's first chunk (offset 0), and 1- and 2-token extends.
RAGGED_PREFILL_MIX = ((4096, 28_672), (2048, 61_440), (1024, 10_000), (512, 0), (1, 5_000),
                      (2, 20_000))
RAGGED_PREFILL_SEED = 1007


def make_ragged_prefill(*, device="cpu", poison=False) -> "PagedInputs":
    """The RAGGED_PREFILL_MIX batch: one sequence per request, its chunk's keys included."""
    q_lens = [q for q, _ in RAGGED_PREFILL_MIX]
    seq_lens = [q + o for q, o in RAGGED_PREFILL_MIX]
    return make_paged(RAGGED_PREFILL_SEED, seq_lens, q_lens, poison=poison, device=device)


def kv_bytes_per_token(num_kv_heads: int = HKV, head_dim: int = HEAD_DIM) -> int:
    """K plus V bytes of one token in one layer (bf16)."""
    return 2 * num_kv_heads * head_dim * 2


# ----------------------------------------------------------------------------------------------
# Audio-text bridge inputs: encoder frames and synthetic adaptor weights.
# ----------------------------------------------------------------------------------------------
D_MODEL = 1024
ADAPTOR_SEED = 1006


@dataclass
class AdaptorInputs:
    """frames bf16 [T_enc, 1024]; w1 bf16 [1024, 4096]; w2 bf16 [1024, 1024] (out, in);
    b1, b2, gamma, beta fp32 [1024]; eps."""
    frames: torch.Tensor
    w1: torch.Tensor
    b1: torch.Tensor
    w2: torch.Tensor
    b2: torch.Tensor
    gamma: torch.Tensor
    beta: torch.Tensor
    eps: float = 1e-5


def make_adaptor(seed: int, num_frames: int, device="cpu") -> AdaptorInputs:
    """Frames ~ N(0, 1) (post-LayerNorm encoder output scale); weights ~ N(0, 1/fan_in);
    biases ~ N(0, 0.02^2); gamma ~ 1 + N(0, 0.1^2); beta ~ N(0, 0.1^2)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    r = lambda *shape: torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    frames = _randn_bf16_chunked((num_frames, D_MODEL), g, device)
    w1 = (r(1024, 4 * D_MODEL) / 64.0).to(torch.bfloat16)
    w2 = (r(1024, 1024) / 32.0).to(torch.bfloat16)
    return AdaptorInputs(frames=frames, w1=w1, b1=0.02 * r(1024), w2=w2, b2=0.02 * r(1024),
                         gamma=1.0 + 0.1 * r(1024), beta=0.1 * r(1024))
