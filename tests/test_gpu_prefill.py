"""Chunked-prefill parity: the CUDA kernel against the fp64 oracle on the same seeded bytes."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits, check_attn, host

pytestmark = pytest.mark.gpu


def run_prefill(pa, inp, layer=0, status=None):
    max_q = int(inp.host_q_lens.max())
    max_s = int(inp.host_seq_lens.max())
    out, lse = pa.attn_prefill_chunk(inp.q[layer], inp.cu_q_lens, inp.k_pools[layer],
                                     inp.v_pools[layer], inp.block_table, inp.seq_lens, max_q,
                                     max_s, inp.scale, status=status)
    torch.cuda.synchronize()
    return out, lse


def oracle_prefill(inp, layer=0, rows=None):
    return oracle.prefill(bits(inp.q[layer]), host(inp.cu_q_lens),
                          bits(inp.k_pools[layer]), bits(inp.v_pools[layer]),
                          inp.host_block_table, inp.host_seq_lens, inp.scale, rows=rows,
                          threads=16)


@pytest.mark.parametrize("q_len,offset", [(1, 0), (1, 999), (15, 0), (16, 16), (17, 100),
                                          (128, 0), (129, 1000), (300, 37), (256, 4096)])
def test_prefill_single_chunk(cuda_lib, q_len, offset):
    inp = W.make_paged(100 + q_len, [offset + q_len], [q_len], poison=True, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_prefill(cuda_lib, inp, status=status)
    ref_o, ref_l = oracle_prefill(inp)
    check_attn(out, lse, ref_o, ref_l, what=f"prefill q_len={q_len} offset={offset}")
    assert cuda_lib.read_device_status(status) == 0


def test_prefill_ragged_chunks(cuda_lib):
    """Several chunks of different lengths and offsets in one call (coalesced prefill)."""
    q_lens = [7, 128, 1, 200, 64]
    offsets = [0, 333, 4095, 16, 1000]
    inp = W.make_paged(200, [o + q for o, q in zip(offsets, q_lens)], q_lens, poison=True,
                       device="cuda")
    out, lse = run_prefill(cuda_lib, inp)
    ref_o, ref_l = oracle_prefill(inp)
    check_attn(out, lse, ref_o, ref_l, what="ragged chunks")


def test_prefill_last_chunk_reduced(cuda_lib):
    """The last-chunk shape scaled down 8x: 512 queries at offset 7,680, every row checked."""
    inp = W.make_paged(201, [7680 + 512], [512], poison=True, device="cuda")
    out, lse = run_prefill(cuda_lib, inp)
    ref_o, ref_l = oracle_prefill(inp)
    check_attn(out, lse, ref_o, ref_l, what="512 @ 7680")


def sampled_rows(n, seed, count=96):
    rng = np.random.default_rng(seed)
    rows = set(range(16)) | set(range(n - 16, n))
    rows |= {r for r in (15, 16, 17, 127, 128, 129, n // 2) if r < n}
    rows |= set(int(x) for x in rng.integers(0, n, size=count))
    return sorted(rows)


def test_prefill_full_size_last_chunk(cuda_lib):
    """4096 queries at offset 61,440 over 65,536 keys, in the bench's launch: every row of every
    head checked (about 2.1 TFLOP of fp64 work for the oracle)."""
    inp = W.make_workload("prefill_4096_at_61440", device="cuda", poison=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_prefill(cuda_lib, inp, status=status)
    ref_o, ref_l = oracle_prefill(inp)
    check_attn(out, lse, ref_o, ref_l, what="prefill_4096_at_61440")
    assert cuda_lib.read_device_status(status) == 0


def test_prefill_ragged_mix_full_size(cuda_lib):
    """The bench's coalesced step: chunks of 4,096 / 2,048 / 1,024 / 512 queries at offsets
    28,672 / 61,440 / 10,000 / 0 and 1- and 2-token extends in one call; sampled rows of every
    chunk (its first and last 16, page and tile edges, random) and both extends in full."""
    inp = W.make_ragged_prefill(device="cuda", poison=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_prefill(cuda_lib, inp, status=status)
    cu = host(inp.cu_q_lens)
    rows = []
    for b in range(len(cu) - 1):
        n = int(cu[b + 1] - cu[b])
        rows += [int(cu[b]) + r for r in (sampled_rows(n, 10 + b, count=24) if n > 40 else range(n))]
    ref_o, ref_l = oracle_prefill(inp, rows=rows)
    check_attn(out, lse, ref_o, ref_l, rows=rows, what="ragged prefill mix")
    assert cuda_lib.read_device_status(status) == 0


def test_prefill_uneven_jobs_level_split(cuda_lib):
    """Chunks whose jobs differ in length (515 / 1,024 / 1,024 / 128 queries at offsets 33,783 /
    36,652 / 26,147 / 31,557). On a 152-SM GB300 the levelled work split gives several CTAs
    whole jobs that exactly fill their share, so their second-phase ranges are empty and lie
    inside jobs cut across many CTAs (the third chunk's query tiles 5 and 6 of KV head 6), which
    the merge must skip. Every row of those tiles and sampled rows of the rest are checked."""
    q_lens = [515, 1024, 1024, 128]
    seq_lens = [34_298, 37_676, 27_171, 31_685]
    inp = W.make_paged(203, seq_lens, q_lens, poison=True, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_prefill(cuda_lib, inp, status=status)
    cu = host(inp.cu_q_lens)
    rows = set(int(cu[2]) + r for r in range(5 * 128, 7 * 128))
    for b in range(len(q_lens)):
        rows |= {int(cu[b]) + r for r in sampled_rows(q_lens[b], 20 + b, count=16)}
    rows = sorted(rows)
    ref_o, ref_l = oracle_prefill(inp, rows=rows)
    check_attn(out, lse, ref_o, ref_l, rows=rows, what="uneven jobs, levelled split")
    assert cuda_lib.read_device_status(status) == 0


def test_prefill_chunk_longer_than_sequence_is_flagged(cuda_lib):
    inp = W.make_paged(202, [50], [20], device="cuda")
    sl = inp.seq_lens.clone()
    sl[0] = 10
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.attn_prefill_chunk(inp.q[0], inp.cu_q_lens, inp.k_pools[0], inp.v_pools[0],
                                inp.block_table, sl, 20, 50, inp.scale, status=status)
    assert cuda_lib.read_device_status(status) & cuda_lib.DEV_ERR_LENGTH


def test_prefill_dominant_key_in_each_column_piece(cuda_lib):
    """Every query of a head pair sees the same scores and one key that dominates them: each row
    that sees the key returns its V row bit for bit. The dominant keys sit in each 32-column
    piece of a 128-key tile (the row max of a piece comes from the TMEM load on tiles that do not
    cross the row's position), on tiles both before the chunk and on its diagonal; the rows that
    do not see their key yet, and the head pair without one, are checked against the oracle."""
    offset, q_len = 1024, 256
    inp = W.make_paged(303, [offset + q_len], [q_len], poison=True, device="cuda")
    q = inp.q[0]
    k = inp.k_pools[0]
    bt = inp.host_block_table
    gen = torch.Generator(device="cuda").manual_seed(5)
    # KV head g -> position of its dominant key (None: no dominant key)
    dominant = {0: 5, 1: 128 + 32 + 5, 2: 256 + 64 + 5, 3: 384 + 96 + 5,
                4: offset + 10, 5: offset + 128 + 70, 6: offset + 127, 7: None}
    for g, t in dominant.items():
        if t is None:
            continue
        q0 = torch.randn(W.HEAD_DIM, generator=gen, device="cuda").to(torch.bfloat16)
        q[:, 2 * g] = q0
        q[:, 2 * g + 1] = q0
        page, slot = int(bt[0, t // W.PAGE]), t % W.PAGE
        k[page, slot, g] = (64.0 * torch.sign(q0.float())).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_prefill(cuda_lib, inp, status=status)
    assert cuda_lib.read_device_status(status) == 0
    v = inp.v_pools[0]
    for g, t in dominant.items():
        if t is None:
            continue
        page, slot = int(bt[0, t // W.PAGE]), t % W.PAGE
        first_row = max(0, t - offset)   # the first query whose position reaches the key
        for h in (2 * g, 2 * g + 1):
            want = v[page, slot, g].expand(q_len - first_row, W.HEAD_DIM)
            assert torch.equal(out[first_row:, h], want), (g, t, h)
    ref_o, ref_l = oracle_prefill(inp)
    check_attn(out, lse, ref_o, ref_l, what="dominant keys")
