"""Randomized parity sweep: many small seeded problems drawn across the calls' argument space.

The fixed cases elsewhere pin the workloads, the documented limits and the hand-picked edges.
This sweep draws 96 problems from a seeded generator: batch sizes, sequence lengths around and
across page and tile edges, chunk lengths and offsets, several chunks per call, split sizes,
the KV-head counts of a partitioned cache (8, 4, 2, 1), NaN-poisoned unused slots. Each problem
runs append -> prefill of its chunks -> decode of its other sequences, and every output is
checked against the oracle (placement bit for bit; attention within the parity tolerance), with
no device status bit set. A failure names the seed of the problem that failed.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits, check_attn, host

pytestmark = pytest.mark.gpu

N_PROBLEMS = 96


def _draw(rng):
    """One problem: (sequence lengths, new tokens per sequence, number of chunked sequences,
    KV heads, split size)."""
    n_chunks = int(rng.integers(1, 5))
    n_dec = int(rng.integers(0, 9))
    edge = [1, 15, 16, 17, 127, 128, 129, 255, 256, 257]
    q_lens, seq_lens = [], []
    for _ in range(n_chunks):
        q = int(rng.choice(edge)) if rng.random() < 0.5 else int(rng.integers(1, 600))
        off = int(rng.choice([0] + edge)) if rng.random() < 0.4 else int(rng.integers(0, 3000))
        q_lens.append(q)
        seq_lens.append(off + q)
    for _ in range(n_dec):
        L = int(rng.choice(edge)) if rng.random() < 0.4 else int(rng.integers(1, 20000))
        q_lens.append(1)
        seq_lens.append(L)
    hk = int(rng.choice([8, 8, 4, 2, 1]))
    split = int(rng.choice([0, 0, 16, 48, 512, 4096]))
    return seq_lens, q_lens, n_chunks, hk, split


@pytest.mark.parametrize("seed", range(N_PROBLEMS))
def test_random_problem(cuda_lib, seed):
    pa = cuda_lib
    rng = np.random.default_rng(7000 + seed)
    seq_lens, q_lens, n_chunks, hk, split = _draw(rng)
    inp = W.make_paged(7000 + seed, seq_lens, q_lens, poison=True, device="cuda")
    dims = (2 * hk, hk, W.HEAD_DIM, W.PAGE)
    # this problem's share of the heads (all 8 KV heads when hk == 8)
    kp = inp.k_pools[0][:, :, :hk].contiguous()
    vp = inp.v_pools[0][:, :, :hk].contiguous()
    k_new = inp.k_new[0][:, :hk].contiguous()
    v_new = inp.v_new[0][:, :hk].contiguous()
    q = inp.q[0][:, :2 * hk].contiguous()
    k_before, v_before = bits(kp).copy(), bits(vp).copy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.kv_append_paged(k_new, v_new, inp.cu_q_lens, inp.start_pos, inp.block_table, kp, vp,
                       status=status, dims=dims)
    cu = host(inp.cu_q_lens)
    rows = int(cu[n_chunks])
    max_s = int(max(seq_lens))
    po, pl = pa.attn_prefill_chunk(q[:rows], inp.cu_q_lens[:n_chunks + 1], kp, vp,
                                   inp.block_table[:n_chunks], inp.seq_lens[:n_chunks],
                                   int(max(q_lens[:n_chunks])), max_s, inp.scale, status=status,
                                   dims=dims)
    n_dec = len(seq_lens) - n_chunks
    if n_dec:
        do, dl = pa.attn_decode_paged(q[rows:].contiguous(), kp, vp, inp.block_table[n_chunks:].contiguous(),
                                      inp.seq_lens[n_chunks:].contiguous(), max_s, inp.scale,
                                      split_tokens=split, status=status, dims=dims)
    torch.cuda.synchronize()
    what = f"seed {seed}: lens {seq_lens}, q_lens {q_lens}, kv heads {hk}, split {split}"
    assert pa.read_device_status(status) == 0, what
    ek, ev = oracle.kv_append(bits(k_new), bits(v_new), cu, host(inp.start_pos),
                              inp.host_block_table, k_before, v_before)
    assert np.array_equal(bits(kp), ek) and np.array_equal(bits(vp), ev), what + " (append)"
    qb = bits(q)
    ro, rl = oracle.prefill(qb[:rows], cu[:n_chunks + 1], ek, ev, inp.host_block_table[:n_chunks],
                            inp.host_seq_lens[:n_chunks], inp.scale, threads=16)
    check_attn(po, pl, ro, rl, what=what + " (prefill)")
    if n_dec:
        ro, rl = oracle.decode(qb[rows:], ek, ev, inp.host_block_table[n_chunks:],
                               inp.host_seq_lens[n_chunks:], inp.scale, threads=16)
        check_attn(do, dl, ro, rl, what=what + " (decode)")
