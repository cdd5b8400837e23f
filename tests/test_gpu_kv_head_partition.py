"""Tensor-parallel partition of the attention by KV head, emulated on one GPU.

A KV cache that outgrows one device can be split by KV head: device r of N holds KV heads
8r/N .. 8(r+1)/N - 1 of every page (pools [pages][16][8/N][128]) and serves the 16/N query
heads that read them. Attention needs no exchange inside the step (each head depends only on
its own K/V); the per-device outputs are gathered along the head axis. Here the "devices" are
separate calls on one GPU with dims (16/N, 8/N, 128, 16), each on its own copies of its heads'
pools: kv_append, prefill of a chunk and decode of other sequences, as in one mixed step. The
appended pools must equal the oracle's placement bit for bit, and the gathered attention
outputs must match the oracle on the whole (unpartitioned) problem.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits, check_attn, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ranks", [2, 4, 8])
def test_kv_head_partition_matches_the_whole(cuda_lib, ranks):
    pa = cuda_lib
    hk, hq = W.HKV // ranks, W.HQ // ranks
    dims = (hq, hk, W.HEAD_DIM, W.PAGE)
    n_chunk = 300
    dec = [3000, 17, 12000, 1000, 20000, 16]
    inp = W.make_paged(70 + ranks, [700 + n_chunk] + dec, [n_chunk] + [1] * len(dec), poison=True,
                       device="cuda")
    max_s = int(inp.host_seq_lens.max())
    k_before, v_before = bits(inp.k_pools[0]).copy(), bits(inp.v_pools[0]).copy()
    pf_o, pf_l, dec_o, dec_l = [], [], {}, {}
    splits = (0, 16, 1024)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pools = []
    for r in range(ranks):
        h0, h1 = r * hk, (r + 1) * hk
        kp = inp.k_pools[0][:, :, h0:h1].contiguous()
        vp = inp.v_pools[0][:, :, h0:h1].contiguous()
        pa.kv_append_paged(inp.k_new[0][:, h0:h1].contiguous(), inp.v_new[0][:, h0:h1].contiguous(),
                           inp.cu_q_lens, inp.start_pos, inp.block_table, kp, vp, status=status,
                           dims=dims)
        q = inp.q[0][:, 2 * h0:2 * h1].contiguous()
        o, l = pa.attn_prefill_chunk(q[:n_chunk], inp.cu_q_lens[:2], kp, vp, inp.block_table[:1],
                                     inp.seq_lens[:1], n_chunk, max_s, inp.scale, status=status,
                                     dims=dims)
        pf_o.append(o)
        pf_l.append(l)
        for split in splits:
            o, l = pa.attn_decode_paged(q[n_chunk:].contiguous(), kp, vp, inp.block_table[1:],
                                        inp.seq_lens[1:], max_s, inp.scale, split_tokens=split,
                                        status=status, dims=dims)
            dec_o.setdefault(split, []).append(o)
            dec_l.setdefault(split, []).append(l)
        pools.append((kp, vp))
    torch.cuda.synchronize()
    assert pa.read_device_status(status) == 0

    ek, ev = oracle.kv_append(bits(inp.k_new[0]), bits(inp.v_new[0]), host(inp.cu_q_lens),
                              host(inp.start_pos), inp.host_block_table, k_before, v_before)
    for r, (kp, vp) in enumerate(pools):
        h0, h1 = r * hk, (r + 1) * hk
        assert np.array_equal(bits(kp), ek[:, :, h0:h1]), f"rank {r} K pool"
        assert np.array_equal(bits(vp), ev[:, :, h0:h1]), f"rank {r} V pool"
    q = bits(inp.q[0])
    ro, rl = oracle.prefill(q[:n_chunk], [0, n_chunk], ek, ev, inp.host_block_table[:1],
                            inp.host_seq_lens[:1], inp.scale, threads=16)
    check_attn(torch.cat(pf_o, dim=1), torch.cat(pf_l, dim=1), ro, rl,
               what=f"prefill over {ranks} head partitions")
    ro, rl = oracle.decode(q[n_chunk:], ek, ev, inp.host_block_table[1:], inp.host_seq_lens[1:],
                           inp.scale, threads=16)
    for split in splits:
        check_attn(torch.cat(dec_o[split], dim=1), torch.cat(dec_l[split], dim=1), ro, rl,
                   what=f"decode over {ranks} head partitions, split_tokens={split}")


@pytest.mark.parametrize("hk", [1, 2, 4])
def test_partitioned_decode_of_long_and_empty_sequences(cuda_lib, hk):
    """One device's share of the heads on long sequences cut into many ranges (each range's
    pages spread over the stage's page slots, so every sequence is merged from its slots'
    partials), plus empty and one-token sequences."""
    pa = cuda_lib
    dims = (2 * hk, hk, W.HEAD_DIM, W.PAGE)
    lens = [70000, 0, 1, 33333, 129]
    inp = W.make_paged(80 + hk, lens, [1] * len(lens), poison=True, device="cuda")
    kp = inp.k_pools[0][:, :, :hk].contiguous()
    vp = inp.v_pools[0][:, :, :hk].contiguous()
    q = inp.q[0][:, :2 * hk].contiguous()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = pa.attn_decode_paged(q, kp, vp, inp.block_table, inp.seq_lens, max(lens), inp.scale,
                                    status=status, dims=dims)
    torch.cuda.synchronize()
    assert pa.read_device_status(status) == 0
    ref_o, ref_l = oracle.decode(bits(q), bits(kp), bits(vp), inp.host_block_table,
                                 inp.host_seq_lens, inp.scale, threads=16)
    check_attn(out, lse, ref_o, ref_l, what=f"{hk} KV heads, long and empty sequences")


@pytest.mark.parametrize("hk,batch", [(4, 48), (2, 88), (1, 100)])
def test_partitioned_decode_single_launch(cuda_lib, hk, batch):
    """A device's share of the heads on a short batch goes through the single-launch path: with
    4 or 2 KV heads these batches have more (sequence, KV head) pairs than the GPU has SMs, so
    a CTA serves two KV heads; with 1 KV head a CTA per sequence. Checked against the oracle and
    against the split path (split_tokens=16) on the same inputs."""
    pa = cuda_lib
    dims = (2 * hk, hk, W.HEAD_DIM, W.PAGE)
    rng = np.random.default_rng(hk)
    lens = [int(x) for x in rng.integers(0, 400, size=batch)]
    lens[0], lens[1] = 400, 0
    inp = W.make_paged(95 + hk, lens, [1] * batch, poison=True, device="cuda")
    kp = inp.k_pools[0][:, :, :hk].contiguous()
    vp = inp.v_pools[0][:, :, :hk].contiguous()
    q = inp.q[0][:, :2 * hk].contiguous()
    assert pa.decode_kernels_per_call(batch, max(lens), dims=dims) == 1
    ref_o, ref_l = oracle.decode(bits(q), bits(kp), bits(vp), inp.host_block_table,
                                 inp.host_seq_lens, inp.scale, threads=16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for split in (0, 16):
        out, lse = pa.attn_decode_paged(q, kp, vp, inp.block_table, inp.seq_lens, max(lens),
                                        inp.scale, split_tokens=split, status=status, dims=dims)
        torch.cuda.synchronize()
        assert pa.read_device_status(status) == 0
        check_attn(out, lse, ref_o, ref_l, what=f"{hk} KV heads, {batch} sequences, split {split}")


def test_unsupported_head_counts_are_rejected(cuda_lib):
    pa = cuda_lib
    inp = W.make_paged(90, [100], [1], device="cuda")
    for dims in ((16, 4, 128, 16), (6, 3, 128, 16), (32, 16, 128, 16)):
        with pytest.raises(pa.PagedAttnError):
            pa.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0], inp.block_table,
                                 inp.seq_lens, 100, inp.scale, dims=dims,
                                 workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
