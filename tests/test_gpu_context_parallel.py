"""Context-parallel split of the decode step, emulated on one GPU.

A long cache can be cut by key range across devices: each device decodes its own range (its
pages of every sequence) and the partial (o, lse) pairs are combined by log-sum-exp. Here the
"devices" are separate calls on one GPU; the exchange is the stacking of their partials, and
attn_merge_lse combines them. The result must match the single-device decode and the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits, check_attn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ranks", [2, 3, 4])
def test_decode_split_by_key_range_and_merged(cuda_lib, ranks):
    pa = cuda_lib
    lens = [30000, 4096, 16, 12345, 70000]
    inp = W.make_paged(40 + ranks, lens, [1] * len(lens), device="cuda")
    B = len(lens)
    bt = inp.host_block_table
    o_parts, l_parts = [], []
    for r in range(ranks):
        # rank r owns pages [p0, p1) of every sequence (whole pages, contiguous key range)
        sub_lens, sub_bt = [], np.zeros_like(bt)
        for b, L in enumerate(lens):
            n_pages = -(-L // 16)
            p0 = n_pages * r // ranks
            p1 = n_pages * (r + 1) // ranks
            k0, k1 = p0 * 16, min(L, p1 * 16)
            sub_lens.append(max(0, k1 - k0))
            sub_bt[b, :p1 - p0] = bt[b, p0:p1]
        sl = torch.tensor(sub_lens, dtype=torch.int32, device="cuda")
        btt = torch.from_numpy(sub_bt).cuda()
        o, l = pa.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0], btt, sl,
                                    max(1, max(sub_lens)), inp.scale)
        o_parts.append(o.float())
        l_parts.append(l)
    merged_o, merged_l = pa.attn_merge_lse(torch.stack(o_parts).contiguous(),
                                           torch.stack(l_parts).contiguous())
    full_o, full_l = pa.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0],
                                          inp.block_table, inp.seq_lens, max(lens), inp.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(bits(inp.q[0]), bits(inp.k_pools[0]), bits(inp.v_pools[0]), bt,
                                 inp.host_seq_lens, inp.scale, threads=16)
    check_attn(merged_o, merged_l, ref_o, ref_l, what=f"{ranks}-way key split, merged")
    check_attn(full_o, full_l, ref_o, ref_l, what="single decode")
