"""kv_append placement (bit-exact) and the public log-sum-exp merge, against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits, check_attn, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("q_lens,starts", [
    ([1], [0]), ([1, 1, 1], [15, 16, 1000]), ([300, 1, 1, 17], [2000, 0, 47, 16]),
    ([4096] + [1] * 31, [32768] + list(range(5000, 5031))),
])
def test_kv_append_bit_exact(cuda_lib, q_lens, starts):
    seq_lens = [s + q for s, q in zip(starts, q_lens)]
    inp = W.make_paged(300 + len(q_lens), seq_lens, q_lens, device="cuda")
    k0, v0 = bits(inp.k_pools[0]), bits(inp.v_pools[0])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.kv_append_paged(inp.k_new[0], inp.v_new[0], inp.cu_q_lens, inp.start_pos,
                             inp.block_table, inp.k_pools[0], inp.v_pools[0], status=status)
    torch.cuda.synchronize()
    ek, ev = oracle.kv_append(bits(inp.k_new[0]), bits(inp.v_new[0]), host(inp.cu_q_lens),
                              host(inp.start_pos), inp.host_block_table, k0, v0)
    assert np.array_equal(bits(inp.k_pools[0]), ek)
    assert np.array_equal(bits(inp.v_pools[0]), ev)
    assert cuda_lib.read_device_status(status) == 0


def test_kv_append_missing_table_entry_is_flagged(cuda_lib):
    inp = W.make_paged(310, [20], [4], device="cuda")
    sp = inp.start_pos.clone()
    sp[0] = inp.block_table.shape[1] * 16 - 2       # last two rows fall past the table row
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = bits(inp.k_pools[0]).copy()
    cuda_lib.kv_append_paged(inp.k_new[0], inp.v_new[0], inp.cu_q_lens, sp, inp.block_table,
                             inp.k_pools[0], inp.v_pools[0], status=status)
    assert cuda_lib.read_device_status(status) & cuda_lib.DEV_ERR_LENGTH
    after = bits(inp.k_pools[0])
    page = inp.host_block_table[0, -1]
    assert np.array_equal(after[page, 14:], bits(inp.k_new[0])[:2])  # in-range rows written
    mask = np.ones(after.shape[:2], bool)
    mask[page, 14:] = False
    assert np.array_equal(after[mask], before[mask])                  # nothing else touched


def test_kv_append_more_packed_rows_than_total_new_is_flagged(cuda_lib):
    """cu_new_lens[batch] = 50 but the call is given total_new = 40 rows: the first 40 rows are
    placed exactly as the oracle places them, the other 10 are not written (no pool byte
    outside the first 40 rows' slots changes) and PA_DEV_ERR_LENGTH is set."""
    inp = W.make_paged(311, [100, 50], [30, 20], device="cuda")
    k0, v0 = bits(inp.k_pools[0]).copy(), bits(inp.v_pools[0]).copy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.kv_append_paged(inp.k_new[0][:40].contiguous(), inp.v_new[0][:40].contiguous(),
                             inp.cu_q_lens, inp.start_pos, inp.block_table, inp.k_pools[0],
                             inp.v_pools[0], status=status)
    assert cuda_lib.read_device_status(status) & cuda_lib.DEV_ERR_LENGTH
    # the oracle's placement of the rows that were given: sequence 1 keeps its first 10 rows
    ek, ev = oracle.kv_append(bits(inp.k_new[0])[:40], bits(inp.v_new[0])[:40],
                              np.array([0, 30, 40]), host(inp.start_pos), inp.host_block_table,
                              k0, v0)
    assert np.array_equal(bits(inp.k_pools[0]), ek)
    assert np.array_equal(bits(inp.v_pools[0]), ev)


@pytest.mark.parametrize("S,R,H", [(1, 5, 16), (3, 7, 16), (40, 2, 3), (2, 1, 1)])
def test_merge_lse(cuda_lib, S, R, H):
    g = torch.Generator(device="cuda").manual_seed(S * 100 + R)
    o = torch.randn(S, R, H, 128, generator=g, device="cuda")
    l = 5 * torch.randn(S, R, H, generator=g, device="cuda")
    if S > 1:
        l[0, 0, 0] = -math.inf          # an empty part
        o[0, 0, 0] = float("nan")       # never read
    if R > 1:
        l[:, 1, 0] = -math.inf          # a row whose parts are all empty
    out, lse = cuda_lib.attn_merge_lse(o, l)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.merge_lse(host(o), host(l))
    check_attn(out, lse, ref_o, ref_l, what=f"merge S={S}")
