"""The calls at the limits they document: the 128K context, 128 prefill chunks per call, a
decode batch of 4,096 sequences, a chunk at offset 0 spanning many tiles, a 128-key-aligned
and a one-past-aligned chunk length."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits, check_attn, host

pytestmark = pytest.mark.gpu


def test_decode_at_the_128k_context(cuda_lib):
    inp = W.make_paged(60, [131072, 7], [1, 1], device="cuda")
    out, lse = cuda_lib.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0],
                                          inp.block_table, inp.seq_lens, 131072, inp.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(bits(inp.q[0]), bits(inp.k_pools[0]), bits(inp.v_pools[0]),
                                 inp.host_block_table, inp.host_seq_lens, inp.scale, threads=16)
    check_attn(out, lse, ref_o, ref_l, what="131,072 keys")


def test_decode_batch_of_4096(cuda_lib):
    rng = np.random.default_rng(61)
    lens = rng.integers(0, 200, size=4096)
    inp = W.make_paged(61, lens, np.ones(4096, np.int64), device="cuda")
    out, lse = cuda_lib.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0],
                                          inp.block_table, inp.seq_lens, 200, inp.scale)
    torch.cuda.synchronize()
    seqs = sorted(set(int(x) for x in rng.integers(0, 4096, 64)) | {0, 4095})
    ref_o, ref_l = oracle.decode(bits(inp.q[0]), bits(inp.k_pools[0]), bits(inp.v_pools[0]),
                                 inp.host_block_table, inp.host_seq_lens, inp.scale, seqs=seqs)
    check_attn(out, lse, ref_o, ref_l, rows=seqs, what="4,096 sequences (sampled)")


@pytest.mark.parametrize("split", [16, 4096])
def test_decode_batch_of_4096_with_a_split_size(cuda_lib, split):
    """A split of one page per range would need more ranges than the workspace holds (64 per
    SM); the range size is raised until it fits, and the result is unchanged. A large split puts
    many short sequences into one range."""
    rng = np.random.default_rng(65)
    lens = rng.integers(0, 400, size=4096)
    inp = W.make_paged(65, lens, np.ones(4096, np.int64), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = cuda_lib.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0],
                                          inp.block_table, inp.seq_lens, 400, inp.scale,
                                          split_tokens=split, status=status)
    torch.cuda.synchronize()
    assert cuda_lib.read_device_status(status) == 0
    seqs = sorted(set(int(x) for x in rng.integers(0, 4096, 96)) | {0, 4095})
    ref_o, ref_l = oracle.decode(bits(inp.q[0]), bits(inp.k_pools[0]), bits(inp.v_pools[0]),
                                 inp.host_block_table, inp.host_seq_lens, inp.scale, seqs=seqs)
    check_attn(out, lse, ref_o, ref_l, rows=seqs, what=f"4,096 sequences, split {split} (sampled)")


def test_prefill_128_chunks_in_one_call(cuda_lib):
    rng = np.random.default_rng(62)
    q_lens = rng.integers(1, 40, size=128)
    offs = rng.integers(0, 300, size=128)
    inp = W.make_paged(62, offs + q_lens, q_lens, device="cuda")
    out, lse = cuda_lib.attn_prefill_chunk(inp.q[0], inp.cu_q_lens, inp.k_pools[0], inp.v_pools[0],
                                           inp.block_table, inp.seq_lens, int(q_lens.max()),
                                           int((offs + q_lens).max()), inp.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.prefill(bits(inp.q[0]), host(inp.cu_q_lens), bits(inp.k_pools[0]),
                                  bits(inp.v_pools[0]), inp.host_block_table,
                                  inp.host_seq_lens, inp.scale, threads=16)
    check_attn(out, lse, ref_o, ref_l, what="128 chunks")


def test_prefill_more_than_128_chunks_is_rejected(cuda_lib):
    inp = W.make_paged(63, [5] * 129, [1] * 129, device="cuda")
    with pytest.raises(cuda_lib.PagedAttnError):
        cuda_lib.attn_prefill_chunk(inp.q[0], inp.cu_q_lens, inp.k_pools[0], inp.v_pools[0],
                                    inp.block_table, inp.seq_lens, 1, 5, inp.scale)


@pytest.mark.parametrize("q_len", [1024, 1025])
def test_prefill_chunk_at_offset_zero(cuda_lib, q_len):
    """The first chunk of a recording: causal over itself only, many diagonal tiles."""
    inp = W.make_paged(64, [q_len], [q_len], device="cuda")
    out, lse = cuda_lib.attn_prefill_chunk(inp.q[0], inp.cu_q_lens, inp.k_pools[0], inp.v_pools[0],
                                           inp.block_table, inp.seq_lens, q_len, q_len, inp.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.prefill(bits(inp.q[0]), host(inp.cu_q_lens), bits(inp.k_pools[0]),
                                  bits(inp.v_pools[0]), inp.host_block_table,
                                  inp.host_seq_lens, inp.scale, threads=16)
    check_attn(out, lse, ref_o, ref_l, what=f"{q_len} rows at offset 0")
