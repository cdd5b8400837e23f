"""CUDA-graph capture of the calls (the decode loop of a serving engine replays one graph per
batch bucket): capture once, refill the static inputs, replay, and compare with the fp64 oracle
and bit for bit with eager calls on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits, check_attn

pytestmark = pytest.mark.gpu


def test_decode_graph_replay_matches_eager(cuda_lib):
    pa = cuda_lib
    lens = [3000, 17, 12000, 1000]
    inp = W.make_paged(31, lens, [1] * 4, device="cuda")
    max_s = 12000
    out = torch.empty_like(inp.q[0])
    lse = torch.empty(4, W.HQ, device="cuda")
    ws = torch.empty(pa.decode_workspace_size(4, max_s), dtype=torch.uint8, device="cuda")
    q_static = inp.q[0].clone()
    pa.attn_decode_paged(q_static, inp.k_pools[0], inp.v_pools[0], inp.block_table, inp.seq_lens,
                         max_s, inp.scale, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.attn_decode_paged(q_static, inp.k_pools[0], inp.v_pools[0], inp.block_table,
                             inp.seq_lens, max_s, inp.scale, out=out, lse=lse, workspace=ws)
    gen = torch.Generator(device="cuda").manual_seed(5)
    for step in range(3):
        q_new = torch.randn(q_static.shape, generator=gen, device="cuda").to(torch.bfloat16)
        q_static.copy_(q_new)
        g.replay()
        ref_o, ref_l = pa.attn_decode_paged(q_new, inp.k_pools[0], inp.v_pools[0],
                                            inp.block_table, inp.seq_lens, max_s, inp.scale)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l), step


def test_mixed_step_graph_replay_matches_eager(cuda_lib):
    pa = cuda_lib
    dec = [900, 5000, 33]
    inp = W.make_paged(32, [512 + 256] + dec, [256, 1, 1, 1], device="cuda")
    max_s = 5000
    k0, v0 = inp.k_pools[0].clone(), inp.v_pools[0].clone()
    pf_ws = torch.empty(pa.prefill_workspace_size(1, 256, max_s), dtype=torch.uint8, device="cuda")
    dec_ws = torch.empty(pa.decode_workspace_size(3, max_s), dtype=torch.uint8, device="cuda")
    po = torch.empty(256, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device="cuda")
    pl = torch.empty(256, W.HQ, device="cuda")
    do = torch.empty(3, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device="cuda")
    dl = torch.empty(3, W.HQ, device="cuda")

    def step():
        pa.kv_append_paged(inp.k_new[0], inp.v_new[0], inp.cu_q_lens, inp.start_pos,
                           inp.block_table, inp.k_pools[0], inp.v_pools[0])
        pa.attn_prefill_chunk(inp.q[0][:256], inp.cu_q_lens[:2], inp.k_pools[0], inp.v_pools[0],
                              inp.block_table[:1], inp.seq_lens[:1], 256, max_s, inp.scale,
                              out=po, lse=pl, workspace=pf_ws)
        pa.attn_decode_paged(inp.q[0][256:], inp.k_pools[0], inp.v_pools[0], inp.block_table[1:],
                             inp.seq_lens[1:], max_s, inp.scale, out=do, lse=dl, workspace=dec_ws)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (po, pl, do, dl, inp.k_pools[0], inp.v_pools[0])]
    inp.k_pools[0].copy_(k0)
    inp.v_pools[0].copy_(v0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (po, pl, do, dl):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip((po, pl, do, dl, inp.k_pools[0], inp.v_pools[0]), eager):
        assert torch.equal(a, b)


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16, 32])
def test_decode_graph_bucket_replays_match_the_oracle(cuda_lib, B):
    """The bench's decode buckets (B sequences of 1,000 cached tokens, the single-sequence one
    being the 1-sequence decode workload): one graph per bucket, replayed for three steps with
    new queries written into its static input; every replay is checked against the oracle."""
    pa = cuda_lib
    L = 1000
    inp = (W.make_workload("decode_b1_l1000", device="cuda", poison=True) if B == 1 else
           W.make_paged(W.CONFIG_SEED["decode_b1_l1000"] + B, np.full(B, L), np.ones(B, np.int64),
                        poison=True, device="cuda"))
    out = torch.empty(B, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, W.HQ, device="cuda")
    ws = torch.empty(pa.decode_workspace_size(B, L), dtype=torch.uint8, device="cuda")
    q_static = inp.q[0].clone()
    call = lambda: pa.attn_decode_paged(q_static, inp.k_pools[0], inp.v_pools[0], inp.block_table,
                                        inp.seq_lens, L, inp.scale, out=out, lse=lse, workspace=ws)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    k, v = bits(inp.k_pools[0]), bits(inp.v_pools[0])
    gen = torch.Generator(device="cuda").manual_seed(100 + B)
    for step in range(3):
        q_static.copy_(torch.randn(q_static.shape, generator=gen, device="cuda").to(torch.bfloat16))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = oracle.decode(bits(q_static), k, v, inp.host_block_table, inp.host_seq_lens,
                                     inp.scale, threads=16)
        check_attn(out, lse, ref_o, ref_l, what=f"bucket {B}, replay {step}")
