"""Decode parity: the CUDA split-KV decode against the fp64 oracle, on the same seeded bytes."""
import math
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits, check_attn, host

pytestmark = pytest.mark.gpu


def run_decode(pa, inp, layer=0, max_seq_len=None, status=None):
    L = inp.host_seq_lens
    max_seq_len = int(L.max()) if max_seq_len is None else max_seq_len
    out, lse = pa.attn_decode_paged(inp.q[layer], inp.k_pools[layer], inp.v_pools[layer],
                                    inp.block_table, inp.seq_lens, max(1, max_seq_len), inp.scale,
                                    status=status)
    torch.cuda.synchronize()
    return out, lse


def oracle_decode(inp, layer=0, seqs=None):
    return oracle.decode(bits(inp.q[layer]), bits(inp.k_pools[layer]), bits(inp.v_pools[layer]),
                         inp.host_block_table, inp.host_seq_lens, inp.scale, seqs=seqs, threads=16)


@pytest.mark.parametrize("lens", [
    [1], [15], [16], [17], [1000],
    [1, 15, 16, 17, 31, 32, 33, 255, 256, 257],
    [0, 5, 0, 300, 0],
    [0],
    list(range(1, 40)),
    [17, 300, 0, 1000, 999, 64] * 4,   # 24 sequences: two KV heads per CTA on the single launch
])
def test_decode_small(cuda_lib, lens):
    inp = W.make_paged(77 + len(lens), lens, [1] * len(lens), poison=True, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_decode(cuda_lib, inp, status=status)
    ref_o, ref_l = oracle_decode(inp)
    check_attn(out, lse, ref_o, ref_l, what=f"decode {lens[:6]}")
    assert cuda_lib.read_device_status(status) == 0


@pytest.mark.parametrize("lens", [[1000] * 2, [1000] * 4, [1000] * 8, [5000, 20, 7000]])
def test_decode_few_sequences_many_partials(cuda_lib, lens):
    """Few sequences, both ways: with the automatic split they go to the single-launch path (a
    cluster of CTAs per sequence and KV head, merged in distributed shared memory); with one page
    per range (split_tokens=16) each is cut into tens of partials merged by 16 warps per head,
    and the last case gives the sequences very different partial counts (two rounds of the warp
    loop for the longest, one partial for the shortest)."""
    inp = W.make_paged(91 + len(lens), lens, [1] * len(lens), poison=True, device="cuda")
    ref_o, ref_l = oracle_decode(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for split in (0, 16):
        out, lse = cuda_lib.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0],
                                              inp.block_table, inp.seq_lens, max(lens), inp.scale,
                                              split_tokens=split, status=status)
        torch.cuda.synchronize()
        check_attn(out, lse, ref_o, ref_l, what=f"decode {lens}, split_tokens={split}")
        assert cuda_lib.read_device_status(status) == 0


@pytest.mark.parametrize("name,scale_down", [("decode_b16_l27k", 10), ("decode_ragged_b64", 10)])
def test_decode_reduced_configs(cuda_lib, name, scale_down):
    L, ql = W.lengths_for(name)
    L = np.maximum(1, L // scale_down)
    inp = W.make_paged(W.CONFIG_SEED[name], L, ql, poison=True, device="cuda",
                       q_scale=4.0 if "ragged" in name else 1.0)
    out, lse = run_decode(cuda_lib, inp)
    ref_o, ref_l = oracle_decode(inp)
    check_attn(out, lse, ref_o, ref_l, what=name)


@pytest.mark.parametrize("name", ["decode_b1_l1000", "decode_b16_l27k", "decode_ragged_b64"])
def test_decode_full_size(cuda_lib, name):
    """The workloads at full size, every sequence checked."""
    inp = W.make_workload(name, device="cuda", poison=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_decode(cuda_lib, inp, status=status)
    ref_o, ref_l = oracle_decode(inp)
    check_attn(out, lse, ref_o, ref_l, what=name)
    assert cuda_lib.read_device_status(status) == 0


def test_decode_dominant_key_is_bit_exact(cuda_lib):
    """One key per (sequence, KV head) dominates: the output is its V row, bit for bit. Pins
    the block table walk, the slot arithmetic and the GQA head map exactly."""
    lens = [37, 300, 16, 1000]
    inp = W.make_paged(5, lens, [1] * 4, device="cuda")
    q = inp.q[0].float()
    k = inp.k_pools[0]
    bt = inp.host_block_table
    rng = np.random.default_rng(5)
    stars = []
    for b, L in enumerate(lens):
        for g in range(W.HKV):
            t = int(rng.integers(0, L))
            stars.append((b, g, t))
            page, slot = int(bt[b, t // W.PAGE]), t % W.PAGE
            # key aligned with both query heads of the group, large enough to dominate
            vec = 64.0 * torch.sign(q[b, 2 * g] + q[b, 2 * g + 1])
            k[page, slot, g] = vec.to(torch.bfloat16)
    out, _ = run_decode(cuda_lib, inp)
    v = inp.v_pools[0]
    for b, g, t in stars:
        page, slot = int(bt[b, t // W.PAGE]), t % W.PAGE
        for h in (2 * g, 2 * g + 1):
            assert torch.equal(out[b, h], v[page, slot, g]), (b, g, t, h)


def test_decode_page_permutation_is_bitwise_invariant(cuda_lib):
    lens = [4000, 123, 2049]
    inp = W.make_paged(9, lens, [1] * 3, device="cuda")
    out1, lse1 = run_decode(cuda_lib, inp)
    # move every page to a new physical slot and rewrite the table
    NP = inp.num_pages
    perm = torch.randperm(NP, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(NP)
    k2 = torch.empty_like(inp.k_pools[0])
    v2 = torch.empty_like(inp.v_pools[0])
    k2[perm.cuda()] = inp.k_pools[0]
    v2[perm.cuda()] = inp.v_pools[0]
    bt2 = perm.to(torch.int32).cuda()[inp.block_table.long()]
    out2, lse2 = cuda_lib.attn_decode_paged(inp.q[0], k2, v2, bt2.contiguous(), inp.seq_lens, 4000,
                                           inp.scale)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_decode_repeat_is_deterministic(cuda_lib):
    inp = W.make_paged(10, [30000, 700, 12000, 5], [1] * 4, device="cuda")
    a = run_decode(cuda_lib, inp)
    b = run_decode(cuda_lib, inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_alone_vs_in_batch(cuda_lib):
    """A sequence decoded alone and inside a batch is split differently; both match."""
    lens = [20000, 3000, 45000]
    inp = W.make_paged(11, lens, [1] * 3, device="cuda")
    out, lse = run_decode(cuda_lib, inp)
    alone, lse_alone = cuda_lib.attn_decode_paged(inp.q[0][2:3].contiguous(), inp.k_pools[0],
                                                  inp.v_pools[0], inp.block_table[2:3].contiguous(),
                                                  inp.seq_lens[2:3].contiguous(), 45000, inp.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_decode(inp, seqs=[2])
    check_attn(out[2:3], lse[2:3], ref_o[2:3], ref_l[2:3], what="in batch")
    check_attn(alone, lse_alone, ref_o[2:3], ref_l[2:3], what="alone")


def test_decode_out_of_range_page_is_flagged_not_read(cuda_lib):
    inp = W.make_paged(12, [100, 40], [1, 1], device="cuda")
    bt = inp.block_table.clone()
    bt[1, 1] = inp.num_pages + 1000      # outside the pool: must be flagged, never dereferenced
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = cuda_lib.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0], bt,
                                          inp.seq_lens, 100, inp.scale, status=status)
    flags = cuda_lib.read_device_status(status)
    assert flags & cuda_lib.DEV_ERR_PAGE_OOB
    ref_o, ref_l = oracle_decode(inp, seqs=[0])
    check_attn(out[:1], lse[:1], ref_o[:1], ref_l[:1], what="untouched sequence")


def test_decode_too_long_sequence_is_flagged(cuda_lib):
    inp = W.make_paged(13, [100, 40], [1, 1], device="cuda")
    sl = inp.seq_lens.clone()
    sl[1] = inp.block_table.shape[1] * 16 + 5
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0], inp.block_table, sl,
                               100, inp.scale, status=status)
    assert cuda_lib.read_device_status(status) & cuda_lib.DEV_ERR_LENGTH


def test_decode_workspace_too_small_is_rejected(cuda_lib):
    inp = W.make_paged(14, [100], [1], device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.PagedAttnError):
        cuda_lib.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0], inp.block_table,
                                   inp.seq_lens, 100, inp.scale, workspace=ws)


SPLITS = [0, 16, 256, 1024, 4096, 2**31 - 1]


@pytest.mark.parametrize("lens", [[4000, 123, 2049, 0, 16, 30000, 1], [1000] * 4 + [70000],
                                  [300, 17, 0, 1000, 1, 64]])
def test_decode_split_count_invariance(cuda_lib, lens):
    """split_tokens in {auto, 16, 256, 1024, 4096, one range}: the key ranges and so the number
    of partials per sequence differ (from one page per range to a single CTA for the whole
    batch); every result matches the oracle, and all agree with each other within the same
    tolerance (the split sizes are whole pages). With the short lengths of the last case the
    automatic choice is the single-launch cluster path."""
    pa = cuda_lib
    inp = W.make_paged(17 + len(lens), lens, [1] * len(lens), poison=True, device="cuda")
    ref_o, ref_l = oracle_decode(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    results = {}
    for split in SPLITS:
        out, lse = pa.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0],
                                        inp.block_table, inp.seq_lens, max(lens), inp.scale,
                                        split_tokens=split, status=status)
        torch.cuda.synchronize()
        check_attn(out, lse, ref_o, ref_l, what=f"split_tokens={split}")
        assert pa.read_device_status(status) == 0, split
        results[split] = (out.clone(), lse.clone())
    base_o = results[0][0].double().cpu().numpy()
    base_l = results[0][1].double().cpu().numpy()
    for split in SPLITS[1:]:
        check_attn(results[split][0], results[split][1], base_o, base_l,
                   what=f"split_tokens={split} vs auto")


def test_decode_split_workspace_grows_with_the_range_count(cuda_lib):
    """A smaller split needs records for more ranges; a workspace sized for auto is rejected
    when the split needs more."""
    pa = cuda_lib
    auto = pa.decode_workspace_size(4, 30000)
    fine = pa.decode_workspace_size(4, 30000, split_tokens=16)
    assert fine > auto
    assert pa.decode_workspace_size(4, 30000, split_tokens=2**31 - 1) < auto
    inp = W.make_paged(16, [30000, 5, 700, 12000], [1] * 4, device="cuda")
    ws = torch.empty(auto, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttnError):
        pa.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0], inp.block_table,
                             inp.seq_lens, 30000, inp.scale, split_tokens=16, workspace=ws)


def test_decode_bounded_wait_gives_up_and_the_next_call_is_correct(cuda_lib):
    """The test hook leaves one ring stage of CTA 0 unfilled and bounds the waits by 1 ms: the
    waiting consumer warps give up, flag PA_DEV_ERR_TIMEOUT and return (the producer drains its
    own copies first). The context stays usable: the next normal call on the same stream
    matches the oracle."""
    pa = cuda_lib
    inp = W.make_paged(15, [3000, 40, 700], [1, 1, 1], device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.debug_decode_starve(True)
    try:
        t0 = time.perf_counter()
        pa.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0], inp.block_table,
                             inp.seq_lens, 3000, inp.scale, status=status)
        flags = pa.read_device_status(status)
        dt = time.perf_counter() - t0
    finally:
        pa.debug_decode_starve(False)
    assert flags & pa.DEV_ERR_TIMEOUT, flags
    assert dt < 1.5, dt
    out, lse = pa.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0], inp.block_table,
                                    inp.seq_lens, 3000, inp.scale, status=status)
    torch.cuda.synchronize()
    assert pa.read_device_status(status) == 0
    ref_o, ref_l = oracle_decode(inp)
    check_attn(out, lse, ref_o, ref_l, what="after the timed-out call")


def test_binding_rejects_misshaped_buffers(cuda_lib):
    """The binding checks shapes the library cannot see through raw pointers (a short block
    table, a small output buffer, pools of the wrong head count) before anything is launched."""
    pa = cuda_lib
    inp = W.make_paged(17, [100, 200], [1, 1], device="cuda")
    q, kp, vp = inp.q[0], inp.k_pools[0], inp.v_pools[0]
    bad = [
        dict(block_table=inp.block_table[:1]),
        dict(seq_lens=inp.seq_lens[:1]),
        dict(out=torch.empty(2, 16, 64, dtype=torch.bfloat16, device="cuda")),
        dict(lse=torch.empty(2, 8, dtype=torch.float32, device="cuda")),
        dict(k_pool=kp[:, :, :4].contiguous()),
    ]
    for kw in bad:
        args = dict(block_table=inp.block_table, seq_lens=inp.seq_lens, k_pool=kp)
        args.update({k: v for k, v in kw.items() if k in args})
        extra = {k: v for k, v in kw.items() if k not in args}
        with pytest.raises(ValueError):
            pa.attn_decode_paged(q, args["k_pool"], vp, args["block_table"], args["seq_lens"],
                                 200, inp.scale, **extra)
    with pytest.raises(ValueError):
        pa.attn_prefill_chunk(q, inp.cu_q_lens, kp, vp, inp.block_table, inp.seq_lens, 1, 200,
                              inp.scale, out=torch.empty(1, 16, 128, dtype=torch.bfloat16,
                                                         device="cuda"))


@pytest.mark.parametrize("L,extra,split", [(30000, 0, 0), (30001, 7, 0), (30000, 100, 0),
                                           (70000, 0, 0), (5000, 0, 256), (12345, 3, 4096)])
def test_decode_one_sequence_against_its_length_bound(cuda_lib, L, extra, split):
    """One sequence through the split-KV kernel with the host's length bound equal to its length,
    above it within the same last page, and pages above it (past the end of the block-table
    row): the block-table entries a CTA loads beside the length are used only when the length
    gives the bound's page count, and every result matches the oracle."""
    pa = cuda_lib
    inp = W.make_paged(400 + L % 97, [L], [1], poison=True, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = pa.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0], inp.block_table,
                                    inp.seq_lens, L + extra, inp.scale, split_tokens=split,
                                    status=status)
    torch.cuda.synchronize()
    assert pa.decode_kernels_per_call(1, L + extra, split) == 2
    ref_o, ref_l = oracle_decode(inp)
    check_attn(out, lse, ref_o, ref_l, what=f"one sequence of {L} keys, bound {L + extra}")
    assert pa.read_device_status(status) == 0
