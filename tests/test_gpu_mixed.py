"""The mixed scheduler step: per layer, append the new tokens, then prefill the chunk and
decode the other sequences, each layer with its own pools; checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits, check_attn, host

pytestmark = pytest.mark.gpu


def mixed_step(pa, inp, layer, chunk_rows, ws=None):
    """append + prefill(first sequence) + decode(the rest) for one layer."""
    B = inp.batch
    pa.kv_append_paged(inp.k_new[layer], inp.v_new[layer], inp.cu_q_lens, inp.start_pos,
                       inp.block_table, inp.k_pools[layer], inp.v_pools[layer])
    q = inp.q[layer]
    max_s = int(inp.host_seq_lens.max())
    po, pl = pa.attn_prefill_chunk(q[:chunk_rows], inp.cu_q_lens[:2], inp.k_pools[layer],
                                   inp.v_pools[layer], inp.block_table[:1], inp.seq_lens[:1],
                                   chunk_rows, max_s, inp.scale)
    do, dl = pa.attn_decode_paged(q[chunk_rows:], inp.k_pools[layer], inp.v_pools[layer],
                                  inp.block_table[1:], inp.seq_lens[1:], max_s, inp.scale,
                                  workspace=ws)
    return po, pl, do, dl


def oracle_mixed(inp, layer, k_before, v_before, chunk_rows, prefill_rows=None, decode_seqs=None):
    k, v = oracle.kv_append(bits(inp.k_new[layer]), bits(inp.v_new[layer]), host(inp.cu_q_lens),
                            host(inp.start_pos), inp.host_block_table, k_before, v_before)
    q = bits(inp.q[layer])
    po, pl = oracle.prefill(q[:chunk_rows], [0, chunk_rows], k, v, inp.host_block_table[:1],
                            inp.host_seq_lens[:1], inp.scale, rows=prefill_rows, threads=16)
    do, dl = oracle.decode(q[chunk_rows:], k, v, inp.host_block_table[1:],
                           inp.host_seq_lens[1:], inp.scale, seqs=decode_seqs, threads=16)
    return po, pl, do, dl


def test_mixed_step_reduced(cuda_lib):
    """Two layers; a 256-query chunk at offset 2,048 plus 7 decodes of 500..9,000 keys."""
    dec = [500, 9000, 1234, 16, 4097, 7777, 31]
    inp = W.make_paged(400, [2048 + 256] + dec, [256] + [1] * 7, layers=2, device="cuda")
    for layer in range(2):
        kb, vb = bits(inp.k_pools[layer]).copy(), bits(inp.v_pools[layer]).copy()
        po, pl, do, dl = mixed_step(cuda_lib, inp, layer, 256)
        torch.cuda.synchronize()
        ro = oracle_mixed(inp, layer, kb, vb, 256)
        check_attn(po, pl, ro[0], ro[1], what=f"layer {layer} prefill")
        check_attn(do, dl, ro[2], ro[3], what=f"layer {layer} decode")


def chunk_rows_256(n, rng):
    """256 rows of a chunk of n: the first and last 16, the rows around every 16-key page edge
    and 128-query tile edge that fall on them, the rest random."""
    rows = set(range(16)) | set(range(n - 16, n))
    edges = set()
    for e in range(128, n, 128):
        edges |= {e - 1, e, e + 1}
    for e in range(16, n, 16 * 37):          # page edges spread across the chunk
        edges |= {e - 1, e}
    rows |= set(sorted(edges)[:96])
    while len(rows) < 256:
        rows.add(int(rng.integers(0, n)))
    return sorted(rows)


def test_mixed_step_full_size(cuda_lib):
    """The 28-layer mixed workload at full size (about 173 GB of pools), in the bench's launch
    configuration: on layers 0 and 27 and two more drawn by seed, every decode sequence and
    256 rows of the chunk (every head; on layer 0 all 4,096 rows) are checked against the oracle,
    which appends the new tokens itself into the pools as they were before the step."""
    free, _ = torch.cuda.mem_get_info()
    L, ql = W.lengths_for("mixed_28l")
    need = 28 * 2 * int((-(-L // 16)).sum() + 16) * 32768 + (8 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free, have {free / 2**30:.0f} GiB")
    inp = W.make_workload("mixed_28l", device="cuda")
    rng = np.random.default_rng(5)
    check_layers = {0, 27} | set(int(x) for x in rng.choice(np.arange(1, 27), size=2, replace=False))
    saved = {l: (bits(inp.k_pools[l]).copy(), bits(inp.v_pools[l]).copy()) for l in check_layers}
    outs = {}
    for layer in range(28):
        r = mixed_step(cuda_lib, inp, layer, 4096)
        if layer in check_layers:
            outs[layer] = tuple(t.clone() for t in r)
    torch.cuda.synchronize()
    rows = chunk_rows_256(4096, rng)
    assert len(rows) == 256
    for layer in sorted(check_layers):
        kb, vb = saved.pop(layer)
        # layer 0: every row of the chunk; the others: the 256 sampled rows
        layer_rows = None if layer == 0 else rows
        ro = oracle_mixed(inp, layer, kb, vb, 4096, prefill_rows=layer_rows)
        po, pl, do, dl = outs[layer]
        check_attn(po, pl, ro[0], ro[1], rows=layer_rows,
                   what=f"layer {layer} prefill ({'all 4,096 rows' if layer_rows is None else '256 rows'})")
        check_attn(do, dl, ro[2], ro[3], what=f"layer {layer} decode (all 31 sequences)")


@pytest.mark.parametrize("split", [(80, 72), (120, 32), (8, 144)])
def test_mixed_step_overlapped_on_two_streams(cuda_lib, split):
    """The bench's whole-step form: after each layer's append, the prefill runs on the current
    stream with its grid capped at split[0] CTAs and the decode on a second stream capped at
    split[1], both captured in one CUDA graph and replayed; every row checked against the
    oracle (reduced sizes, two layers)."""
    dec = [500, 9000, 1234, 16, 4097, 7777, 31]
    inp = W.make_paged(400, [2048 + 256] + dec, [256] + [1] * 7, layers=2, device="cuda")
    kb = [bits(inp.k_pools[l]).copy() for l in range(2)]
    vb = [bits(inp.v_pools[l]).copy() for l in range(2)]
    max_s = int(inp.host_seq_lens.max())
    dev = inp.q[0].device
    side = torch.cuda.Stream(device=dev)
    outs = [(torch.empty(256, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev),
             torch.empty(256, W.HQ, dtype=torch.float32, device=dev),
             torch.empty(7, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev),
             torch.empty(7, W.HQ, dtype=torch.float32, device=dev)) for _ in range(2)]
    dws = torch.empty(cuda_lib.decode_workspace_size(7, max_s), dtype=torch.uint8, device=dev)
    pws = torch.empty(max(256, cuda_lib.prefill_workspace_size(1, 256, max_s)), dtype=torch.uint8,
                      device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        stream = torch.cuda.current_stream()
        for layer in range(2):
            cuda_lib.kv_append_paged(inp.k_new[layer], inp.v_new[layer], inp.cu_q_lens,
                                     inp.start_pos, inp.block_table, inp.k_pools[layer],
                                     inp.v_pools[layer], status=status, stream=stream)
            side.wait_stream(stream)
            po, pl, do, dl = outs[layer]
            q = inp.q[layer]
            cuda_lib.attn_prefill_chunk(q[:256], inp.cu_q_lens[:2], inp.k_pools[layer],
                                        inp.v_pools[layer], inp.block_table[:1], inp.seq_lens[:1],
                                        256, max_s, inp.scale, out=po, lse=pl, workspace=pws,
                                        status=status, stream=stream, max_ctas=split[0])
            cuda_lib.attn_decode_paged(q[256:], inp.k_pools[layer], inp.v_pools[layer],
                                       inp.block_table[1:], inp.seq_lens[1:], max_s, inp.scale,
                                       out=do, lse=dl, workspace=dws, status=status, stream=side,
                                       max_ctas=split[1])
            stream.wait_stream(side)

    g = torch.cuda.CUDAGraph()
    s0 = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s0):
        with torch.cuda.graph(g):
            step()
    g.replay()  # the append is idempotent: the same tokens land in the same slots
    torch.cuda.synchronize()
    assert cuda_lib.read_device_status(status) == 0
    for layer in range(2):
        ro = oracle_mixed(inp, layer, kb[layer], vb[layer], 256)
        po, pl, do, dl = outs[layer]
        check_attn(po, pl, ro[0], ro[1], what=f"overlapped layer {layer} prefill {split}")
        check_attn(do, dl, ro[2], ro[3], what=f"overlapped layer {layer} decode {split}")
