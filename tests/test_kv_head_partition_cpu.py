"""The exchange of a KV-head (tensor-parallel) partition on CPU with gloo (world size 2).

Each rank holds half of the KV heads of every page and the query heads that read them,
computes its heads' decode and chunked-prefill attention with the oracle, and the ranks
all-gather their outputs along the head axis. The gathered result must equal the
single-process oracle on all heads: attention of one head depends only on its own K/V, so the
partition needs no other exchange."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    rng = np.random.default_rng(11)
    Hq, Hkv, D, P = 16, 8, 128, 16
    lens = [70, 300, 1, 33]
    q_lens = [20, 1, 1, 1]
    n_pages = [-(-L // P) for L in lens]
    NP = sum(n_pages) + 2
    perm = rng.permutation(NP)
    bt = np.zeros((len(lens), max(n_pages)), dtype=np.int32)
    off = 0
    for b, n in enumerate(n_pages):
        bt[b, :n] = perm[off:off + n]
        off += n
    k = rng.standard_normal((NP, P, Hkv, D))
    v = rng.standard_normal((NP, P, Hkv, D))
    q = rng.standard_normal((sum(q_lens), Hq, D))
    return q, k, v, bt, np.array(lens), np.array(q_lens), 0.088


def _attention(q, k, v, bt, lens, q_lens, scale):
    import oracle
    n = int(q_lens[0])
    po, pl = oracle.prefill(q[:n], [0, n], k, v, bt[:1], lens[:1], scale)
    do, dl = oracle.decode(q[n:], k, v, bt[1:], lens[1:], scale)
    return np.concatenate([po, do]), np.concatenate([pl, dl])


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v, bt, lens, q_lens, scale = _inputs()
    hk = k.shape[2] // world
    h0, h1 = rank * hk, (rank + 1) * hk
    o, lse = _attention(q[:, 2 * h0:2 * h1], k[:, :, h0:h1], v[:, :, h0:h1], bt, lens, q_lens, scale)
    o_t, l_t = torch.from_numpy(np.ascontiguousarray(o)), torch.from_numpy(np.ascontiguousarray(lse))
    o_all = [torch.empty_like(o_t) for _ in range(world)]
    l_all = [torch.empty_like(l_t) for _ in range(world)]
    dist.all_gather(o_all, o_t)
    dist.all_gather(l_all, l_t)
    out[rank] = (torch.cat(o_all, dim=1).numpy(), torch.cat(l_all, dim=1).numpy())
    dist.destroy_process_group()


def test_two_rank_head_split_gathers_to_the_whole():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    ref_o, ref_l = _attention(*_inputs())
    for r in range(world):
        mo, ml = out[r]
        assert np.array_equal(mo, ref_o) and np.array_equal(ml, ref_l)
