"""The exchange step of a context-parallel decode on CPU with gloo (world size 2): each rank
holds half of every sequence's keys, computes its partial (o, lse) with the oracle, the ranks
all-gather the partials, and every rank merges them by log-sum-exp. The merged result must
equal the single-process oracle on the whole cache."""
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
    rng = np.random.default_rng(9)
    Hq, Hkv, D, P = 16, 8, 128, 16
    lens = [37, 300, 1]
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
    q = rng.standard_normal((len(lens), Hq, D))
    return q, k, v, bt, np.array(lens), 0.088


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    q, k, v, bt, lens, scale = _inputs()
    sub_lens, sub_bt = [], np.zeros_like(bt)
    for b, L in enumerate(lens):
        n = -(-L // 16)
        p0, p1 = n * rank // world, n * (rank + 1) // world
        sub_lens.append(max(0, min(L, p1 * 16) - p0 * 16))
        sub_bt[b, :p1 - p0] = bt[b, p0:p1]
    o, lse = oracle.decode(q, k, v, sub_bt, sub_lens, scale)
    o_t, l_t = torch.from_numpy(o), torch.from_numpy(lse)
    o_all = [torch.empty_like(o_t) for _ in range(world)]
    l_all = [torch.empty_like(l_t) for _ in range(world)]
    dist.all_gather(o_all, o_t)
    dist.all_gather(l_all, l_t)
    mo, ml = oracle.merge_lse(torch.stack(o_all).numpy(), torch.stack(l_all).numpy())
    out[rank] = (mo, ml)
    dist.destroy_process_group()


def test_two_rank_key_split_merges_to_the_whole():
    import oracle
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
    q, k, v, bt, lens, scale = _inputs()
    ref_o, ref_l = oracle.decode(q, k, v, bt, lens, scale)
    for r in range(world):
        mo, ml = out[r]
        np.testing.assert_allclose(mo, ref_o, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(ml, ref_l, rtol=1e-13)
