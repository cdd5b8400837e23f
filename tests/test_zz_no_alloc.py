"""attn_decode_paged_noalloc: decode for callers that cannot allocate device memory.

Such callers (an engine whose KV-cache pool already holds all free HBM, a plugin host without
an allocator, a loop where cudaMalloc may synchronize the device) get a decode whose scratch is
a fixed array inside the library. This file is collected last on purpose. The test calls the
entry point through the C ABI twice in a row, on different batches, and compares each result
with attn_decode_paged's (which uses a caller-provided workspace) within the parity tolerance.
"""
import ctypes

import pytest
import torch

import workloads as W
from helpers import ATOL, LSE_ATOL, RTOL

pytestmark = pytest.mark.gpu


def _noalloc_call(lib, pa, inp, max_seq_len, out, lse):
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    return lib.attn_decode_paged_noalloc(
        pa.Dims(*pa.DEFAULT_DIMS), P(inp.q[0].data_ptr()), P(inp.k_pools[0].data_ptr()),
        P(inp.v_pools[0].data_ptr()), inp.k_pools[0].shape[0], P(inp.block_table.data_ptr()),
        inp.block_table.shape[1], P(inp.seq_lens.data_ptr()), inp.batch, max_seq_len,
        ctypes.c_float(inp.scale), P(out.data_ptr()), P(lse.data_ptr()), None, stream)


def _close(a, b, atol, rtol):
    a, b = a.float(), b.float()
    return bool(torch.all((a - b).abs() <= atol + rtol * b.abs()))


def test_noalloc_decode_matches_workspace_decode_twice(cuda_lib):
    pa = cuda_lib
    lib = pa.load()
    cases = [([30000, 700, 12000, 5, 0, 45000], 21), ([1000] * 9 + [60000], 22)]
    for lens, seed in cases:
        inp = W.make_paged(seed, lens, [1] * len(lens), device="cuda")
        max_s = max(lens)
        out = torch.full_like(inp.q[0], float("nan"))
        lse = torch.full((inp.batch, W.HQ), float("nan"), device="cuda")
        rc = _noalloc_call(lib, pa, inp, max_s, out, lse)
        assert rc == 0, lib.pa_last_error()
        ref_o, ref_l = pa.attn_decode_paged(inp.q[0], inp.k_pools[0], inp.v_pools[0],
                                            inp.block_table, inp.seq_lens, max_s, inp.scale)
        torch.cuda.synchronize()
        assert _close(out, ref_o, ATOL, RTOL)
        fin = torch.isfinite(ref_l)
        assert torch.equal(fin, torch.isfinite(lse))
        assert bool(torch.all((lse[fin] - ref_l[fin]).abs() <= LSE_ATOL))


def test_noalloc_rejects_batches_beyond_its_scratch(cuda_lib):
    pa = cuda_lib
    lib = pa.load()
    inp = W.make_paged(23, [16] * 2000, [1] * 2000, device="cuda")
    out = torch.empty_like(inp.q[0])
    lse = torch.empty(inp.batch, W.HQ, device="cuda")
    rc = _noalloc_call(lib, pa, inp, 16, out, lse)
    assert rc == 3
    assert b"built-in" in lib.pa_last_error()
