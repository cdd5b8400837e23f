"""Shared test helpers: moving bytes to the oracle and the parity tolerance.

Tolerance (the decode/prefill outputs are bf16, accumulation fp32): every output element must
satisfy |gpu - ref| <= 4e-3 + 8e-3 * |ref| against the unrounded fp64 oracle, and every LSE
|gpu - ref| <= 1e-3. Block-table indexing and KV append placement are compared bit for bit.
"""
import numpy as np
import torch

ATOL = 4e-3
RTOL = 8e-3
LSE_ATOL = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> int16 numpy array of its bit patterns (the oracle widens them exactly)."""
    return t.detach().view(torch.int16).cpu().numpy()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def check_attn(out, lse, ref_o, ref_lse, rows=None, what=""):
    """Compare GPU (out bf16 [R, H, D], lse fp32 [R, H]) against oracle fp64 arrays.

    ``rows`` restricts the comparison to those row indices (the oracle computed only them)."""
    o = out.detach().float().cpu().numpy().astype(np.float64)
    ref_o = np.asarray(ref_o)
    ref_lse = np.asarray(ref_lse)
    if rows is not None:
        rows = np.asarray(rows)
        o, ref_o, ref_lse = o[rows], ref_o[rows], ref_lse[rows]
    err = np.abs(o - ref_o)
    bound = ATOL + RTOL * np.abs(ref_o)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} output elements out of tolerance, e.g. "
                             + ", ".join(f"{tuple(i)} gpu={o[tuple(i)]:.6g} ref={ref_o[tuple(i)]:.6g}"
                                         for i in idx))
    if lse is not None:
        l = lse.detach().cpu().numpy().astype(np.float64)
        if rows is not None:
            l = l[rows]
        inf_ref = np.isneginf(ref_lse)
        assert np.array_equal(np.isneginf(l), inf_ref), f"{what}: -inf LSE pattern differs"
        d = np.abs(l[~inf_ref] - ref_lse[~inf_ref])
        assert d.size == 0 or d.max() <= LSE_ATOL, f"{what}: LSE error {d.max():.3g} > {LSE_ATOL}"
    return float(err.max()) if err.size else 0.0
