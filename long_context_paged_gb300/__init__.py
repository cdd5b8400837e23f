"""GB300-native paged GQA attention: Python binding of ``libpagedattn.so``.

Thin ctypes marshalling over the C ABI in ``include/pagedattn.h``: every computation runs in
the library's CUDA kernels. PyTorch only provides device memory and streams. There is no CPU
or fallback path: if the shared library has not been built, ``load()`` raises.

Calls (same names as the C ABI):

* ``kv_append_paged``   write new tokens' K/V rows into their page slots
* ``attn_decode_paged`` one decode step over a paged KV cache (split-KV + log-sum-exp merge)
* ``attn_prefill_chunk`` causal attention of query chunks over their cached prefix + themselves
* ``attn_merge_lse``    combine partial results over disjoint key sets
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "load", "PagedAttnError", "Dims", "DEFAULT_DIMS",
    "kv_append_paged", "attn_decode_paged", "attn_decode_paged_noalloc", "attn_prefill_chunk",
    "attn_merge_lse", "adaptor_mlp_merge4", "adaptor_workspace_size", "LaunchOpts",
    "decode_workspace_size", "decode_kernels_per_call", "prefill_workspace_size",
    "read_device_status", "debug_decode_starve",
    "DEV_ERR_PAGE_OOB", "DEV_ERR_LENGTH", "DEV_ERR_TIMEOUT", "DEV_ERR_INTERNAL", "lib_path",
]

DEV_ERR_PAGE_OOB = 1
DEV_ERR_LENGTH = 2
DEV_ERR_TIMEOUT = 4
DEV_ERR_INTERNAL = 8

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def lib_path() -> str:
    return os.path.join(_HERE, "_lib", "libpagedattn.so")


class Dims(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32)]


DEFAULT_DIMS = (16, 8, 128, 16)


class PagedAttnError(RuntimeError):
    def __init__(self, call: str, code: int):
        lib = load()
        text = lib.pa_status_string(code).decode()
        detail = lib.pa_last_error().decode()
        super().__init__(f"{call} failed: {text} ({code}){': ' + detail if detail else ''}")
        self.code = code


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float

class LaunchOpts(ctypes.Structure):
    """pa_launch_opts: max_ctas > 0 caps a call's persistent grid (0 = one CTA per SM)."""
    _fields_ = [("max_ctas", ctypes.c_int32)]


def _opts(max_ctas):
    if max_ctas is None:
        return None, None
    m = int(max_ctas)
    if m < 0:
        raise ValueError("max_ctas must be >= 0")
    o = LaunchOpts(m)
    return o, ctypes.byref(o)


_SIGS = {
    "kv_append_paged": (_I32, [Dims, _P, _P, _I32, _P, _P, _I32, _P, _I32, _P, _P, _I64, _P, _P]),
    "pa_decode_workspace_size": (_SZ, [Dims, _I32, _I32, _I32]),
    "pa_decode_kernels_per_call": (_I32, [Dims, _I32, _I32, _I32]),
    "attn_decode_paged": (_I32, [Dims, _P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _F, _I32, _P, _P,
                                 _P, _SZ, _P, _P]),
    "pa_debug_decode_starve": (_I32, [_I32]),
    "attn_decode_paged_noalloc": (_I32, [Dims, _P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _F, _P,
                                         _P, _P, _P]),
    "pa_prefill_workspace_size": (_SZ, [Dims, _I32, _I32, _I32]),
    "attn_prefill_chunk": (_I32, [Dims, _P, _P, _I32, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32,
                                  _F, _P, _P, _P, _SZ, _P, _P]),
    "attn_decode_paged_ex": (_I32, [Dims, _P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _F, _I32, _P,
                                    _P, _P, _SZ, _P, _P, _P]),
    "attn_prefill_chunk_ex": (_I32, [Dims, _P, _P, _I32, _P, _P, _I64, _P, _I32, _P, _I32, _I32,
                                     _I32, _F, _P, _P, _P, _SZ, _P, _P, _P]),
    "attn_merge_lse": (_I32, [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "pa_adaptor_workspace_size": (_SZ, [_I32]),
    "adaptor_mlp_merge4": (_I32, [_I32, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P, _SZ, _P, _P]),
    "pa_read_device_status": (_I32, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
    "pa_status_string": (ctypes.c_char_p, [_I32]),
    "pa_last_error": (ctypes.c_char_p, []),
    "pa_version": (_I32, []),
}


def load():
    """Load the built library (raises if it is missing: there is no fallback)."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


# ----------------------------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------------------------
def _dims(dims):
    return Dims(*(dims or DEFAULT_DIMS))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _check(call, code):
    if code != 0:
        raise PagedAttnError(call, code)


def _on_device(call, *tensors):
    """Every tensor must live on the current CUDA device: the library launches there, and a
    pointer into another GPU's memory would be read by the wrong device."""
    dev = torch.cuda.current_device()
    for t in tensors:
        if t is not None and t.device.index != dev:
            raise ValueError(f"{call}: tensors must be on the current CUDA device (cuda:{dev}), "
                             f"got {t.device}")


def _shape(name, t, shape):
    """t must have this shape (None entries match anything)."""
    if t.dim() != len(shape) or any(w is not None and d != w for d, w in zip(t.shape, shape)):
        raise ValueError(f"{name} must have shape {tuple('*' if w is None else w for w in shape)}, "
                         f"got {tuple(t.shape)}")


def _rows_at_least(name, t, n):
    if t.shape[0] < n:
        raise ValueError(f"{name} must have at least {n} rows, got {t.shape[0]}")


def _heads(dims):
    """(query heads, KV heads) of a shape the library supports, else None: the library itself
    then rejects the call (PA_ERR_UNSUPPORTED) and the shape checks below are skipped."""
    d = _dims(dims)
    if (d.head_dim == 128 and d.page_size == 16 and d.num_kv_heads in (1, 2, 4, 8)
            and d.num_q_heads == 2 * d.num_kv_heads):
        return d.num_q_heads, d.num_kv_heads
    return None


def _pools(k_pool, v_pool, hkv):
    _shape("k_pool", k_pool, (None, 16, hkv, 128))
    _shape("v_pool", v_pool, tuple(k_pool.shape))


def _given(t, name, dtype, shape):
    """A caller-provided output buffer: dtype, layout and shape checked, since the kernels write
    every element of it."""
    if t is not None:
        _need(t, name, dtype)
        _shape(name, t, shape)


# ----------------------------------------------------------------------------------------------
# the four calls
# ----------------------------------------------------------------------------------------------
def kv_append_paged(k_new, v_new, cu_new_lens, start_pos, block_table, k_pool, v_pool, *,
                    status=None, stream=None, dims=None):
    """Write rows of k_new/v_new [T, Hkv, D] into the pools at their block-table slots."""
    for t, n, d in ((k_new, "k_new", torch.bfloat16), (v_new, "v_new", torch.bfloat16),
                    (cu_new_lens, "cu_new_lens", torch.int32), (start_pos, "start_pos", torch.int32),
                    (block_table, "block_table", torch.int32), (k_pool, "k_pool", torch.bfloat16),
                    (v_pool, "v_pool", torch.bfloat16)):
        _need(t, n, d)
    B = start_pos.shape[0]
    _rows_at_least("cu_new_lens", cu_new_lens, B + 1)
    _rows_at_least("block_table", block_table, B)
    heads = _heads(dims)
    if heads is not None:
        _shape("k_new", k_new, (None, heads[1], 128))
        _shape("v_new", v_new, tuple(k_new.shape))
        _pools(k_pool, v_pool, heads[1])
    if status is not None:
        _need(status, "status", torch.int32)
    _on_device("kv_append_paged", k_new, v_new, cu_new_lens, start_pos, block_table, k_pool,
               v_pool, status)
    lib = load()
    _check("kv_append_paged", lib.kv_append_paged(
        _dims(dims), _ptr(k_new), _ptr(v_new), k_new.shape[0], _ptr(cu_new_lens), _ptr(start_pos),
        start_pos.shape[0], _ptr(block_table), block_table.shape[1], _ptr(k_pool), _ptr(v_pool),
        k_pool.shape[0], _ptr(status), _stream(stream)))


def decode_workspace_size(batch: int, max_seq_len: int, split_tokens: int = 0, dims=None) -> int:
    return int(load().pa_decode_workspace_size(_dims(dims), batch, max_seq_len, split_tokens))


def decode_kernels_per_call(batch: int, max_seq_len: int, split_tokens: int = 0, dims=None) -> int:
    """Kernels one attn_decode_paged call launches (1: single-launch short-batch path, 2: split
    kernel + merge; 0 for an empty or unsupported call)."""
    return int(load().pa_decode_kernels_per_call(_dims(dims), batch, max_seq_len, split_tokens))


def prefill_workspace_size(batch: int, max_q_len: int, max_seq_len: int, dims=None) -> int:
    return int(load().pa_prefill_workspace_size(_dims(dims), batch, max_q_len, max_seq_len))


def _workspace(nbytes, device, workspace):
    if workspace is not None:
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def attn_decode_paged(q, k_pool, v_pool, block_table, seq_lens, max_seq_len: int,
                      softmax_scale: float, *, split_tokens: int = 0, out=None, lse=None,
                      workspace=None, status=None, stream=None, want_lse=True, dims=None,
                      max_ctas=None):
    """Decode attention: q [B, Hq, D] over each sequence's cached keys. Returns (out, lse).

    split_tokens: keys per split-KV range (whole pages); 0 = one equal share per SM.
    max_ctas: cap on the persistent grid (attn_decode_paged_ex); None = the plain call."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B = q.shape[0]
    _rows_at_least("block_table", block_table, B)
    _rows_at_least("seq_lens", seq_lens, B)
    heads = _heads(dims)
    if heads is not None:
        _shape("q", q, (B, heads[0], 128))
        _pools(k_pool, v_pool, heads[1])
        _given(out, "out", torch.bfloat16, (B, heads[0], 128))
        _given(lse, "lse", torch.float32, (B, heads[0]))
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(B, q.shape[1], dtype=torch.float32, device=q.device)
    ws_bytes = decode_workspace_size(B, max_seq_len, split_tokens, dims)
    workspace = _workspace(ws_bytes, q.device, workspace)
    if status is not None:
        _need(status, "status", torch.int32)
    _on_device("attn_decode_paged", q, k_pool, v_pool, block_table, seq_lens, out, lse,
               workspace, status)
    lib = load()
    args = (_dims(dims), _ptr(q), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(block_table),
            block_table.shape[1], _ptr(seq_lens), B, int(max_seq_len), float(softmax_scale),
            int(split_tokens), _ptr(out), _ptr(lse), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    keep, ref = _opts(max_ctas)
    if ref is None:
        _check("attn_decode_paged", lib.attn_decode_paged(*args))
    else:
        _check("attn_decode_paged_ex", lib.attn_decode_paged_ex(*args, ref))
    del keep
    return out, lse


def attn_decode_paged_noalloc(q, k_pool, v_pool, block_table, seq_lens, max_seq_len: int,
                              softmax_scale: float, *, out, lse=None, status=None, stream=None,
                              dims=None):
    """attn_decode_paged with the library's fixed scratch array instead of a workspace.

    For callers that cannot allocate device memory: out (and lse, if wanted) must be given;
    nothing is allocated here or in the library. Calls that overlap on the GPU race on the
    shared scratch and must be serialized by the caller."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    B = q.shape[0]
    _rows_at_least("block_table", block_table, B)
    _rows_at_least("seq_lens", seq_lens, B)
    heads = _heads(dims)
    if heads is not None:
        _shape("q", q, (B, heads[0], 128))
        _pools(k_pool, v_pool, heads[1])
        _given(out, "out", torch.bfloat16, (B, heads[0], 128))
        _given(lse, "lse", torch.float32, (B, heads[0]))
    if status is not None:
        _need(status, "status", torch.int32)
    _on_device("attn_decode_paged_noalloc", q, k_pool, v_pool, block_table, seq_lens, out, lse,
               status)
    lib = load()
    _check("attn_decode_paged_noalloc", lib.attn_decode_paged_noalloc(
        _dims(dims), _ptr(q), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), q.shape[0], int(max_seq_len), float(softmax_scale),
        _ptr(out), _ptr(lse), _ptr(status), _stream(stream)))
    return out, lse


def attn_prefill_chunk(q, cu_q_lens, k_pool, v_pool, block_table, seq_lens, max_q_len: int,
                       max_seq_len: int, softmax_scale: float, *, out=None, lse=None,
                       workspace=None, status=None, stream=None, want_lse=True, dims=None,
                       max_ctas=None):
    """Chunked prefill: q [Tq, Hq, D] packed by cu_q_lens. Returns (out, lse).

    max_ctas: cap on the persistent grid (attn_prefill_chunk_ex); None = the plain call."""
    _need(q, "q", torch.bfloat16, 3)
    _need(cu_q_lens, "cu_q_lens", torch.int32, 1)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B = seq_lens.shape[0]
    Tq = q.shape[0]
    _rows_at_least("cu_q_lens", cu_q_lens, B + 1)
    _rows_at_least("block_table", block_table, B)
    heads = _heads(dims)
    if heads is not None:
        _shape("q", q, (Tq, heads[0], 128))
        _pools(k_pool, v_pool, heads[1])
        _given(out, "out", torch.bfloat16, (Tq, heads[0], 128))
        _given(lse, "lse", torch.float32, (Tq, heads[0]))
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    ws_bytes = prefill_workspace_size(B, max_q_len, max_seq_len, dims)
    if ws_bytes > 0:
        workspace = _workspace(ws_bytes, q.device, workspace)
    if status is not None:
        _need(status, "status", torch.int32)
    _on_device("attn_prefill_chunk", q, cu_q_lens, k_pool, v_pool, block_table, seq_lens, out,
               lse, workspace, status)
    lib = load()
    args = (_dims(dims), _ptr(q), _ptr(cu_q_lens), q.shape[0], _ptr(k_pool), _ptr(v_pool),
            k_pool.shape[0], _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B,
            int(max_q_len), int(max_seq_len), float(softmax_scale), _ptr(out), _ptr(lse),
            _ptr(workspace),
            0 if workspace is None else workspace.numel() * workspace.element_size(),
            _ptr(status), _stream(stream))
    keep, ref = _opts(max_ctas)
    if ref is None:
        _check("attn_prefill_chunk", lib.attn_prefill_chunk(*args))
    else:
        _check("attn_prefill_chunk_ex", lib.attn_prefill_chunk_ex(*args, ref))
    del keep
    return out, lse


def attn_merge_lse(o_parts, lse_parts, *, out=None, lse_out=None, stream=None):
    """o_parts fp32 [S, R, H, D], lse_parts fp32 [S, R, H] -> (out bf16 [R, H, D], lse [R, H])."""
    _need(o_parts, "o_parts", torch.float32, 4)
    _need(lse_parts, "lse_parts", torch.float32, 3)
    S, R, H, D = o_parts.shape
    _shape("lse_parts", lse_parts, (S, R, H))
    _given(out, "out", torch.bfloat16, (R, H, D))
    _given(lse_out, "lse_out", torch.float32, (R, H))
    if out is None:
        out = torch.empty(R, H, D, dtype=torch.bfloat16, device=o_parts.device)
    if lse_out is None:
        lse_out = torch.empty(R, H, dtype=torch.float32, device=o_parts.device)
    _on_device("attn_merge_lse", o_parts, lse_parts, out, lse_out)
    lib = load()
    _check("attn_merge_lse", lib.attn_merge_lse(S, R, H, D, _ptr(o_parts), _ptr(lse_parts),
                                                _ptr(out), _ptr(lse_out), _stream(stream)))
    return out, lse_out


def adaptor_workspace_size(num_frames: int) -> int:
    return int(load().pa_adaptor_workspace_size(num_frames))


def adaptor_mlp_merge4(frames, w1, b1, w2, b2, gamma, beta, eps: float = 1e-5, *, out=None,
                       workspace=None, status=None, stream=None):
    """Decoder embeddings from encoder frames [T_enc, 1024]: 4x merge, Linear-SiLU-Linear-
    LayerNorm. Returns out bf16 [T_enc / 4, 1024]."""
    _need(frames, "frames", torch.bfloat16, 2)
    _need(w1, "w1", torch.bfloat16, 2)
    _need(w2, "w2", torch.bfloat16, 2)
    for t, n in ((b1, "b1"), (b2, "b2"), (gamma, "gamma"), (beta, "beta")):
        _need(t, n, torch.float32, 1)
    n_frames = frames.shape[0]
    T = n_frames // 4
    _shape("frames", frames, (n_frames, 1024))
    _shape("w1", w1, (1024, 4096))
    _shape("w2", w2, (1024, 1024))
    for t, n in ((b1, "b1"), (b2, "b2"), (gamma, "gamma"), (beta, "beta")):
        _shape(n, t, (1024,))
    _given(out, "out", torch.bfloat16, (T, 1024))
    if out is None:
        out = torch.empty(T, 1024, dtype=torch.bfloat16, device=frames.device)
    if workspace is None:
        workspace = torch.empty(max(256, adaptor_workspace_size(n_frames)), dtype=torch.uint8,
                                device=frames.device)
    if status is not None:
        _need(status, "status", torch.int32)
    _on_device("adaptor_mlp_merge4", frames, w1, b1, w2, b2, gamma, beta, out, workspace, status)
    lib = load()
    _check("adaptor_mlp_merge4", lib.adaptor_mlp_merge4(
        n_frames, _ptr(frames), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2), _ptr(gamma), _ptr(beta),
        float(eps), _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream)))
    return out


def debug_decode_starve(enable: bool) -> None:
    """Test hook: later decode launches of this thread leave one ring stage empty and bound
    their waits by 1 ms, so the bounded-wait give-up path runs (status PA_DEV_ERR_TIMEOUT)."""
    _check("pa_debug_decode_starve", load().pa_debug_decode_starve(1 if enable else 0))


def read_device_status(status, stream=None) -> int:
    """Wait for the stream, return the device status bits and clear them."""
    _need(status, "status", torch.int32)
    flags = ctypes.c_uint32(0)
    _check("pa_read_device_status", load().pa_read_device_status(_ptr(status), ctypes.byref(flags),
                                                                 _stream(stream)))
    return int(flags.value)
