"""Host-side checks of the C ABI (no GPU needed): the library builds for sm_103a, loads, and
exports every function that include/*.h declares; argument errors are rejected before any
CUDA call."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from long_context_paged_gb300 import build as b
    b.build()
    import long_context_paged_gb300 as pa
    return pa.load()


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("kv_append_paged", "attn_decode_paged", "attn_prefill_chunk", "attn_merge_lse"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert lib.pa_status_string(0) == b"ok"
    assert lib.pa_status_string(3) == b"workspace too small"
    assert lib.pa_version() >= 100


def test_argument_errors_are_rejected_before_launch(lib):
    import long_context_paged_gb300 as pa
    bad_dims = pa.Dims(16, 8, 64, 16)
    good = pa.Dims(*pa.DEFAULT_DIMS)
    null = None
    # unsupported shape
    assert lib.attn_decode_paged(bad_dims, null, null, null, 1, null, 1, null, 1, 16, 1.0, 0,
                                 null, null, null, 0, null, null) == 2
    assert lib.attn_prefill_chunk(pa.Dims(16, 4, 128, 16), null, null, 1, null, null, 1, null, 1,
                                  null, 1, 1, 16, 1.0, null, null, null, 0, null, null) == 2
    assert lib.kv_append_paged(pa.Dims(16, 8, 128, 32), null, null, 1, null, null, 1, null, 1,
                               null, null, 1, null, null) == 2
    # negative sizes / null pointers
    assert lib.attn_decode_paged(good, null, null, null, 1, null, 1, null, -1, 16, 1.0, 0,
                                 null, null, null, 0, null, null) == 1
    assert lib.attn_decode_paged(good, null, null, null, 1, null, 1, null, 2, 16, 1.0, 0,
                                 null, null, null, 0, null, null) == 1
    assert lib.attn_decode_paged(good, null, null, null, 1, null, 1, null, 1, 200000, 1.0, 0,
                                 null, null, null, 0, null, null) == 1
    assert lib.kv_append_paged(good, null, null, -3, null, null, 1, null, 1,
                               null, null, 1, null, null) == 1
    assert lib.attn_merge_lse(2, 3, 4, 130, null, null, null, null, null) == 2
    assert lib.attn_merge_lse(-1, 3, 4, 128, null, null, null, null, null) == 1
    # empty work is a no-op success
    assert lib.attn_decode_paged(good, null, null, null, 1, null, 1, null, 0, 16, 1.0, 0,
                                 null, null, null, 0, null, null) == 0
    assert lib.attn_merge_lse(1, 0, 16, 128, null, null, null, null, null) == 0
    assert lib.pa_read_device_status(null, null, null) == 1


def test_decode_kernels_per_call_query(lib):
    """pa_decode_kernels_per_call: 0 for unsupported dims or an empty or invalid call, else 1
    (single-launch path) or 2 (split + merge); explicit split sizes always take the split path.
    It launches nothing, so it runs without a GPU (where it can only answer 2)."""
    import long_context_paged_gb300 as pa
    good = pa.Dims(*pa.DEFAULT_DIMS)
    assert lib.pa_decode_kernels_per_call(pa.Dims(16, 8, 64, 16), 1, 1000, 0) == 0
    assert lib.pa_decode_kernels_per_call(good, 0, 1000, 0) == 0
    assert lib.pa_decode_kernels_per_call(good, 1, -1, 0) == 0
    assert lib.pa_decode_kernels_per_call(good, 1, 1000, -1) == 0
    assert lib.pa_decode_kernels_per_call(good, 1, 1000, 0) in (1, 2)
    assert lib.pa_decode_kernels_per_call(good, 1, 1000, 256) == 2
    assert lib.pa_decode_kernels_per_call(good, 64, 90000, 0) == 2


def test_prefill_argument_errors_are_rejected_before_launch(lib):
    """attn_prefill_chunk's checks, each before any CUDA call. Every case here must be rejected:
    the pointers are fake (aligned, non-null host addresses) and are never dereferenced."""
    import long_context_paged_gb300 as pa
    good = pa.Dims(*pa.DEFAULT_DIMS)
    null = None
    a = ctypes.c_void_p(1 << 20)     # fake 16-byte-aligned address
    mis = ctypes.c_void_p((1 << 20) + 8)

    def call(q=a, cu=a, total_q=128, k=a, v=a, num_pages=64, bt=a, bt_stride=8, sl=a, batch=1,
             max_q=128, max_s=1024, scale=0.0884, out=a):
        return lib.attn_prefill_chunk(good, q, cu, total_q, k, v, num_pages, bt, bt_stride, sl,
                                      batch, max_q, max_s, scale, out, null, null, 0, null, null)

    INVALID, UNSUPPORTED, OK = 1, 2, 0
    # sizes and scale
    assert call(batch=-1) == INVALID
    assert call(total_q=-1) == INVALID
    assert call(bt_stride=0) == INVALID
    assert call(num_pages=0) == INVALID
    assert call(max_q=-1) == INVALID
    assert call(max_q=2048, max_s=1024) == INVALID          # chunk longer than any sequence
    assert call(max_s=131073) == INVALID                    # past the 128K context
    for scale in (0.0, -1.0, float("nan"), float("inf")):
        assert call(scale=scale) == INVALID
    # missing or misaligned pointers
    for kw in ("q", "cu", "k", "v", "bt", "sl", "out"):
        assert call(**{kw: null}) == INVALID, kw
    for kw in ("q", "k", "v", "out"):
        assert call(**{kw: mis}) == INVALID, kw
    # limits of the kernel
    assert call(batch=129, max_q=1, total_q=129) == UNSUPPORTED   # at most 128 chunks per call
    assert call(total_q=1 << 24) == UNSUPPORTED
    assert call(num_pages=1 << 27) == UNSUPPORTED                # token index past 2^31
    # empty work is a no-op success, whatever the pointers
    assert call(batch=0, q=null, out=null) == OK
    assert call(total_q=0, q=null, out=null) == OK
    assert call(max_q=0, q=null, out=null) == OK


def test_decode_and_append_argument_errors_are_rejected_before_launch(lib):
    """attn_decode_paged and kv_append_paged checks, each before any CUDA call. Every case here
    must be rejected: the pointers are fake (aligned, non-null host addresses), never read."""
    import long_context_paged_gb300 as pa
    good = pa.Dims(*pa.DEFAULT_DIMS)
    null = None
    a = ctypes.c_void_p(1 << 20)
    ws = ctypes.c_void_p(1 << 21)    # 256-byte aligned
    mis = ctypes.c_void_p((1 << 20) + 8)
    INVALID, OK = 1, 0

    def decode(q=a, k=a, v=a, num_pages=64, bt=a, bt_stride=8, sl=a, batch=1, max_s=1024,
               scale=0.0884, split=0, out=a, work=ws):
        return lib.attn_decode_paged(good, q, k, v, num_pages, bt, bt_stride, sl, batch, max_s,
                                     scale, split, out, null, work, 1 << 30, null, null)

    assert decode(batch=-1) == INVALID
    assert decode(batch=4097) == INVALID                    # past the largest decode batch
    assert decode(bt_stride=0) == INVALID
    assert decode(num_pages=0) == INVALID
    assert decode(max_s=-1) == INVALID
    assert decode(max_s=131073) == INVALID
    assert decode(scale=float("nan")) == INVALID
    assert decode(split=-1) == INVALID                      # split size must be >= 0 (0 = auto)
    for kw in ("q", "k", "v", "bt", "sl", "out", "work"):
        assert decode(**{kw: null}) == INVALID, kw
    for kw in ("q", "k", "v", "out"):
        assert decode(**{kw: mis}) == INVALID, kw
    assert decode(work=ctypes.c_void_p((1 << 21) + 128)) == INVALID   # workspace not 256-aligned
    assert decode(batch=0, q=null, work=null) == OK

    def append(k_new=a, v_new=a, total=16, cu=a, start=a, batch=1, bt=a, bt_stride=8, kp=a,
               vp=a, num_pages=64):
        return lib.kv_append_paged(good, k_new, v_new, total, cu, start, batch, bt, bt_stride,
                                   kp, vp, num_pages, null, null)

    assert append(total=-1) == INVALID
    assert append(batch=-1) == INVALID
    assert append(bt_stride=0) == INVALID
    assert append(num_pages=0) == INVALID
    for kw in ("k_new", "v_new", "cu", "start", "bt", "kp", "vp"):
        assert append(**{kw: null}) == INVALID, kw
    for kw in ("k_new", "v_new", "kp", "vp"):
        assert append(**{kw: mis}) == INVALID, kw
    assert append(total=0, k_new=null) == OK
    assert append(batch=0, k_new=null) == OK


def test_adaptor_argument_errors_are_rejected_before_launch(lib):
    """adaptor_mlp_merge4 validates everything on the host; the fake pointers below are never
    dereferenced because every case returns before anything is launched."""
    vp, fp = ctypes.c_void_p, ctypes.c_void_p
    A = 1 << 12                      # a 16-byte aligned fake address
    ok = [vp(A), vp(A), fp(A), vp(A), fp(A), fp(A), fp(A)]   # frames, w1, b1, w2, b2, gamma, beta

    def call(num_frames, ptrs=ok, eps=1e-5, out=vp(A), ws=vp(A), ws_bytes=1 << 30):
        return lib.adaptor_mlp_merge4(num_frames, *ptrs, ctypes.c_float(eps), out, ws,
                                      ctypes.c_size_t(ws_bytes), None, None)

    assert call(6) == 1                                  # not a multiple of the 4x merge
    assert call(-4) == 1
    assert call(8, eps=-1.0) == 1
    assert call(0) == 0                                  # empty work is a no-op success
    assert call(8, ptrs=[None] + ok[1:]) == 1            # null input
    misaligned_gamma = ok[:5] + [fp(A + 4)] + ok[6:]
    assert call(8, ptrs=misaligned_gamma) == 1           # gamma / beta are read as 16-byte vectors
    assert call(8, out=vp(A + 8)) == 1
    need = lib.pa_adaptor_workspace_size(8)
    assert need == 2 * 1024 * 2 + 256                    # bf16 hidden rows of the 2 merged tokens
    assert call(8, ws_bytes=need - 1) == 3               # workspace too small
    assert lib.pa_adaptor_workspace_size(-1) == 0


def test_grid_cap_argument_errors_are_rejected_before_launch(lib):
    """attn_decode_paged_ex / attn_prefill_chunk_ex: a negative max_ctas is an argument error,
    returned before any CUDA call (so this runs without a GPU)."""
    import long_context_paged_gb300 as pa
    good = pa.Dims(16, 8, 128, 16)
    null = None
    bad = pa.LaunchOpts(-1)
    assert lib.attn_decode_paged_ex(good, null, null, null, 1, null, 1, null, 1, 16, 1.0, 0,
                                    null, null, null, 0, null, null, ctypes.byref(bad)) == 1
    assert lib.attn_prefill_chunk_ex(good, null, null, 1, null, null, 1, null, 1, null, 1, 1, 16,
                                     1.0, null, null, null, 0, null, null, ctypes.byref(bad)) == 1
    # unsupported head shapes stay PA_ERR_UNSUPPORTED whatever the cap
    ok = pa.LaunchOpts(8)
    assert lib.attn_decode_paged_ex(pa.Dims(16, 8, 64, 16), null, null, null, 1, null, 1, null, 1,
                                    16, 1.0, 0, null, null, null, 0, null, null,
                                    ctypes.byref(ok)) == 2
    assert lib.attn_prefill_chunk_ex(pa.Dims(16, 4, 128, 16), null, null, 1, null, null, 1, null,
                                     1, null, 1, 1, 16, 1.0, null, null, null, 0, null, null,
                                     ctypes.byref(ok)) == 2
    with pytest.raises(ValueError):
        pa._opts(-2)
