"""Python binding of libfa (exact attention forward on GB300, sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libfa.so``.  The names mirror the C ABI in ``include/fa.h``.
If the library has not been built, every entry point raises -- there is no
fallback implementation.

Tensors are [B, N, H, d] (batch, sequence, head, head dim) and contiguous;
LSE is float32 [B, H, N].
"""
from __future__ import annotations

import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_TOO_LARGE = 4
FA_ERR_CUDA = 5
FA_ERR_TIMEOUT = 6

FA_BF16 = 0
FA_FP16 = 1

FA_SCALE_TILE = 0
FA_SCALE_HEAD = 1
FA_SCALE_TENSOR = 2

# Every symbol include/fa.h declares (checked by the tests).
EXPORTS = ("fa_fwd", "fa_fwd_gqa", "fa_fwd_gqa_packed", "fa_fwd_ext", "fa_fwd_splitkv", "fa_splitkv_workspace_floats",
           "fa_splitkv_auto", "fa_quantize_fp8", "fa_quantize_fp8_granular", "fa_fwd_fp8", "fa_fwd_fp8_gqa", "fa_bwd", "fa_bwd_ext", "fa_bwd_noalloc",
           "fa_check_status", "fa_status_detail", "fa_selftest_wait_timeout",
           "fa_status_string", "fa_version")

_lib = None


class FaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def load():
    """Load libfa.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
            "(the CUDA path has no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_gqa.restype = i
    lib.fa_fwd_gqa_packed.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_gqa_packed.restype = i
    lib.fa_fwd_ext.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, f, vp, i, vp]
    lib.fa_fwd_ext.restype = i
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_splitkv_workspace_floats.argtypes = [i, i, i, i, i]
    lib.fa_splitkv_workspace_floats.restype = ctypes.c_longlong
    lib.fa_splitkv_auto.argtypes = [i, i, i, i]
    lib.fa_splitkv_auto.restype = i
    lib.fa_quantize_fp8.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
    lib.fa_quantize_fp8.restype = i
    lib.fa_quantize_fp8_granular.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.fa_quantize_fp8_granular.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_fwd_fp8_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_fp8_gqa.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_ext.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i,
                               f, vp, vp, i, vp]
    lib.fa_bwd_ext.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_selftest_wait_timeout.argtypes = [vp, vp]
    lib.fa_selftest_wait_timeout.restype = i
    lib.fa_check_status.argtypes = [vp]
    lib.fa_check_status.restype = i
    lib.fa_status_detail.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.fa_status_detail.restype = None
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_version.argtypes = []
    lib.fa_version.restype = i
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def status_string(code: int) -> str:
    return load().fa_status_string(int(code)).decode()


def fa_fwd(q, k, v, o, lse, B: int, H: int, N: int, d: int, alpha: float,
           causal: int, dtype: int, stream=None) -> int:
    """Direct call of the C entry point; returns the fa_status code.

    Pointer arguments may be torch tensors or integer device addresses;
    ``lse`` may be None.  ``stream`` is a torch stream, a raw cudaStream_t
    integer, or None for torch's current stream."""
    return load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                         int(B), int(H), int(N), int(d), float(alpha),
                         int(causal), int(dtype), _stream(stream))


def fa_fwd_gqa(q, k, v, o, lse, B: int, H: int, H_kv: int, N: int, d: int, alpha: float,
               causal: int, dtype: int, stream=None) -> int:
    """Direct call of the C entry point: K/V with H_kv heads shared by groups
    of H / H_kv query heads (see include/fa.h)."""
    return load().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                             int(H_kv), int(N), int(d), float(alpha), int(causal), int(dtype),
                             _stream(stream))


def fa_fwd_gqa_packed(q, k, v, o, lse, B: int, H: int, H_kv: int, N: int, d: int,
                      alpha: float, causal: int, dtype: int, stream=None) -> int:
    """Direct call of the C entry point: fa_fwd_gqa with the query heads of
    each K/V head packed into the rows of one Q tile (see include/fa.h)."""
    return load().fa_fwd_gqa_packed(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                    int(H), int(H_kv), int(N), int(d), float(alpha),
                                    int(causal), int(dtype), _stream(stream))


def fa_fwd_ext(q, k, v, o, lse, B: int, H: int, H_kv: int, N: int, d: int, alpha: float,
               window_left: int, window_right: int, softcap: float, sinks, dtype: int,
               stream=None) -> int:
    """Direct call of the C entry point: local window, softcap and per-head
    sinks (see include/fa.h); ``sinks`` may be None."""
    return load().fa_fwd_ext(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                             int(H_kv), int(N), int(d), float(alpha), int(window_left),
                             int(window_right), float(softcap), _ptr(sinks), int(dtype),
                             _stream(stream))


def attention_ext(q, k, v, window=(-1, -1), softcap: float = 0.0, sinks=None,
                  alpha: float | None = None, out=None, lse=None, want_lse: bool = True,
                  stream=None):
    """Forward with the score and mask variants for torch tensors on the GPU:
    window = (left, right) key bounds around the diagonal (-1: none),
    softcap c (0: none), sinks float32 [H] on the GPU or None.  K/V may have
    fewer heads than Q (grouped).  Returns (O, LSE or None)."""
    import torch
    if q.dtype == torch.bfloat16:
        dt = FA_BF16
    elif q.dtype == torch.float16:
        dt = FA_FP16
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    B, N, H, d = q.shape
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    rc = fa_fwd_ext(q, k, v, out, lse, B, H, k.shape[2], N, d, alpha, int(window[0]),
                    int(window[1]), float(softcap), sinks, dt, stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_ext")
    return out, lse


def fa_fwd_splitkv(q, k, v, o, lse, B: int, H: int, N: int, d: int, alpha: float, causal: int,
                   dtype: int, n_splits: int, workspace, stream=None) -> int:
    """Direct call of the C entry point (see include/fa.h)."""
    return load().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                                 int(N), int(d), float(alpha), int(causal), int(dtype),
                                 int(n_splits), _ptr(workspace), _stream(stream))


def fa_splitkv_workspace_floats(B: int, H: int, N: int, d: int, n_splits: int) -> int:
    return load().fa_splitkv_workspace_floats(int(B), int(H), int(N), int(d), int(n_splits))


def fa_splitkv_auto(B: int, H: int, N: int, d: int) -> int:
    return load().fa_splitkv_auto(int(B), int(H), int(N), int(d))


def attention_splitkv(q, k, v, causal: bool = False, alpha: float | None = None,
                      n_splits: int = 0, want_lse: bool = True, stream=None):
    """Split-KV forward for torch tensors on the GPU (n_splits 0: the
    library's choice for this device).  Returns (O, LSE or None)."""
    import torch
    dt = FA_BF16 if q.dtype == torch.bfloat16 else FA_FP16
    B, N, H, d = q.shape
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    if n_splits <= 0:
        n_splits = fa_splitkv_auto(B, H, N, d)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if want_lse else None
    ws = torch.empty((fa_splitkv_workspace_floats(B, H, N, d, n_splits),), dtype=torch.float32,
                     device=q.device)
    rc = fa_fwd_splitkv(q, k, v, out, lse, B, H, N, d, alpha, int(bool(causal)), dt, n_splits,
                        ws, stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv")
    return out, lse


def fa_quantize_fp8(x, x8, scales, hadamard_signs, B: int, H: int, N: int,
                    d: int, stream=None) -> int:
    """Direct call of the C entry point (see include/fa.h)."""
    return load().fa_quantize_fp8(_ptr(x), _ptr(x8), _ptr(scales), _ptr(hadamard_signs),
                                  int(B), int(H), int(N), int(d), _stream(stream))


def fa_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B: int, H: int,
               N: int, d: int, alpha: float, causal: int, stream=None) -> int:
    """Direct call of the C entry point (see include/fa.h)."""
    return load().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale),
                             _ptr(v_scale), _ptr(o), _ptr(lse), int(B), int(H), int(N),
                             int(d), float(alpha), int(causal), _stream(stream))


def fa_quantize_fp8_granular(x, x8, scales, hadamard_signs, B: int, H: int, N: int,
                             d: int, granularity: int, stream=None) -> int:
    """Direct call of the C entry point (see include/fa.h)."""
    return load().fa_quantize_fp8_granular(_ptr(x), _ptr(x8), _ptr(scales),
                                           _ptr(hadamard_signs), int(B), int(H), int(N),
                                           int(d), int(granularity), _stream(stream))


def quantize_fp8(x, hadamard_signs=None, stream=None, granularity: int = FA_SCALE_TILE):
    """bf16 [B,N,H,d] on the GPU -> (uint8 e4m3 codes, float scales [B,H,ceil(N/128)]);
    ``granularity`` FA_SCALE_HEAD / FA_SCALE_TENSOR give one scale per head /
    per tensor, repeated over the tiles."""
    import torch
    B, N, H, d = x.shape
    x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    sc = torch.empty((B, H, (N + 127) // 128), dtype=torch.float32, device=x.device)
    if granularity == FA_SCALE_TILE:
        rc = fa_quantize_fp8(x, x8, sc, hadamard_signs, B, H, N, d, stream)
    else:
        rc = fa_quantize_fp8_granular(x, x8, sc, hadamard_signs, B, H, N, d, granularity,
                                      stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_quantize_fp8")
    return x8, sc


def fa_fwd_fp8_gqa(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B: int, H: int, H_kv: int,
                   N: int, d: int, alpha: float, causal: int, stream=None) -> int:
    """Direct call of the C entry point: fa_fwd_fp8 with K/V (codes and
    scales) over H_kv heads (see include/fa.h)."""
    return load().fa_fwd_fp8_gqa(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale),
                                 _ptr(v_scale), _ptr(o), _ptr(lse), int(B), int(H), int(H_kv),
                                 int(N), int(d), float(alpha), int(causal), _stream(stream))


def attention_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool = False,
                  alpha: float | None = None, out=None, lse=None, want_lse: bool = True,
                  stream=None):
    """FP8 forward on quantized inputs; returns (O bf16, LSE or None).  K/V
    may have fewer heads than Q (fa_fwd_fp8_gqa)."""
    import torch
    B, N, H, d = q8.shape
    H_kv = k8.shape[2]
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q8.shape, dtype=torch.bfloat16, device=q8.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    if H_kv == H:
        rc = fa_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, out, lse, B, H, N, d, alpha,
                        int(bool(causal)), stream)
    else:
        rc = fa_fwd_fp8_gqa(q8, k8, v8, q_scale, k_scale, v_scale, out, lse, B, H, H_kv, N, d,
                            alpha, int(bool(causal)), stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_fp8")
    return out, lse


def bwd_workspace_floats(B: int, H: int, N: int) -> int:
    """Size of fa_bwd's workspace: float [2][B][H][ceil(N/128)*128]."""
    return 2 * B * H * ((N + 127) // 128) * 128


def fa_bwd(q, k, v, o, dout, lse, workspace, dq, dk, dv, B: int, H: int, N: int, d: int,
           alpha: float, causal: int, dtype: int, stream=None) -> int:
    """Direct call of the C entry point (see include/fa.h)."""
    return load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                         _ptr(workspace), _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(H), int(N),
                         int(d), float(alpha), int(causal), int(dtype), _stream(stream))


def fa_bwd_ext(q, k, v, o, dout, lse, workspace, dq, dk, dv, B: int, H: int, H_kv: int, N: int,
               d: int, alpha: float, window_left: int, window_right: int, softcap: float, sinks,
               dsinks, dtype: int, stream=None) -> int:
    """Direct call of the C entry point: the backward of fa_fwd_ext with a
    local window and softcap; sinks/dsinks may be None (see include/fa.h)."""
    return load().fa_bwd_ext(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                             _ptr(workspace), _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(H),
                             int(H_kv), int(N), int(d), float(alpha), int(window_left),
                             int(window_right), float(softcap), _ptr(sinks), _ptr(dsinks), int(dtype),
                             _stream(stream))


def attention_backward_ext(q, k, v, o, lse, dout, window=(-1, -1), softcap: float = 0.0,
                           sinks=None, alpha: float | None = None, stream=None):
    """Gradients (dQ, dK, dV, dsinks or None) for the forward of
    ``attention_ext`` with a window, softcap and optional sinks."""
    import torch
    if q.dtype == torch.bfloat16:
        dt = FA_BF16
    elif q.dtype == torch.float16:
        dt = FA_FP16
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    B, N, H, d = q.shape
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty((bwd_workspace_floats(B, H, N),), dtype=torch.float32, device=q.device)
    ds = None if sinks is None else torch.empty((H,), dtype=torch.float32, device=q.device)
    rc = fa_bwd_ext(q, k, v, o, dout, lse, ws, dq, dk, dv, B, H, k.shape[2], N, d, alpha,
                    int(window[0]),
                    int(window[1]), float(softcap), sinks, ds, dt, stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_ext")
    return dq, dk, dv, ds


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B: int, H: int, N: int, d: int,
                   alpha: float, causal: int, dtype: int, stream=None) -> int:
    """Direct call of the C entry point: fa_bwd with the library's own
    16 MiB device workspace, for callers that must not allocate (see
    include/fa.h; overlapping calls race on that workspace)."""
    return load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                 _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d),
                                 float(alpha), int(causal), int(dtype), _stream(stream))


def attention_backward(q, k, v, o, lse, dout, causal: bool = False,
                       alpha: float | None = None, stream=None):
    """Gradients (dQ, dK, dV) for torch tensors on the GPU; ``o`` and ``lse``
    come from ``attention`` on the same inputs.  Allocates the outputs and
    the workspace with torch; raises FaError on a non-OK status."""
    import torch
    if q.dtype == torch.bfloat16:
        dt = FA_BF16
    elif q.dtype == torch.float16:
        dt = FA_FP16
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    B, N, H, d = q.shape
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty((bwd_workspace_floats(B, H, N),), dtype=torch.float32, device=q.device)
    rc = fa_bwd(q, k, v, o, dout, lse, ws, dq, dk, dv, B, H, N, d, alpha,
                int(bool(causal)), dt, stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv


def fa_selftest_wait_timeout(result, stream=None) -> int:
    """Direct call of the C entry point: a kernel whose bounded waits run
    out (no fault); result is a device uint32 tensor of 2 elements."""
    return load().fa_selftest_wait_timeout(_ptr(result), _stream(stream))


def fa_check_status(stream=None) -> int:
    return load().fa_check_status(_stream(stream))


def fa_status_detail() -> list[int]:
    out = (ctypes.c_uint32 * 4)()
    load().fa_status_detail(out)
    return list(out)


def fa_version() -> int:
    return load().fa_version()


def attention(q, k, v, causal: bool = False, alpha: float | None = None,
              out=None, lse=None, want_lse: bool = True, stream=None,
              pack_gqa: bool = False):
    """Convenience wrapper over ``fa_fwd`` for torch tensors on the GPU
    (``fa_fwd_gqa`` when K/V have fewer heads than Q; ``fa_fwd_gqa_packed``
    with ``pack_gqa``).

    Allocates O (and LSE) with torch when not given, launches, and raises
    FaError on a non-OK status.  Returns (O, LSE or None)."""
    import torch
    if q.dtype == torch.bfloat16:
        dt = FA_BF16
    elif q.dtype == torch.float16:
        dt = FA_FP16
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    B, N, H, d = q.shape
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    H_kv = k.shape[2]
    if H_kv == H:
        rc = fa_fwd(q, k, v, out, lse, B, H, N, d, alpha, int(bool(causal)), dt, stream)
    else:
        call = fa_fwd_gqa_packed if pack_gqa else fa_fwd_gqa
        rc = call(q, k, v, out, lse, B, H, H_kv, N, d, alpha, int(bool(causal)), dt, stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return out, lse
