"""FP64 CPU oracle for exact attention (forward and gradients) -- TEST
INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``exact_attention_forward_fa_gb300``) never imports, links or
executes anything here, and this package imports nothing from it.

The arithmetic lives in ``fa_oracle.c`` (plain C11, FP64, built here with
gcc).  This module only marshals numpy arrays into it.  What each function
computes, and the passage it follows, is stated in ``fa_oracle.c``:

* ``attention`` / ``attention_rows`` / ``attention_probs``: the plain
  definition (materialised S and P rows), "FlashAttention-3 on Hopper"
  sec. 3.1, 3.2, 4.6, 4.7.
* ``attention_online``: the tiled online recurrence with the conditional
  rescale rule, "FlashAttention-3 on Hopper" sec. 4.2 and "FlashAttention
  v1-v4" (conditional rescale).
* ``attention_gqa``: grouped key/value heads (GQA/MQA), each query head with
  its own key/value head h // (H / H_kv), "FlashAttention-3 on Hopper" ch. 11.
* ``attention_ext`` / ``attention_ext_head``: the variants -- local
  (sliding-window) masks, tanh softcap and a per-head sink logit,
  "FlashAttention-3 on Hopper" sec. 4.6 (sinks) and 4.7 (local masks,
  transform before mask), "03 FA3" sec. 5 (softcap).
* ``attention_bwd`` / ``attention_bwd_head``: the gradients dQ, dK, dV from
  the definition, "FlashAttention-3 on Hopper" sec. 7.1.
* ``attention_bwd_ext`` / ``attention_bwd_ext_head``: the gradients of the
  variants (window, softcap, sink), including the sink logit's gradient.
* ``hadamard_rotate``, ``e4m3_encode`` / ``e4m3_decode``,
  ``quantize_e4m3_tiles``: the FP8 pre-pass pieces, "FlashAttention-3 on
  Hopper" sec. 6.1, 6.3, 6.4.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into liboracle.so (gcc, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
           "-Wall", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    lib.oracle_attention_head.argtypes = [
        _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_double,
        ctypes.c_int, _ip, ctypes.c_int, _dp, ctypes.c_long, _dp, _dp]
    lib.oracle_attention_head.restype = ctypes.c_int
    lib.oracle_attention_fwd.argtypes = [
        _dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_attention_fwd.restype = ctypes.c_int
    lib.oracle_attention_bwd_head.argtypes = [
        _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
        ctypes.c_double, ctypes.c_int, _dp, ctypes.c_long, _dp, ctypes.c_long,
        _dp, ctypes.c_long]
    lib.oracle_attention_bwd_head.restype = ctypes.c_int
    lib.oracle_attention_bwd.argtypes = [
        _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_attention_bwd.restype = ctypes.c_int
    lib.oracle_attention_online_head.argtypes = [
        _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_double,
        ctypes.c_int, _ip, _ip, ctypes.c_int, ctypes.c_double, _dp,
        ctypes.c_long, _dp, ctypes.POINTER(ctypes.c_long)]
    lib.oracle_attention_online_head.restype = ctypes.c_int
    lib.oracle_attention_ext_head.argtypes = [
        _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_double,
        ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp, _ip, ctypes.c_int,
        _dp, ctypes.c_long, _dp]
    lib.oracle_attention_ext_head.restype = ctypes.c_int
    lib.oracle_attention_ext_fwd.argtypes = [
        _dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, _dp, ctypes.c_int]
    lib.oracle_attention_ext_fwd.restype = ctypes.c_int
    lib.oracle_attention_bwd_ext_head.argtypes = [
        _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
        ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp, _dp, _dp, _dp, _dp]
    lib.oracle_attention_bwd_ext_head.restype = ctypes.c_int
    lib.oracle_hadamard_rotate.argtypes = [
        _dp, _dp, ctypes.c_long, ctypes.c_int, ctypes.c_long, _dp]
    lib.oracle_hadamard_rotate.restype = ctypes.c_int
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint]
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint
    lib.oracle_quantize_e4m3_tiles.argtypes = [
        _dp, ctypes.POINTER(ctypes.c_ubyte), ctypes.POINTER(ctypes.c_float),
        ctypes.c_long, ctypes.c_int, ctypes.c_long, ctypes.c_int]
    lib.oracle_quantize_e4m3_tiles.restype = ctypes.c_int
    _lib = lib
    return lib


def _f64(x) -> np.ndarray:
    """Exact widening to a C-contiguous float64 array (bf16/fp16/fp32 -> f64)."""
    if hasattr(x, "detach"):                      # a torch tensor
        import torch
        x = x.detach().to("cpu").to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def attention(q, k, v, alpha: float, causal: bool, n_threads: int = 1):
    """O [B,N,H,d] and LSE [B,H,N] in float64 from Q/K/V [B,N,H,d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, H, d = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((B, H, N), dtype=np.float64)
    rc = _load().oracle_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                      _ptr(lse), B, H, N, d, float(alpha),
                                      int(bool(causal)), int(n_threads))
    if rc:
        raise RuntimeError(f"oracle_attention_fwd failed ({rc})")
    return o, lse


def attention_gqa(q, k, v, alpha: float, causal: bool, n_threads: int = 1):
    """Grouped key/value heads: q [B,N,H,d], k/v [B,N,H_kv,d] with H_kv
    dividing H; query head h attends with key/value head h // (H // H_kv).
    The definition is the per-head attention with each query head's own key
    and value head, so K and V are repeated per query head and the plain
    definition is applied ("FlashAttention-3 on Hopper", ch. 11)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    H, H_kv = q.shape[2], k.shape[2]
    if H_kv < 1 or H % H_kv:
        raise ValueError("H_kv must divide H")
    g = H // H_kv
    return attention(q, np.repeat(k, g, axis=2), np.repeat(v, g, axis=2), alpha, causal,
                     n_threads)


def attention_ext(q, k, v, alpha: float, window=(-1, -1), softcap: float = 0.0,
                  sinks=None, n_threads: int = 1):
    """The variants on [B,N,H,d] tensors: window = (wl, wr) hides key j from
    query i when j > i + wr (wr >= 0) or j < i - wl (wl >= 0), -1 = no bound;
    softcap c > 0 replaces each visible score s by c tanh(s / c); sinks [H]
    (or None) is one extra logit per head in every row's softmax denominator.
    k, v may have H_kv heads dividing H (query head h uses h // (H / H_kv)).
    Returns O [B,N,H,d] and LSE [B,H,N] in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, H, d = q.shape
    H_kv = k.shape[2]
    if H_kv < 1 or H % H_kv:
        raise ValueError("H_kv must divide H")
    if H_kv != H:
        k = np.ascontiguousarray(np.repeat(k, H // H_kv, axis=2))
        v = np.ascontiguousarray(np.repeat(v, H // H_kv, axis=2))
    o = np.zeros_like(q)
    lse = np.zeros((B, H, N), dtype=np.float64)
    sk = None if sinks is None else np.ascontiguousarray(_f64(sinks).reshape(H))
    wl, wr = int(window[0]), int(window[1])
    rc = _load().oracle_attention_ext_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(alpha),
        wl, wr, float(softcap), _ptr(sk) if sk is not None else None,
        int(n_threads))
    if rc:
        raise RuntimeError(f"oracle_attention_ext_fwd failed ({rc})")
    return o, lse


def attention_ext_head(q, k, v, alpha: float, window=(-1, -1),
                       softcap: float = 0.0, sink=None, rows=None):
    """One head of ``attention_ext``: q [Nq,d], k/v [Nk,d], sink a scalar or
    None; the diagonal is bottom-right aligned, i + (Nk - Nq).  With ``rows``
    only those query rows are computed."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Nq, d = q.shape
    Nk = k.shape[0]
    if rows is None:
        n, rows_arr = Nq, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        n = len(rows_arr)
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    sk = None if sink is None else np.array([float(sink)], dtype=np.float64)
    rc = _load().oracle_attention_ext_head(
        _ptr(q), _ptr(k), _ptr(v), Nq, Nk, d, d, d, d, float(alpha),
        int(window[0]), int(window[1]), float(softcap),
        _ptr(sk) if sk is not None else None,
        rows_arr.ctypes.data_as(_ip) if rows_arr is not None else None, n,
        _ptr(o), d, _ptr(lse))
    if rc:
        raise RuntimeError(f"oracle_attention_ext_head failed ({rc})")
    return o, lse


def attention_ext_rows(q, k, v, alpha: float, b: int, h: int, rows,
                       window=(-1, -1), softcap: float = 0.0, sinks=None):
    """Rows ``rows`` of head (b, h) of [B,N,H,d] tensors with the variants;
    k, v may have fewer (grouped) heads."""
    H, H_kv = q.shape[2], k.shape[2]
    hk = h // (H // H_kv)
    sink = None if sinks is None else float(_f64(sinks).reshape(-1)[h])
    return attention_ext_head(_f64(q[b, :, h, :]), _f64(k[b, :, hk, :]),
                              _f64(v[b, :, hk, :]), alpha, window, softcap, sink,
                              rows)


def attention_bwd(q, k, v, dout, alpha: float, causal: bool, n_threads: int = 1):
    """Gradients (dQ, dK, dV) [B,N,H,d] in float64 of attention with the
    upstream gradient dO [B,N,H,d]."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, N, H, d = q.shape
    dq, dk, dv = np.zeros_like(q), np.zeros_like(q), np.zeros_like(q)
    rc = _load().oracle_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                      _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                      float(alpha), int(bool(causal)),
                                      int(n_threads))
    if rc:
        raise RuntimeError(f"oracle_attention_bwd failed ({rc})")
    return dq, dk, dv


def attention_bwd_ext_head(q, k, v, dout, alpha: float, window=(-1, -1),
                           softcap: float = 0.0, sink=None):
    """One head of the variants' gradients: q/dout [Nq,d], k/v [Nk,d], sink a
    scalar or None.  Returns (dQ, dK, dV, dsigma) with dsigma 0 without a
    sink."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    Nq, d = q.shape
    Nk = k.shape[0]
    dq, dk, dv = np.zeros((Nq, d)), np.zeros((Nk, d)), np.zeros((Nk, d))
    sk = None if sink is None else np.array([float(sink)])
    ds = np.zeros(1)
    rc = _load().oracle_attention_bwd_ext_head(
        _ptr(q), _ptr(k), _ptr(v), _ptr(dout), Nq, Nk, d, float(alpha), int(window[0]),
        int(window[1]), float(softcap), _ptr(sk) if sk is not None else None, _ptr(dq),
        _ptr(dk), _ptr(dv), _ptr(ds))
    if rc:
        raise RuntimeError(f"oracle_attention_bwd_ext_head failed ({rc})")
    return dq, dk, dv, float(ds[0])


def attention_bwd_ext(q, k, v, dout, alpha: float, window=(-1, -1), softcap: float = 0.0,
                      sinks=None, n_threads: int = 1):
    """The variants' gradients on [B,N,H,d] tensors: (dQ, dK, dV, dsinks [H]),
    dsinks summed over the batch (zeros without sinks).  k, v may have H_kv
    heads dividing H: query head h uses K/V head h // (H / H_kv), and dK, dV
    of a K/V head are the sums over its query heads (a shared input's
    gradient is the sum of its uses).  Heads are independent and run on a
    thread pool."""
    from concurrent.futures import ThreadPoolExecutor
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, N, H, d = q.shape
    H_kv = k.shape[2]
    if H_kv < 1 or H % H_kv:
        raise ValueError("H_kv must divide H")
    g = H // H_kv
    if g > 1:
        k = np.ascontiguousarray(np.repeat(k, g, axis=2))
        v = np.ascontiguousarray(np.repeat(v, g, axis=2))
    dq, dk, dv = np.zeros_like(q), np.zeros_like(q), np.zeros_like(q)
    sk = None if sinks is None else _f64(sinks).reshape(H)
    dsink = np.zeros((B, H))

    def one(bh):
        b, h = bh
        g = attention_bwd_ext_head(q[b, :, h], k[b, :, h], v[b, :, h], dout[b, :, h], alpha,
                                   window, softcap, None if sk is None else sk[h])
        dq[b, :, h], dk[b, :, h], dv[b, :, h] = g[0], g[1], g[2]
        dsink[b, h] = g[3]

    with ThreadPoolExecutor(max_workers=max(1, int(n_threads))) as ex:
        list(ex.map(one, [(b, h) for b in range(B) for h in range(H)]))
    if g > 1:
        dk = dk.reshape(B, N, H_kv, g, d).sum(axis=3)
        dv = dv.reshape(B, N, H_kv, g, d).sum(axis=3)
    return dq, dk, dv, dsink.sum(axis=0)


def attention_bwd_head(q, k, v, dout, alpha: float, causal: bool):
    """One head: q/dout [Nq,d], k/v [Nk,d] -> (dQ [Nq,d], dK, dV [Nk,d])."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    Nq, d = q.shape
    Nk = k.shape[0]
    dq = np.zeros((Nq, d))
    dk = np.zeros((Nk, d))
    dv = np.zeros((Nk, d))
    rc = _load().oracle_attention_bwd_head(
        _ptr(q), _ptr(k), _ptr(v), _ptr(dout), Nq, Nk, d, d, d, d, d,
        float(alpha), int(bool(causal)), _ptr(dq), d, _ptr(dk), d, _ptr(dv), d)
    if rc:
        raise RuntimeError(f"oracle_attention_bwd_head failed ({rc})")
    return dq, dk, dv


def attention_head(q, k, v, alpha: float, causal: bool, rows=None,
                   want_probs: bool = False):
    """One head: q [Nq,d], k/v [Nk,d].  Returns (O, LSE[, P]).

    With ``rows`` only those query rows are computed (O has len(rows) rows).
    Causal masking is bottom-right aligned: key j is hidden from query i
    when j > i + (Nk - Nq).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Nq, d = q.shape
    Nk = k.shape[0]
    if rows is None:
        n = Nq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        n = len(rows_arr)
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    probs = np.zeros((Nq, Nk), dtype=np.float64) if want_probs else None
    rc = _load().oracle_attention_head(
        _ptr(q), _ptr(k), _ptr(v), Nq, Nk, d, d, d, d, float(alpha),
        int(bool(causal)),
        rows_arr.ctypes.data_as(_ip) if rows_arr is not None else None,
        n, _ptr(o), d, _ptr(lse), _ptr(probs) if want_probs else None)
    if rc:
        raise RuntimeError(f"oracle_attention_head failed ({rc})")
    return (o, lse, probs) if want_probs else (o, lse)


def attention_rows(q, k, v, alpha: float, causal: bool, b: int, h: int, rows):
    """Rows ``rows`` of head (b, h) of [B,N,H,d] tensors (torch or numpy)."""
    def head(x):
        x = x[b, :, h, :]
        return _f64(x)
    return attention_head(head(q), head(k), head(v), alpha, causal, rows=rows)


def attention_online(q, k, v, alpha: float, causal: bool, tiles, tau: float):
    """Tiled online recurrence over key tiles ``tiles`` = [(lo, hi), ...]
    in processing order.  Returns (O, LSE, number of reference moves)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Nq, d = q.shape
    Nk = k.shape[0]
    lo = np.ascontiguousarray(np.array([t[0] for t in tiles], dtype=np.int32))
    hi = np.ascontiguousarray(np.array([t[1] for t in tiles], dtype=np.int32))
    o = np.zeros((Nq, d), dtype=np.float64)
    lse = np.zeros((Nq,), dtype=np.float64)
    nres = ctypes.c_long(0)
    rc = _load().oracle_attention_online_head(
        _ptr(q), _ptr(k), _ptr(v), Nq, Nk, d, d, d, d, float(alpha),
        int(bool(causal)), lo.ctypes.data_as(_ip), hi.ctypes.data_as(_ip),
        len(tiles), float(tau), _ptr(o), d, _ptr(lse), ctypes.byref(nres))
    if rc:
        raise RuntimeError(f"oracle_attention_online_head failed ({rc})")
    return o, lse, int(nres.value)


def hadamard_rotate(x, signs):
    """x [..., d] -> x (1/sqrt d) H diag(signs), H Sylvester-ordered."""
    x = _f64(x)
    d = x.shape[-1]
    flat = np.ascontiguousarray(x.reshape(-1, d))
    y = np.zeros_like(flat)
    s = _f64(signs).reshape(d)
    rc = _load().oracle_hadamard_rotate(_ptr(flat), _ptr(y), flat.shape[0], d,
                                        d, _ptr(s))
    if rc:
        raise RuntimeError("oracle_hadamard_rotate failed")
    return y.reshape(x.shape)


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.vectorize(lambda t: lib.oracle_e4m3_decode(int(t)),
                        otypes=[np.float64])(c)


def e4m3_encode(x) -> np.ndarray:
    lib = _load()
    a = np.asarray(x, dtype=np.float64)
    return np.vectorize(lambda t: lib.oracle_e4m3_encode(float(t)),
                        otypes=[np.uint8])(a)


def quantize_e4m3_tiles(x, tile_rows: int = 128):
    """x [n_rows, d] (one head) -> (codes uint8 [n_rows, d], scales f32)."""
    x = _f64(x)
    n, d = x.shape
    codes = np.zeros((n, d), dtype=np.uint8)
    n_tiles = (n + tile_rows - 1) // tile_rows
    scales = np.zeros((n_tiles,), dtype=np.float32)
    rc = _load().oracle_quantize_e4m3_tiles(
        _ptr(x), codes.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)),
        scales.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), n, d, d,
        tile_rows)
    if rc:
        raise RuntimeError("oracle_quantize_e4m3_tiles failed")
    return codes, scales
