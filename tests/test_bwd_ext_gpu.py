"""GPU parity of the variants' backward (fa_bwd_ext, through the C ABI)
against the FP64 oracle gradients of the variants ("FlashAttention-3 on
Hopper", sec. 7.8 local attention and score modifiers in the backward;
sec. 4.6 sinks; "03 FA3" sec. 5 softcap).

The forward runs first on the GPU (fa_fwd_ext gives O and LSE, with the
sinks when given); the oracle computes dQ, dK, dV and the sink logits'
gradient from the definition on the same 16-bit inputs and dO.

Tolerances are the plain backward's (tests/test_bwd_gpu.py): rel-RMSE
<= 1.5 u and max |g - g_ref| <= 4 u max |g_ref| with u = 2^-8 (bf16) or
2^-10 (fp16).  The sink gradient dsigma = -sum_i P_i,sink D_i sums terms
whose D_i carries the 16-bit rounding of O, so its bound is
4 u sum_i |P_i,sink D_i| (that sum taken from the oracle's values).

Exact pins: the window (-1, 0) reproduces fa_bwd's causal bits and
(-1, -1) its unmasked bits (same tiles, order and masks).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_fa_gb300 import synth

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 4
ULP = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -10}


def _inputs(B, H, N, d, dtype, seed):
    q, k, v = synth.qkv(B, H, N, d, seed=seed, dtype=dtype)
    do = torch.from_numpy(synth.normal((B, N, H, d), seed=seed + 3)).to(q.dtype)
    return q, k, v, do


def _gpu(fa, q, k, v, do, window, sinks, alpha, softcap=0.0):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    sk = None if sinks is None else torch.from_numpy(np.asarray(sinks, np.float32)).to(dev)
    o, lse = fa.attention_ext(qd, kd, vd, window=window, softcap=softcap, sinks=sk, alpha=alpha)
    dq, dk, dv, ds = fa.attention_backward_ext(qd, kd, vd, o, lse, dod, window=window,
                                               softcap=softcap, sinks=sk, alpha=alpha)
    assert fa.fa_check_status() == fa.FA_OK
    g = [x.float().cpu().numpy().astype(np.float64) for x in (dq, dk, dv)]
    return g, (None if ds is None else ds.cpu().numpy().astype(np.float64))


def _check(got, ref, u, rms_units=1.5):
    for g, r in zip(got, ref):
        assert np.all(np.isfinite(g))
        scale = np.abs(r).max()
        err = np.abs(g - r)
        if scale == 0.0:
            assert err.max() <= 1e-5
            continue
        rms = np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(r ** 2))
        assert rms <= rms_units * u, f"rel-RMSE {rms:.3e}"
        assert err.max() <= 4 * u * scale, f"max {err.max() / scale:.3e} of max|ref|"


def _dsink_bound(q, k, v, do, alpha, window, sinks, u, softcap=0.0):
    """4 u sum_{b,i} |P_i,sink D_i| per head, from the oracle's O and LSE."""
    o, lse = oracle.attention_ext(q, k, v, alpha, window=window, softcap=softcap, sinks=sinks,
                                  n_threads=THREADS)
    D = np.sum(oracle._f64(do) * o, axis=-1)                  # [B, N, H]
    p = np.exp(np.asarray(sinks, np.float64)[None, :, None] - lse)   # [B, H, N]
    return 4 * u * np.sum(np.abs(p * np.transpose(D, (0, 2, 1))), axis=(0, 2))


CASES = [
    # (B, H, N, d, window, sinks, dtype)
    (2, 2, 1000, 128, (256, 0), False, "bf16"),      # sliding causal window
    (2, 2, 1000, 64, (256, 0), False, "bf16"),
    (1, 2, 1000, 128, (100, 100), False, "bf16"),    # narrower than a tile, both sides
    (1, 2, 1000, 64, (0, 0), False, "bf16"),         # the diagonal alone
    (1, 2, 1000, 64, (127, 0), False, "bf16"),       # tile-boundary windows
    (1, 2, 1000, 128, (128, 1), False, "bf16"),
    (1, 2, 777, 64, (-1, 300), False, "fp16"),       # right bound only
    (1, 2, 777, 128, (300, -1), False, "bf16"),      # left bound only
    (1, 2, 513, 128, (5, 700), False, "bf16"),
    (1, 3, 1000, 128, (-1, 0), True, "bf16"),        # sinks, causal shape
    (2, 2, 700, 64, (200, 0), True, "bf16"),         # sinks and a window
    (1, 2, 300, 128, (64, 64), True, "fp16"),
    (1, 1, 1, 128, (0, 0), True, "bf16"),            # N = 1
    (1, 1, 129, 64, (-1, -1), False, "bf16"),
]


@pytest.mark.parametrize("B,H,N,d,window,sinks,dtype", CASES)
def test_bwd_ext_parity(gpu_lib, B, H, N, d, window, sinks, dtype):
    q, k, v, do = _inputs(B, H, N, d, dtype, seed=synth.BASE_SEED + 5 * N + d)
    sk = synth.sinks(H, seed=N + 1) if sinks else None
    a = synth.default_alpha(d)
    g, ds = _gpu(gpu_lib, q, k, v, do, window, sk, a)
    dq, dk, dv, dsr = oracle.attention_bwd_ext(q, k, v, do, a, window, 0.0, sk,
                                               n_threads=THREADS)
    _check(g, (dq, dk, dv), ULP[dtype])
    if sinks:
        bound = _dsink_bound(q, k, v, do, a, window, sk, ULP[dtype])
        assert np.all(np.abs(ds - dsr) <= bound + 1e-6), (ds, dsr, bound)
    else:
        assert ds is None


SOFTCAP_CASES = [
    # (B, H, N, d, window, softcap, sinks, dtype)
    (2, 2, 1000, 128, (-1, -1), 50.0, False, "bf16"),  # softcap alone
    (1, 2, 1000, 128, (-1, 0), 5.0, False, "bf16"),    # a tight softcap, causal shape
    (1, 2, 777, 64, (256, 0), 30.0, True, "bf16"),     # with a window and sinks
    (1, 2, 513, 128, (100, 100), 20.0, False, "fp16"),
    (1, 3, 1000, 64, (-1, 0), 50.0, True, "bf16"),
]


@pytest.mark.parametrize("B,H,N,d,window,softcap,sinks,dtype", SOFTCAP_CASES)
def test_bwd_ext_softcap_parity(gpu_lib, B, H, N, d, window, softcap, sinks, dtype):
    # Scores pass through c tanh(s / c): dS carries 1 - t^2.  tanh.approx.f32
    # (abs error 8e-6) moves P by at most c * 8e-6 relative, far below u.
    q, k, v, do = _inputs(B, H, N, d, dtype, seed=synth.BASE_SEED + 3 * N + d)
    q = (q.float() * 2.0).to(q.dtype)      # wider scores, so the cap bends them
    sk = synth.sinks(H, seed=N + 2) if sinks else None
    a = synth.default_alpha(d)
    g, ds = _gpu(gpu_lib, q, k, v, do, window, sk, a, softcap)
    dq, dk, dv, dsr = oracle.attention_bwd_ext(q, k, v, do, a, window, softcap, sk,
                                               n_threads=THREADS)
    _check(g, (dq, dk, dv), ULP[dtype])
    if sinks:
        bound = _dsink_bound(q, k, v, do, a, window, sk, ULP[dtype], softcap)
        assert np.all(np.abs(ds - dsr) <= bound + 1e-6), (ds, dsr, bound)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_ext_windows_reproduce_plain_bits(gpu_lib, d):
    B, H, N = 2, 2, 1000
    dev = torch.device("cuda")
    q, k, v, do = (x.to(dev) for x in _inputs(B, H, N, d, "bf16", seed=41))
    for causal, window in ((True, (-1, 0)), (False, (-1, -1))):
        o, lse = gpu_lib.attention(q, k, v, causal=causal)
        g1 = gpu_lib.attention_backward(q, k, v, o, lse, do, causal=causal)
        g2 = gpu_lib.attention_backward_ext(q, k, v, o, lse, do, window=window)
        for x, y in zip(g1, g2[:3]):
            assert torch.equal(x, y)


def test_bwd_ext_deterministic_with_sinks(gpu_lib):
    B, H, N, d = 2, 3, 900, 128
    dev = torch.device("cuda")
    q, k, v, do = (x.to(dev) for x in _inputs(B, H, N, d, "bf16", seed=43))
    sk = torch.from_numpy(synth.sinks(H, seed=7)).to(dev)
    o, lse = gpu_lib.attention_ext(q, k, v, window=(300, 0), sinks=sk)
    r1 = gpu_lib.attention_backward_ext(q, k, v, o, lse, do, window=(300, 0), sinks=sk)
    r2 = gpu_lib.attention_backward_ext(q, k, v, o, lse, do, window=(300, 0), sinks=sk)
    for x, y in zip(r1, r2):
        assert torch.equal(x, y)


def test_bwd_ext_b4_h16_n4096_d128_window_two_heads(gpu_lib):
    # The bench workload with a (1024, 0) window; two (b, h) heads are
    # compared in full against the oracle (dK and dV of a head need all of
    # its query rows).
    B, H, N, d = 4, 16, 4096, 128
    window = (1024, 0)
    q, k, v, do = _inputs(B, H, N, d, "bf16", seed=synth.BASE_SEED + 77)
    a = synth.default_alpha(d)
    g, _ = _gpu(gpu_lib, q, k, v, do, window, None, a)
    for b, h in [(0, 0), (3, 15)]:
        ref = oracle.attention_bwd_ext_head(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], a,
                                            window, 0.0, None)
        _check([x[b, :, h] for x in g], ref[:3], ULP["bf16"])


GQA_CASES = [
    # (B, H, H_kv, N, d, window, softcap, sinks)
    (2, 8, 2, 1000, 128, (-1, -1), 0.0, False),
    (1, 8, 1, 777, 64, (256, 0), 0.0, False),          # multi-query
    (1, 4, 2, 513, 128, (-1, 0), 30.0, True),
    (1, 6, 3, 300, 64, (64, 64), 0.0, True),
]


@pytest.mark.parametrize("B,H,H_kv,N,d,window,softcap,sinks", GQA_CASES)
def test_bwd_ext_grouped_heads(gpu_lib, B, H, H_kv, N, d, window, softcap, sinks):
    # dK, dV of a K/V head sum the gradients of its H / H_kv query heads.
    t = torch.bfloat16
    seed = synth.BASE_SEED + 11 * N + H_kv
    q = torch.from_numpy(synth.normal((B, N, H, d), seed=seed)).to(t)
    k = torch.from_numpy(synth.normal((B, N, H_kv, d), seed=seed + 1)).to(t)
    v = torch.from_numpy(synth.normal((B, N, H_kv, d), seed=seed + 2)).to(t)
    do = torch.from_numpy(synth.normal((B, N, H, d), seed=seed + 3)).to(t)
    sk = synth.sinks(H, seed=N + 3) if sinks else None
    a = synth.default_alpha(d)
    g, ds = _gpu(gpu_lib, q, k, v, do, window, sk, a, softcap)
    assert g[1].shape == (B, N, H_kv, d) and g[2].shape == (B, N, H_kv, d)
    dq, dk, dv, dsr = oracle.attention_bwd_ext(q, k, v, do, a, window, softcap, sk,
                                               n_threads=THREADS)
    _check(g, (dq, dk, dv), ULP["bf16"])
    if sinks:
        bound = _dsink_bound(q, k, v, do, a, window, sk, ULP["bf16"], softcap)
        assert np.all(np.abs(ds - dsr) <= bound + 1e-6), (ds, dsr, bound)
