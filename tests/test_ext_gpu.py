"""GPU parity of the score and mask variants (fa_fwd_ext) against the FP64
oracle: local / sliding-window masks ("FlashAttention-3 on Hopper",
sec. 4.7), tanh softcap ("03 FA3", sec. 5) and per-head sinks
("FlashAttention-3 on Hopper", sec. 4.6), alone and combined, with grouped
K/V heads, both 16-bit dtypes, d = 64 and 128, ragged N and windows at and
around tile boundaries.

Tolerances are those of the plain forward (O max-abs 1e-2, O RMSE 2e-3,
LSE max-abs 1e-3).  With a softcap the kernel's tanh is tanh.approx.f32,
whose absolute error (at most 8.0e-6 = 2^-16.9, measured on a GB300 over
2^24 points of [-10, 10]) moves a score by at most c * 8e-6 -- 4e-4 at
c = 50, below the 2^-9 relative rounding of the 16-bit P -- so the same
bounds hold.

Exact pins: the window (-1, 0) reproduces fa_fwd's causal bits and
(-1, -1) its unmasked bits (same tiles, same order, same masks); a sink of
-inf reproduces the no-sink bits.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_fa_gb300 import synth

pytestmark = pytest.mark.gpu

O_MAX, O_RMSE, LSE_MAX = 1e-2, 2e-3, 1e-3
THREADS = os.cpu_count() or 4
DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def _inputs(B, H, H_kv, N, d, dtype, seed):
    t = DT[dtype]
    q = torch.from_numpy(synth.normal((B, N, H, d), seed=seed)).to(t)
    k = torch.from_numpy(synth.normal((B, N, H_kv, d), seed=seed + 1)).to(t)
    v = torch.from_numpy(synth.normal((B, N, H_kv, d), seed=seed + 2)).to(t)
    return q, k, v


def _run(fa, q, k, v, window, softcap, sinks, alpha):
    dev = torch.device("cuda")
    sk = None if sinks is None else torch.from_numpy(np.asarray(sinks, np.float32)).to(dev)
    o, lse = fa.attention_ext(q.to(dev), k.to(dev), v.to(dev), window=window,
                              softcap=softcap, sinks=sk, alpha=alpha)
    assert fa.fa_check_status() == fa.FA_OK
    return o, lse


def _check(o_gpu, lse_gpu, o_ref, lse_ref):
    o = o_gpu.astype(np.float64)
    assert np.all(np.isfinite(o))
    err = np.abs(o - o_ref)
    rmse = float(np.sqrt(np.mean(err ** 2)))
    assert err.max() <= O_MAX, f"O max-abs {err.max():.3e}"
    assert rmse <= O_RMSE, f"O rmse {rmse:.3e}"
    lerr = np.abs(lse_gpu.astype(np.float64) - lse_ref)
    assert lerr.max() <= LSE_MAX, f"LSE max-abs {lerr.max():.3e}"


EXT_CASES = [
    # (B, H, H_kv, N, d, window, softcap, sinks, dtype)
    (2, 4, 4, 1000, 128, (256, 0), 0.0, False, "bf16"),     # sliding causal window
    (2, 4, 4, 1000, 64, (256, 0), 0.0, False, "bf16"),
    (1, 2, 2, 1000, 128, (100, 100), 0.0, False, "bf16"),   # symmetric, narrower than a tile
    (1, 2, 2, 1000, 128, (0, 0), 0.0, False, "bf16"),       # the diagonal alone
    (1, 2, 2, 1000, 64, (127, 0), 0.0, False, "bf16"),      # tile-boundary windows
    (1, 2, 2, 1000, 64, (128, 0), 0.0, False, "bf16"),
    (1, 2, 2, 1000, 128, (129, 1), 0.0, False, "bf16"),
    (1, 2, 2, 777, 64, (-1, 300), 0.0, False, "fp16"),      # right bound only
    (1, 2, 2, 777, 128, (300, -1), 0.0, False, "bf16"),     # left bound only
    (1, 2, 2, 513, 128, (5, 700), 0.0, False, "bf16"),
    (2, 4, 4, 1000, 128, (-1, 0), 50.0, False, "bf16"),     # causal + softcap
    (1, 2, 2, 1000, 128, (-1, -1), 5.0, False, "bf16"),     # a tight softcap
    (1, 2, 2, 1000, 64, (300, 40), 5.0, False, "fp16"),
    (1, 4, 4, 1000, 128, (-1, 0), 0.0, True, "bf16"),       # sinks
    (1, 4, 4, 1000, 64, (128, 0), 30.0, True, "bf16"),      # all three
    (2, 8, 2, 1000, 128, (512, 0), 50.0, True, "bf16"),     # all three + GQA
    (1, 8, 1, 300, 64, (64, 64), 0.0, True, "fp16"),        # multi-query + sinks
    (1, 1, 1, 1, 128, (0, 0), 0.0, True, "bf16"),           # N = 1
    (1, 1, 1, 129, 128, (-1, -1), 0.0, False, "bf16"),
    (1, 3, 3, 2048, 128, (1000, 0), 0.0, True, "bf16"),
]


@pytest.mark.parametrize("B,H,H_kv,N,d,window,softcap,sinks,dtype", EXT_CASES)
def test_ext_parity(gpu_lib, B, H, H_kv, N, d, window, softcap, sinks, dtype):
    q, k, v = _inputs(B, H, H_kv, N, d, dtype, seed=synth.BASE_SEED + N + d)
    sk = synth.sinks(H, seed=N) if sinks else None
    a = synth.default_alpha(d)
    o, lse = _run(gpu_lib, q, k, v, window, softcap, sk, a)
    o_ref, lse_ref = oracle.attention_ext(q, k, v, a, window=window, softcap=softcap,
                                          sinks=sk, n_threads=THREADS)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


@pytest.mark.parametrize("H_kv", [4, 2])
@pytest.mark.parametrize("d", [64, 128])
def test_ext_windows_reproduce_plain_bits(gpu_lib, d, H_kv):
    B, H, N = 2, 4, 1000
    q, k, v = (x.cuda() for x in _inputs(B, H, H_kv, N, d, "bf16", seed=17))
    for causal, window in ((True, (-1, 0)), (False, (-1, -1))):
        o1, l1 = gpu_lib.attention(q, k, v, causal=causal)
        o2, l2 = gpu_lib.attention_ext(q, k, v, window=window)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_sink_minus_infinity_is_no_sink(gpu_lib):
    B, H, N, d = 1, 3, 700, 128
    q, k, v = (x.cuda() for x in _inputs(B, H, H, N, d, "bf16", seed=23))
    sk = torch.full((H,), -math.inf, dtype=torch.float32, device="cuda")
    o1, l1 = gpu_lib.attention_ext(q, k, v, window=(200, 0), softcap=20.0)
    o2, l2 = gpu_lib.attention_ext(q, k, v, window=(200, 0), softcap=20.0, sinks=sk)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("sigma", [12.0, 60.0, 100.0])
def test_dominant_sink(gpu_lib, sigma):
    # e^sigma far above every row sum: O -> 0 and LSE -> sigma.  At 100 the
    # sink term 2^(sigma log2 e - r) overflows FP32; the kernel then gives
    # O = 0 (the true O is below 1e-40) and still forms LSE stably.
    B, H, N, d = 1, 2, 600, 64
    q, k, v = _inputs(B, H, H, N, d, "bf16", seed=29)
    sk = np.full((H,), sigma, dtype=np.float32)
    a = synth.default_alpha(d)
    o, lse = _run(gpu_lib, q, k, v, (100, 0), 0.0, sk, a)
    o_ref, lse_ref = oracle.attention_ext(q, k, v, a, window=(100, 0), sinks=sk,
                                          n_threads=THREADS)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


def test_sampled_b4_h16_n4096_d128_sliding_softcap_sinks(gpu_lib):
    B, H, N, d = 4, 16, 4096, 128
    window, softcap = (1024, 0), 50.0
    q, k, v = synth.qkv(B, H, N, d, seed=synth.BASE_SEED + 99)
    sk = synth.sinks(H, seed=99)
    a = synth.default_alpha(d)
    o, lse = _run(gpu_lib, q, k, v, window, softcap, sk, a)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    rng = np.random.default_rng(5)
    for b, h in [(0, 0), (3, 15), (1, 7)]:
        rows = sorted(set([0, 1, 127, 128, 1023, 1024, 1025, N // 2, N - 1] +
                          rng.integers(0, N, size=16).tolist()))
        o_ref, l_ref = oracle.attention_ext_rows(q, k, v, a, b, h, rows, window, softcap, sk)
        _check(o[b, rows, h, :], lse[b, h, rows], o_ref, l_ref)


def test_sampled_long_sequence_window_and_sinks(gpu_lib):
    # N = 2^16 + 1 with a sliding window: far-apart rows see disjoint keys.
    B, H, N, d = 1, 2, 65537, 128
    window = (4096, 0)
    q, k, v = synth.qkv(B, H, N, d, seed=synth.BASE_SEED + 123)
    sk = synth.sinks(H, seed=123)
    a = synth.default_alpha(d)
    o, lse = _run(gpu_lib, q, k, v, window, 0.0, sk, a)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    rows = [0, 4095, 4096, 4097, 32768, 65535, 65536]
    for h in range(H):
        o_ref, l_ref = oracle.attention_ext_rows(q, k, v, a, 0, h, rows, window, 0.0, sk)
        _check(o[0, rows, h, :], lse[0, h, rows], o_ref, l_ref)
