"""GPU parity of the backward pass: fa_bwd (through the C ABI) against the
FP64 oracle gradients ("FlashAttention-3 on Hopper", sec. 7.1).

The forward runs first on the GPU (fa_fwd gives O and LSE); the oracle
computes dQ, dK, dV from the definition on the same 16-bit inputs and dO.

Tolerances, from the arithmetic: each gradient passes through three
roundings of at most half a 16-bit ulp -- the rounding of P or dS before the
GEMM that consumes it, the rounding of O inside D = rowsum(dO o O), and the
rounding of the output -- on top of FP32 accumulation.  With u the relative
spacing of the type (2^-8 bf16, 2^-10 fp16) that gives a relative RMS error
below u (measured ~0.6 u) and an elementwise error below a few u of the
tensor's largest value.  The tests use rel-RMSE <= 1.5 u and
max |g - g_ref| <= 4 u max |g_ref|.  Gradients that are zero in exact
arithmetic (one visible key) must come out below 1e-5 in absolute value.
"""
import os
from concurrent.futures import ThreadPoolExecutor

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


def _gpu_grads(fa, q, k, v, do, causal, alpha):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fa.attention(qd, kd, vd, causal=causal, alpha=alpha)
    g = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, alpha=alpha)
    assert fa.fa_check_status() == fa.FA_OK
    return [x.float().cpu().numpy().astype(np.float64) for x in g]


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


CASES = [
    # (B, H, N, d, causal, dtype)
    (1, 1, 128, 64, False, "bf16"),
    (1, 1, 128, 128, True, "bf16"),
    (1, 1, 1, 128, True, "bf16"),
    (1, 1, 1, 64, False, "bf16"),
    (1, 2, 127, 64, True, "bf16"),
    (2, 2, 257, 64, True, "bf16"),
    (1, 2, 300, 128, False, "bf16"),
    (1, 2, 300, 128, True, "bf16"),
    (2, 8, 1024, 64, False, "bf16"),       # B2 H8 N1024 d64
    (2, 8, 1024, 64, True, "bf16"),
    (2, 8, 1000, 64, True, "bf16"),        # N not a tile multiple
    (1, 2, 1000, 128, True, "bf16"),
    (1, 2, 513, 128, True, "fp16"),
    (1, 2, 513, 64, False, "fp16"),
]


@pytest.mark.parametrize("B,H,N,d,causal,dtype", CASES)
def test_bwd_parity(gpu_lib, B, H, N, d, causal, dtype):
    q, k, v, do = _inputs(B, H, N, d, dtype, seed=N + d)
    a = synth.default_alpha(d)
    got = _gpu_grads(gpu_lib, q, k, v, do, causal, a)
    ref = oracle.attention_bwd(q, k, v, do, a, causal, n_threads=THREADS)
    _check(got, ref, ULP[dtype])


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_sampled_b4_h16_n4096_d128(gpu_lib, causal):
    # The full workload in the bench's launch configuration; the oracle
    # recomputes the gradients of four sampled heads from the definition.
    B, H, N, d = 4, 16, 4096, 128
    q, k, v, do = _inputs(B, H, N, d, "bf16", seed=synth.BASE_SEED)
    a = synth.default_alpha(d)
    got = _gpu_grads(gpu_lib, q, k, v, do, causal, a)
    heads = [(0, 0), (1, 7), (2, 11), (3, 15)]

    def ref(bh):
        b, h = bh
        return oracle.attention_bwd_head(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h],
                                         a, causal)

    with ThreadPoolExecutor(len(heads)) as ex:
        refs = list(ex.map(ref, heads))
    for (b, h), r in zip(heads, refs):
        _check([g[b, :, h] for g in got], r, ULP["bf16"])


def test_bwd_deterministic_and_causal_row_zero(gpu_lib):
    fa = gpu_lib
    B, H, N, d = 1, 2, 777, 128
    q, k, v, do = _inputs(B, H, N, d, "bf16", seed=5)
    a = synth.default_alpha(d)
    g1 = _gpu_grads(fa, q, k, v, do, True, a)
    g2 = _gpu_grads(fa, q, k, v, do, True, a)
    for x, y in zip(g1, g2):
        assert np.array_equal(x, y)
    # Query 0 sees only key 0, so its softmax is constant: dQ row 0 is zero
    # (up to the rounding difference of D and dP).
    assert np.abs(g1[0][:, 0]).max() <= 1e-5


@pytest.mark.parametrize("alpha", [0.03, 0.5])
def test_bwd_other_scales_and_wide_scores(gpu_lib, alpha):
    # With wide scores the softmax rows are nearly one-hot, so dS = P o
    # (dP - D) is a small difference of nearly equal terms: the rounding of
    # O inside D (half an ulp of O) no longer shrinks with the gradient, and
    # the relative RMS error is allowed 3 u instead of 1.5 u.
    B, H, N, d = 1, 2, 500, 64
    q, k, v, do = _inputs(B, H, N, d, "bf16", seed=21)
    q = (q.float() * 3).to(torch.bfloat16)
    for causal in (False, True):
        got = _gpu_grads(gpu_lib, q, k, v, do, causal, alpha)
        ref = oracle.attention_bwd(q, k, v, do, alpha, causal, n_threads=THREADS)
        _check(got, ref, ULP["bf16"], rms_units=3.0)


def test_bwd_unsupported_head_dim_is_rejected(gpu_lib):
    fa = gpu_lib
    x = torch.zeros((1, 128, 1, 256), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device="cuda")
    rc = fa.fa_bwd(x, x, x, x, x, lse, lse, x, x, x, 1, 1, 128, 256, 0.0625, 0, fa.FA_BF16)
    assert rc == fa.FA_ERR_UNSUPPORTED


def test_bwd_long_sequence_sampled_dq_and_dk_sum(gpu_lib):
    # N = 2^15 + 5, non-causal: dQ of a query row depends on that row alone,
    # so sampled rows are checked against the oracle gradient of those rows
    # over all keys; dK, dV are checked through a property that holds at any
    # size: sum_j dK_j = alpha sum_i (sum_j dS_ij) q_i = 0 because every row
    # of dS sums to zero (sum_j P_ij (dP_ij - D_i) = D_i - D_i).
    B, H, N, d = 1, 1, 32773, 128
    q, k, v, do = _inputs(B, H, N, d, "bf16", seed=77)
    a = synth.default_alpha(d)
    dq, dk, dv = _gpu_grads(gpu_lib, q, k, v, do, False, a)
    rows = [0, 1, 127, 128, 16384, N - 2, N - 1]
    ref = oracle.attention_bwd_head(q[0, rows, 0], k[0, :, 0], v[0, :, 0], do[0, rows, 0],
                                    a, False)
    _check([dq[0, rows, 0]], [ref[0]], ULP["bf16"])
    s = dk[0, :, 0].sum(axis=0)
    assert np.all(np.abs(s) <= 4 * ULP["bf16"] * np.abs(dk[0, :, 0]).sum(axis=0) / np.sqrt(N) + 1e-3)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_back_to_back_launches_stay_in_step(gpu_lib, d):
    # Many causal launches queued without a host synchronisation between
    # them, the way a training loop issues them.  Each CTA's roles hand
    # tiles over through barriers whose phases must each hold one tile's
    # arrivals; a warp that ran a tile ahead onto a shared barrier once
    # made a phase complete early and left a wait that never ended (it ran
    # out its bound and set the status word).  Every launch must leave the
    # status word clear and give the same bits.
    fa = gpu_lib
    dev = torch.device("cuda")
    B, H, N = 4, 32 if d == 64 else 16, 4096
    q, k, v, do = (x.to(dev) for x in _inputs(B, H, N, d, "bf16", seed=91))
    o, lse = fa.attention(q, k, v, causal=True)
    first = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    same = torch.ones((), dtype=torch.bool, device=dev)
    for _ in range(60):
        g = fa.attention_backward(q, k, v, o, lse, do, causal=True)
        for x, y in zip(g, first):
            same &= (x == y).all()
    assert fa.fa_check_status() == fa.FA_OK
    assert bool(same.item())
    assert all(bool(torch.isfinite(x).all()) for x in first)
