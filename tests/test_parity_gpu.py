"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle.

Tolerances (stated for unit-variance inputs): O max-abs <= 1e-2, O RMSE
<= 2e-3, LSE max-abs <= 1e-3.  Small and ragged shapes are compared element
by element in full.  At full size, the N = 4096 and N = 16384 points of the
16k-token sequence sweep (B = 16384 / N; d = 64, 128, 256; plain and causal)
are compared element by element on every O and LSE value; N = 4096, d = 128
is the bench's own workload (same seed, same launch configuration).  The
other sweep points are compared on sampled (b, h, row) outputs that the
oracle computes one by one.  Exact pins: causal row 0 reproduces V[0] bit for bit, a constant V
gives that constant, and two launches give identical bits.
"""
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


def _run(fa, q, k, v, causal, alpha, want_lse=True, stream=None, pack_gqa=False):
    dev = torch.device("cuda")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=causal,
                          alpha=alpha, want_lse=want_lse, stream=stream, pack_gqa=pack_gqa)
    assert fa.fa_check_status() == fa.FA_OK
    return o, lse


def _check(o_gpu, lse_gpu, o_ref, lse_ref, scale_aware=False):
    o = o_gpu.astype(np.float64)
    err = np.abs(o - o_ref)
    rmse = float(np.sqrt(np.mean(err ** 2)))
    assert np.all(np.isfinite(o))
    if scale_aware:
        # Inputs far from unit variance make |O| reach several units, where
        # the spacing of BF16 values alone exceeds 1e-2: allow one BF16 ulp
        # of the value (2^-8 |O|) on top of the unit-scale bound.
        bound = O_MAX + 2.0 ** -8 * np.abs(o_ref)
        assert np.all(err <= bound), f"O err/bound {(err / bound).max():.3f}"
    else:
        assert err.max() <= O_MAX, f"O max-abs {err.max():.3e}"
    assert rmse <= O_RMSE, f"O rmse {rmse:.3e}"
    if lse_gpu is not None:
        lerr = np.abs(lse_gpu.astype(np.float64) - lse_ref)
        assert lerr.max() <= LSE_MAX, f"LSE max-abs {lerr.max():.3e}"
    return float(err.max()), rmse


FULL_CASES = [
    # (B, H, N, d, causal, dtype)
    (1, 1, 128, 64, False, "bf16"),        # the smallest workload (one tile)
    (2, 8, 1024, 64, False, "bf16"),       # B2 H8 N1024 d64
    (2, 8, 1024, 64, True, "bf16"),
    (2, 8, 1000, 64, False, "bf16"),       # N not a tile multiple
    (2, 8, 1000, 64, True, "bf16"),
    (1, 1, 1, 64, False, "bf16"),
    (1, 1, 1, 128, True, "bf16"),
    (1, 2, 127, 128, True, "bf16"),
    (2, 3, 129, 64, True, "bf16"),
    (1, 2, 255, 64, False, "bf16"),
    (1, 1, 257, 128, True, "bf16"),
    (1, 2, 300, 128, False, "bf16"),
    (3, 1, 384, 128, True, "bf16"),
    (1, 2, 513, 128, False, "fp16"),
    (1, 2, 513, 128, True, "fp16"),
    (1, 1, 640, 64, True, "fp16"),
    (1, 1, 1, 256, True, "bf16"),          # head dim 256: one Q tile per unit
    (1, 1, 64, 256, False, "bf16"),
    (2, 1, 129, 256, True, "bf16"),
    (1, 2, 300, 256, False, "bf16"),
    (1, 2, 300, 256, True, "bf16"),
    (1, 2, 513, 256, False, "fp16"),
    (2, 2, 1000, 256, True, "bf16"),
]


@pytest.mark.parametrize("B,H,N,d,causal,dtype", FULL_CASES)
def test_full_parity(gpu_lib, B, H, N, d, causal, dtype):
    q, k, v = synth.qkv(B, H, N, d, seed=synth.BASE_SEED + N, dtype=dtype)
    alpha = synth.default_alpha(d)
    o, lse = _run(gpu_lib, q, k, v, causal, alpha)
    o_ref, lse_ref = oracle.attention(q, k, v, alpha, causal, n_threads=THREADS)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


def _sampled(fa, B, H, N, d, causal, n_heads=3, n_rows=24, seed=0):
    q, k, v = synth.qkv(B, H, N, d, seed=synth.BASE_SEED + 7 * N + d)
    alpha = synth.default_alpha(d)
    o, lse = _run(fa, q, k, v, causal, alpha)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    rng = np.random.default_rng(seed + N + d)
    heads = {(0, 0), (B - 1, H - 1)}
    while len(heads) < min(n_heads, B * H):
        heads.add((int(rng.integers(B)), int(rng.integers(H))))
    for b, h in sorted(heads):
        rows = sorted(set([0, 1, 127, 128, N // 2, N - 1] +
                          rng.integers(0, N, size=n_rows).tolist()))
        o_ref, lse_ref = oracle.attention_rows(q, k, v, alpha, causal, b, h, rows)
        _check(o[b, rows, h, :], lse[b, h, rows], o_ref, lse_ref)


def test_sampled_b4_h16_n4096_d128(gpu_lib):
    _sampled(gpu_lib, 4, 16, 4096, 128, False)


# Every element at full size: the N = 4096 and N = 16384 points of the sweep
# at each head dim (hidden 2048, 16k tokens), plain and causal.
FULL_SIZE = [(n, d, h, c) for n in (4096, 16384)
             for (d, h) in ((64, 32), (128, 16), (256, 8)) for c in (False, True)]


@pytest.mark.parametrize("N,d,H,causal", FULL_SIZE)
def test_full_size_every_element(gpu_lib, N, d, H, causal):
    B = 16384 // N
    q, k, v = synth.qkv(B, H, N, d, seed=synth.BASE_SEED)
    alpha = synth.default_alpha(d)
    o, lse = _run(gpu_lib, q, k, v, causal, alpha)
    o_ref, lse_ref = oracle.attention(q, k, v, alpha, causal, n_threads=THREADS)
    mx, rmse = _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)
    print(f"full B{B} H{H} N{N} d{d} causal={causal}: O max-abs {mx:.3e} rmse {rmse:.3e}")


SWEEP = [(n, d, h, c) for n in (512, 1024, 2048, 4096, 8192, 16384)
         for (d, h) in ((64, 32), (128, 16), (256, 8)) for c in (False, True)]


@pytest.mark.parametrize("N,d,H,causal", SWEEP)
def test_sampled_sequence_sweep(gpu_lib, N, d, H, causal):
    _sampled(gpu_lib, 16384 // N, H, N, d, causal, n_heads=2, n_rows=16)


def test_unsupported_head_dim_is_rejected(gpu_lib):
    fa = gpu_lib
    x = torch.zeros((1, 128, 1, 96), dtype=torch.bfloat16, device="cuda")
    rc = fa.fa_fwd(x, x, x, x, None, 1, 1, 128, 96, 0.1, 0, fa.FA_BF16)
    assert rc == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("d", [64, 128, 256])
def test_causal_row_zero_is_v0_exactly(gpu_lib, d):
    B, H, N = 2, 3, 700
    q, k, v = synth.qkv(B, H, N, d, seed=11)
    o, lse = _run(gpu_lib, q, k, v, True, synth.default_alpha(d))
    assert torch.equal(o[:, 0].cpu(), v[:, 0])
    s0 = synth.default_alpha(d) * (q[:, 0].double() * k[:, 0].double()).sum(-1)
    assert torch.allclose(lse[:, :, 0].cpu().double(), s0, atol=1e-5, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_give_the_constant(gpu_lib, causal):
    B, H, N, d = 1, 2, 1000, 128
    q, k, _ = synth.qkv(B, H, N, d, seed=5)
    v = torch.full((B, N, H, d), 0.71875, dtype=torch.bfloat16)   # exact in bf16
    o, _ = _run(gpu_lib, q, k, v, causal, synth.default_alpha(d))
    of = o.float().cpu()
    # sum_j p_j c / sum_j p_j = c up to FP32 rounding, then one bf16 rounding
    assert (of - 0.71875).abs().max().item() <= 2.0 ** -8


def test_deterministic_bits_lse_optional_and_side_stream(gpu_lib):
    fa = gpu_lib
    B, H, N, d = 2, 4, 1536, 128
    q, k, v = synth.qkv(B, H, N, d, seed=3)
    a = synth.default_alpha(d)
    o1, l1 = _run(fa, q, k, v, False, a)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = _run(fa, q, k, v, False, a, stream=s)
    s.synchronize()
    o3, l3 = _run(fa, q, k, v, False, a, want_lse=False)
    assert l3 is None
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_causal_dynamic_order_repeats_bits(gpu_lib, d):
    # Causal launches hand units to CTAs dynamically (which CTA runs which
    # tile differs between launches); every launch must give the same bits,
    # with one K/V head per query head and with grouped K/V heads.
    B, H, N = 3, 8, 1300
    q, k, v = (x.cuda() for x in synth.qkv(B, H, N, d, seed=21))
    a = synth.default_alpha(d)
    runs = [gpu_lib.attention(q, k, v, causal=True, alpha=a) for _ in range(3)]
    kg, vg = k[:, :, :2].contiguous(), v[:, :, :2].contiguous()
    runs_g = [gpu_lib.attention(q, kg, vg, causal=True, alpha=a) for _ in range(3)]
    assert gpu_lib.fa_check_status() == gpu_lib.FA_OK
    for rs in (runs, runs_g):
        for o, l in rs[1:]:
            assert torch.equal(o, rs[0][0]) and torch.equal(l, rs[0][1])


@pytest.mark.parametrize("B,H,N,d", [(32, 64, 640, 64), (4, 16, 4096, 128), (2, 8, 2000, 256)])
def test_dynamic_order_writes_every_row(gpu_lib, B, H, N, d):
    # Causal launches have one CTA per unit and let running CTAs take over
    # the others (up to 6144 here).  O and LSE start as NaN: a unit that no
    # CTA ran would leave NaN rows, one that ran twice would still give the
    # same values, so every row must come out finite and equal to a
    # launch's own bits on the second run.
    fa = gpu_lib
    q, k, v = (x.cuda() for x in synth.qkv(B, H, N, d, seed=33))
    a = synth.default_alpha(d)
    outs = []
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        assert fa.fa_fwd(q, k, v, o, lse, B, H, N, d, a, 1, fa.FA_BF16) == fa.FA_OK
        outs.append((o, lse))
    assert fa.fa_check_status() == fa.FA_OK
    for o, lse in outs:
        assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_dynamic_order_backward_writes_every_row(gpu_lib):
    # The causal backward's two main kernels take the same dynamic order:
    # dQ, dK, dV start as NaN and must come out finite everywhere.
    fa = gpu_lib
    B, H, N, d = 8, 16, 1500, 128
    q, k, v = (x.cuda() for x in synth.qkv(B, H, N, d, seed=34))
    do = torch.from_numpy(synth.normal((B, N, H, d), seed=35)).to(q.dtype).cuda()
    a = synth.default_alpha(d)
    o, lse = fa.attention(q, k, v, causal=True, alpha=a)
    g = [torch.full_like(q, float("nan")) for _ in range(3)]
    ws = torch.empty((fa.bwd_workspace_floats(B, H, N),), dtype=torch.float32, device="cuda")
    assert fa.fa_bwd(q, k, v, o, do, lse, ws, *g, B, H, N, d, a, 1, fa.FA_BF16) == fa.FA_OK
    assert fa.fa_check_status() == fa.FA_OK
    assert all(bool(torch.isfinite(x).all()) for x in g)


def _offset16(n, dtype):
    """A device buffer of n elements that starts 16 bytes past a 32-byte
    boundary (torch allocations are 256-byte aligned)."""
    shift = 16 // torch.empty((), dtype=dtype).element_size()
    buf = torch.empty((n + shift,), dtype=dtype, device="cuda")
    out = buf[shift:]
    assert out.data_ptr() % 32 == 16
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_outputs_at_16_byte_offsets_match_aligned_bits(gpu_lib, causal):
    # The API promises 16-byte alignment only: the O stores and the split
    # partials must give the same bits there as at a 256-byte boundary.
    fa = gpu_lib
    B, H, N, d = 2, 3, 700, 64
    q, k, v = (x.cuda() for x in synth.qkv(B, H, N, d, seed=12))
    a = synth.default_alpha(d)
    o1, l1 = fa.attention(q, k, v, causal=causal, alpha=a)
    o2 = _offset16(q.numel(), q.dtype).view(q.shape)
    l2 = torch.empty_like(l1)
    assert fa.fa_fwd(q, k, v, o2, l2, B, H, N, d, a, int(causal), fa.FA_BF16) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    S = 2
    ws = _offset16(fa.fa_splitkv_workspace_floats(B, H, N, d, S), torch.float32)
    o3 = torch.empty_like(q)
    l3 = torch.empty_like(l1)
    assert fa.fa_fwd_splitkv(q, k, v, o3, l3, B, H, N, d, a, int(causal), fa.FA_BF16, S,
                             ws) == fa.FA_OK
    o4, l4 = fa.attention_splitkv(q, k, v, causal=causal, alpha=a, n_splits=S)
    assert fa.fa_check_status() == fa.FA_OK
    assert torch.equal(o3, o4) and torch.equal(l3, l4)


@pytest.mark.parametrize("alpha", [0.03, 0.5])
def test_other_scales_and_wide_scores(gpu_lib, alpha):
    # Scores with a wide spread move the reference point often (tau = 8).
    B, H, N, d = 1, 2, 777, 64
    q, k, v = synth.qkv(B, H, N, d, seed=21)
    q = (q.float() * 3).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = _run(gpu_lib, q, k, v, causal, alpha)
        o_ref, lse_ref = oracle.attention(q, k, v, alpha, causal, n_threads=THREADS)
        _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
               scale_aware=True)


@pytest.mark.parametrize("lift", [2.0, 5.0])
@pytest.mark.parametrize("d", [64, 128])
def test_late_spike_moves_the_reference(gpu_lib, d, lift):
    # Key 0 scores far above every other key for most rows.  Key tiles are
    # visited from the last to the first, so the spike arrives on the final
    # tile: depending on the row the reference point either stays (P up to
    # 2^16) or moves late, rescaling everything accumulated before it.
    B, H, N = 1, 2, 700
    q, k, v = synth.qkv(B, H, N, d, seed=33)
    u = torch.ones(d) / d ** 0.5
    q = (q.float() + lift * u).to(torch.bfloat16)
    k = k.clone()
    k[:, 0] = (5.0 * d ** 0.5 * u).to(torch.bfloat16)
    a = synth.default_alpha(d)
    for causal in (False, True):
        o, lse = _run(gpu_lib, q, k, v, causal, a)
        o_ref, lse_ref = oracle.attention(q, k, v, a, causal, n_threads=THREADS)
        _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
               scale_aware=True)


def test_outputs_beyond_n_untouched(gpu_lib):
    # Rows >= N of the last tile are computed but never stored.
    fa = gpu_lib
    B, H, N, d = 1, 1, 200, 128
    q, k, v = synth.qkv(B, H, N, d, seed=9)
    big = torch.full((B, N + 64, H, d), 7.0, dtype=torch.bfloat16, device="cuda")
    o = big[:, :N]                                  # contiguous prefix view
    lse = torch.full((B, H, N + 64), 9.0, dtype=torch.float32, device="cuda")
    rc = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), o, lse, B, H, N, d,
                   synth.default_alpha(d), 0, fa.FA_BF16)
    assert rc == fa.FA_OK and fa.fa_check_status() == fa.FA_OK
    assert torch.all(big[:, N:] == 7.0)
    assert torch.all(lse[:, :, N:] == 9.0)


GQA_CASES = [
    # (B, H, H_kv, N, d, causal)
    (2, 8, 2, 1000, 128, True),
    (2, 8, 2, 1000, 128, False),
    (1, 8, 1, 513, 64, True),           # multi-query
    (1, 6, 3, 257, 64, False),
    (1, 4, 2, 300, 256, True),
    (1, 4, 1, 129, 256, False),
]


@pytest.mark.parametrize("B,H,H_kv,N,d,causal", GQA_CASES)
def test_gqa_parity(gpu_lib, B, H, H_kv, N, d, causal):
    # Grouped key/value heads: query head h attends with K/V head
    # h // (H // H_kv) ("FlashAttention-3 on Hopper", ch. 11).
    q = torch.from_numpy(synth.normal((B, N, H, d), seed=N + 1)).to(torch.bfloat16)
    k = torch.from_numpy(synth.normal((B, N, H_kv, d), seed=N + 2)).to(torch.bfloat16)
    v = torch.from_numpy(synth.normal((B, N, H_kv, d), seed=N + 3)).to(torch.bfloat16)
    a = synth.default_alpha(d)
    o, lse = _run(gpu_lib, q, k, v, causal, a)
    o_ref, lse_ref = oracle.attention_gqa(q, k, v, a, causal, n_threads=THREADS)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


PACK_CASES = [
    # (B, H, H_kv, N, d, causal, dtype): group g = H / H_kv query heads per
    # K/V head share each Q tile of 128 / g positions
    (2, 8, 4, 1000, 128, True, torch.bfloat16),      # g = 2
    (2, 8, 2, 1000, 128, False, torch.bfloat16),     # g = 4
    (1, 8, 1, 513, 64, True, torch.bfloat16),        # g = 8 (multi-query)
    (1, 16, 1, 77, 64, False, torch.bfloat16),       # g = 16, one partial tile
    (1, 32, 1, 300, 128, True, torch.float16),       # g = 32: 4 positions a tile
    (1, 64, 1, 130, 64, True, torch.bfloat16),       # g = 64: 2 positions a tile
    (1, 4, 2, 1, 64, False, torch.bfloat16),         # one position
    (2, 16, 2, 2048, 128, True, torch.bfloat16),     # many units, longest first
]


@pytest.mark.parametrize("B,H,H_kv,N,d,causal,dtype", PACK_CASES)
def test_gqa_packed_parity(gpu_lib, B, H, H_kv, N, d, causal, dtype):
    # Packed grouped heads: tile row p holds position m R + p / g of query
    # head h g + p % g; every row must still equal the definition.
    q = torch.from_numpy(synth.normal((B, N, H, d), seed=N + 11)).to(dtype)
    k = torch.from_numpy(synth.normal((B, N, H_kv, d), seed=N + 12)).to(dtype)
    v = torch.from_numpy(synth.normal((B, N, H_kv, d), seed=N + 13)).to(dtype)
    a = synth.default_alpha(d)
    o, lse = _run(gpu_lib, q, k, v, causal, a, pack_gqa=True)
    o_ref, lse_ref = oracle.attention_gqa(q, k, v, a, causal, n_threads=THREADS)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


def test_gqa_packed_matches_unpacked_closely(gpu_lib):
    # The same rows through both layouts: the per-row arithmetic is the
    # same, only the warp-wide rescale decisions see other rows, so the
    # results agree to a few ulp of the output, not bit for bit.
    B, H, H_kv, N, d = 2, 16, 4, 1500, 128
    q = torch.from_numpy(synth.normal((B, N, H, d), seed=5)).to(torch.bfloat16)
    k = torch.from_numpy(synth.normal((B, N, H_kv, d), seed=6)).to(torch.bfloat16)
    v = torch.from_numpy(synth.normal((B, N, H_kv, d), seed=7)).to(torch.bfloat16)
    a = synth.default_alpha(d)
    for causal in (False, True):
        o1, l1 = _run(gpu_lib, q, k, v, causal, a)
        o2, l2 = _run(gpu_lib, q, k, v, causal, a, pack_gqa=True)
        assert float((o1.float() - o2.float()).abs().max()) <= 2 ** -7
        assert float((l1 - l2).abs().max()) <= 1e-4


def test_gqa_packed_with_one_head_per_group_is_the_plain_forward(gpu_lib):
    # g = 1: fa_fwd_gqa_packed takes the plain layout, so its bits equal fa_fwd's.
    fa = gpu_lib
    B, H, N, d = 2, 3, 700, 128
    q, k, v = (x.cuda() for x in synth.qkv(B, H, N, d, seed=17))
    a = synth.default_alpha(d)
    outs = []
    for call in ("fa_fwd", "fa_fwd_gqa_packed"):
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        if call == "fa_fwd":
            rc = fa.fa_fwd(q, k, v, o, lse, B, H, N, d, a, 1, fa.FA_BF16)
        else:
            rc = fa.fa_fwd_gqa_packed(q, k, v, o, lse, B, H, H, N, d, a, 1, fa.FA_BF16)
        assert rc == fa.FA_OK and fa.fa_check_status() == fa.FA_OK
        outs.append((o, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


SPLIT_CASES = [
    # (B, H, N, d, causal, n_splits)
    (1, 2, 1000, 128, True, 3),
    (1, 2, 1000, 128, False, 2),
    (2, 1, 777, 64, True, 5),
    (1, 1, 300, 64, False, 4),
    (1, 1, 128, 128, False, 2),        # one key tile: one split holds nothing
    (1, 3, 4096, 128, True, 7),
]


@pytest.mark.parametrize("B,H,N,d,causal,S", SPLIT_CASES)
def test_splitkv_parity(gpu_lib, B, H, N, d, causal, S):
    # Split-KV ("FlashAttention-3 on Hopper", ch. 10): partials over split
    # key ranges, merged by their LSEs, equal the one-pass definition.
    q, k, v = synth.qkv(B, H, N, d, seed=N + S)
    a = synth.default_alpha(d)
    dev = torch.device("cuda")
    o, lse = gpu_lib.attention_splitkv(q.to(dev), k.to(dev), v.to(dev), causal=causal,
                                       alpha=a, n_splits=S)
    assert gpu_lib.fa_check_status() == gpu_lib.FA_OK
    o_ref, lse_ref = oracle.attention(q, k, v, a, causal, n_threads=THREADS)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


def test_splitkv_one_split_equals_fa_fwd(gpu_lib):
    # One split is the whole key range: the combine weight is exactly 1, so
    # the result is fa_fwd's, bit for bit.
    B, H, N, d = 2, 2, 700, 128
    q, k, v = (x.cuda() for x in synth.qkv(B, H, N, d, seed=3))
    for causal in (False, True):
        o1, l1 = gpu_lib.attention(q, k, v, causal=causal)
        o2, l2 = gpu_lib.attention_splitkv(q, k, v, causal=causal, n_splits=1)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("N,d,causal", [(65537, 128, False), (65537, 64, True), (131072, 128, True)])
def test_sampled_long_sequences(gpu_lib, N, d, causal):
    # Long sequences: 64-bit row offsets, a ragged last tile (N = 2^16 + 1),
    # 512-1024 key tiles per unit; rows sampled across the whole range.
    _sampled(gpu_lib, 1, 2, N, d, causal, n_heads=2, n_rows=12)


def test_sampled_many_units(gpu_lib):
    # B32 H64 N640: 2048 heads, 6144 work units -- many waves of the
    # persistent grid; heads sampled at both ends and in between.
    _sampled(gpu_lib, 32, 64, 640, 64, True, n_heads=4, n_rows=8)
