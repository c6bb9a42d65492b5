"""GPU checks of the FP8 path: the quantization pre-pass against the
oracle's block quantization, and the FP8 forward against FP64 attention.

* Quantization ("FlashAttention-3 on Hopper", sec. 6.3-6.4): scales equal
  amax/448 of the (rotated) tile -- exactly without rotation, to 2^-20
  relative with it (the kernel's FP32 Walsh-Hadamard butterflies round);
  codes equal the round-to-nearest e4m3 code of y/scale (the kernel forms
  y * (1/scale) in FP32, within one rounding of the quotient), except where
  y/scale lies within 2^-18 of a rounding boundary, where either neighbour
  is valid.
* FP8 forward on the outlier distribution (N(0,1) + 0.1% N(0,100)), the
  metric of the FA3 numerical-error experiment: O RMSE against the FP64
  oracle on the unquantized inputs <= 1.5e-2 with block scales and the
  Hadamard rotation; the rotation lowers the error.
* A bound derived from the arithmetic, against FP64 attention on the
  dequantized (rotated) inputs, i.e. the operands the tensor core sees: the
  kernel differs only by the e4m3 rounding of P' (relative 2^-4 for normal
  values, absolute 2^-10 below 2^-6) and FP32 accumulation.  P' is formed
  as 2^(x - r + c), so a row's terms sum to at least 2^c (c = 4), and
      |O_gpu - O_deq| <= (2^-4 + n_keys 2^-10 / (ratio_min 2^c)) max_j |v_j - O_deq|
                        + 2^-8 |O_deq| + 1e-3.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_fa_gb300 import synth

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 4


def _quant(fa, x, signs, granularity=0):
    dev = torch.device("cuda")
    s = None if signs is None else torch.from_numpy(signs).to(dev)
    x8, sc = fa.quantize_fp8(x.to(dev), s, granularity=granularity)
    assert fa.fa_check_status() == fa.FA_OK
    return x8.cpu().numpy(), sc.cpu().numpy()


def _check_codes(got, xh, y, scale_rows, rotate):
    """Codes of one head against the oracle's e4m3 encoding, given the
    per-row scales the kernel used (float32 [rows, 1])."""
    if not rotate:
        # Same decision in the kernel's precision: the FP32 product
        # x * (1 / scale), then round-to-nearest-even to e4m3 -> bit exact.
        inv = np.float32(1.0) / scale_rows
        q32 = (xh.astype(np.float32) * inv).astype(np.float64)
        assert np.array_equal(got, oracle.e4m3_encode(q32))
    else:
        # The rotated values carry FP32 butterfly rounding: the code is the
        # RNE code of y/scale, or a neighbour where y/scale lies within
        # 2^-18 of a rounding boundary.
        v = y / scale_rows.astype(np.float64)
        lo = oracle.e4m3_encode(v * (1 - 2.0 ** -18) - 2.0 ** -40)
        hi = oracle.e4m3_encode(v * (1 + 2.0 ** -18) + 2.0 ** -40)
        mid = oracle.e4m3_encode(v)
        ok = (got == mid) | (got == lo) | (got == hi)
        assert np.all(ok), np.argwhere(~ok)[:5]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("rotate", [False, True])
def test_quantize_matches_oracle(gpu_lib, d, rotate):
    B, H, N = 2, 3, 300
    x = torch.from_numpy(synth.normal((B, N, H, d), seed=77 + d, outliers=True)).to(torch.bfloat16)
    signs = synth.hadamard_signs(d, seed=5) if rotate else None
    x8, sc = _quant(gpu_lib, x, signs)
    for b in range(B):
        for h in range(H):
            xh = x[b, :, h, :].double().numpy()
            y = oracle.hadamard_rotate(xh, signs) if rotate else xh
            codes_ref, sc_ref = oracle.quantize_e4m3_tiles(y, 128)
            rel = np.abs(sc[b, h] - sc_ref) / sc_ref
            assert np.all(rel <= (2.0 ** -20 if rotate else 0.0)), rel.max()
            scale_rows = np.repeat(sc[b, h], 128)[:N, None]          # float32
            _check_codes(x8[b, :, h, :], xh, y, scale_rows, rotate)


@pytest.mark.parametrize("granularity", ["head", "tensor"])
@pytest.mark.parametrize("rotate", [False, True])
def test_quantize_granular_matches_oracle(gpu_lib, granularity, rotate):
    # One scale per head (the oracle's block quantization with one tile of
    # N rows) or per tensor (one tile of all B N H rows: the maximum is
    # order-free), repeated over the per-tile layout.
    fa = gpu_lib
    B, H, N, d = 2, 3, 300, 128
    g = fa.FA_SCALE_HEAD if granularity == "head" else fa.FA_SCALE_TENSOR
    x = torch.from_numpy(synth.normal((B, N, H, d), seed=91, outliers=True)).to(torch.bfloat16)
    signs = synth.hadamard_signs(d, seed=6) if rotate else None
    x8, sc = _quant(fa, x, signs, g)
    xd = x.double().numpy()
    y = oracle.hadamard_rotate(xd, signs) if rotate else xd
    tol = 2.0 ** -20 if rotate else 0.0
    if g == fa.FA_SCALE_TENSOR:
        _, s_all = oracle.quantize_e4m3_tiles(y.reshape(-1, d), B * N * H)
    for b in range(B):
        for h in range(H):
            if g == fa.FA_SCALE_HEAD:
                _, s_ref = oracle.quantize_e4m3_tiles(y[b, :, h, :], N)
            else:
                s_ref = s_all
            assert s_ref.shape == (1,)
            rel = np.abs(sc[b, h] - s_ref[0]) / s_ref[0]
            assert np.all(rel <= tol), rel.max()
            assert np.all(sc[b, h] == sc[b, h, 0])
            scale_rows = np.repeat(sc[b, h], 128)[:N, None]
            _check_codes(x8[b, :, h, :], xd[b, :, h, :], y[b, :, h, :], scale_rows, rotate)


def test_quantize_e4m3_ties_round_to_even(gpu_lib):
    # A tile with amax 448 has scale 1, so its codes are e4m3(x) directly:
    # every exact midpoint between e4m3 neighbours must go to the even code.
    vals = oracle.e4m3_decode(np.arange(0x7e))
    mids = (vals[:-1] + vals[1:]) / 2
    bf = torch.tensor(mids).to(torch.bfloat16).double().numpy()
    ties = bf[bf == mids]
    x = np.zeros((1, 128, 1, 64), dtype=np.float32)
    x.reshape(-1)[:len(ties)] = ties
    x.reshape(-1)[-1] = 448.0
    x8, sc = _quant(gpu_lib, torch.from_numpy(x).to(torch.bfloat16), None)
    assert sc.item() == 1.0
    assert np.array_equal(x8.reshape(-1)[:len(ties)], oracle.e4m3_encode(ties))


def _fp8_run(fa, q, k, v, causal, signs, granularity=0, v_granularity=None):
    # The FP8 pipeline: Q and K with per-tile scales (block quantization),
    # V with one scale per head unless stated otherwise (v_granularity).
    dev = torch.device("cuda")
    s = None if signs is None else torch.from_numpy(signs).to(dev)
    if v_granularity is None:
        v_granularity = max(granularity, fa.FA_SCALE_HEAD)
    q8, qs = fa.quantize_fp8(q.to(dev), s, granularity=granularity)
    k8, ks = fa.quantize_fp8(k.to(dev), s, granularity=granularity)
    v8, vs = fa.quantize_fp8(v.to(dev), None, granularity=v_granularity)
    d = q.shape[-1]
    o, lse = fa.attention_fp8(q8, k8, v8, qs, ks, vs, causal=causal, alpha=synth.default_alpha(d))
    assert fa.fa_check_status() == fa.FA_OK
    return (o.float().cpu().numpy(), lse.cpu().numpy(),
            (q8.cpu().numpy(), qs.cpu().numpy(), k8.cpu().numpy(), ks.cpu().numpy(),
             v8.cpu().numpy(), vs.cpu().numpy()))


def _dequant(codes, scales):
    B, N, H, d = codes.shape
    vals = oracle.e4m3_decode(codes)
    rows = np.repeat(scales, 128, axis=2)[:, :, :N]          # [B, H, N]
    return vals * np.transpose(rows, (0, 2, 1))[:, :, :, None]


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_rmse_gate_and_rotation_helps(gpu_lib, causal, d):
    B, H, N = 1, 4, 1024
    q, k, v = synth.qkv(B, H, N, d, seed=synth.BASE_SEED + 5, outliers=True)
    a = synth.default_alpha(d)
    o_ref, lse_ref = oracle.attention(q, k, v, a, causal, n_threads=THREADS)
    o_rot, lse_rot, _ = _fp8_run(gpu_lib, q, k, v, causal, synth.hadamard_signs(d))
    o_plain, _, _ = _fp8_run(gpu_lib, q, k, v, causal, None)
    rmse_rot = float(np.sqrt(np.mean((o_rot - o_ref) ** 2)))
    rmse_plain = float(np.sqrt(np.mean((o_plain - o_ref) ** 2)))
    print(f"FP8 RMSE d={d} causal={causal}: rotated {rmse_rot:.3e}, unrotated {rmse_plain:.3e}")
    assert np.all(np.isfinite(o_rot))
    assert rmse_rot <= 1.5e-2
    assert rmse_rot < rmse_plain


@pytest.mark.parametrize("v_gran", ["tile", "head"])
@pytest.mark.parametrize("B,H,N,d,causal", [(1, 2, 300, 128, False), (1, 2, 300, 128, True),
                                             (2, 3, 1000, 128, True), (1, 1, 129, 128, False),
                                             (1, 2, 300, 256, False), (1, 2, 300, 256, True),
                                             (2, 3, 1000, 256, True), (1, 1, 129, 256, False),
                                             (1, 1, 1, 256, True), (3, 1, 640, 256, False)])
def test_fp8_kernel_against_dequantized_inputs(gpu_lib, B, H, N, d, causal, v_gran):
    # Per-tile V scales are folded into P' (any ratio v_j / v_max <= 1);
    # one V scale per head makes that ratio 1.
    q, k, v = synth.qkv(B, H, N, d, seed=N + 3, outliers=True)
    signs = synth.hadamard_signs(d, seed=N)
    vg = gpu_lib.FA_SCALE_TILE if v_gran == "tile" else gpu_lib.FA_SCALE_HEAD
    o, lse, (q8, qs, k8, ks, v8, vs) = _fp8_run(gpu_lib, q, k, v, causal, signs,
                                                v_granularity=vg)
    qd, kd, vd = _dequant(q8, qs), _dequant(k8, ks), _dequant(v8, vs)
    a = synth.default_alpha(d)
    o_deq, lse_deq = oracle.attention(qd, kd, vd, a, causal, n_threads=THREADS)
    ratio_min = (vs / vs.max(axis=2, keepdims=True)).min()
    for b in range(B):
        for h in range(H):
            vv = vd[b, :, h, :]
            od = o_deq[b, :, h, :]
            # max over keys j of |v_j - O_i| per column, without the [N, N, d] array
            spread = np.maximum(vv.max(axis=0)[None, :] - od, od - vv.min(axis=0)[None, :])
            c_off = 4                              # the kernel's exponent offset
            w = 2.0 ** -4 + N * 2.0 ** -10 / (ratio_min * 2.0 ** c_off)
            bound = w * spread + 2.0 ** -8 * np.abs(od) + 1e-3
            err = np.abs(o[b, :, h, :] - od)
            assert np.all(err <= bound), (err / bound).max()
    assert np.abs(lse - lse_deq).max() < 5e-2


@pytest.mark.parametrize("B,H,N,d,causal", [(4, 16, 4096, 128, False), (4, 16, 4096, 128, True),
                                             (4, 8, 4096, 256, False), (4, 8, 4096, 256, True),
                                             (1, 8, 16384, 256, False)])
def test_fp8_full_size_rmse_every_element(gpu_lib, B, H, N, d, causal):
    # Hidden 2048, 16k tokens, with outliers, in the bench's launch
    # configuration: RMSE over every O element against FP64 attention on
    # the unquantized inputs, the metric of the FA3 numerical-error
    # experiment.  d = 256, N = 16384 is the pages' FP8 headline point.
    q, k, v = synth.qkv(B, H, N, d, seed=synth.BASE_SEED, outliers=True)
    o, _, _ = _fp8_run(gpu_lib, q, k, v, causal, synth.hadamard_signs(d))
    a = synth.default_alpha(d)
    o_ref, _ = oracle.attention(q, k, v, a, causal, n_threads=THREADS)
    assert np.all(np.isfinite(o))
    rmse = float(np.sqrt(np.mean((o - o_ref) ** 2)))
    print(f"FP8 RMSE B{B} H{H} N{N} d{d} causal={causal} (all elements): {rmse:.3e}")
    assert rmse <= 1.5e-2


def test_fp8_ablation_block_scales_and_rotation(gpu_lib):
    # The FA3 numerical-error ablation (the FlashAttention-3 review on
    # diycv.top, "numerical error"): O RMSE against FP64 attention on the
    # unquantized outlier inputs for block scales (Q, K per 128-row tile, V
    # per head) vs one scale per tensor, each with and without the Hadamard
    # rotation, at B4 H16 N4096 d128.  The pages report 9.1e-3 (block +
    # rotation), 9.3e-3 (per tensor + rotation) and 2.4e-2 (no rotation).
    # Checked here: the rotation lowers the error at either granularity;
    # without the rotation block scales beat one scale per tensor; with it
    # the two agree within the pages' own 2.2 % gap (e4m3's precision is
    # relative, so once the rotation has spread the outliers the scale only
    # decides which values fall to subnormals).  A further arm keeps
    # per-tile V scales, whose fold into P' rounds the dominant terms of P'
    # (reported; it must still pass the 1.5e-2 gate).
    fa = gpu_lib
    B, H, N, d = 4, 16, 4096, 128
    q, k, v = synth.qkv(B, H, N, d, seed=synth.BASE_SEED, outliers=True)
    a = synth.default_alpha(d)
    o_ref, _ = oracle.attention(q, k, v, a, False, n_threads=THREADS)
    rm = {}
    for name, g in (("block", fa.FA_SCALE_TILE), ("tensor", fa.FA_SCALE_TENSOR)):
        for rot in (True, False):
            o, _, _ = _fp8_run(fa, q, k, v, False, synth.hadamard_signs(d) if rot else None, g)
            assert np.all(np.isfinite(o))
            rm[(name, rot)] = float(np.sqrt(np.mean((o - o_ref) ** 2)))
    o, _, _ = _fp8_run(fa, q, k, v, False, synth.hadamard_signs(d),
                       v_granularity=fa.FA_SCALE_TILE)
    rm_vtile = float(np.sqrt(np.mean((o - o_ref) ** 2)))
    print("FP8 ablation RMSE: " + ", ".join(
        f"{n}{'+rot' if r else ''} {x:.3e}" for (n, r), x in rm.items())
          + f"; block+rot with per-tile V scales {rm_vtile:.3e}")
    assert rm_vtile <= 1.5e-2
    assert rm[("block", True)] <= 1.5e-2
    assert rm[("block", True)] < rm[("block", False)]
    assert rm[("tensor", True)] < rm[("tensor", False)]
    assert rm[("block", False)] < rm[("tensor", False)]
    assert abs(rm[("block", True)] - rm[("tensor", True)]) <= 0.022 * rm[("tensor", True)]


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,H_kv", [(8, 2), (6, 1)])
def test_fp8_gqa_equals_expanded_heads_and_meets_the_gate(gpu_lib, d, causal, H, H_kv):
    # Grouped K/V heads (fa_fwd_fp8_gqa): query head h reads K/V head
    # h / (H / H_kv).  Repeating each K/V head's codes and scales for its
    # query heads and running fa_fwd_fp8 is the same arithmetic, so the bits
    # must agree; and the result meets the FP8 RMSE gate against FP64
    # grouped attention on the unquantized inputs.
    fa = gpu_lib
    dev = torch.device("cuda")
    B, N, g = 2, 700, H // H_kv
    q, k, v = synth.qkv(B, H, N, d, seed=N + d + H_kv, outliers=True)
    k, v = k[:, :, :H_kv].contiguous(), v[:, :, :H_kv].contiguous()
    s = torch.from_numpy(synth.hadamard_signs(d)).to(dev)
    q8, qs = fa.quantize_fp8(q.to(dev), s)
    k8, ks = fa.quantize_fp8(k.to(dev), s)
    v8, vs = fa.quantize_fp8(v.to(dev), None, granularity=fa.FA_SCALE_HEAD)
    a = synth.default_alpha(d)
    o_g, l_g = fa.attention_fp8(q8, k8, v8, qs, ks, vs, causal=causal, alpha=a)
    rep = lambda x, dim: x.repeat_interleave(g, dim=dim).contiguous()
    o_e, l_e = fa.attention_fp8(q8, rep(k8, 2), rep(v8, 2), qs, rep(ks, 1), rep(vs, 1),
                                causal=causal, alpha=a)
    assert fa.fa_check_status() == fa.FA_OK
    assert torch.equal(o_g, o_e) and torch.equal(l_g, l_e)
    o_ref, _ = oracle.attention_gqa(q, k, v, a, causal, n_threads=THREADS)
    rmse = float(np.sqrt(np.mean((o_g.float().cpu().numpy() - o_ref) ** 2)))
    assert rmse <= 1.5e-2, rmse


def test_fp8_gqa_rejects_bad_groups(gpu_lib):
    fa = gpu_lib
    x8 = torch.zeros((1, 128, 6, 128), dtype=torch.uint8, device="cuda")
    sc = torch.ones((1, 6, 1), dtype=torch.float32, device="cuda")
    o = torch.empty((1, 128, 6, 128), dtype=torch.bfloat16, device="cuda")
    for H_kv in (0, 4):
        assert fa.fa_fwd_fp8_gqa(x8, x8, x8, sc, sc, sc, o, None, 1, 6, H_kv, 128, 128, 0.1,
                                 0) == fa.FA_ERR_INVALID_ARG

