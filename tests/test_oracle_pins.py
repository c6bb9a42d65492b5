"""Pins for the FP64 oracle: it is checked against things other than itself.

* 50-digit decimal brute force of the definition on tiny inputs (all masks,
  Nq != Nk bottom-right causal, empty rows);
* closed forms: identical keys (uniform softmax), causal row 0, one key;
* invariants: rows of P sum to 1, P = exp(S - LSE), shift of every key by a
  constant vector, joint permutation of keys and values;
* the tiled online recurrence with the conditional-rescale rule (random tile
  sizes, shuffled order, tau = 0 and tau = 8) equals the one-pass definition;
* Hadamard rotation against scipy's Hadamard matrix, orthogonality, and the
  invariance of attention under Q -> QM, K -> KM;
* e4m3 decode/encode against torch.float8_e4m3fn;
* block quantization: scale = amax / 448 and half-ulp reconstruction;
* a stored golden case (tests/golden) written by oracle-only script;
* planted mistakes (swapped or transposed operands, a wrong scale) fail the
  brute-force pin, so the pins are sensitive to them;
* gradients: central finite differences of L = sum(O * dO) through the
  forward definition, fp64 torch autograd through plain ops, the invariants
  sum_j dK_j = 0, D_i = dO_i . O_i and dV = P^T dO, and planted mistakes
  (swapped operands, a dropped scale, an ignored mask) that the
  finite-difference pin rejects.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from tests import _brute

RNG = np.random.default_rng(1234)


def _rand(*shape, scale=1.0):
    return (RNG.standard_normal(shape) * scale).astype(np.float32).astype(np.float64)


def _close_to_brute(o, lse, bo, bl, tol=1e-13):
    for i in range(len(bo)):
        if bl[i] is None:
            assert lse[i] == -math.inf
            assert np.all(o[i] == 0.0)
            continue
        assert abs(lse[i] - float(bl[i])) <= tol * max(1.0, abs(float(bl[i])))
        for c in range(len(bo[i])):
            assert abs(o[i][c] - float(bo[i][c])) <= tol * max(1.0, abs(float(bo[i][c])))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk,d", [(1, 1, 1), (3, 3, 2), (5, 5, 4), (8, 8, 3),
                                     (4, 7, 2), (7, 4, 4), (6, 2, 3)])
def test_brute_force_tiny(nq, nk, d, causal):
    q, k, v = _rand(nq, d), _rand(nk, d), _rand(nk, d)
    alpha = float(np.float32(RNG.uniform(0.2, 1.5)))
    o, lse = oracle.attention_head(q, k, v, alpha, causal)
    bo, bl = _brute.attention(q.tolist(), k.tolist(), v.tolist(), alpha, causal)
    _close_to_brute(o, lse, bo, bl)


def test_brute_force_empty_rows_exist():
    # Nq > Nk with bottom-right causal alignment hides every key from the
    # first Nq - Nk rows: O = 0, LSE = -inf.
    q, k, v = _rand(6, 3), _rand(2, 3), _rand(2, 3)
    o, lse = oracle.attention_head(q, k, v, 0.7, True)
    assert np.all(np.isneginf(lse[:4])) and np.all(np.isfinite(lse[4:]))
    assert np.all(o[:4] == 0.0)
    bo, bl = _brute.attention(q.tolist(), k.tolist(), v.tolist(), 0.7, True)
    _close_to_brute(o, lse, bo, bl)


def test_batched_matches_per_head():
    B, N, H, d = 2, 9, 3, 4
    q, k, v = _rand(B, N, H, d), _rand(B, N, H, d), _rand(B, N, H, d)
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, 0.5, causal, n_threads=3)
        for b in range(B):
            for h in range(H):
                oh, lh = oracle.attention_head(q[b, :, h], k[b, :, h], v[b, :, h], 0.5, causal)
                assert np.array_equal(o[b, :, h], oh)
                assert np.array_equal(lse[b, h], lh)
                rows = [8, 0, 3]
                orr, lr = oracle.attention_rows(q, k, v, 0.5, causal, b, h, rows)
                assert np.array_equal(orr, oh[rows]) and np.array_equal(lr, lh[rows])


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_and_lse_identity(causal):
    N, d = 40, 16
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    alpha = 0.25
    o, lse, p = oracle.attention_head(q, k, v, alpha, causal, want_probs=True)
    assert np.allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    s = alpha * (q @ k.T)
    if causal:
        s = np.where(np.triu(np.ones((N, N), bool), 1), -np.inf, s)
        assert np.all(p[np.triu(np.ones((N, N), bool), 1)] == 0.0)
    # Backward-recompute identity: P_ij = exp(S_ij - LSE_i).
    assert np.allclose(p, np.exp(s - lse[:, None]), rtol=1e-13, atol=0)
    # O = P V
    assert np.allclose(o, p @ v, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_closed_form(causal):
    N, d = 37, 8
    q, v = _rand(N, d), _rand(N, d)
    krow = _rand(d)
    k = np.tile(krow, (N, 1))
    alpha = 0.3
    o, lse = oracle.attention_head(q, k, v, alpha, causal)
    for i in range(N):
        vis = i + 1 if causal else N
        assert np.allclose(o[i], v[:vis].mean(axis=0), rtol=1e-13, atol=1e-15)
        expect = alpha * float(q[i] @ krow) + math.log(vis)
        assert abs(lse[i] - expect) <= 1e-13 * max(1.0, abs(expect))


def test_causal_row_zero_and_single_key():
    N, d = 20, 5
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    o, lse = oracle.attention_head(q, k, v, 0.9, True)
    assert np.array_equal(o[0], v[0])
    assert lse[0] == pytest.approx(0.9 * float(q[0] @ k[0]), rel=1e-15, abs=1e-15)
    o1, l1 = oracle.attention_head(q[:3], k[:1], v[:1], 0.9, False)
    assert np.array_equal(o1, np.tile(v[0], (3, 1)))
    assert np.allclose(l1, 0.9 * (q[:3] @ k[0]), rtol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tau", [0.0, 8.0])
def test_online_tiled_equals_one_pass(causal, tau):
    N, d = 150, 12
    # Large score spread so that the reference point has to move often.
    q, k, v = _rand(N, d, scale=3.0), _rand(N, d, scale=3.0), _rand(N, d)
    alpha = 0.4
    cuts = sorted(set(RNG.integers(1, N, size=9).tolist()))
    bounds = [0] + cuts + [N]
    tiles = [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]
    tiles.append((5, 5))                      # an empty tile is harmless
    order = RNG.permutation(len(tiles))
    tiles = [tiles[i] for i in order]
    o1, l1 = oracle.attention_head(q, k, v, alpha, causal)
    o2, l2, moves = oracle.attention_online(q, k, v, alpha, causal, tiles, tau)
    assert np.allclose(o2, o1, rtol=1e-12, atol=1e-14)
    assert np.allclose(l2, l1, rtol=1e-12, atol=1e-14)
    if tau == 0.0:
        assert moves > 0
    else:
        _, _, moves0 = oracle.attention_online(q, k, v, alpha, causal, tiles, 0.0)
        assert moves < moves0                 # the threshold skips rescales


def test_online_descending_tiles_of_128():
    # The kernel's own visiting order: 128-key tiles, last (ragged) tile first.
    N, d = 1000, 16
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    tiles = [(j * 128, min(N, j * 128 + 128)) for j in range((N + 127) // 128)][::-1]
    for causal in (False, True):
        o1, l1 = oracle.attention_head(q, k, v, 0.25, causal)
        o2, l2, _ = oracle.attention_online(q, k, v, 0.25, causal, tiles, 8.0)
        assert np.allclose(o2, o1, rtol=1e-12, atol=1e-14)
        assert np.allclose(l2, l1, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    N, d = 33, 6
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    c = _rand(d)
    alpha = 0.5
    o1, l1 = oracle.attention_head(q, k, v, alpha, causal)
    o2, l2 = oracle.attention_head(q, k + c, v, alpha, causal)
    assert np.allclose(o2, o1, rtol=1e-12, atol=1e-14)
    assert np.allclose(l2, l1 + alpha * (q @ c), rtol=1e-12, atol=1e-13)


def test_key_value_permutation_invariance():
    N, d = 29, 7
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    perm = RNG.permutation(N)
    o1, l1 = oracle.attention_head(q, k, v, 0.6, False)
    o2, l2 = oracle.attention_head(q, k[perm], v[perm], 0.6, False)
    assert np.allclose(o2, o1, rtol=1e-12, atol=1e-14)
    assert np.allclose(l2, l1, rtol=1e-13)


@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_hadamard_rotation_matches_scipy_and_is_orthogonal(d):
    signs = np.where(RNG.random(d) < 0.5, -1.0, 1.0)
    x = _rand(5, d)
    y = oracle.hadamard_rotate(x, signs)
    M = scipy.linalg.hadamard(d).astype(np.float64) * signs[None, :] / math.sqrt(d)
    assert np.allclose(y, x @ M, rtol=1e-13, atol=1e-13)
    Mo = oracle.hadamard_rotate(np.eye(d), signs)
    assert np.allclose(Mo @ Mo.T, np.eye(d), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_invariant_under_rotation(causal):
    N, d = 50, 32
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    signs = np.where(RNG.random(d) < 0.5, -1.0, 1.0)
    o1, l1 = oracle.attention_head(q, k, v, 0.2, causal)
    o2, l2 = oracle.attention_head(oracle.hadamard_rotate(q, signs),
                                   oracle.hadamard_rotate(k, signs), v, 0.2, causal)
    assert np.allclose(o2, o1, rtol=1e-11, atol=1e-13)
    assert np.allclose(l2, l1, rtol=1e-12, atol=1e-13)


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7e] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_round_to_nearest_even():
    vals = np.concatenate([
        RNG.standard_normal(4000) * 30.0,
        RNG.standard_normal(1000) * 0.01,
        oracle.e4m3_decode(np.arange(0x7e)),                     # exact codes
        (oracle.e4m3_decode(np.arange(0x7d)) + oracle.e4m3_decode(np.arange(1, 0x7e))) / 2,  # ties
        [0.0, 447.9, 448.0, 463.9, -463.9]])
    vals = vals.astype(np.float32).astype(np.float64)     # torch casts from float32
    ours = oracle.e4m3_encode(vals)
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    # Beyond the largest finite value we saturate (torch would give NaN).
    assert oracle.e4m3_encode(np.array([1e6, -500.0])).tolist() == [0x7e, 0xfe]


def test_block_quantization_scale_and_reconstruction():
    x = _rand(300, 16)
    x[130:140, 3] *= 40.0                      # an outlier cluster in tile 1
    x[256:, :] = 0.0                           # an all-zero last tile
    codes, scales = oracle.quantize_e4m3_tiles(x, 128)
    assert scales.shape == (3,)
    for t in range(2):
        amax = np.abs(x[t * 128:(t + 1) * 128]).max()
        assert scales[t] == np.float32(amax / 448.0)
    assert scales[2] == 1.0 and np.all(codes[256:] == 0)
    rec = oracle.e4m3_decode(codes) * np.repeat(scales.astype(np.float64), 128)[:300, None]
    # e4m3 has 3 mantissa bits: relative half-ulp 2^-4 for normals, and an
    # absolute half-ulp of 2^-10 * scale in the subnormal range.
    err = np.abs(rec - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4,
                       2.0 ** -10 * np.repeat(scales.astype(np.float64), 128)[:300, None])
    assert np.all(err <= bound * (1 + 1e-12))
    assert np.abs(oracle.e4m3_decode(codes[:256])).max() <= 448.0


def test_golden_fixture():
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_attention.json")
    with open(path) as f:
        g = json.load(f)
    for case in g["cases"]:
        q, k, v = (np.array(case[n], dtype=np.float64) for n in ("q", "k", "v"))
        o, lse = oracle.attention_head(q, k, v, case["alpha"], case["causal"])
        assert np.allclose(o, np.array(case["o"]), rtol=1e-14, atol=1e-15)
        assert np.allclose(lse, np.array(case["lse"]), rtol=1e-14, atol=1e-15)


def _brute_fails(q, k, v, alpha, causal, o, lse):
    bo, bl = _brute.attention(q.tolist(), k.tolist(), v.tolist(), alpha, causal)
    try:
        _close_to_brute(o, lse, bo, bl)
    except AssertionError:
        return True
    return False


def test_planted_mistakes_are_caught():
    N, d = 6, 3
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    a = 0.8
    # swapped K and V operands
    o, l = oracle.attention_head(q, v, k, a, False)
    assert _brute_fails(q, k, v, a, False, o, l)
    # transposed (Q and K exchanged)
    o, l = oracle.attention_head(k, q, v, a, False)
    assert _brute_fails(q, k, v, a, False, o, l)
    # missing scale (alpha dropped)
    o, l = oracle.attention_head(q, k, v, 1.0, False)
    assert _brute_fails(q, k, v, a, False, o, l)
    # wrong mask direction
    o, l = oracle.attention_head(q[::-1].copy(), k[::-1].copy(), v[::-1].copy(), a, True)
    assert _brute_fails(q, k, v, a, True, o[::-1], l[::-1])
    # sign error in the scores
    o, l = oracle.attention_head(-q, k, v, a, False)
    assert _brute_fails(q, k, v, a, False, o, l)


# ---------------------------------------------------------------------------
# Gradients ("FlashAttention-3 on Hopper", sec. 7.1)
# ---------------------------------------------------------------------------

def _loss(q, k, v, dout, a, causal):
    """L = sum(O * dO), whose gradients are the ones the backward returns."""
    o, _ = oracle.attention_head(q, k, v, a, causal)
    return float(np.sum(o * dout))


def _fd_grads(q, k, v, dout, a, causal, eps=1e-5):
    """Central finite differences of L with respect to every input element."""
    out = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(args[which])
        for idx in np.ndindex(g.shape):
            x0 = args[which][idx]
            args[which][idx] = x0 + eps
            lp = _loss(*args, dout, a, causal)
            args[which][idx] = x0 - eps
            lm = _loss(*args, dout, a, causal)
            args[which][idx] = x0
            g[idx] = (lp - lm) / (2 * eps)
        out.append(g)
    return out


def _fd_agrees(grads, fd, tol=1e-7):
    return all(np.allclose(g, f, rtol=tol, atol=tol) for g, f in zip(grads, fd))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk,d", [(1, 1, 1), (3, 3, 2), (5, 5, 3), (4, 6, 2), (6, 3, 3)])
def test_bwd_matches_finite_differences(nq, nk, d, causal):
    q, k, v, dout = _rand(nq, d), _rand(nk, d), _rand(nk, d), _rand(nq, d)
    a = 0.9
    grads = oracle.attention_bwd_head(q, k, v, dout, a, causal)
    assert _fd_agrees(grads, _fd_grads(q, k, v, dout, a, causal))


def _torch_grads(q, k, v, dout, a, causal):
    """The same gradients by fp64 autograd through plain torch ops."""
    t = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v)]
    s = a * t[0] @ t[1].T
    if causal:
        nq, nk = s.shape
        i = torch.arange(nq)[:, None]
        j = torch.arange(nk)[None, :]
        s = s.masked_fill(j > i + (nk - nq), float("-inf"))
    o = torch.softmax(s, dim=-1) @ t[2]
    o.backward(torch.tensor(dout, dtype=torch.float64))
    return [x.grad.numpy() for x in t]


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_matches_torch_autograd(causal):
    B, H, N, d = 1, 2, 37, 8
    q, k, v, dout = (_rand(B, N, H, d) for _ in range(4))
    a = 0.35
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, a, causal, n_threads=2)
    for h in range(H):
        ref = _torch_grads(q[0, :, h], k[0, :, h], v[0, :, h], dout[0, :, h], a, causal)
        for got, want in zip((dq[0, :, h], dk[0, :, h], dv[0, :, h]), ref):
            assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_invariants(causal):
    # Each row of dS sums to zero, so the key gradients sum to zero; and
    # D_i = <P_i, dP_i> equals dO_i . O_i (sec. 7.1.2), which the GPU uses.
    N, d = 29, 6
    q, k, v, dout = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
    a = 0.6
    dq, dk, dv = oracle.attention_bwd_head(q, k, v, dout, a, causal)
    assert np.abs(dk.sum(axis=0)).max() <= 1e-12
    o, _, p = oracle.attention_head(q, k, v, a, causal, want_probs=True)
    d_from_p = np.sum(p * (dout @ v.T), axis=1)
    assert np.allclose(np.sum(dout * o, axis=1), d_from_p, rtol=1e-12, atol=1e-12)
    # dV is linear in dO with the probabilities as weights: dV = P^T dO
    assert np.allclose(dv, p.T @ dout, rtol=1e-12, atol=1e-12)


def test_bwd_planted_mistakes_are_caught():
    N, d = 5, 3
    q, k, v, dout = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
    a = 0.8
    fd = _fd_grads(q, k, v, dout, a, True)
    assert _fd_agrees(oracle.attention_bwd_head(q, k, v, dout, a, True), fd)
    # swapped K and V
    assert not _fd_agrees(oracle.attention_bwd_head(q, v, k, dout, a, True), fd)
    # dO and V exchanged (dP built from the wrong operand)
    assert not _fd_agrees(oracle.attention_bwd_head(q, k, dout, v, a, True), fd)
    # scale dropped
    assert not _fd_agrees(oracle.attention_bwd_head(q, k, v, dout, 1.0, True), fd)
    # mask ignored
    assert not _fd_agrees(oracle.attention_bwd_head(q, k, v, dout, a, False), fd)


# ---------------------------------------------------------------------------
# Grouped key/value heads ("FlashAttention-3 on Hopper", ch. 11)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 2), (6, 3), (4, 1)])
def test_gqa_maps_query_head_to_its_kv_head(H, H_kv):
    # Each query head h must attend with key/value head h // (H // H_kv):
    # checked head by head against the one-head definition (a mapping by
    # h % H_kv, or a shared head for all, fails this).
    B, N, d = 2, 9, 3
    q = _rand(B, N, H, d)
    k, v = _rand(B, N, H_kv, d), _rand(B, N, H_kv, d)
    a = 0.7
    for causal in (False, True):
        o, lse = oracle.attention_gqa(q, k, v, a, causal)
        g = H // H_kv
        for b in range(B):
            for h in range(H):
                oh, lh = oracle.attention_head(q[b, :, h], k[b, :, h // g], v[b, :, h // g],
                                               a, causal)
                assert np.array_equal(o[b, :, h], oh) and np.array_equal(lse[b, h], lh)
    with pytest.raises(ValueError):
        oracle.attention_gqa(q, _rand(B, N, H + 1, d), _rand(B, N, H + 1, d), a, False)
