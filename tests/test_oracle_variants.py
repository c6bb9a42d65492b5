"""Pins for the oracle's score and mask variants (local windows, softcap,
sinks): "FlashAttention-3 on Hopper" sec. 4.6 (learnable sinks folded into
the row sum) and sec. 4.7 (local attention's left boundary; a score
transformation precedes the mask); "03 FA3" sec. 5 (softcap c tanh(s / c)).

The variant oracle is checked against things other than itself:

* the 50-digit decimal brute force of tests/_brute.py on tiny inputs, over
  windows, softcaps, sinks and Nq != Nk (bottom-right diagonal);
* reductions to the plain, already pinned definition: (-1, 0) is causal,
  (-1, -1) is no mask, and a window row equals plain attention over the
  sliced key range;
* closed forms: all-zero queries with a sink, identical keys under softcap;
* limits: a sink at -800 is no sink, a softcap of 1e8 is no softcap, and a
  softcapped LSE lies within [-c, c] + log(visible keys);
* masked keys and values do not influence the result at all;
* planted mistakes (window off by one, swapped window sides, wrong softcap,
  the sink of another head) fail the brute-force pin;
* gradients (dQ, dK, dV and the sink logit's): central finite differences
  of L = sum(O * dO) through the variant forward, the plain gradient oracle
  for (-1, 0) and (-1, -1), and planted mistakes (softcap factor, window,
  sink dropped or changed) that the finite-difference pin rejects.
"""
import math

import numpy as np
import pytest

import oracle
from tests import _brute

RNG = np.random.default_rng(4321)


def _rand(*shape, scale=1.0):
    return (RNG.standard_normal(shape) * scale).astype(np.float32).astype(np.float64)


def _agree(o, lse, bo, bl, tol=1e-13):
    for i in range(len(bo)):
        if bl[i] is None:
            if not (lse[i] == -math.inf and np.all(o[i] == 0.0)):
                return False
            continue
        if abs(lse[i] - float(bl[i])) > tol * max(1.0, abs(float(bl[i]))):
            return False
        for c in range(len(bo[i])):
            if abs(o[i][c] - float(bo[i][c])) > tol * max(1.0, abs(float(bo[i][c]))):
                return False
    return True


WINDOWS = [(-1, -1), (-1, 0), (0, 0), (1, 2), (2, -1), (0, -1), (3, 1), (-1, 2)]
SOFTCAPS = [0.0, 0.7, 5.0]
SINKS = [None, 0.3, -1.0, 4.0]


@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("nq,nk,d", [(1, 1, 1), (5, 5, 3), (8, 8, 2), (4, 7, 2), (7, 4, 3)])
def test_brute_force_windows(nq, nk, d, window):
    q, k, v = _rand(nq, d), _rand(nk, d), _rand(nk, d)
    alpha = float(np.float32(RNG.uniform(0.3, 1.4)))
    for softcap, sink in [(0.0, None), (0.7, None), (0.0, 0.3), (5.0, -1.0)]:
        o, lse = oracle.attention_ext_head(q, k, v, alpha, window, softcap, sink)
        bo, bl = _brute.attention_ext(q.tolist(), k.tolist(), v.tolist(), alpha,
                                      window[0], window[1], softcap, sink)
        assert _agree(o, lse, bo, bl), (window, softcap, sink)


@pytest.mark.parametrize("softcap", SOFTCAPS)
@pytest.mark.parametrize("sink", SINKS)
def test_brute_force_softcap_and_sinks(softcap, sink):
    nq, nk, d = 6, 6, 4
    q, k, v = _rand(nq, d, scale=2.0), _rand(nk, d), _rand(nk, d)
    o, lse = oracle.attention_ext_head(q, k, v, 0.9, (2, 0), softcap, sink)
    bo, bl = _brute.attention_ext(q.tolist(), k.tolist(), v.tolist(), 0.9, 2, 0,
                                  softcap, sink)
    assert _agree(o, lse, bo, bl)


def test_rows_without_keys_with_and_without_sink():
    # Nq > Nk with a right bound: the first rows see no key.
    q, k, v = _rand(6, 3), _rand(2, 3), _rand(2, 3)
    o, lse = oracle.attention_ext_head(q, k, v, 0.7, (-1, 0))
    assert np.all(np.isneginf(lse[:4])) and np.all(o[:4] == 0.0)
    o, lse = oracle.attention_ext_head(q, k, v, 0.7, (-1, 0), 0.0, 1.25)
    assert np.all(lse[:4] == 1.25) and np.all(o[:4] == 0.0)
    bo, bl = _brute.attention_ext(q.tolist(), k.tolist(), v.tolist(), 0.7, -1, 0, 0.0, 1.25)
    assert _agree(o, lse, bo, bl)


@pytest.mark.parametrize("causal", [False, True])
def test_reduces_to_plain_definition(causal):
    B, N, H, d = 2, 23, 3, 8
    q, k, v = _rand(B, N, H, d), _rand(B, N, H, d), _rand(B, N, H, d)
    o, lse = oracle.attention(q, k, v, 0.4, causal)
    oe, le = oracle.attention_ext(q, k, v, 0.4, window=(-1, 0) if causal else (-1, -1))
    assert np.allclose(oe, o, rtol=1e-13, atol=1e-15)
    assert np.allclose(le, lse, rtol=1e-14, atol=0)


@pytest.mark.parametrize("window", [(5, 0), (0, 4), (7, 3), (-1, 2), (3, -1)])
def test_window_row_is_attention_over_the_slice(window):
    N, d = 31, 6
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    wl, wr = window
    o, lse = oracle.attention_ext_head(q, k, v, 0.6, window, 0.0, None)
    for i in range(N):
        lo = 0 if wl < 0 else max(0, i - wl)
        hi = N if wr < 0 else min(N, i + wr + 1)
        os_, ls = oracle.attention_head(q[i:i + 1], k[lo:hi], v[lo:hi], 0.6, False)
        assert np.allclose(o[i], os_[0], rtol=1e-13, atol=1e-15)
        assert abs(lse[i] - ls[0]) <= 1e-13 * max(1.0, abs(ls[0]))


def test_masked_keys_do_not_matter():
    N, d = 20, 5
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    window = (3, 1)
    o, lse = oracle.attention_ext_head(q, k, v, 0.8, window, 2.0, 0.5)
    for i in range(N):
        hidden = [j for j in range(N) if j > i + 1 or j < i - 3]
        if not hidden:
            continue
        k2, v2 = k.copy(), v.copy()
        k2[hidden] = _rand(len(hidden), d, scale=50.0)
        v2[hidden] = _rand(len(hidden), d, scale=50.0)
        o2, l2 = oracle.attention_ext_head(q, k2, v2, 0.8, window, 2.0, 0.5, rows=[i])
        assert np.array_equal(o2[0], o[i]) and l2[0] == lse[i]


@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (2, 1)])
def test_sink_closed_form_with_zero_queries(window):
    # q = 0: every visible score is 0 (also after softcap), so with n visible
    # keys O = sum(v) / (n + e^sigma) and LSE = log(n + e^sigma).
    N, d, sigma = 9, 4, 1.7
    q, k, v = np.zeros((N, d)), _rand(N, d), _rand(N, d)
    wl, wr = window
    for softcap in (0.0, 3.0):
        o, lse = oracle.attention_ext_head(q, k, v, 0.5, window, softcap, sigma)
        for i in range(N):
            vis = [j for j in range(N)
                   if not ((wr >= 0 and j > i + wr) or (wl >= 0 and j < i - wl))]
            den = len(vis) + math.exp(sigma)
            assert np.allclose(o[i], v[vis].sum(axis=0) / den, rtol=1e-13, atol=1e-15)
            assert abs(lse[i] - math.log(den)) <= 1e-14 * max(1.0, math.log(den))


def test_softcap_identical_keys_closed_form():
    # Identical keys: every visible score is the same value t, so P is uniform
    # and LSE = t + log(n) with t = c tanh(alpha q.k / c).
    N, d, c, alpha = 15, 6, 2.5, 0.9
    q, v = _rand(N, d, scale=3.0), _rand(N, d)
    krow = _rand(d)
    k = np.tile(krow, (N, 1))
    o, lse = oracle.attention_ext_head(q, k, v, alpha, (4, 0), c, None)
    for i in range(N):
        lo = max(0, i - 4)
        n = i + 1 - lo
        t = c * np.tanh(alpha * float(q[i] @ krow) / c)
        assert np.allclose(o[i], v[lo:i + 1].mean(axis=0), rtol=1e-13, atol=1e-15)
        assert abs(lse[i] - (t + math.log(n))) <= 1e-13 * max(1.0, abs(lse[i]))


def test_limits_sink_and_softcap():
    N, d = 17, 8
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    o0, l0 = oracle.attention_ext_head(q, k, v, 0.5, (6, 2), 0.0, None)
    o1, l1 = oracle.attention_ext_head(q, k, v, 0.5, (6, 2), 0.0, -800.0)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    o2, l2 = oracle.attention_ext_head(q, k, v, 0.5, (6, 2), 1e8, None)
    assert np.allclose(o2, o0, rtol=1e-12, atol=1e-14)
    assert np.allclose(l2, l0, rtol=1e-12, atol=1e-14)
    # large scores: the softcapped scores lie in [-c, c]
    c = 1.5
    o3, l3 = oracle.attention_ext_head(q * 40, k, v, 0.5, (-1, -1), c, None)
    assert np.all(l3 <= c + math.log(N) + 1e-12)
    assert np.all(l3 >= -c + math.log(N) - 1e-12)


def test_whole_tensor_matches_heads_with_grouping_and_sinks():
    B, N, H, H_kv, d = 2, 13, 4, 2, 4
    q = _rand(B, N, H, d)
    k, v = _rand(B, N, H_kv, d), _rand(B, N, H_kv, d)
    sinks = _rand(H)
    o, lse = oracle.attention_ext(q, k, v, 0.7, window=(3, 2), softcap=1.5,
                                  sinks=sinks, n_threads=3)
    for b in range(B):
        for h in range(H):
            hk = h // (H // H_kv)
            oh, lh = oracle.attention_ext_head(q[b, :, h], k[b, :, hk], v[b, :, hk], 0.7,
                                               (3, 2), 1.5, float(sinks[h]))
            assert np.array_equal(o[b, :, h], oh) and np.array_equal(lse[b, h], lh)
            orr, lr = oracle.attention_ext_rows(q, k, v, 0.7, b, h, [12, 0, 5],
                                                (3, 2), 1.5, sinks)
            assert np.array_equal(orr, oh[[12, 0, 5]]) and np.array_equal(lr, lh[[12, 0, 5]])


def test_invalid_arguments():
    q = _rand(3, 2)
    with pytest.raises(RuntimeError):
        oracle.attention_ext_head(q, q, q, 1.0, (-2, 0))
    with pytest.raises(RuntimeError):
        oracle.attention_ext_head(q, q, q, 1.0, (0, 0), -1.0)


def test_planted_mistakes_are_caught():
    N, d = 7, 3
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    a, win, c, sink = 0.8, (2, 1), 1.3, 0.4

    def fails(o, lse):
        bo, bl = _brute.attention_ext(q.tolist(), k.tolist(), v.tolist(), a,
                                      win[0], win[1], c, sink)
        return not _agree(o, lse, bo, bl)

    assert not fails(*oracle.attention_ext_head(q, k, v, a, win, c, sink))
    assert fails(*oracle.attention_ext_head(q, k, v, a, (3, 1), c, sink))    # left off by one
    assert fails(*oracle.attention_ext_head(q, k, v, a, (2, 2), c, sink))    # right off by one
    assert fails(*oracle.attention_ext_head(q, k, v, a, (1, 2), c, sink))    # sides swapped
    assert fails(*oracle.attention_ext_head(q, k, v, a, win, c * 1.1, sink))  # softcap value
    assert fails(*oracle.attention_ext_head(q, k, v, a, win, 0.0, sink))     # softcap dropped
    assert fails(*oracle.attention_ext_head(q, k, v, a, win, c, -0.4))       # another sink
    assert fails(*oracle.attention_ext_head(q, k, v, a, win, c, None))       # sink dropped
    assert fails(*oracle.attention_ext_head(q, k, v, 1.0, win, c, sink))     # alpha dropped


# ---------------------------------------------------------------------------
# Gradients of the variants ("FlashAttention-3 on Hopper", sec. 7.1)
# ---------------------------------------------------------------------------

def _ext_loss(q, k, v, dout, a, window, softcap, sink):
    o, _ = oracle.attention_ext_head(q, k, v, a, window, softcap, sink)
    return float(np.sum(o * dout))


def _ext_fd(q, k, v, dout, a, window, softcap, sink, eps=1e-5):
    grads = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(args[which])
        for idx in np.ndindex(g.shape):
            x0 = args[which][idx]
            args[which][idx] = x0 + eps
            lp = _ext_loss(*args, dout, a, window, softcap, sink)
            args[which][idx] = x0 - eps
            lm = _ext_loss(*args, dout, a, window, softcap, sink)
            args[which][idx] = x0
            g[idx] = (lp - lm) / (2 * eps)
        grads.append(g)
    if sink is None:
        grads.append(0.0)
    else:
        lp = _ext_loss(q, k, v, dout, a, window, softcap, sink + eps)
        lm = _ext_loss(q, k, v, dout, a, window, softcap, sink - eps)
        grads.append((lp - lm) / (2 * eps))
    return grads


def _grads_agree(g, fd, tol=1e-7):
    return (all(np.allclose(x, y, rtol=tol, atol=tol) for x, y in zip(g[:3], fd[:3]))
            and abs(g[3] - fd[3]) <= tol * max(1.0, abs(fd[3])))


@pytest.mark.parametrize("window,softcap,sink", [
    ((-1, -1), 0.0, None), ((-1, 0), 0.0, None), ((1, 0), 0.0, None), ((2, 1), 0.0, 0.4),
    ((-1, -1), 1.5, None), ((1, 2), 0.8, -0.3), ((-1, 0), 2.0, 1.2), ((0, 0), 0.0, 0.7)])
@pytest.mark.parametrize("nq,nk,d", [(5, 5, 3), (4, 6, 2)])
def test_bwd_ext_matches_finite_differences(nq, nk, d, window, softcap, sink):
    q, k, v, dout = _rand(nq, d), _rand(nk, d), _rand(nk, d), _rand(nq, d)
    a = 0.9
    g = oracle.attention_bwd_ext_head(q, k, v, dout, a, window, softcap, sink)
    assert _grads_agree(g, _ext_fd(q, k, v, dout, a, window, softcap, sink))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_ext_reduces_to_plain_gradients(causal):
    N, d = 9, 4
    q, k, v, dout = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
    g = oracle.attention_bwd_ext_head(q, k, v, dout, 0.6, (-1, 0) if causal else (-1, -1))
    ref = oracle.attention_bwd_head(q, k, v, dout, 0.6, causal)
    for x, y in zip(g[:3], ref):
        assert np.allclose(x, y, rtol=1e-13, atol=1e-15)
    assert g[3] == 0.0


def test_bwd_ext_whole_tensor_matches_heads():
    B, N, H, d = 2, 7, 3, 4
    q, k, v, dout = (_rand(B, N, H, d) for _ in range(4))
    sinks = _rand(H)
    dq, dk, dv, ds = oracle.attention_bwd_ext(q, k, v, dout, 0.5, (2, 0), 1.5, sinks, n_threads=3)
    tot = np.zeros(H)
    for b in range(B):
        for h in range(H):
            g = oracle.attention_bwd_ext_head(q[b, :, h], k[b, :, h], v[b, :, h], dout[b, :, h],
                                              0.5, (2, 0), 1.5, float(sinks[h]))
            assert np.array_equal(dq[b, :, h], g[0]) and np.array_equal(dk[b, :, h], g[1])
            assert np.array_equal(dv[b, :, h], g[2])
            tot[h] += g[3]
    assert np.allclose(ds, tot, rtol=1e-15, atol=0)


def test_bwd_ext_planted_mistakes_are_caught():
    N, d = 6, 3
    q, k, v, dout = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
    a, win, c, sink = 0.8, (2, 1), 1.3, 0.5
    fd = _ext_fd(q, k, v, dout, a, win, c, sink)
    assert _grads_agree(oracle.attention_bwd_ext_head(q, k, v, dout, a, win, c, sink), fd)
    assert not _grads_agree(oracle.attention_bwd_ext_head(q, k, v, dout, a, win, 0.0, sink), fd)
    assert not _grads_agree(oracle.attention_bwd_ext_head(q, k, v, dout, a, (3, 1), c, sink), fd)
    assert not _grads_agree(oracle.attention_bwd_ext_head(q, k, v, dout, a, win, c, None), fd)
    assert not _grads_agree(oracle.attention_bwd_ext_head(q, k, v, dout, a, win, c, -0.5), fd)


def test_bwd_ext_grouped_heads_match_finite_differences():
    # Grouped K/V heads: the gradient of a shared K/V head is the sum over
    # its query heads; checked by differentiating the grouped forward.
    B, N, H, H_kv, d = 1, 4, 4, 2, 2
    q, dout = _rand(B, N, H, d), _rand(B, N, H, d)
    k, v = _rand(B, N, H_kv, d), _rand(B, N, H_kv, d)
    a, win, c = 0.7, (2, 0), 1.5

    def loss(kk, vv):
        o, _ = oracle.attention_ext(q, kk, vv, a, window=win, softcap=c)
        return float(np.sum(o * dout))

    _, dk, dv, _ = oracle.attention_bwd_ext(q, k, v, dout, a, win, c, None)
    assert dk.shape == k.shape and dv.shape == v.shape
    eps = 1e-5
    for x, g in ((k, dk), (v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + eps
            lp = loss(k, v)
            x[idx] = x0 - eps
            lm = loss(k, v)
            x[idx] = x0
            fd[idx] = (lp - lm) / (2 * eps)
        assert np.allclose(g, fd, rtol=1e-7, atol=1e-7)
