"""50-digit decimal brute force of the attention definition, for pinning the
FP64 oracle on tiny inputs.  Independent of ``oracle/``: it shares no code
with it, only the definition ("FlashAttention-3 on Hopper", sec. 3.1 with
masks as -inf, sec. 4.6 for LSE and empty rows, sec. 4.7 for the
bottom-right causal predicate col > row + (Nk - Nq))."""
from __future__ import annotations

from decimal import Decimal, getcontext


def attention(q, k, v, alpha, causal):
    """q: Nq x d, k/v: Nk x d (nested lists of floats).  Returns (O, LSE)
    as nested lists of Decimal; an empty row gives zeros and LSE None."""
    getcontext().prec = 50
    Nq, Nk = len(q), len(k)
    d = len(q[0]) if Nq else 0
    a = Decimal(alpha)
    O, L = [], []
    for i in range(Nq):
        scores = {}
        for j in range(Nk):
            if causal and j > i + (Nk - Nq):
                continue
            dot = sum((Decimal(q[i][c]) * Decimal(k[j][c]) for c in range(d)),
                      Decimal(0))
            scores[j] = a * dot
        if not scores:
            O.append([Decimal(0)] * d)
            L.append(None)
            continue
        m = max(scores.values())
        w = {j: (s - m).exp() for j, s in scores.items()}
        tot = sum(w.values(), Decimal(0))
        O.append([sum((w[j] * Decimal(v[j][c]) for j in w), Decimal(0)) / tot
                  for c in range(len(v[0]))])
        L.append(m + tot.ln())
    return O, L


def _tanh(x):
    """tanh at the context's precision from exp: (e^2x - 1) / (e^2x + 1)."""
    if x < 0:
        return -_tanh(-x)
    e = (2 * x).exp()
    return (e - 1) / (e + 1)


def attention_ext(q, k, v, alpha, wl, wr, softcap, sink):
    """The variants ("FlashAttention-3 on Hopper", sec. 4.6 sinks, sec. 4.7
    local masks with the transform before the mask; "03 FA3" sec. 5
    softcap), with the bottom-right aligned diagonal i + (Nk - Nq): key j is
    hidden from query i when j > diag + wr (wr >= 0) or j < diag - wl
    (wl >= 0); a visible score s becomes c tanh(s / c) when softcap c > 0;
    the sink (None or a float) is one more logit in the denominator with no
    value.  Returns (O, LSE) as Decimals; a row with neither a visible key
    nor a sink gives zeros and LSE None."""
    getcontext().prec = 50
    Nq, Nk = len(q), len(k)
    d = len(q[0]) if Nq else 0
    a = Decimal(alpha)
    O, L = [], []
    for i in range(Nq):
        diag = i + (Nk - Nq)
        scores = {}
        for j in range(Nk):
            if wr >= 0 and j > diag + wr:
                continue
            if wl >= 0 and j < diag - wl:
                continue
            s = a * sum((Decimal(q[i][c]) * Decimal(k[j][c]) for c in range(d)),
                        Decimal(0))
            if softcap > 0:
                cc = Decimal(softcap)
                s = cc * _tanh(s / cc)
            scores[j] = s
        terms = list(scores.values()) + ([Decimal(sink)] if sink is not None else [])
        if not terms:
            O.append([Decimal(0)] * len(v[0]))
            L.append(None)
            continue
        m = max(terms)
        w = {j: (s - m).exp() for j, s in scores.items()}
        tot = sum(w.values(), Decimal(0))
        if sink is not None:
            tot += (Decimal(sink) - m).exp()
        O.append([sum((w[j] * Decimal(v[j][c]) for j in w), Decimal(0)) / tot
                  for c in range(len(v[0]))])
        L.append(m + tot.ln())
    return O, L
