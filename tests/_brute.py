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
