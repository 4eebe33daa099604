"""Pure-Python dense attention brute force -- TEST INFRASTRUCTURE.

softmax(q K^T * scale) V for one query over contiguous K/V, in Python floats
(IEEE double) with nothing but loops and math.exp.  It knows nothing about
pages, blocks or tables, so agreement with the paged oracle on small inputs
pins the paging (the "Decode-only block-table attention" item of the ForgeLLM
README's feature list promises exactly the dense result without building
padded K/V).  Use only on small inputs.
"""
from __future__ import annotations

import math
from typing import List, Sequence


def attention(q: Sequence[float], K: Sequence[Sequence[float]], V: Sequence[Sequence[float]],
              scale: float) -> List[float]:
    """One query row q[D]; K, V are [L][D]; returns the [D] output (zeros when L == 0)."""
    D = len(q)
    L = len(K)
    if L == 0:
        return [0.0] * D
    s = [scale * sum(q[c] * K[t][c] for c in range(D)) for t in range(L)]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = sum(e)
    return [sum(e[t] * V[t][c] for t in range(L)) / z for c in range(D)]

