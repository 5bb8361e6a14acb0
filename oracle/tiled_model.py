"""Tile-by-tile online-softmax model of attention, fp64, for one head.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It is not the
oracle: the oracle is the three-pass definition in ``oracle.c``.  This model
exists to pin the intermediate quantities that the worked example prints --
running maximum, rescale factor and running denominator after each key
tile -- and to show that the recurrence reaches the three-pass result.

It takes the steps in the order of the worked example in "Deep Learning -
Flash Attention" (ricojia.github.io, "An Example", steps 4-6) and of the
tiling steps in "FlashAttention" (ai360xpert.com, "Tiling and online
softmax"): for each query block Q_i, stream the key/value blocks K_j, V_j;
compute the tile scores S_ij = Q_i K_j^T * scale; update the row maximum
m_new = max(m_old, rowmax S_ij); rescale by alpha = exp(m_old - m_new); form
the unnormalised weights P_ij = exp(S_ij - m_new); update
l_new = alpha * l_old + rowsum(P_ij) and O_new = alpha * O_old + P_ij V_j;
after the last block divide O by l.
"""
from __future__ import annotations

import numpy as np


def tiled_attention(Q, K, V, scale, block_q=2, block_k=2, causal=False, trace=None):
    """O [N, d_v] and LSE [N] of one head; ``trace`` (a list) receives one dict
    per (query block, key block) step with m, alpha and l after that step."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    N = Q.shape[0]
    O = np.zeros((N, V.shape[1]))
    lse = np.zeros(N)
    for qs in range(0, N, block_q):
        qe = min(qs + block_q, N)
        m = np.full(qe - qs, -np.inf)
        l = np.zeros(qe - qs)
        acc = np.zeros((qe - qs, V.shape[1]))
        for ks in range(0, K.shape[0], block_k):
            ke = min(ks + block_k, K.shape[0])
            S = (Q[qs:qe] @ K[ks:ke].T) * scale
            if causal:  # key j visible to query i when j <= i
                qi = np.arange(qs, qe)[:, None]
                kj = np.arange(ks, ke)[None, :]
                S = np.where(kj <= qi, S, -np.inf)
            m_new = np.maximum(m, S.max(axis=1))
            # a row that has seen no key yet keeps weight 0 (exp(-inf) = 0)
            base = np.where(np.isfinite(m_new), m_new, 0.0)
            alpha = np.exp(m - base)
            P = np.exp(S - base[:, None])
            l = alpha * l + P.sum(axis=1)
            acc = alpha[:, None] * acc + P @ V[ks:ke]
            m = m_new
            if trace is not None:
                trace.append({"q_block": qs // block_q, "k_block": ks // block_k,
                              "S": S.copy(), "m": m.copy(), "alpha": alpha.copy(),
                              "l": l.copy()})
        O[qs:qe] = acc / l[:, None]
        lse[qs:qe] = m + np.log(l)
    return O, lse
