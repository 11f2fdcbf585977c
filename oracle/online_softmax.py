"""The online-softmax recurrence, taken literally, and the merge of partial states.

Test infrastructure (see ``oracle/__init__``).

[P4] equation (4): for a new block of scores s_j, with running maximum m and
running normaliser l,
    m' = max(m, max_j s_j),     l' = e^{m - m'} l + sum_j e^{s_j - m'},
and the weighted-value accumulator is rescaled by the same factor e^{m - m'}
before the block's e^{s_j - m'} v_j are added.  [P3] §"分块 Attention 计算"
states that the blocks are read one by one and reduced with this online
softmax; [P1] §"Attention計算" states the result equals the softmax over the
concatenation of all blocks.

``merge_partials`` applies the same recurrence to summaries (m_p, l_p, acc_p)
of consecutive token ranges, which is what a split-K reduction computes: each
partial is one "block" whose contribution is already summed.

Pins: agreement with ``attention.dense_decode_attention`` to 1e-12 for many
block sizes and for x30 / x1000 logits ([P4]'s own binary64 record reports a
largest error of 2.22e-16 over 8 cases); the merge of any split equals the
single pass (``tests/test_oracle_pins.py``).
"""

from __future__ import annotations

import math

import numpy as np


def partial_state(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, block_size: int):
    """Run the recurrence over rows of K/V in blocks; return (m, l, acc) un-normalised."""
    q = np.asarray(q, dtype=np.float64)
    d_v = V.shape[-1]
    m = -math.inf
    l = 0.0
    acc = np.zeros(d_v, dtype=np.float64)
    n = K.shape[0]
    for start in range(0, n, block_size):
        Kj = K[start:start + block_size]
        Vj = V[start:start + block_size]
        s = float(scale) * (Kj @ q)
        m_new = max(m, float(s.max()))
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        p = np.exp(s - m_new)
        l = alpha * l + float(p.sum())
        acc = alpha * acc + p @ Vj
        m = m_new
    return m, l, acc


def online_softmax_attention(q, K, V, scale: float, block_size: int) -> np.ndarray:
    """softmax(scale K q) V computed block by block with the recurrence."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[-1], dtype=np.float64)
    m, l, acc = partial_state(q, K, V, scale, block_size)
    return acc / l


def merge_partials(parts) -> np.ndarray:
    """Merge [(m_p, l_p, acc_p), ...] of consecutive ranges into the final output.

    Each partial is folded in with the recurrence: the running state is
    rescaled by e^{m - m'} and the partial by e^{m_p - m'}.
    """
    m = -math.inf
    l = 0.0
    acc = None
    for (mp, lp, accp) in parts:
        if lp == 0.0:
            continue
        m_new = max(m, mp)
        a_old = math.exp(m - m_new) if m != -math.inf else 0.0
        a_new = math.exp(mp - m_new)
        l = a_old * l + a_new * lp
        accp = np.asarray(accp, dtype=np.float64)
        acc = a_new * accp if acc is None else a_old * acc + a_new * accp
        m = m_new
    if acc is None:
        raise ValueError("no non-empty partial")
    return acc / l
