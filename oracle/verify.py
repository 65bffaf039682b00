"""Verification of a drafted block: greedy prefix match and lossless
rejection sampling.

Test infrastructure only (see the package docstring).

Source: "DFlash vs DFlash 2" blog, section "The problem: one expensive token
at a time".  The target scores the whole block in one pass and accepts the
longest valid prefix.  Greedy: a draft survives if it equals the target's
choice.  Sampling: a draft y ~ q survives with probability
alpha(y) = min(1, p(y)/q(y)); at the first rejection a correction is drawn
from the residual proportional to [p - q]+; if every draft survives, the
target emits one bonus token from its next distribution.  tau counts all
committed tokens of the cycle, bonus included.

Shapes (gamma = block size, G = gamma - 1 drafted tokens):
  draft      int [B, G]            y_1 .. y_G
  p / target float32 [B, gamma, V] row i is the target at the position of y_{i+1};
                                   row G is the bonus row
  q          float32 [B, G, V]
Result: accept_len int32 [B] (n, 0 <= n <= G) and tokens int32 [B, gamma]
with tokens[:n] = y_1..y_n, tokens[n] = the correction or bonus and the
rest -1.  tau = n + 1.

Readings taken here where the pages are silent:
  * greedy ties go to the lowest id;
  * the accept test u < p/q is evaluated as u*q(y) < p(y) in float64 with
    u = u24 * 2^-24, which is exact (24-bit times 24-bit mantissas);
  * the residual r = max(0, p - q) is formed in float32 (one rounding) and
    drawn from with the fixed-point inverse CDF; a residual of zero mass
    (possible only when p = q on the fixed-point grid) falls back to p.
"""

import numpy as np

from . import fixedpoint, philox


def greedy(target_logits, draft):
    t = np.asarray(target_logits, dtype=np.float32)
    y = np.asarray(draft, dtype=np.int64)
    B, gamma, _ = t.shape
    G = gamma - 1
    assert y.shape == (B, G)
    a = np.argmax(t, axis=-1)           # first maximum = lowest id
    accept_len = np.zeros(B, dtype=np.int32)
    tokens = np.full((B, gamma), -1, dtype=np.int32)
    for b in range(B):
        n = 0
        while n < G and y[b, n] == a[b, n]:
            n += 1
        accept_len[b] = n
        tokens[b, :n] = y[b, :n]
        tokens[b, n] = a[b, n]
    return accept_len, tokens


def sampled(p, q, draft, seeds, step):
    p = np.asarray(p, dtype=np.float32)
    q = np.asarray(q, dtype=np.float32)
    y = np.asarray(draft, dtype=np.int64)
    seeds = np.asarray(seeds, dtype=np.uint64)
    B, gamma, V = p.shape
    G = gamma - 1
    assert q.shape == (B, G, V) and y.shape == (B, G) and seeds.shape == (B,)
    rows = np.arange(B)

    # accept tests at every drafted position (a uniform per position)
    pos = np.arange(G, dtype=np.uint64)[None, :]
    u24 = philox.uniform24(seeds[:, None], step, pos, philox.PURPOSE_ACCEPT)
    u = u24.astype(np.float64) * 2.0 ** -24
    py = p[rows[:, None], np.arange(G)[None, :], y].astype(np.float64)
    qy = q[rows[:, None], np.arange(G)[None, :], y].astype(np.float64)
    accepted = u * qy < py                       # [B, G]

    # n = number of leading accepted drafts
    rejected_any = ~accepted.all(axis=1) if G > 0 else np.zeros(B, dtype=bool)
    n = np.where(rejected_any, np.argmin(accepted, axis=1) if G > 0 else 0, G)

    # distribution of the committed token at position n
    j = np.minimum(n, G - 1) if G > 0 else np.zeros(B, dtype=np.int64)
    p_row = p[rows, n]                            # target row at position n
    if G > 0:
        resid = np.maximum(p[rows, j] - q[rows, j], np.float32(0.0))  # float32
        R_res = fixedpoint.to_fixed(resid)
    else:
        R_res = np.zeros((B, V), dtype=np.uint64)
    R_p = fixedpoint.to_fixed(p_row)
    use_resid = rejected_any & (R_res.sum(axis=1, dtype=np.uint64) > 0)
    R = np.where(use_resid[:, None], R_res, R_p)
    u64 = philox.uniform64(seeds, step, n.astype(np.uint64), philox.PURPOSE_RESIDUAL)
    last = fixedpoint.sample_rows(R, u64)

    accept_len = n.astype(np.int32)
    y_pad = np.concatenate([y, np.full((B, 1), -1, dtype=np.int64)], axis=1)
    tokens = np.where(np.arange(gamma)[None, :] < n[:, None], y_pad, -1)
    tokens[rows, n] = last
    return accept_len, tokens.astype(np.int32)


def acceptance_probability(p_row, q_row):
    """Probability that a draft y ~ q is accepted: sum_v min(p_v, q_v)."""
    return float(np.minimum(np.asarray(p_row, np.float64), np.asarray(q_row, np.float64)).sum())


def expected_tau(beta):
    """E[tau] = 1 + sum_k prod_{i<=k} beta_i for per-position acceptance beta."""
    return 1.0 + float(np.cumprod(np.asarray(beta, dtype=np.float64)).sum())
