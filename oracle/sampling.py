"""Sampling-distribution preparation and the drafter's own draw.

Test infrastructure only (see the package docstring).

* ``probs``: p = top_p(softmax(logits / T)).  The model card
  "Beam-1.0-501B-A23B-DFlash2" (section "Acceptance length") samples at
  temperature 0.7 and top-p 0.99.  The pages do not define top-p; it is
  read here as the usual nucleus rule: order the ids by (probability desc, id
  asc), keep the shortest prefix whose probability mass reaches top_p, zero
  the rest and renormalise.  The same preparation is applied to the target's
  p and the drafter's q.
* ``draft_draw``: the drafter proposes y ~ q ("DFlash vs DFlash 2", section
  "The problem: one expensive token at a time": "proposes token y from
  distribution q"), one inverse-CDF draw per position with Philox purpose 0.
"""

import numpy as np

from . import fixedpoint, philox


def softmax(logits, temperature=1.0):
    """Row softmax of logits / temperature in float64."""
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def top_p_keep(p, top_p):
    """Boolean mask of the kept ids of each row of p (float64 [..., V])."""
    p = np.asarray(p, dtype=np.float64)
    V = p.shape[-1]
    flat = p.reshape(-1, V)
    keep = np.zeros_like(flat, dtype=bool)
    for r in range(flat.shape[0]):
        row = flat[r]
        # order: probability descending, ties by id ascending
        order = np.lexsort((np.arange(V), -row))
        csum = np.cumsum(row[order])
        # shortest prefix whose mass reaches top_p of the row's total
        n_keep = int(np.searchsorted(csum, top_p * csum[-1], side="left")) + 1
        keep[r, order[:min(n_keep, V)]] = True
    return keep.reshape(p.shape)


def probs(logits, temperature=1.0, top_p=1.0):
    """p = top_p(softmax(logits / T)), renormalised; float64 [..., V]."""
    p = softmax(logits, temperature)
    if top_p < 1.0:
        keep = top_p_keep(p, top_p)
        p = np.where(keep, p, 0.0)
        p = p / p.sum(axis=-1, keepdims=True)
    return p


def draft_draw(q, seeds, step):
    """y_i ~ q_i for each request b and draft position i.

    q: float32 [B, G, V] (G = gamma - 1 drafted positions); seeds uint64 [B];
    step: uint64 scalar.  Returns int64 [B, G].
    """
    q = np.asarray(q, dtype=np.float32)
    B, G, _ = q.shape
    pos = np.arange(G, dtype=np.uint64)[None, :]
    u = philox.uniform64(np.asarray(seeds, dtype=np.uint64)[:, None], step, pos,
                         philox.PURPOSE_DRAFT)
    return fixedpoint.sample_rows(fixedpoint.to_fixed(q), u)
