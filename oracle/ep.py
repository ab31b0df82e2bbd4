"""Oracle of expert-parallel dispatch and combine (test infrastructure).

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests, smoke()
and the benchmark's CPU legs are the only callers; the CUDA library never
imports it and it imports nothing from the CUDA package.

Expert parallelism splits the E experts of the layer over n ranks in equal
contiguous ranges (rank d owns experts [d*E/n, (d+1)*E/n)).  The pages name it
only as the multi-GPU form that other PRs build on (the DeepEP dispatch of the
quant-info page's related PRs; the TP/EP question of the LoRA-MoE page's
review).  The steps written out here:

  dispatch: every (token, slot) pair p = t*K + k with expert e in [0, E) goes
            to rank e // (E/n); a rank's pairs are sent in increasing p.  Pairs
            with an expert id outside [0, E) are dropped (status "index").
  compute:  the owner computes w * (expert e's LoRA-MoE output for x_t) for each
            received pair, with e taken relative to its first expert.
  combine:  y_t = sum over k in increasing order of the returned rows of t's
            pairs (dropped pairs add nothing).

Everything is plain Python over small inputs; no step is blocked or fused.
"""
from __future__ import annotations

import numpy as np

OK = 0
INDEX = -3


def ep_dispatch(topk_ids, num_experts: int, n_ranks: int):
    """Send order of the pairs by destination rank.

    Returns (status, order, counts, pos):
      order  int32 [valid pairs]: pair ids, rank 0's first, each rank's in increasing p
      counts int32 [n_ranks]:     pairs sent to each rank
      pos    int32 [P]:           place of pair p in `order`, -1 for a dropped pair
    """
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    P = ids.size
    if n_ranks < 1 or num_experts < 1 or num_experts % n_ranks != 0:
        return -1, None, None, None
    per = num_experts // n_ranks
    status = OK
    dest = []
    counts = [0] * n_ranks
    for p in range(P):
        e = int(ids[p])
        if e < 0 or e >= num_experts:
            dest.append(-1)
            status = INDEX
            continue
        d = e // per
        dest.append(d)
        counts[d] += 1
    starts = [0] * n_ranks
    for d in range(1, n_ranks):
        starts[d] = starts[d - 1] + counts[d - 1]
    order = [0] * sum(counts)
    pos = [-1] * P
    for p in range(P):
        d = dest[p]
        if d < 0:
            continue
        order[starts[d]] = p
        pos[p] = starts[d]
        starts[d] += 1
    return (status, np.asarray(order, dtype=np.int32), np.asarray(counts, dtype=np.int32),
            np.asarray(pos, dtype=np.int32))


def ep_combine(rows, pos, num_tokens: int, topk: int):
    """y[t] = sum over k of rows[pos[t*K + k]] (k increasing, skipping -1), fp64."""
    rows = np.asarray(rows, dtype=np.float64)
    H = rows.shape[1] if rows.ndim == 2 else 0
    y = np.zeros((num_tokens, H), dtype=np.float64)
    for t in range(num_tokens):
        for k in range(topk):
            q = int(pos[t * topk + k])
            if q >= 0:
                y[t] += rows[q]
    return y
