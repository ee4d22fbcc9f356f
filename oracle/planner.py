"""Plain CPU oracle of the anchor-guided selection planner (numpy, fp64).

TEST INFRASTRUCTURE ONLY: the test suite may import this module; the library never does, and
it shares no code with it.

Method: DiTango (gist.science/paper/2607.15650), Methodology 1, Anchor-Guided Selection
Planner. The page states the ingredients and leaves the formulas open; this module takes the
plainest reading of each:

  * Error modeling: the error of reusing a state is a function of the partition's importance w
    and of the temporal error growth delta -> here their product, e[i, j] = w[i, j] * delta[i].
  * Anchor steps compute every pair and update the importance weights -> w[i, j] is the share
    of query partition i's attention mass that KV partition j holds at the anchor: per query
    row, the merge weight exp(lse_ij - lse_i) of state (i, j) (lse_i = log-sum-exp over j), so
    each row's weights sum to 1; w[i, :] averages them over the rows of partition i (and over
    batch and heads).
  * Online prediction: between anchors, the change of the always-computed local state stands
    in for the drift of the remote ones -> delta[i] = ||O_ii(t) - O_ii(anchor)|| /
    ||O_ii(anchor)||, Frobenius norms over the rows of partition i (batch, heads, channels).
  * Group-wise strategy: spatially adjacent partitions are grouped and decided together ->
    KV partitions form contiguous groups of g; for each query partition i and group G the
    predicted error is the sum of e[i, j] over the members j != i; groups whose error exceeds
    tau are recomputed, largest error first, while the count of computed pairs stays within
    the budget. A group holding a pair that was never computed is always recomputed (nothing
    to reuse); the local pair (i, i) is always computed.
"""
from __future__ import annotations

import numpy as np


def importance(lse: np.ndarray, offsets) -> np.ndarray:
    """w [P, P] from the per-pair lse of every query row at an anchor step.

    lse: [B, H, P, N]: lse[b, h, j, r] is the lse of state (partition(r), j) of row r.
    """
    lse = np.asarray(lse, dtype=np.float64)
    B, H, P, N = lse.shape
    offsets = np.asarray(offsets, dtype=np.int64)
    w = np.zeros((P, P), dtype=np.float64)
    for i in range(P):
        r0, r1 = int(offsets[i]), int(offsets[i + 1])
        block = lse[:, :, :, r0:r1]                        # [B, H, P, rows]
        top = block.max(axis=2, keepdims=True)
        tot = top + np.log(np.exp(block - top).sum(axis=2, keepdims=True))
        share = np.exp(block - tot)                        # merge weight of each state
        w[i] = share.sum(axis=(0, 1, 3)) / (B * H * (r1 - r0))
    return w


def drift(O_now: np.ndarray, O_anchor: np.ndarray, offsets) -> np.ndarray:
    """delta [P]: relative Frobenius change of each partition's local (diagonal) states.

    O_now, O_anchor: [B, H, N, d], row r holding the state (partition(r), partition(r)).
    A partition whose anchor states are all zero gets delta = 0.
    """
    a = np.asarray(O_now, dtype=np.float64)
    b = np.asarray(O_anchor, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    P = len(offsets) - 1
    out = np.zeros(P, dtype=np.float64)
    for i in range(P):
        r0, r1 = int(offsets[i]), int(offsets[i + 1])
        num = ((a[:, :, r0:r1] - b[:, :, r0:r1]) ** 2).sum()
        den = (b[:, :, r0:r1] ** 2).sum()
        out[i] = np.sqrt(num / den) if den > 0 else 0.0
    return out


def groups(P: int, g: int):
    """Contiguous groups of g KV partitions (the last may be shorter)."""
    return [list(range(s, min(s + g, P))) for s in range(0, P, g)]


def select(w: np.ndarray, delta: np.ndarray, tau: float, g: int, budget: int,
           valid: np.ndarray) -> np.ndarray:
    """Reuse mask [P, P] (1 = reuse) for the next step.

    Candidates are the (query partition i, group G) pairs with at least one member j != i.
    Groups with a never-computed member are recomputed first (in (i, G) order); the others
    are considered by decreasing predicted error sum_{j in G, j != i} w[i, j] * delta[i] (ties:
    lower i, then lower G) and recomputed if that error exceeds tau and the computed pairs
    (counting the P local ones) stay within `budget` (budget < 0: no limit).
    """
    P = w.shape[0]
    valid = np.asarray(valid, dtype=bool)
    mask = np.ones((P, P), dtype=np.uint8)
    np.fill_diagonal(mask, 0)
    computed = P
    forced, ranked = [], []
    for i in range(P):
        for k, grp in enumerate(groups(P, g)):
            members = [j for j in grp if j != i]
            if not members:
                continue
            err = 0.0
            for j in members:  # in ascending j, the order the library sums in
                err += float(w[i, j]) * float(delta[i])
            if any(not valid[i, j] for j in members):
                forced.append((i, k, members))
            else:
                ranked.append((-err, i, k, members, err))
    for i, k, members in forced:
        for j in members:
            mask[i, j] = 0
        computed += len(members)
    ranked.sort(key=lambda c: (c[0], c[1], c[2]))
    for _, i, k, members, err in ranked:
        if not err > tau:
            continue
        if budget >= 0 and computed + len(members) > budget:
            continue
        for j in members:
            mask[i, j] = 0
        computed += len(members)
    return mask
