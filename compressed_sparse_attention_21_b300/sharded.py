"""Sharded decode across ranks: the host-side collective logic.

A decode step over a context too long for one GPU splits each sequence's
compressed entries along the entry axis ("DeepSeek-V4 core architecture",
§2.4: 1M-token contexts; §2.2 step 2 and step 3 define what is computed).
Rank r of R owns a contiguous range of every sequence's CSA entries and of
its HCA entries; the raw tail of each query's open block belongs to the last
rank.  One step, per query:

1. every rank scores its visible entries with the lightning indexer and keeps
   its local top-k as (score, global entry index);
2. the ranks all-gather their candidates (k per rank); the global top-k is
   the top-k of the union, by score descending then index ascending -- exact,
   because a rank's local top-k holds every member of the global top-k that
   the rank owns;
3. every rank attends, over its own entries among the global selection (CSA)
   and over its HCA range (plus the raw tail on the last rank), and returns a
   partial output with its log-sum-exp per head;
4. the partials are merged: lse = log sum_r exp(lse_r),
   o = sum_r exp(lse_r - lse) o_r.

The per-rank compute is passed in as callables (scores of an entry range,
attention over a key set); this module holds the collective steps and the
merges, which use only torch.distributed all_gather.  The collectives carry
k (score, index) pairs and H x d partial outputs per query; no multicast.
"""
from __future__ import annotations

import math
from typing import Callable, Sequence

import numpy as np


def shard_bounds(n: int, world: int, rank: int) -> tuple:
    """Contiguous range [j0, j1) of n entries owned by `rank` (sizes differ by at most one)."""
    base, extra = divmod(n, world)
    j0 = rank * base + min(rank, extra)
    return j0, j0 + base + (1 if rank < extra else 0)


def local_topk(scores: np.ndarray, j0: int, k: int) -> tuple:
    """The k best (score, global index) of one rank's scores for entries j0 .. j0 + len - 1.

    Order: score descending, then index ascending; fewer than k when the rank
    has fewer entries.  Returns (scores, indices) in that order."""
    idx = np.arange(j0, j0 + len(scores), dtype=np.int64)
    order = np.lexsort((idx, -np.asarray(scores, np.float64)))[:k]
    return np.asarray(scores, np.float64)[order], idx[order]


def global_topk(cand_scores: Sequence[np.ndarray], cand_idx: Sequence[np.ndarray], k: int) -> np.ndarray:
    """Merge the ranks' candidates: the top-k by (score desc, index asc) of their union,
    returned in ascending index order and padded with -1 to k entries."""
    s = np.concatenate([np.asarray(x, np.float64) for x in cand_scores]) if cand_scores else np.zeros(0)
    j = np.concatenate([np.asarray(x, np.int64) for x in cand_idx]) if cand_idx else np.zeros(0, np.int64)
    order = np.lexsort((j, -s))[:k]
    sel = np.sort(j[order])
    out = np.full(k, -1, np.int64)
    out[:len(sel)] = sel
    return out


def lse_merge(o_parts: Sequence[np.ndarray], lse_parts: Sequence[np.ndarray]) -> tuple:
    """Combine per-rank partial attention outputs.

    o_parts[r]: [H, d] output over rank r's keys (normalised by its own sum);
    lse_parts[r]: [H] natural-log sum of exp(logits) over those keys (-inf when
    the rank had no key).  Returns (o [H, d], lse [H]) over all ranks' keys."""
    lse = np.stack([np.asarray(x, np.float64) for x in lse_parts])        # [R, H]
    o = np.stack([np.asarray(x, np.float64) for x in o_parts])            # [R, H, d]
    m = lse.max(0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse - m_safe[None])                                        # exp(-inf) = 0
    tot = w.sum(0)
    out_lse = m_safe + np.log(tot)
    out_o = (w[:, :, None] * o).sum(0) / tot[:, None]
    return out_o, out_lse


def all_gather_arrays(arr: np.ndarray, group=None) -> list:
    """all_gather of a numpy array whose shape may differ across ranks in its first axis."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    t = torch.from_numpy(np.ascontiguousarray(arr))
    n = torch.tensor([t.shape[0]], dtype=torch.int64)
    sizes = [torch.zeros_like(n) for _ in range(world)]
    dist.all_gather(sizes, n, group=group)
    cap = int(max(int(x) for x in sizes))
    pad = torch.zeros((cap,) + tuple(t.shape[1:]), dtype=t.dtype)
    pad[:t.shape[0]] = t
    bufs = [torch.zeros_like(pad) for _ in range(world)]
    dist.all_gather(bufs, pad, group=group)
    return [b[:int(s)].numpy() for b, s in zip(bufs, sizes)]


def sharded_decode_query(t: int, n_csa: int, n_hca: int, m_csa: int, m_hca: int, top_k: int,
                         score_range: Callable[[int, int], np.ndarray],
                         attend_csa: Callable[[np.ndarray, bool], tuple],
                         attend_hca: Callable[[int, int, bool], tuple],
                         group=None) -> dict:
    """One query at position t on this rank (collective: every rank calls it for the same query).

    n_csa / n_hca: the sequence's CSA / HCA entry counts (the ranks split them);
    m_csa / m_hca: the ratios.  score_range(j0, j1) -> indexer scores of visible
    entries j0 .. j1 - 1; attend_csa(entry_ids, with_tail) -> (o [H, d], lse [H])
    over those CSA entries (plus the raw tail of the CSA block if with_tail);
    attend_hca(j0, j1, with_tail) -> the same over HCA entries j0 .. j1 - 1.
    Returns the merged selection idx [top_k] and both merged outputs and LSEs."""
    import torch.distributed as dist
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    last = rank == world - 1
    # 1-2: local top-k over this rank's visible CSA entries, all-gather, global top-k
    n_vis = (t + 1) // m_csa
    j0, j1 = shard_bounds(n_csa, world, rank)
    v1 = min(j1, n_vis)
    s = score_range(j0, v1) if v1 > j0 else np.zeros(0)
    ls, li = local_topk(s, j0, top_k)
    all_s = all_gather_arrays(ls.astype(np.float64), group)
    all_i = all_gather_arrays(li.astype(np.int64), group)
    idx = global_topk(all_s, all_i, top_k)
    # 3: partial attention over this rank's selected entries and HCA range
    mine = idx[(idx >= j0) & (idx < j1)]
    oC, lC = attend_csa(mine, last and (t + 1) % m_csa > 0)
    nh_vis = (t + 1) // m_hca
    h0, h1 = shard_bounds(n_hca, world, rank)
    oH, lH = attend_hca(h0, min(h1, nh_vis), last and (t + 1) % m_hca > 0)
    # 4: LSE merge of the partials
    parts = all_gather_arrays(np.concatenate([oC.ravel(), lC, oH.ravel(), lH])[None], group)
    H, d = oC.shape
    oCs, lCs, oHs, lHs = [], [], [], []
    for p in parts:
        p = p[0]
        oCs.append(p[:H * d].reshape(H, d))
        lCs.append(p[H * d:H * d + H])
        oHs.append(p[H * d + H:2 * H * d + H].reshape(H, d))
        lHs.append(p[2 * H * d + H:])
    oC_m, lC_m = lse_merge(oCs, lCs)
    oH_m, lH_m = lse_merge(oHs, lHs)
    return {"idx": idx, "oC": oC_m, "lseC": lC_m, "oH": oH_m, "lseH": lH_m}


def empty_partial(H: int, d: int) -> tuple:
    """The partial of a rank without keys: output 0, log-sum-exp -inf."""
    return np.zeros((H, d)), np.full(H, -math.inf)
