"""Sharded decode on CPU ranks (gloo, world size 2) against the unsharded oracle.

Each rank owns a contiguous half of every sequence's CSA and HCA entries and
computes with the oracle: local indexer scores and top-k, then attention over
its share of the global selection and of the HCA entries (the raw tail on the
last rank).  The collective steps are those of
compressed_sparse_attention_21_b300.sharded: an all-gather of (score, index)
candidates, the global top-k of their union, and the log-sum-exp merge of the
partial outputs.  The merged result must equal the oracle run on the whole
problem: identical index sets, outputs and LSEs within 1e-12.
"""
import math
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from compressed_sparse_attention_21_b300 import sharded  # noqa: E402
from compressed_sparse_attention_21_b300 import workloads as wl  # noqa: E402

LENGTHS = [1203, 9, 777, 4099, 300]
N_Q = [1, 1, 3, 2, 5]          # decode steps and short chunks: the last n_q positions
SHAPE = dict(H=4, d=16, HI=2, dI=8, top_k=16, mC=4, mH=128)


def _problem():
    w = wl.Workload("sharded", len(LENGTHS), LENGTHS, False, H=SHAPE["H"], d=SHAPE["d"], HI=SHAPE["HI"],
                    dI=SHAPE["dI"], top_k=SHAPE["top_k"], mC=SHAPE["mC"], mH=SHAPE["mH"], seed=77)
    return wl.to_numpy(wl.make_problem(w, n_q=N_Q))


def _bf16(bits):
    import torch
    b = np.ascontiguousarray(bits, np.uint16)
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = _problem()
        H, d, k, mC, mH = SHAPE["H"], SHAPE["d"], SHAPE["top_k"], SHAPE["mC"], SHAPE["mH"]
        out = []
        for b, (L, nq) in enumerate(zip(LENGTHS, N_Q)):
            cu_kv, cu_q, cu_csa, cu_hca = p["cu_kv"], p["cu_q"], p["cu_csa"], p["cu_hca"]
            for i in range(nq):
                qi = int(cu_q[b]) + i
                t = L - nq + i
                qI, qv = p["qI"][qi], p["q"][qi]

                def score_range(j0, j1):
                    return oracle.index_scores(qI, p["kI"][cu_csa[b] + j0:cu_csa[b] + j1])

                def tail_rows(m):
                    r = (t + 1) % m
                    return _bf16(p["kv"][cu_kv[b] + t - r + 1:cu_kv[b] + t + 1])

                def attend(keys):
                    if len(keys) == 0:
                        return sharded.empty_partial(H, d)
                    return oracle.attend(qv, keys, p["scale"])

                def attend_csa(ids, with_tail):
                    keys = [oracle.compress_selected(cu_kv, cu_csa, p["kv"], p["gate"], mC, cu_csa[b] + ids)] \
                        if len(ids) else []
                    if with_tail:
                        keys.append(tail_rows(mC))
                    return attend(np.concatenate(keys) if keys else np.zeros((0, d)))

                def attend_hca(h0, h1, with_tail):
                    keys = [oracle.compress_selected(cu_kv, cu_hca, p["kv"], p["gate"], mH,
                                                     cu_hca[b] + np.arange(h0, h1))] if h1 > h0 else []
                    if with_tail:
                        keys.append(tail_rows(mH))
                    return attend(np.concatenate(keys) if keys else np.zeros((0, d)))

                r = sharded.sharded_decode_query(t, int(cu_csa[b + 1] - cu_csa[b]), int(cu_hca[b + 1] - cu_hca[b]),
                                                 mC, mH, k, score_range, attend_csa, attend_hca)
                out.append(r)
        q.put((rank, out))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_sharded_decode_equals_the_unsharded_oracle(orc):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    got = dict(q.get(timeout=300) for _ in range(2))
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    ref = orc.hybrid_queries(_problem())
    for rank in (0, 1):
        res = got[rank]
        assert len(res) == ref["idx"].shape[0]
        for row, r in enumerate(res):
            assert np.array_equal(r["idx"], ref["idx"][row]), (rank, row)
            for key in ("oC", "lseC", "oH", "lseH"):
                assert np.abs(r[key] - ref[key][row]).max() <= 1e-12, (rank, row, key)


def test_global_topk_equals_topk_of_the_union(orc):
    # the merged selection of per-shard top-k lists is the top-k of all scores,
    # ties to the lower index (checked against the oracle's own top-k with planted ties)
    rng = np.random.default_rng(5)
    s = np.round(rng.standard_normal(301), 1)          # many equal scores
    for world in (1, 2, 3, 5):
        for k in (1, 7, 40, 400):
            parts_s, parts_i = [], []
            for r in range(world):
                j0, j1 = sharded.shard_bounds(len(s), world, r)
                ls, li = sharded.local_topk(s[j0:j1], j0, k)
                parts_s.append(ls)
                parts_i.append(li)
            assert np.array_equal(sharded.global_topk(parts_s, parts_i, k), orc.topk(s, k)), (world, k)


def test_lse_merge_equals_attention_over_all_keys(orc):
    rng = np.random.default_rng(6)
    H, d = 3, 8
    q = wl.bits(__import__("torch").randn(H, d).to(__import__("torch").bfloat16))
    keys = rng.standard_normal((23, d))
    o_all, l_all = orc.attend(q, keys, 1 / math.sqrt(d))
    cuts = [0, 5, 5, 17, 23]                                  # an empty part included
    o_p, l_p = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b > a:
            o, l = orc.attend(q, keys[a:b], 1 / math.sqrt(d))
        else:
            o, l = sharded.empty_partial(H, d)
        o_p.append(o)
        l_p.append(l)
    o_m, l_m = sharded.lse_merge(o_p, l_p)
    assert np.abs(o_m - o_all).max() <= 1e-13 and np.abs(l_m - l_all).max() <= 1e-13


def test_shard_bounds_cover_every_entry_once():
    for n in (0, 1, 2, 7, 262144):
        for world in (1, 2, 3, 8):
            spans = [sharded.shard_bounds(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans[:-1], spans[1:]))
            sizes = [j1 - j0 for j0, j1 in spans]
            assert max(sizes) - min(sizes) <= 1
