"""GPU parity: every step of the CUDA path against the fp64 oracle, through the C ABI.

Small ragged cases cover tiles, ragged tails, lengths below one block, exact
block boundaries and n(t) <= k; the five workloads run at full size (the
128K prefill on a sampled query set, every other workload on every query).
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_21_b300 import _lib as csa
from compressed_sparse_attention_21_b300 import build as csa_build
from compressed_sparse_attention_21_b300 import workloads as wl

from . import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    csa_build.build()
    csa.load()
    oracle.build()
    yield
    assert csa.check_device_error() == 0


def problem(lengths, n_q, H=8, d=128, HI=2, dI=32, k=16, mC=4, mH=128, seed=0, gate_std=1.0):
    w = wl.Workload("case", len(lengths), list(lengths), False, H=H, d=d, HI=HI, dI=dI, top_k=k, mC=mC,
                    mH=mH, gate_std=gate_std, seed=seed)
    return wl.make_problem(w, n_q=n_q)


RAGGED = [1, 3, 4, 5, 127, 128, 129, 300, 1000]


# ---------------------------------------------------------------------------
# a1: compression
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("d", [128, 512])
@pytest.mark.parametrize("ratio,side", [(1, "csa"), (2, "csa"), (4, "csa"), (8, "csa"), (32, "csa"),
                                        (64, "hca"), (128, "hca"), (4, "hca")])
def test_compress_prefill(d, ratio, side):
    p = problem(RAGGED, RAGGED, d=d, mC=ratio if side == "csa" else 4, mH=ratio if side == "hca" else 128,
                seed=ratio)
    g = P.GpuProblem(p)
    inp = wl.to_numpy(p)
    cu = inp["cu_csa"] if side == "csa" else inp["cu_hca"]
    out = torch.full((int(cu[-1]), d), float("nan"), dtype=torch.bfloat16, device="cuda")
    (csa.csa_compress if side == "csa" else csa.hca_compress)(g.full, g.kv, g.gate, out, ratio=ratio)
    torch.cuda.synchronize()
    ref = oracle.compress_packed(inp["cu_kv"], cu, inp["kv"], inp["gate"], ratio)
    got = P.bf16_to_f64(out)
    err, ratio_to_bound = P.entry_err(got, ref)
    assert ratio_to_bound <= 1.0, err
    # tighter: one bf16 rounding of an fp32 weighted sum (see parity.entry_ulp_check)
    mix = oracle.compress_packed(inp["cu_kv"], cu, P.abs_bits(inp["kv"]), inp["gate"], ratio)
    assert P.entry_ulp_check(got, ref, mix, ratio) <= 1.0


def test_compress_fused_and_decode_append():
    lengths = [4, 127, 128, 260, 512, 777]
    p = problem(lengths, [1] * len(lengths), d=512, seed=3)
    g = P.GpuProblem(p)
    inp = wl.to_numpy(p)
    ref_c = oracle.compress_packed(inp["cu_kv"], inp["cu_csa"], inp["kv"], inp["gate"], 4)
    ref_h = oracle.compress_packed(inp["cu_kv"], inp["cu_hca"], inp["kv"], inp["gate"], 128)
    # decode layout: only the block closed by the newest token may be written
    h = csa.Hybrid(g.layout, g.kv, g.gate, g.qI, g.kI, g.q, p["top_k"], p["scale"],
                   csa_cache=torch.full((g.layout.total_csa, 512), 7.0, dtype=torch.bfloat16, device="cuda"),
                   hca_cache=torch.full((g.layout.total_hca, 512), 7.0, dtype=torch.bfloat16, device="cuda"))
    h()
    torch.cuda.synchronize()
    got_c, got_h = P.bf16_to_f64(h.csa_cache), P.bf16_to_f64(h.hca_cache)
    for b, L in enumerate(lengths):
        for j in range(L // 4):
            row = inp["cu_csa"][b] + j
            if (j + 1) * 4 == L:
                assert P.entry_err(got_c[row], ref_c[row])[1] <= 1.0
            else:
                assert (got_c[row] == 7.0).all(), (b, j)
        for j in range(L // 128):
            row = inp["cu_hca"][b] + j
            if (j + 1) * 128 == L:
                assert P.entry_err(got_h[row], ref_h[row])[1] <= 1.0
            else:
                assert (got_h[row] == 7.0).all(), (b, j)


# ---------------------------------------------------------------------------
# a2/a3: indexer + top-k, both paths
# ---------------------------------------------------------------------------
def _check_index(p, idx, score, fp8=None):
    """fp8: the oracle's (codes, scales) of the keys; the oracle then scores and selects on them."""
    inp = wl.to_numpy(p)
    idx = idx.cpu().numpy()
    score = score.cpu().numpy()
    total_q = int(inp["cu_q"][-1])
    orc = oracle.hybrid_queries(inp, do_hca=False) if fp8 is None else None
    kinds = {"equal": 0, "tie": 0, "fp32tie": 0}
    for qi in range(total_q):
        b = int(np.searchsorted(inp["cu_q"], qi, side="right") - 1)
        L = inp["cu_kv"][b + 1] - inp["cu_kv"][b]
        t = L - (inp["cu_q"][b + 1] - inp["cu_q"][b]) + (qi - inp["cu_q"][b])
        n = int((t + 1) // p["mC"])
        rows = slice(inp["cu_csa"][b], inp["cu_csa"][b] + n)
        kseq = inp["kI"][rows]
        if fp8 is None:
            s = oracle.index_scores(inp["qI"][qi], kseq) if n else np.zeros(0)
            o_idx, dq = orc["idx"][qi], None
        else:
            s = oracle.index_scores_fp8(inp["qI"][qi], fp8[0][rows], fp8[1][rows]) if n else np.zeros(0)
            o_idx, dq = oracle.topk(s, p["top_k"]), P.fp8_dequant(fp8[0][rows], fp8[1][rows])
        kind, _ = P.check_topk_row(idx[qi], o_idx, s, n, p["top_k"], inp["qI"][qi], kseq, dq)
        kinds[kind] += 1
        v = idx[qi] >= 0
        # returned scores are the fp32 scores of the returned indices
        assert np.allclose(score[qi][v], s[idx[qi][v]], rtol=1e-5, atol=1e-3)
        assert np.isneginf(score[qi][~v]).all()
    return kinds


@pytest.mark.parametrize("HI,dI,k", [(2, 32, 64), (4, 64, 512), (4, 64, 1024), (1, 128, 7)])
def test_index_topk_multi_cta_path(HI, dI, k):
    lengths = [1, 5, 100, 4096, 5001, 20000, 70001]
    p = problem(lengths, [1] * len(lengths), HI=HI, dI=dI, k=k, seed=11)
    g = P.GpuProblem(p)
    idx, score = csa.lightning_index_topk(g.layout, g.qI, g.kI, k)
    torch.cuda.synchronize()
    kinds = _check_index(p, idx, score)
    assert kinds["equal"] >= len(lengths) - 1


@pytest.mark.parametrize("HI,dI,k", [(2, 32, 64), (4, 64, 512), (4, 64, 7), (1, 128, 100)])
def test_index_topk_prefill_paths(HI, dI, k):
    # 2200 queries, rows of at most 375 entries: the prefill paths (tensor-memory
    # score tiles for d_I = 64, mma.sync tiles otherwise) keep every entry
    lengths = [1500, 700]
    p = problem(lengths, lengths, HI=HI, dI=dI, k=k, seed=12)
    g = P.GpuProblem(p)
    idx, score = csa.lightning_index_topk(g.layout, g.qI, g.kI, k)
    torch.cuda.synchronize()
    _check_index(p, idx, score)


def _check_index_rows(p, idx, score, rows):
    """_check_index on the listed query rows only (long prefills)."""
    inp = wl.to_numpy(p)
    kinds = {"equal": 0, "tie": 0, "fp32tie": 0}
    for qi in rows:
        b = int(np.searchsorted(inp["cu_q"], qi, side="right") - 1)
        L = inp["cu_kv"][b + 1] - inp["cu_kv"][b]
        t = L - (inp["cu_q"][b + 1] - inp["cu_q"][b]) + (qi - inp["cu_q"][b])
        n = int((t + 1) // p["mC"])
        kseq = inp["kI"][inp["cu_csa"][b]:inp["cu_csa"][b] + n]
        s = oracle.index_scores(inp["qI"][qi], kseq) if n else np.zeros(0)
        kind, _ = P.check_topk_row(idx[qi], oracle.topk(s, p["top_k"]), s, n, p["top_k"], inp["qI"][qi], kseq)
        kinds[kind] += 1
        v = idx[qi] >= 0
        assert np.allclose(score[qi][v], s[idx[qi][v]], rtol=1e-5, atol=1e-3)
    return kinds


@pytest.mark.parametrize("k", [64, 512, 1024])
def test_index_topk_prefill_sampled_threshold(k):
    # rows longer than the candidate buffer (n > 4096): the sampled threshold,
    # the candidate filter and the warp selection; three sequences share the
    # first 128-query block of the tensor-memory path
    lengths = [60, 5, 20000, 3000]
    p = problem(lengths, lengths, HI=4, dI=64, k=k, seed=14)
    g = P.GpuProblem(p)
    idx, score = csa.lightning_index_topk(g.layout, g.qI, g.kI, k)
    torch.cuda.synchronize()
    idx, score = idx.cpu().numpy(), score.cpu().numpy()
    rng = np.random.default_rng(15)
    total = sum(lengths)
    rows = np.unique(np.concatenate([np.arange(0, 200), np.arange(16380, 16420), np.arange(20060, 20070),
                                     np.arange(total - 40, total), rng.integers(0, total, 300)]))
    kinds = _check_index_rows(p, idx, score, rows)
    assert kinds["equal"] >= len(rows) - 3, kinds


@pytest.mark.parametrize("dI", [32, 64])
@pytest.mark.parametrize("queries", ["decode", "prefill", "prefill_overflow"])
def test_index_topk_all_ties_lowest_index_wins(queries, dI):
    # prefill_overflow: rows longer than the prefill path's candidate buffer, all
    # scores equal, so the exact fallback selection must run
    lengths = {"prefill": [3000, 4100], "decode": [3000, 4100, 9000], "prefill_overflow": [17000]}[queries]
    queries = "prefill" if queries.startswith("prefill") else queries
    p = problem(lengths, lengths if queries == "prefill" else [1] * len(lengths), HI=2, dI=dI, k=64, seed=13)
    p["kI"] = torch.ones_like(p["kI"])      # every entry scores the same
    g = P.GpuProblem(p)
    idx, _ = csa.lightning_index_topk(g.layout, g.qI, g.kI, 64)
    idx = idx.cpu().numpy()
    for qi in range(idx.shape[0]):
        b = int(np.searchsorted(g.layout.host["cu_q"], qi, side="right") - 1)
        L = lengths[b]
        t = L - g.layout.n_q[b] + (qi - g.layout.host["cu_q"][b])
        n = (t + 1) // 4
        want = list(range(min(64, n))) + [-1] * (64 - min(64, n))
        assert list(idx[qi]) == want


def test_index_topk_prefill_fallback_then_next_sequence():
    # the 128-query block at 16384 holds the last 16 queries of a sequence whose
    # keys all tie (rows of 4097-4100 entries overflow the candidate buffer, so
    # the exact fallback runs and reuses the query tiles' space) and then the first
    # 112 queries of a sequence with ordinary keys, scored after the fallback
    lengths = [16400, 2000]
    k = 8
    p = problem(lengths, lengths, HI=2, dI=64, k=k, seed=16)
    n0 = lengths[0] // 4
    p["kI"][:n0] = 1.0
    g = P.GpuProblem(p)
    idx, score = csa.lightning_index_topk(g.layout, g.qI, g.kI, k)
    torch.cuda.synchronize()
    idx, score = idx.cpu().numpy(), score.cpu().numpy()
    for qi in range(16300, lengths[0]):
        n = (qi + 1) // 4
        assert list(idx[qi]) == list(range(min(k, n))) + [-1] * (k - min(k, n)), qi
    rows = np.arange(lengths[0], lengths[0] + 400)
    kinds = _check_index_rows(p, idx, score, rows)
    assert kinds["equal"] >= len(rows) - 2, kinds


# ---------------------------------------------------------------------------
# f2: FP8 indexer keys
# ---------------------------------------------------------------------------
def _plant_fp8_rows(kI):
    """Rows that exercise the quantiser's special cases (kI: [n, dI] bf16, n >= 6)."""
    dI = kI.shape[1]
    kI[0] = 0.0                                        # all zero: codes 0, scale 0
    kI[1] = 0.0
    kI[1, dI - 1] = -2.5                               # one non-zero: it maps to -448
    kI[2, 0] = 1.0
    kI[2, 1:] = -1e-6                                  # far below the smallest subnormal: -0
    kI[3] = torch.tensor(([448.0, 1.0625, 1.1875, 17.0, 2.0 ** -10, 3 * 2.0 ** -10, -1.0625, -0.0]
                          * dI)[:dI])                  # scale 1: exact midpoints, ties to even
    kI[4] = -kI[4].abs()
    kI[4, 0] = -kI[4].abs().max() * 2                  # the largest magnitude is negative
    kI[5] *= 1e-30                                     # tiny but normal row scale
    return kI


@pytest.mark.parametrize("dI", [32, 64, 128])
def test_quantize_index_keys_bit_exact(dI):
    lengths = [1, 4, 5, 27, 1000, 4099]                # 1282 rows: several blocks of 8 and a ragged tail
    p = problem(lengths, [1] * len(lengths), HI=2, dI=dI, seed=40 + dI)
    p["kI"] = _plant_fp8_rows(p["kI"].clone())
    g = P.GpuProblem(p)
    codes, scale = csa.quantize_index_keys(g.full, g.kI)
    torch.cuda.synchronize()
    o_codes, o_scale = oracle.quantize_index_keys(wl.bits(p["kI"]))
    got_c, got_s = codes.cpu().numpy(), scale.cpu().numpy()
    assert got_c.shape == o_codes.shape
    bad = np.argwhere(got_c != o_codes)
    assert len(bad) == 0, f"{len(bad)} codes differ, first {bad[:4].tolist()}"
    assert np.array_equal(got_s.view(np.uint32), o_scale.view(np.uint32))


def closed_rows(lengths, n_q, m):
    """Entry rows closed by the query positions: entry j of a sequence exists once
    its m tokens do, so the query at t = (j+1)m - 1 closes it."""
    rows, e0 = [], 0
    for L, nq in zip(lengths, n_q):
        rows += [e0 + (t + 1) // m - 1 for t in range(L - nq, L) if (t + 1) % m == 0]
        e0 += L // m
    return np.array(rows, dtype=np.int64)


@pytest.mark.parametrize("dI", [32, 64, 128])
@pytest.mark.parametrize("case", ["decode", "chunked", "prefill"])
def test_quantize_closed_index_keys(dI, case):
    lengths = [4, 5, 8, 127, 128, 4096, 4099, 1000]
    n_q = {"decode": [1] * 8, "chunked": [4, 1, 8, 37, 64, 300, 3, 999], "prefill": lengths}[case]
    p = problem(lengths, n_q, HI=2, dI=dI, seed=60 + dI)
    p["kI"] = _plant_fp8_rows(p["kI"].clone())
    g = P.GpuProblem(p)
    n = g.full.total_csa
    codes = torch.full((n, dI), 0x55, dtype=torch.uint8, device="cuda")
    scale = torch.full((n,), -1.0, dtype=torch.float32, device="cuda")
    csa.quantize_closed_index_keys(g.layout, g.kI, codes, scale)
    torch.cuda.synchronize()
    assert csa.check_device_error() == 0
    rows = closed_rows(lengths, n_q, 4)
    o_codes, o_scale = oracle.quantize_index_keys(wl.bits(p["kI"]))
    got_c, got_s = codes.cpu().numpy(), scale.cpu().numpy()
    assert np.array_equal(got_c[rows], o_codes[rows])
    assert np.array_equal(got_s[rows].view(np.uint32), o_scale[rows].view(np.uint32))
    other = np.setdiff1d(np.arange(n), rows)
    assert (got_c[other] == 0x55).all() and (got_s[other] == -1.0).all(), "a row no query closes was written"
    if case == "prefill":   # every entry is closed by some position: the same as quantising every row
        assert len(rows) == n


@pytest.mark.parametrize("HI,dI,k", [(2, 32, 64), (4, 64, 512), (4, 128, 1024), (1, 128, 7)])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_index_topk_fp8(HI, dI, k, mode):
    if mode == "decode":
        lengths = [1, 5, 100, 4096, 5001, 20000, 70001]
        n_q = [1] * len(lengths)
    else:
        lengths = [1500, 700]
        n_q = lengths
    p = problem(lengths, n_q, HI=HI, dI=dI, k=k, seed=50 + dI)
    g = P.GpuProblem(p)
    codes, scale = csa.quantize_index_keys(g.full, g.kI)
    idx, score = csa.lightning_index_topk_fp8(g.layout, g.qI, codes, scale, k)
    torch.cuda.synchronize()
    fp8 = oracle.quantize_index_keys(wl.bits(p["kI"]))
    kinds = _check_index(p, idx, score, fp8=fp8)
    if mode == "decode":
        assert kinds["equal"] >= len(lengths) - 1


@pytest.mark.parametrize("case", ["decode_small", "chunked"])
def test_hybrid_fp8_small(case):
    if case == "decode_small":
        p = problem([4, 4097, 8191, 30001], [1] * 4, H=128, d=512, HI=4, dI=64, k=256, seed=35)
    else:
        p = problem([1000, 2000], [37, 300], H=64, d=512, HI=4, dI=64, k=64, seed=36)
    g = P.GpuProblem(p)
    h = g.hybrid(prebuilt=True, fp8=True)
    rep = P.check_hybrid(p, h, fp8=oracle.quantize_index_keys(wl.bits(p["kI"])))
    assert rep["topk"]["equal"] >= rep["queries"] - 2
    o1 = h.o_csa.clone()
    h()
    torch.cuda.synchronize()
    assert torch.equal(o1, h.o_csa)


def test_workload_decode_64k_fp8_every_query():
    w = wl.WORKLOADS["decode_64k"]
    p = wl.make_problem(w)
    g = P.GpuProblem(p)
    h = g.hybrid(prebuilt=True, fp8=True)
    rep = P.check_hybrid(p, h, check_entries="sampled", fp8=oracle.quantize_index_keys(wl.bits(p["kI"])))
    assert csa.check_device_error() == 0
    print("decode_64k fp8", rep)


# ---------------------------------------------------------------------------
# a4/a5: attention, on the oracle's own selection
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("H,d", [(8, 128), (8, 512), (64, 512), (128, 512), (64, 128)])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_attend_parity(H, d, mode):
    # decode: 20000 gives the dense branch 188 keys, split over several CTAs
    lengths = [1, 3, 4, 129, 1000, 5003, 20000] if mode == "decode" else [1, 130, 257]
    n_q = [1] * len(lengths) if mode == "decode" else lengths
    k = 64 if mode == "prefill" else 128
    p = problem(lengths, n_q, H=H, d=d, k=k, seed=H + d)
    g = P.GpuProblem(p)
    inp = wl.to_numpy(p)
    csa_cache, hca_cache = g.build_caches()
    orc_hca = oracle.compress_packed(inp["cu_kv"], inp["cu_hca"], inp["kv"], inp["gate"], 128)
    orc = oracle.hybrid_queries(inp, hca_entries=orc_hca)
    idx = torch.from_numpy(orc["idx"]).cuda()
    oC, lC = csa.sparse_mqa_attend(g.layout, g.q, csa_cache, g.kv, idx, k, p["scale"])
    oH, lH = csa.hca_dense_attend(g.layout, g.q, hca_cache, g.kv, p["scale"])
    torch.cuda.synchronize()
    P.assert_att(P.bf16_to_f64(oC), orc["oC"], "sparse")
    P.assert_att(P.bf16_to_f64(oH), orc["oH"], "dense")
    assert np.abs(lC.cpu().numpy() - orc["lseC"]).max() <= 1e-2
    assert np.abs(lH.cpu().numpy() - orc["lseH"]).max() <= 1e-2


def test_attend_invisible_index_is_reported_and_skipped():
    p = problem([64, 64], [1, 1], k=8, seed=21)
    g = P.GpuProblem(p)
    csa_cache, _ = g.build_caches()
    idx = torch.full((2, 8), -1, dtype=torch.int32, device="cuda")
    idx[:, 0] = 3
    idx[1, 1] = 16                           # n(63) = 16: index 16 is not visible
    csa.sparse_mqa_attend(g.layout, g.q, csa_cache, g.kv, idx, 8, p["scale"])
    assert csa.check_device_error() == 6
    assert csa.check_device_error() == 0    # reading clears it


def test_attend_persistent_invisible_index_is_reported_and_skipped():
    # a prefill-sized call (d = 512, 64 heads, more queries than SMs) runs the
    # persistent kernel; one row names an entry its query cannot see: the call
    # reports it, skips that key, and every other row still matches the oracle
    lengths = [300, 200]
    k = 16
    p = problem(lengths, lengths, H=64, d=512, k=k, seed=23)
    g = P.GpuProblem(p)
    inp = wl.to_numpy(p)
    csa_cache, _ = g.build_caches()
    orc = oracle.hybrid_queries(inp)
    idx_np = orc["idx"].copy()
    bad_row = 299                                    # t = 299 of sequence 0 sees entries 0 .. 74
    assert idx_np[bad_row, -1] >= 0
    idx_np[bad_row, -1] = 80                         # not visible
    idx = torch.from_numpy(idx_np).cuda()
    oC, _ = csa.sparse_mqa_attend(g.layout, g.q, csa_cache, g.kv, idx, k, p["scale"])
    torch.cuda.synchronize()
    assert csa.check_device_error() == 6
    assert csa.check_device_error() == 0
    got = P.bf16_to_f64(oC)
    keep = np.ones(got.shape[0], bool)
    keep[bad_row] = False
    P.assert_att(got[keep], orc["oC"][keep], "sparse, rows without the invisible index")


# ---------------------------------------------------------------------------
# f4: sliding-window attention over the raw tokens
# ---------------------------------------------------------------------------
def _swa_check(p, window, eval_q=None):
    g = P.GpuProblem(p)
    inp = wl.to_numpy(p)
    o, lse = csa.swa_attend(g.layout, g.q, g.kv, window, p["scale"])
    torch.cuda.synchronize()
    assert csa.check_device_error() == 0
    ref_o, ref_l = oracle.swa_queries(inp["cu_kv"], inp["cu_q"], inp["kv"], inp["q"], window, p["scale"],
                                      eval_q=eval_q)
    got_o, got_l = P.bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)
    if eval_q is not None:
        got_o, got_l = got_o[eval_q], got_l[eval_q]
    P.assert_att(got_o, ref_o, f"swa w={window}")
    assert np.abs(got_l - ref_l).max() <= 1e-2, window


@pytest.mark.parametrize("H,d", [(8, 128), (8, 512), (64, 512), (128, 512), (64, 128)])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
@pytest.mark.parametrize("window", [1, 64, 65, 300, 1 << 20])
def test_swa_parity(H, d, mode, window):
    # decode: one query per sequence, its window split over several CTAs;
    # prefill: every position (d = 512 with 64 heads runs the persistent kernel);
    # windows of one token, one tile, one tile and one key, several tiles, all
    lengths = [1, 3, 4, 129, 1000, 5003] if mode == "decode" else [1, 130, 257, 70]
    n_q = [1] * len(lengths) if mode == "decode" else lengths
    _swa_check(problem(lengths, n_q, H=H, d=d, seed=H + d + window % 97), window)


def test_swa_bench_config_sampled():
    # the sliding-window call exactly as bench.py times it (32768-token prefill,
    # 64 heads, d = 512, window 4096, its seeded inputs), checked on the window's
    # boundary positions and a random sample
    import bench
    cfg = bench.SWA_PREFILL
    L, H, d, win = cfg["length"], cfg["H"], cfg["d"], cfg["window"]
    q = wl.randn(cfg["seed"], 4, (L, H, d), std=1.0)
    kv = wl.randn(cfg["seed"], 0, (L, d), std=1.0)
    layout = csa.Layout([L], [L], 4, 128, device="cuda")
    scale = 1.0 / float(d) ** 0.5
    o, lse = csa.swa_attend(layout, q.cuda(), kv.cuda(), win, scale)
    torch.cuda.synchronize()
    assert csa.check_device_error() == 0
    rng = np.random.default_rng(3)
    eval_q = np.unique(np.concatenate([[0, 1, 63, 64, 4094, 4095, 4096, 4097, 20000, L - 1],
                                       rng.integers(0, L, 22)])).astype(np.int64)
    ref_o, ref_l = oracle.swa_queries(np.array([0, L]), np.array([0, L]), wl.bits(kv), wl.bits(q), win, scale,
                                      eval_q=eval_q)
    P.assert_att(P.bf16_to_f64(o)[eval_q], ref_o, "swa bench config")
    assert np.abs(lse.cpu().numpy()[eval_q] - ref_l).max() <= 1e-2


@pytest.mark.parametrize("window", [4096, 700])
def test_swa_prefill_many_queries_per_cta(window):
    # 4096 + 1500 queries on at most 148 CTAs: the persistent kernel takes each
    # next query ahead of its loads; checked on every 7th query
    lengths = [4096, 1500]
    p = problem(lengths, lengths, H=64, d=512, seed=window)
    _swa_check(p, window, eval_q=np.arange(0, sum(lengths), 7))


def test_swa_chunked_and_decode_layouts_without_queries():
    # chunked and decode sequences beside one with no queries, and a call
    # with no queries at all
    p = problem([900, 64, 77, 3000], [17, 0, 1, 64], H=64, d=512, seed=5)
    _swa_check(p, 128)
    e = problem([5, 9], [0, 0], H=64, d=512, seed=6)
    g = P.GpuProblem(e)
    o, lse = csa.swa_attend(g.layout, g.q, g.kv, 8, e["scale"])
    torch.cuda.synchronize()
    assert o.numel() == 0 and csa.check_device_error() == 0


# ---------------------------------------------------------------------------
# f3: inverse-RoPE correction of the attention output
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("H,d,d_rope", [(1, 128, 8), (8, 128, 64), (8, 128, 128), (64, 512, 64), (128, 512, 512)])
@pytest.mark.parametrize("base", [10000.0, 500.0])
def test_inverse_rope_parity(H, d, d_rope, base):
    # prefill, decode, chunked and query-free sequences, and one decode query
    # at position 2^20 - 1 (angles up to 2^20 radians)
    lengths, n_q = [300, 1 << 20, 50, 9, 4000], [300, 1, 0, 9, 17]
    layout = csa.Layout(lengths, n_q, 4, 128, device="cuda")
    rng = np.random.default_rng(H + d_rope)
    x = torch.from_numpy(rng.standard_normal((layout.total_q, H, d)).astype(np.float32)).to(torch.bfloat16)
    out = x.cuda()
    csa.inverse_rope(layout, out, d_rope, base)
    torch.cuda.synchronize()
    assert csa.check_device_error() == 0
    got = P.bf16_to_f64(out)
    xin = P.bf16_to_f64(x)
    ref = oracle.inverse_rope(np.array(layout.host["cu_kv"]), np.array(layout.host["cu_q"]), xin, d_rope, base)
    assert np.array_equal(got[:, :, :d - d_rope], xin[:, :, :d - d_rope])   # untouched dims, bit for bit
    pair = np.repeat(np.maximum(np.abs(xin[:, :, d - d_rope::2]), np.abs(xin[:, :, d - d_rope + 1::2])), 2, axis=-1)
    err = np.abs(got[:, :, d - d_rope:] - ref[:, :, d - d_rope:])
    # one bf16 rounding (half a bf16 spacing) of an fp32 rotation with fp32 sine and cosine
    bound = P.half_ulp_bf16(ref[:, :, d - d_rope:]) * 1.001 + 2.0 ** -20 * pair
    assert (err <= bound).all(), (err - bound).max()


def test_inverse_rope_bench_config_sampled():
    # the call exactly as bench.py times it (a 32768-token prefill's output, 64
    # heads, d = 512, d_rope = 64, its seeded input), checked on sampled rows:
    # each sampled query as a one-query sequence ending at its position
    import bench
    cfg = bench.ROPE_CFG
    L, H, d, dr = cfg["length"], cfg["H"], cfg["d"], cfg["d_rope"]
    x = wl.randn(cfg["seed"], 0, (L, H, d), std=1.0)
    out = x.cuda()
    csa.inverse_rope(csa.Layout([L], [L], 4, 128, device="cuda"), out, dr, cfg["base"])
    torch.cuda.synchronize()
    assert csa.check_device_error() == 0
    rows = np.unique(np.concatenate([[0, 1, 2, 4095, L - 1], np.random.default_rng(4).integers(0, L, 40)]))
    cu_kv = np.concatenate([[0], np.cumsum(rows + 1)]).astype(np.int64)
    cu_q = np.arange(len(rows) + 1, dtype=np.int64)
    xin = P.bf16_to_f64(x[torch.from_numpy(rows)])
    ref = oracle.inverse_rope(cu_kv, cu_q, xin, dr, cfg["base"])
    got = P.bf16_to_f64(out[torch.from_numpy(rows).cuda()])
    pair = np.repeat(np.maximum(np.abs(xin[:, :, d - dr::2]), np.abs(xin[:, :, d - dr + 1::2])), 2, axis=-1)
    assert np.array_equal(got[:, :, :d - dr], xin[:, :, :d - dr])
    err = np.abs(got[:, :, d - dr:] - ref[:, :, d - dr:])
    bound = P.half_ulp_bf16(ref[:, :, d - dr:]) * 1.001 + 2.0 ** -20 * pair
    assert (err <= bound).all(), (err - bound).max()


# ---------------------------------------------------------------------------
# a6: the hybrid step
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["prefill_small", "decode_small", "chunked"])
def test_hybrid_small(case):
    if case == "prefill_small":
        p = problem([1, 200, 513], [1, 200, 513], H=64, d=512, HI=4, dI=64, k=32, seed=31)
    elif case == "decode_small":
        p = problem([4, 4097, 8191, 30001], [1] * 4, H=128, d=512, HI=4, dI=64, k=256, seed=32)
    else:
        p = problem([1000, 2000], [37, 300], H=64, d=512, HI=4, dI=64, k=64, seed=33)
    g = P.GpuProblem(p)
    h = g.hybrid(prebuilt=case != "prefill_small")
    rep = P.check_hybrid(p, h)
    assert rep["topk"]["equal"] >= rep["queries"] - 2
    # a second call on the same workspace gives the same answer (counters were left clean)
    o1 = h.o_csa.clone()
    h()
    torch.cuda.synchronize()
    assert torch.equal(o1, h.o_csa)


def test_hybrid_on_two_streams_at_once():
    # Two hybrid steps issued back to back on two streams (each with its own
    # buffers and workspace) run concurrently, each with the helper stream and
    # events of its own stream: both give exactly the results they give alone.
    cases = [problem([4097, 8191, 30001], [1] * 3, H=64, d=512, HI=4, dI=64, k=256, seed=35),
             problem([1000, 5000, 65536], [1] * 3, H=64, d=512, HI=4, dI=64, k=512, seed=36)]
    hs = [P.GpuProblem(p).hybrid(prebuilt=True) for p in cases]
    ref = [(h.idx.clone(), h.o_csa.clone(), h.o_hca.clone()) for h in hs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(20):
        for h, s in zip(hs, streams):
            with torch.cuda.stream(s):
                h()
    torch.cuda.synchronize()
    for h, (idx, oC, oH) in zip(hs, ref):
        assert torch.equal(h.idx, idx) and torch.equal(h.o_csa, oC) and torch.equal(h.o_hca, oH)
    assert csa.check_device_error() == 0


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("nseq", [3, 1200])
def test_hybrid_without_complete_blocks(fp8, nseq):
    # no sequence reaches one block: no CSA or HCA entry exists, every query
    # attends only the raw tokens of its own open block, and the selection is
    # empty.  1200 sequences give 2400 queries, the size at which the bf16
    # indexer takes its prefill paths (FP8 keys must still take their own).
    lengths = ([1, 2, 3] * (nseq // 3))[:nseq]
    p = problem(lengths, lengths, H=64, d=512, HI=4, dI=64, k=32, seed=70)
    g = P.GpuProblem(p)
    assert g.full.total_csa == 0 and g.full.total_hca == 0
    h = g.hybrid(prebuilt=False, fp8=fp8)
    P.check_hybrid(p, h, fp8=oracle.quantize_index_keys(wl.bits(p["kI"])) if fp8 else None)
    assert (h.idx.cpu() == -1).all()
    assert csa.check_device_error() == 0


def test_hybrid_with_query_free_sequences():
    # sequences without queries contribute entries to the packed arrays but no output rows
    p = problem([300, 1000, 77, 4099], [0, 5, 0, 1], H=64, d=512, HI=4, dI=64, k=64, seed=71)
    g = P.GpuProblem(p)
    h = g.hybrid(prebuilt=True)
    rep = P.check_hybrid(p, h)
    assert rep["queries"] == 6
    assert csa.check_device_error() == 0


def test_calls_without_queries_do_nothing():
    # total_q = 0: every call succeeds without launching and leaves its outputs alone
    p = problem([100, 37], [0, 0], H=64, d=512, HI=4, dI=64, k=16, seed=72)
    g = P.GpuProblem(p)
    assert g.layout.total_q == 0
    idx, _ = csa.lightning_index_topk(g.layout, g.qI, g.kI, 16)
    codes, scale = csa.quantize_index_keys(g.full, g.kI)
    idx8, _ = csa.lightning_index_topk_fp8(g.layout, g.qI, codes, scale, 16)
    sentinel = torch.full((g.full.total_csa, 64), 7, dtype=torch.uint8, device="cuda")
    sc = torch.full((g.full.total_csa,), 3.0, device="cuda")
    csa.quantize_closed_index_keys(g.layout, g.kI, sentinel, sc)
    h = g.hybrid(prebuilt=True)
    torch.cuda.synchronize()
    assert idx.shape[0] == 0 and idx8.shape[0] == 0 and h.o_csa.shape[0] == 0
    assert (sentinel == 7).all() and (sc == 3.0).all()
    assert csa.check_device_error() == 0


def test_hybrid_ratio_one_is_dense_causal():
    # m_C = 1, k >= L: the CSA branch is dense causal MQA (and so is HCA with m_H = 1)
    L = 300
    p = problem([L], [L], H=8, d=128, k=512, mC=1, mH=1, seed=34)
    g = P.GpuProblem(p)
    h = g.hybrid(prebuilt=False)
    q = P.bf16_to_f64(g.q).transpose(1, 0, 2)[None]
    kvf = P.bf16_to_f64(g.kv)[None, None].repeat(8, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(kvf),
                                                           torch.from_numpy(kvf), is_causal=True,
                                                           scale=p["scale"])[0].permute(1, 0, 2).numpy()
    P.assert_att(P.bf16_to_f64(h.o_csa), ref, "CSA m=1")
    P.assert_att(P.bf16_to_f64(h.o_hca), ref, "HCA m=1")


# ---------------------------------------------------------------------------
# the five workloads at full size
# ---------------------------------------------------------------------------
def sample_queries(L, n, seed):
    """Boundary-heavy query sample for a long prefill (positions t of one sequence)."""
    fixed = set(range(16)) | set(range(L - 16, L))
    fixed |= {t for t in range(512) if t % 4 in (2, 3) or t % 128 in (126, 127)}
    fixed |= set(range(4090, 4111)) | set(range(8180, 8201))
    fixed = sorted(t for t in fixed if t < L)
    rng = np.random.default_rng(seed + 100)
    rest = np.setdiff1d(np.arange(L), fixed)
    extra = rng.choice(rest, size=max(0, n - len(fixed)), replace=False)
    return np.sort(np.concatenate([fixed, extra]).astype(np.int64))[:max(n, len(fixed))]


def _workload_check(name, eval_q=None, entries="all"):
    w = wl.WORKLOADS[name]
    p = wl.make_problem(w)
    g = P.GpuProblem(p)
    h = g.hybrid(prebuilt=w.decode)
    rep = P.check_hybrid(p, h, eval_q=eval_q, check_entries=entries)
    assert csa.check_device_error() == 0
    print(name, rep)
    # swaps accepted only by the fp32 error band (a k-th score near zero) stay rare:
    # at most 1% of the queries (and 2 on a small batch)
    assert rep["topk"]["fp32tie"] <= max(2, rep["queries"] // 100), rep["topk"]
    return rep


def test_workload_prefill_4k_every_query():
    rep = _workload_check("prefill_4k")
    assert rep["queries"] == 4096


def test_workload_decode_64k_every_query():
    _workload_check("decode_64k", entries="sampled")


@pytest.mark.slow
def test_workload_ragged_decode_every_query():
    _workload_check("ragged_decode", entries="sampled")


@pytest.mark.slow
def test_workload_decode_1m_every_query():
    _workload_check("decode_1m", entries="sampled")


@pytest.mark.slow
def test_workload_prefill_128k_sampled_queries():
    eval_q = sample_queries(131072, 1024, wl.WORKLOADS["prefill_128k"].seed)
    rep = _workload_check("prefill_128k", eval_q=eval_q, entries="sampled")
    assert rep["queries"] >= 1024
