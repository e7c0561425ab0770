"""Parity helpers: run the CUDA path through the C ABI and compare it with the
fp64 oracle on the same seeded inputs.

Acceptance (per query or entry):
  * compressed entries: max abs error <= 1e-2, or half a bf16 ulp of the
    value (+1e-5) where that is larger (|e| >= 4: the bf16 cache format
    cannot hold such values to 1e-2);
  * top-k: the index sets are equal, except swaps whose oracle scores lie
    within 1e-4 relative of the oracle's k-th score; every index is visible,
    none repeats, and there are exactly min(k, n(t)) of them.  Swaps outside
    that band but inside the fp32 forward-error bound of the score the
    library computes (an fp32 sum over heads of q_h . k) are counted apart
    and reported; they arise where the k-th score sits near zero;
  * attention: max abs error <= 2e-2 and relative L2 error <= 5e-3, checked
    end-to-end where the selections agree and always on the GPU's own
    selection (the oracle re-run with the GPU's indices);
  * FP8 indexer keys: the library's E4M3 codes and fp32 scales equal the
    oracle's bit for bit; the oracle then selects on its own fp64 scores of
    the dequantised keys and the top-k rule above applies to those scores,
    with one more fp32 rounding (the scale) in the error band.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from compressed_sparse_attention_21_b300 import _lib as csa
from compressed_sparse_attention_21_b300 import workloads as wl

ENTRY_TOL = 1e-2
ATT_ABS_TOL = 2e-2
ATT_REL_TOL = 5e-3
TOPK_REL_TOL = 1e-4
U32 = 2.0 ** -24


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def half_ulp_bf16(x):
    """Half the bf16 spacing at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 8)


def entry_err(gpu, ref):
    """Max abs error of stored bf16 entries, and the worst ratio to the allowed bound.

    The bound is 1e-2, widened to half a bf16 ulp of the value (plus 1e-5 for
    the fp32 accumulation) where the storage format alone cannot meet 1e-2:
    for |e| >= 4 one bf16 rounding can move a value by up to 2^-6.
    """
    err = np.abs(gpu - ref)
    if err.size == 0:
        return 0.0, 0.0
    bound = np.maximum(ENTRY_TOL, half_ulp_bf16(np.maximum(np.abs(gpu), np.abs(ref))) + 1e-5)
    return float(err.max()), float((err / bound).max())


def entry_ulp_check(gpu, ref, abs_mix, m):
    """Entries against the arithmetic they come from: an fp32 softmax-weighted
    sum of m bf16 tokens, rounded to bf16 once.

    |gpu - ref| <= 1 bf16 ulp of ref (the final rounding, with a binade step to
    spare) + (m + 4) * 2^-23 * sum_t w_t |c_t| (the fp32 exponentials, the
    weighted sum and the normalisation).  abs_mix is the oracle's entry of the
    same block on |c|, i.e. sum_t w_t |c_t|.  A dropped or doubled token, a
    wrong weight or a misplaced block moves an entry far beyond this bound.
    Returns the worst ratio of error to bound."""
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
    bound = ulp + (m + 4) * 2.0 ** -23 * abs_mix + 1e-30
    err = np.abs(gpu - ref)
    return float((err / bound).max()) if err.size else 0.0


def abs_bits(bits):
    """bf16 bit patterns of |x| (sign bit cleared)."""
    return np.ascontiguousarray(bits, np.uint16) & np.uint16(0x7FFF)


class GpuProblem:
    """Device copies of a seeded problem and the two layouts it needs."""

    def __init__(self, p, device="cuda"):
        self.p = p
        self.device = device
        dv = lambda t: t.to(device, non_blocking=False).contiguous()
        self.kv, self.gate, self.qI, self.kI, self.q = (dv(p[k]) for k in ("kv", "gate", "qI", "kI", "q"))
        self.layout = csa.Layout(p["lengths"], p["n_q"], p["mC"], p["mH"], device=device)
        self.full = csa.Layout(p["lengths"], p["lengths"], p["mC"], p["mH"], device=device)

    def build_caches(self):
        """Compress every complete block (a prefill-shaped call) into fresh caches."""
        d = self.p["d"]
        csa_cache = torch.zeros((self.full.total_csa, d), dtype=torch.bfloat16, device=self.device)
        hca_cache = torch.zeros((self.full.total_hca, d), dtype=torch.bfloat16, device=self.device)
        if self.full.total_csa:
            csa.csa_compress(self.full, self.kv, self.gate, csa_cache)
        if self.full.total_hca:
            csa.hca_compress(self.full, self.kv, self.gate, hca_cache)
        return csa_cache, hca_cache

    def hybrid(self, prebuilt=True, skip_compress=False, with_scores=True, fp8=False):
        caches = self.build_caches() if prebuilt else (None, None)
        k_idx_fp8 = csa.quantize_index_keys(self.full, self.kI) if fp8 else None
        h = csa.Hybrid(self.layout, self.kv, self.gate, self.qI, self.kI, self.q, self.p["top_k"],
                       self.p["scale"], csa_cache=caches[0], hca_cache=caches[1],
                       skip_compress=skip_compress, with_scores=with_scores, k_idx_fp8=k_idx_fp8)
        h()
        torch.cuda.synchronize()
        return h


def oracle_inputs(p):
    return wl.to_numpy(p)


def score_abs_bound(qI_bits, kI_bits, js, dequant=None):
    """sum_h sum_i |q_hi k_ji| for the listed entries (the fp32 error scale)."""
    q = np.abs(oracle_f64(qI_bits)).sum(0)                 # [dI]
    k = np.abs(dequant(js) if dequant is not None else oracle_f64(kI_bits[js]))   # [len(js), dI]
    return k @ q


_E4M3 = None


def e4m3_table():
    """Value of every E4M3 code, from the oracle's decoder (fp64, exact)."""
    global _E4M3
    if _E4M3 is None:
        _E4M3 = np.array([oracle.e4m3_decode(c) for c in range(256)], np.float64)
    return _E4M3


def fp8_dequant(codes, scale):
    """js -> scale_j * e4m3(codes_j) for rows js of one sequence's FP8 keys."""
    tab = e4m3_table()
    return lambda js: scale[js].astype(np.float64)[:, None] * tab[codes[js]]


def oracle_f64(bits):
    b = np.ascontiguousarray(bits, np.uint16)
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()


def check_topk_row(gpu_row, orc_row, scores, n_vis, k, qI_bits, kI_seq_bits, dequant=None):
    """Returns ('equal'|'tie'|'fp32tie', n_swaps); raises AssertionError on a real mismatch.

    dequant: for FP8 keys, a callable js -> [len(js), dI] fp64 dequantised keys
    (then kI_seq_bits is unused); the fp32 score has one more rounding (the scale)."""
    g = gpu_row[gpu_row >= 0]
    o = orc_row[orc_row >= 0]
    want = min(k, n_vis)
    assert len(g) == want, f"{len(g)} indices, expected {want}"
    assert (gpu_row[want:] == -1).all(), "padding must be -1"
    assert len(np.unique(g)) == len(g), "duplicate index"
    assert (g >= 0).all() and (g < n_vis).all(), "index not visible"
    assert (np.diff(g) > 0).all(), "indices must ascend"
    gs, os_ = set(g.tolist()), set(o.tolist())
    if gs == os_:
        return "equal", 0
    diff = np.array(sorted(gs ^ os_), dtype=np.int64)
    kth = scores[o].min()
    band = TOPK_REL_TOL * abs(kth)
    gap = np.abs(scores[diff] - kth)
    if (gap <= band).all():
        return "tie", len(diff) // 2
    # fp32 forward-error band of the library's score (head sum, then a dI-term dot)
    HI, dI = qI_bits.shape
    n_terms = HI + dI + 2 + (1 if dequant is not None else 0)
    gam = n_terms * U32 / (1 - n_terms * U32)
    j_k = int(o[np.argmin(scores[o])])
    bnd = gam * score_abs_bound(qI_bits, kI_seq_bits, np.concatenate([diff, [j_k]]), dequant)
    tol = bnd[:-1] + bnd[-1]
    bad = gap > np.maximum(band, tol)
    assert not bad.any(), \
        f"top-k mismatch beyond tie tolerance: gaps {gap[bad][:5]} (band {band}, fp32 {tol[bad][:5]})"
    return "fp32tie", len(diff) // 2


def att_err(gpu, ref):
    g = gpu.astype(np.float64)
    diff = g - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300)) if diff.size else 0.0
    return max_abs, rel


def assert_att(gpu, ref, what):
    m, r = att_err(gpu, ref)
    assert m <= ATT_ABS_TOL and r <= ATT_REL_TOL, f"{what}: max abs {m:.3g}, rel L2 {r:.3g}"
    return m, r


def check_hybrid(p, h: "csa.Hybrid", eval_q=None, check_entries="all", entry_sample=None, seed=0,
                 fp8=None):
    """Compare a finished hybrid run with the oracle on `eval_q` (default: all queries).

    fp8: the oracle's (codes, scales) of the indexer keys when the run used the
    FP8 indexer; the oracle then selects on its FP8 scores.
    Returns a report dict (errors, tie counts)."""
    inp = oracle_inputs(p)
    total_q = int(inp["cu_q"][-1])
    eval_q = np.arange(total_q, dtype=np.int64) if eval_q is None else np.asarray(eval_q, np.int64)
    rep = {"queries": len(eval_q)}

    # --- compressed entries (caches) ---
    gpu_hca = h.hca_cache.cpu()
    if check_entries == "all":
        gpu_csa = h.csa_cache.cpu()
        orc_csa = oracle.compress_packed(inp["cu_kv"], inp["cu_csa"], inp["kv"], inp["gate"], p["mC"])
        e_csa, r_csa = entry_err(bf16_to_f64(gpu_csa), orc_csa)
    else:
        rng = np.random.default_rng(seed)
        n_csa = h.csa_cache.shape[0]
        ent = np.unique(np.concatenate([rng.integers(0, n_csa, entry_sample or 4096), [0, n_csa - 1]]))
        orc = oracle.compress_selected(inp["cu_kv"], inp["cu_csa"], inp["kv"], inp["gate"], p["mC"], ent)
        sel = h.csa_cache[torch.from_numpy(ent).to(h.csa_cache.device)].cpu()
        e_csa, r_csa = entry_err(bf16_to_f64(sel), orc)
    orc_hca = oracle.compress_packed(inp["cu_kv"], inp["cu_hca"], inp["kv"], inp["gate"], p["mH"])
    e_hca, r_hca = entry_err(bf16_to_f64(gpu_hca), orc_hca)
    assert r_csa <= 1.0, f"CSA entries max abs {e_csa}"
    assert r_hca <= 1.0, f"HCA entries max abs {e_hca}"
    rep["entry_err_csa"], rep["entry_err_hca"] = e_csa, e_hca

    # --- oracle on its own selection ---
    cu_kv, cu_q, cu_csa = inp["cu_kv"], inp["cu_q"], inp["cu_csa"]

    def visible(qi):
        b = int(np.searchsorted(cu_q, qi, side="right") - 1)
        L = cu_kv[b + 1] - cu_kv[b]
        t = L - (cu_q[b + 1] - cu_q[b]) + (qi - cu_q[b])
        return b, int((t + 1) // p["mC"])

    def fp8_row(qi):
        b, n_vis = visible(qi)
        codes, scale = fp8[0][cu_csa[b]:cu_csa[b] + n_vis], fp8[1][cu_csa[b]:cu_csa[b] + n_vis]
        s = oracle.index_scores_fp8(inp["qI"][qi], codes, scale) if n_vis else np.zeros(0)
        return s, fp8_dequant(codes, scale)

    if fp8 is None:
        orc = oracle.hybrid_queries(inp, eval_q=eval_q, hca_entries=orc_hca)
    else:
        orc_idx = np.stack([oracle.topk(fp8_row(qi)[0], p["top_k"]) for qi in eval_q])
        orc = oracle.hybrid_queries(inp, eval_q=eval_q, given_idx=orc_idx, hca_entries=orc_hca)
        orc["idx"] = orc_idx
    rows = torch.from_numpy(eval_q).to(h.idx.device)
    gpu_idx = h.idx[rows].cpu().numpy()
    gpu_oC = bf16_to_f64(h.o_csa[rows])
    gpu_oH = bf16_to_f64(h.o_hca[rows])
    gpu_lC = h.lse_csa[rows].cpu().numpy()
    gpu_lH = h.lse_hca[rows].cpu().numpy()

    # --- top-k ---
    kinds = {"equal": 0, "tie": 0, "fp32tie": 0}
    swapped = []
    for r, qi in enumerate(eval_q):
        b, n_vis = visible(qi)
        kI_seq = inp["kI"][cu_csa[b]:cu_csa[b] + n_vis]
        if fp8 is None:
            scores, dq = (oracle.index_scores(inp["qI"][qi], kI_seq) if n_vis else np.zeros(0)), None
        else:
            scores, dq = fp8_row(qi)
        kind, _ = check_topk_row(gpu_idx[r], orc["idx"][r], scores, n_vis, p["top_k"], inp["qI"][qi], kI_seq,
                                 dq)
        kinds[kind] += 1
        if kind != "equal":
            swapped.append(r)
    rep["topk"] = kinds

    # --- attention: HCA end-to-end; CSA end-to-end where selections agree ---
    rep["hca_abs"], rep["hca_rel"] = assert_att(gpu_oH, orc["oH"], "HCA output")
    assert np.abs(gpu_lH - orc["lseH"]).max() <= 1e-2, "HCA lse"
    same = np.setdiff1d(np.arange(len(eval_q)), swapped)
    if len(same):
        rep["csa_abs"], rep["csa_rel"] = assert_att(gpu_oC[same], orc["oC"][same], "CSA output (end-to-end)")
        assert np.abs(gpu_lC[same] - orc["lseC"][same]).max() <= 1e-2, "CSA lse"
    # --- CSA attention on the GPU's own selection (every query) ---
    orc_g = oracle.hybrid_queries(inp, eval_q=eval_q, given_idx=gpu_idx, do_hca=False)
    rep["csa_given_abs"], rep["csa_given_rel"] = assert_att(gpu_oC, orc_g["oC"], "CSA output (GPU selection)")
    assert np.abs(gpu_lC - orc_g["lseC"]).max() <= 1e-2, "CSA lse (GPU selection)"
    return rep
