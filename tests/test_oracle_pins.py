"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a closed form, a textbook/library
routine, brute force on a tiny input, or an invariant that the definitions
of the CSA/HCA path fix (DeepSeek-V4 core architecture, §2.2 CSA steps 1-3
and §2.3 HCA), so that a dropped term, a wrong sign, an off-by-one in the
block/visibility arithmetic or a transposed operand fails at least one.
"""
import math
import os

import numpy as np
import pytest
import torch

from compressed_sparse_attention_21_b300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf(x):
    """float array -> bf16 bit patterns (exact when x is bf16-representable)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return wl.bits(t)


def f(bits):
    """bf16 bit patterns -> float64 values (exact)."""
    b = np.ascontiguousarray(bits, np.uint16)
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()


def tiny_problem(L, d=8, H=2, HI=2, dI=4, mC=4, mH=128, k=4, seed=0, n_q=None, gate_std=1.0):
    w = wl.Workload("tiny", 1, [L], False, H=H, d=d, HI=HI, dI=dI, top_k=k, mC=mC, mH=mH,
                    gate_std=gate_std, seed=seed)
    return wl.to_numpy(wl.make_problem(w, n_q=n_q))


def sdpa_causal(q_bits, kv_bits, scale):
    """Dense causal MQA through torch's library routine, fp64 on the CPU.

    q: [L, H, d]; kv: [L, d] shared by all heads (key = value)."""
    q = torch.from_numpy(f(q_bits)).permute(1, 0, 2)[None]          # [1, H, L, d]
    kv = torch.from_numpy(f(kv_bits))[None, None].expand(1, q.shape[1], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(q, kv, kv, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()                             # [L, H, d]


# ----------------------------------------------------------------------------
# compression (§2.2 step 1; §2.3)
# ----------------------------------------------------------------------------

def test_compress_closed_form_weights(orc):
    # logits 0, ln2, ln3, ln4 -> weights 1/10, 2/10, 3/10, 4/10 exactly
    z = np.log(np.array([1.0, 2.0, 3.0, 4.0])).astype(np.float32)
    c = np.array([[1, -2], [0.5, 4], [-1, 8], [2, 0.25]], np.float32)
    e = orc.compress(bf(c), z, 4)
    zf = z.astype(np.float64)
    w = np.exp(zf) / np.exp(zf).sum()          # the fp32-rounded logits, exactly
    assert np.allclose(w, [0.1, 0.2, 0.3, 0.4], atol=1e-7)
    expect = (w[:, None] * c.astype(np.float64)).sum(0)
    assert np.allclose(e[0], expect, rtol=0, atol=1e-15)


def test_compress_uniform_logits_is_mean_pooling(orc):
    rng = np.random.default_rng(1)
    L, d, m = 64, 16, 4
    c = bf(rng.standard_normal((L, d)))
    z = np.repeat(rng.standard_normal(L // m), m).astype(np.float32)   # constant per block
    e = orc.compress(c, z, m)
    mean = f(c).reshape(L // m, m, d).mean(1)
    assert np.allclose(e, mean, rtol=0, atol=1e-14)


def test_compress_block_alignment_and_trailing_block(orc):
    # c_t = t in every channel, uniform logits: entry j = mean(4j .. 4j+3) = 4j + 1.5
    L, d = 10, 3
    c = bf(np.repeat(np.arange(L, dtype=np.float32)[:, None], d, 1))
    e = orc.compress(c, np.zeros(L, np.float32), 4)
    assert e.shape == (2, d)                         # tokens 8, 9 form no entry
    assert np.array_equal(e[:, 0], [1.5, 5.5])


def test_compress_invariances(orc):
    rng = np.random.default_rng(2)
    L, d, m = 32, 8, 4
    c = bf(rng.standard_normal((L, d)))
    z = rng.standard_normal(L).astype(np.float32)
    e = orc.compress(c, z, m)
    # shift all logits of a block by a constant (exactly representable shift)
    e2 = orc.compress(c, (z + np.float32(3.0)).astype(np.float32), m)
    assert np.allclose(e, e2, atol=1e-12)
    # permute (c, z) pairs inside each block
    perm = np.concatenate([j * m + rng.permutation(m) for j in range(L // m)])
    e3 = orc.compress(c[perm], z[perm], m)
    assert np.allclose(e, e3, atol=1e-14)


def test_compress_dominant_logit_and_ratio_one(orc):
    rng = np.random.default_rng(3)
    L, d = 8, 5
    c = bf(rng.standard_normal((L, d)))
    z = np.zeros(L, np.float32)
    z[2] = 50.0
    z[5] = 50.0
    e = orc.compress(c, z, 4)
    # the other weights are exp(-50) ~ 2e-22
    assert np.allclose(e[0], f(c)[2], rtol=0, atol=1e-19)
    assert np.allclose(e[1], f(c)[5], rtol=0, atol=1e-19)
    assert np.array_equal(orc.compress(c, rng.standard_normal(L).astype(np.float32), 1), f(c))


def test_compress_hca_ratio(orc):
    rng = np.random.default_rng(4)
    L, d = 300, 4
    c = bf(rng.standard_normal((L, d)))
    z = rng.standard_normal(L).astype(np.float32)
    e = orc.compress(c, z, 128)
    assert e.shape == (2, d)
    # brute force for block 1, straight from the definition in plain Python
    zs = [float(v) for v in z[128:256]]
    mx = max(zs)
    ws = [math.exp(v - mx) for v in zs]
    tot = sum(ws)
    cf = f(c)
    for x in range(d):
        ref = sum(ws[i] / tot * cf[128 + i, x] for i in range(128))
        assert abs(e[1, x] - ref) < 1e-13


# ----------------------------------------------------------------------------
# indexer and top-k (§2.2 step 2)
# ----------------------------------------------------------------------------

def test_index_scores_brute_force(orc):
    rng = np.random.default_rng(5)
    HI, dI, n = 3, 5, 7
    qI = bf(rng.standard_normal((HI, dI)))
    kI = bf(rng.standard_normal((n, dI)))
    s = orc.index_scores(qI, kI)
    qf, kf = f(qI), f(kI)
    for j in range(n):
        ref = 0.0
        for h in range(HI):
            for i in range(dI):
                ref += qf[h, i] * kf[j, i]
        assert abs(s[j] - ref) < 1e-12


def test_index_scores_single_head_is_dot_and_head_sum(orc):
    rng = np.random.default_rng(6)
    dI, n = 64, 50
    q1 = bf(rng.standard_normal((1, dI)))
    kI = bf(rng.standard_normal((n, dI)))
    assert np.allclose(orc.index_scores(q1, kI), f(kI) @ f(q1)[0], rtol=0, atol=1e-12)
    q4 = bf(rng.standard_normal((4, dI)))
    # the head sum can be taken first: sum_h q_h . k = (sum_h q_h) . k
    assert np.allclose(orc.index_scores(q4, kI), f(kI) @ f(q4).sum(0), rtol=0, atol=1e-11)


def test_topk_brute_force_with_ties(orc):
    rng = np.random.default_rng(7)
    for trial in range(50):
        n = int(rng.integers(0, 40))
        k = int(rng.integers(1, 20))
        s = rng.integers(-3, 4, n).astype(np.float64)          # many ties
        got = orc.topk(s, k)
        order = sorted(range(n), key=lambda j: (-s[j], j))[:k]
        want = sorted(order) + [-1] * (k - len(order))
        assert list(got) == want, (trial, s, k)


def test_topk_all_equal_takes_lowest_indices(orc):
    got = orc.topk(np.zeros(100), 10)
    assert list(got) == list(range(10))


# ----------------------------------------------------------------------------
# attention (§2.2 step 3; §2.3)
# ----------------------------------------------------------------------------

def test_attend_single_key(orc):
    rng = np.random.default_rng(8)
    H, d = 3, 6
    q = bf(rng.standard_normal((H, d)))
    key = rng.standard_normal((1, d))
    o, lse = orc.attend(q, key, 0.5)
    assert np.allclose(o, np.repeat(key, H, 0), atol=1e-15)
    assert np.allclose(lse, 0.5 * f(q) @ key[0], atol=1e-14)


def test_attend_matches_library_sdpa(orc):
    rng = np.random.default_rng(9)
    H, d, n = 4, 16, 37
    q = bf(rng.standard_normal((H, d)))
    keys = rng.standard_normal((n, d))
    o, lse = orc.attend(q, keys, 1 / math.sqrt(d))
    qt = torch.from_numpy(f(q))[None, :, None, :]            # [1, H, 1, d]
    kt = torch.from_numpy(keys)[None, None].expand(1, H, n, d)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, kt, scale=1 / math.sqrt(d))
    assert np.allclose(o, ref[0, :, 0].numpy(), atol=1e-13)
    logits = (torch.from_numpy(f(q)) @ torch.from_numpy(keys).T) / math.sqrt(d)
    assert np.allclose(lse, torch.logsumexp(logits, -1).numpy(), atol=1e-13)


def test_csa_ratio_one_full_topk_is_dense_causal_mqa(orc):
    # m_C = 1 and k >= n: every token is its own entry and all are selected
    L = 40
    p = tiny_problem(L, d=16, H=3, mC=1, k=64, seed=10)
    out = orc.hybrid_queries(p, do_hca=False)
    ref = sdpa_causal(p["q"], p["kv"], p["scale"])
    assert np.allclose(out["oC"], ref, atol=1e-12)
    assert (out["idx"][:, :L] >= -1).all()


def test_hca_short_sequence_is_dense_causal_mqa(orc):
    L = 100                                        # < 128: no HCA entry, only raw tail
    p = tiny_problem(L, d=16, H=2, seed=11)
    out = orc.hybrid_queries(p, do_csa=False)
    assert np.allclose(out["oH"], sdpa_causal(p["q"], p["kv"], p["scale"]), atol=1e-12)


def test_hca_ratio_one_is_dense_causal_mqa(orc):
    L = 33
    p = tiny_problem(L, d=8, H=2, mH=1, seed=12)
    out = orc.hybrid_queries(p, do_csa=False)
    assert np.allclose(out["oH"], sdpa_causal(p["q"], p["kv"], p["scale"]), atol=1e-12)


def test_outputs_in_convex_hull_of_keys(orc):
    L = 300
    p = tiny_problem(L, d=8, H=4, k=8, seed=13)
    out = orc.hybrid_queries(p)
    kvf = f(p["kv"])
    lo, hi = kvf.min(0) - 1e-12, kvf.max(0) + 1e-12   # entries are convex mixes of tokens
    assert (out["oC"] >= lo).all() and (out["oC"] <= hi).all()
    assert (out["oH"] >= lo).all() and (out["oH"] <= hi).all()


def test_key_counts_via_lse(orc):
    # q = 0 makes every logit 0, so lse = log(number of keys):
    # CSA: min(k, n_C) + r_C, HCA: n_H + r_H  (visibility and own-block tail)
    L, k = 300, 16
    p = tiny_problem(L, d=4, H=1, k=k, seed=14)
    p["q"] = np.zeros_like(p["q"])
    out = orc.hybrid_queries(p)
    for t in range(L):
        nC, rC = (t + 1) // 4, (t + 1) % 4
        nH, rH = (t + 1) // 128, (t + 1) % 128
        assert abs(out["lseC"][t, 0] - math.log(min(k, nC) + rC)) < 1e-12, t
        assert abs(out["lseH"][t, 0] - math.log(nH + rH)) < 1e-12, t
        assert (out["idx"][t] >= 0).sum() == min(k, nC)


def test_visibility_boundary(orc):
    # entry j = 5 gets a huge indexer score; t = 4j+2 must not see it, t = 4j+3 must.
    j = 5
    p = tiny_problem(64, d=4, H=1, HI=1, dI=4, k=2, seed=15)
    p["qI"] = bf(np.ones((64, 1, 4)))
    kI = np.zeros((16, 4), np.float32)
    kI[j] = 100.0
    p["kI"] = bf(kI)
    out = orc.hybrid_queries(p, eval_q=np.array([4 * j + 2, 4 * j + 3]), do_hca=False)
    assert j not in out["idx"][0] and j in out["idx"][1]


def test_causality_future_perturbation(orc):
    L, t = 260, 150
    p = tiny_problem(L, d=8, H=2, k=8, seed=16)
    base = orc.hybrid_queries(p, eval_q=np.array([t]))
    q2 = dict(p)
    rng = np.random.default_rng(17)
    kv = p["kv"].copy()
    kv[t + 1:] = bf(rng.standard_normal((L - t - 1, 8)))
    gate = p["gate"].copy()
    gate[t + 1:] = 9.0
    kI = p["kI"].copy()
    kI[(t + 1) // 4:] = bf(100 * np.ones((kI.shape[0] - (t + 1) // 4, kI.shape[1])))
    q = p["q"].copy()
    q[t + 1:] = 0
    q2.update(kv=kv, gate=gate, kI=kI, q=q)
    pert = orc.hybrid_queries(q2, eval_q=np.array([t]))
    for key in ("idx", "oC", "lseC", "oH", "lseH"):
        assert np.array_equal(base[key], pert[key]), key


def test_given_idx_reproduces_own_selection(orc):
    p = tiny_problem(200, d=8, H=2, k=8, seed=18)
    own = orc.hybrid_queries(p, do_hca=False)
    again = orc.hybrid_queries(p, given_idx=own["idx"], do_hca=False)
    assert np.array_equal(own["oC"], again["oC"])


def test_structural_counts_golden(orc):
    """Golden structural constants printed on the pages (see the fixture's citations)."""
    rows = {}
    with open(os.path.join(GOLDEN, "structural_counts.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split("=")
                rows[key.strip()] = int(val)
    L = rows["context_tokens"]
    # one token dimension and one head keep this cheap; q = 0 -> lse = log(#keys)
    inp = dict(cu_kv=np.array([0, L]), cu_q=np.array([0, 1]),
               cu_csa=np.array([0, L // 4]), cu_hca=np.array([0, L // 128]),
               kv=bf(np.ones((L, 1))), gate=np.zeros(L, np.float32),
               qI=bf(np.ones((1, 1, 1))), kI=bf(np.ones((L // 4, 1))),
               q=bf(np.zeros((1, 1, 1))), mC=4, mH=128, top_k=L, scale=1.0)
    out = orc.hybrid_queries(inp)
    n_csa = int((out["idx"][0] >= 0).sum())
    assert n_csa == rows["csa_entries"]
    assert abs(out["lseH"][0, 0] - math.log(rows["hca_entries"])) < 1e-9
    assert rows["csa_entries"] * 4 == L and rows["hca_entries"] * 128 == L


# ----------------------------------------------------------------------------
# FP8 indexer keys (DeepSeek-V4 core architecture, §9 key innovations, row 5:
# the indexer's QK product is quantised).  The E4M3 format's definition and
# torch's float8_e4m3fn conversion pin the codec; closed forms pin the scaling.
# ----------------------------------------------------------------------------

def test_e4m3_decode_matches_torch_for_every_code(orc):
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([orc.e4m3_decode(c) for c in range(256)])
    assert np.array_equal(got, ref, equal_nan=True)
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6
    assert np.signbit(got[0x80]) and got[0x80] == 0.0


def test_e4m3_encode_round_trip_and_saturation(orc):
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert orc.e4m3_encode(orc.e4m3_decode(c)) == c, hex(c)
    assert orc.e4m3_encode(449.0) == 0x7E and orc.e4m3_encode(1e30) == 0x7E
    assert orc.e4m3_encode(-470.0) == 0xFE
    assert orc.e4m3_encode(-1e-9) == 0x80 and orc.e4m3_encode(1e-9) == 0x00


def test_e4m3_encode_ties_to_even(orc):
    # midpoints between neighbouring codes go to the code with an even mantissa
    assert orc.e4m3_encode(1.0625) == 0x38           # 1.0 (m=0) | 1.125 (m=1)
    assert orc.e4m3_encode(1.1875) == 0x3A           # 1.125 (m=1) | 1.25 (m=2)
    assert orc.e4m3_encode(17.0) == orc.e4m3_encode(16.0)
    assert orc.e4m3_encode(2.0 ** -10) == 0x00       # half the smallest subnormal
    assert orc.e4m3_encode(3 * 2.0 ** -10) == 0x02   # subnormal m=1 | m=2
    assert orc.e4m3_encode(-1.0625) == 0xB8
    # 0.25 ulp off a midpoint goes to the nearer side
    assert orc.e4m3_encode(1.0625 + 2.0 ** -6) == 0x39


def test_e4m3_encode_matches_torch_on_random_and_midpoint_values(orc):
    rng = np.random.default_rng(17)
    tab = np.array([orc.e4m3_decode(c) for c in range(0x7F)])
    mids = (tab[:-1] + tab[1:]) / 2
    x = np.concatenate([rng.uniform(-448, 448, 4000), rng.standard_normal(4000) * 0.01,
                        mids, -mids, tab, -tab]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in x], np.uint8)
    bad = np.flatnonzero(got != ref)
    assert len(bad) == 0, (x[bad[:4]], got[bad[:4]], ref[bad[:4]])


def test_quantize_index_keys_hand_example(orc):
    k = bf([[0.5, -1.0, 0.25, 0.0], [0.0, 0.0, 0.0, 0.0], [448.0, 17.0, -1.0625, 2.0 ** -10]])
    codes, scale = orc.quantize_index_keys(k)
    # row 0: a = 1, inv = 448: 224 = 1.75*2^7, -448, 112 = 1.75*2^6, 0
    assert codes[0].tolist() == [0x76, 0xFE, 0x6E, 0x00]
    assert scale[0] == np.float32(1.0) / np.float32(448.0)
    assert codes[1].tolist() == [0, 0, 0, 0] and scale[1] == 0.0
    # row 2: a = 448, inv = 1, scale = 1: the values themselves, ties to even
    assert codes[2].tolist() == [0x7E, orc.e4m3_encode(16.0), 0xB8, 0x00] and scale[2] == 1.0


def test_quantize_index_keys_matches_fp32_torch_route(orc):
    # the same steps through torch's float32 arithmetic and its E4M3 conversion
    rng = np.random.default_rng(18)
    for dI in (32, 64, 128):
        kb = bf(rng.standard_normal((300, dI)) * rng.uniform(1e-3, 1e3, (300, 1)))
        codes, scale = orc.quantize_index_keys(kb)
        kf = torch.from_numpy(f(kb)).float()
        a = kf.abs().amax(1)
        inv = torch.tensor(448.0, dtype=torch.float32) / a
        ref = (kf * inv[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes, ref)
        assert np.array_equal(scale, (a / torch.tensor(448.0, dtype=torch.float32)).numpy())


def test_quantize_dequantize_error_bound(orc):
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 in the normal range,
    # absolute error <= 2^-10 * scale in the subnormal range; the row max survives
    rng = np.random.default_rng(19)
    kb = bf(rng.standard_normal((200, 64)))
    codes, scale = orc.quantize_index_keys(kb)
    tab = np.array([orc.e4m3_decode(c) for c in range(256)])
    kq = scale.astype(np.float64)[:, None] * tab[codes]
    kf = f(kb)
    err = np.abs(kq - kf)
    bound = np.maximum(2.0 ** -4 * np.abs(kf), 2.0 ** -10 * scale[:, None]) * (1 + 2.0 ** -20)
    assert (err <= bound).all()
    amax = np.abs(kf).max(1)
    assert np.allclose(np.abs(kq).max(1), amax, rtol=2.0 ** -22, atol=0)


def test_index_scores_fp8_is_dot_with_dequantised_keys(orc):
    rng = np.random.default_rng(20)
    HI, dI, n = 3, 32, 40
    qI = bf(rng.standard_normal((HI, dI)))
    kb = bf(rng.standard_normal((n, dI)))
    codes, scale = orc.quantize_index_keys(kb)
    tab = np.array([orc.e4m3_decode(c) for c in range(256)])
    kq = scale.astype(np.float64)[:, None] * tab[codes]
    s = orc.index_scores_fp8(qI, codes, scale)
    assert np.allclose(s, kq @ f(qI).sum(0), rtol=1e-12, atol=1e-12)
    # keys that E4M3 holds exactly with scale 1 (row max 448) score as the bf16 indexer does
    kx = bf(np.concatenate([np.full((n, 1), 448.0), rng.integers(-8, 9, (n, dI - 1)) / 4.0], 1))
    c2, s2 = orc.quantize_index_keys(kx)
    assert (s2 == 1.0).all()
    assert np.array_equal(orc.index_scores_fp8(qI, c2, s2), orc.index_scores(qI, kx))


def test_quantize_is_exactly_invariant_to_power_of_two_row_scaling(orc):
    # k -> 2^e k (exact in bf16) leaves a * inv unchanged in fp32, so the codes
    # stay and the scale moves by exactly 2^e: catches a wrong amax, a wrong row
    # or a scale formula that is not a / 448
    rng = np.random.default_rng(21)
    kb = bf(rng.standard_normal((50, 64)))
    c0, s0 = orc.quantize_index_keys(kb)
    for e in (-20, -3, 1, 7, 30):
        c1, s1 = orc.quantize_index_keys(bf(f(kb) * 2.0 ** e))
        assert np.array_equal(c1, c0)
        assert np.array_equal(s1, (s0.astype(np.float64) * 2.0 ** e).astype(np.float32))


def test_quantize_sign_flip_flips_only_sign_bits(orc):
    rng = np.random.default_rng(22)
    kb = bf(rng.standard_normal((40, 32)))
    c0, s0 = orc.quantize_index_keys(kb)
    c1, s1 = orc.quantize_index_keys(bf(-f(kb)))
    assert np.array_equal(c1, c0 ^ 0x80) and np.array_equal(s1, s0)


def test_e4m3_encode_is_monotone(orc):
    rng = np.random.default_rng(23)
    x = np.sort(np.concatenate([rng.uniform(-500, 500, 3000), rng.standard_normal(3000) * 1e-2]))
    tab = np.array([orc.e4m3_decode(c) for c in range(256)])
    vals = np.array([tab[orc.e4m3_encode(float(v))] for v in x])
    assert (np.diff(vals) >= 0).all()
    # and the nearest: no finite code lies strictly closer to x
    fin = tab[np.isfinite(tab)]
    for v, q in zip(x[::50], vals[::50]):
        assert abs(q - v) <= np.min(np.abs(fin - np.clip(v, -448, 448))) + abs(v - np.clip(v, -448, 448)) + 1e-12


def test_attention_ignores_the_order_of_the_selected_indices(orc):
    p = tiny_problem(64, d=8, H=2, HI=2, dI=4, mC=4, k=8, seed=24, n_q=[3])
    base = orc.hybrid_queries(p, do_hca=False)
    rng = np.random.default_rng(24)
    perm = np.stack([rng.permutation(row) for row in base["idx"]])
    again = orc.hybrid_queries(p, given_idx=perm, do_hca=False)
    assert np.allclose(again["oC"], base["oC"], rtol=0, atol=1e-12)
    assert np.allclose(again["lseC"], base["lseC"], rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# packed batches and query positions (§2.2 step 1: one entry per m tokens of a
# sequence; queries are a sequence's last n_q positions)
# ----------------------------------------------------------------------------

def packed_problem(lengths, n_q, d=8, H=2, HI=2, dI=4, mC=4, mH=16, k=5, seed=0):
    w = wl.Workload("packed", len(lengths), list(lengths), False, H=H, d=d, HI=HI, dI=dI, top_k=k, mC=mC,
                    mH=mH, seed=seed)
    return wl.to_numpy(wl.make_problem(w, n_q=n_q))


def one_sequence(p, b):
    """Sequence b of a packed problem as a batch of one (every offset 0)."""
    cu = {key: p[key] for key in ("cu_kv", "cu_q", "cu_csa", "cu_hca")}
    kv0, kv1 = cu["cu_kv"][b], cu["cu_kv"][b + 1]
    q0, q1 = cu["cu_q"][b], cu["cu_q"][b + 1]
    c0, c1 = cu["cu_csa"][b], cu["cu_csa"][b + 1]
    h0, h1 = cu["cu_hca"][b], cu["cu_hca"][b + 1]
    s = dict(p)
    s.update(cu_kv=np.array([0, kv1 - kv0]), cu_q=np.array([0, q1 - q0]), cu_csa=np.array([0, c1 - c0]),
             cu_hca=np.array([0, h1 - h0]), kv=p["kv"][kv0:kv1], gate=p["gate"][kv0:kv1], qI=p["qI"][q0:q1],
             q=p["q"][q0:q1], kI=p["kI"][c0:c1])
    return s


def test_packed_batch_equals_each_sequence_alone(orc):
    # Prefill, decode and chunked sequences packed together (and one without
    # queries): every query's selection, outputs and LSEs equal those of its
    # sequence run alone, bit for bit.  A wrong cu_kv / cu_csa / cu_hca / cu_q
    # offset, or a query assigned to the wrong sequence, reads another
    # sequence's tokens, entries or indexer keys and fails here.
    lengths = [70, 1, 45, 130, 9, 64]
    n_q = [70, 1, 0, 12, 9, 1]
    p = packed_problem(lengths, n_q, seed=40)
    packed = orc.hybrid_queries(p)
    row = 0
    for b, nq in enumerate(n_q):
        if nq == 0:
            continue
        alone = orc.hybrid_queries(one_sequence(p, b))
        for key in ("idx", "oC", "lseC", "oH", "lseH"):
            assert np.array_equal(packed[key][row:row + nq], alone[key]), (b, key)
        row += nq
    assert row == packed["idx"].shape[0]


def test_decode_and_chunked_queries_equal_the_same_positions_of_a_prefill(orc):
    # The queries of a sequence are its last n_q positions: t = L - n_q + i.
    # The same tokens with n_q = L (prefill), n_q = 1 (decode) and n_q = 7
    # (chunked) give, for each position, the same result bit for bit, when the
    # query rows of the shorter layouts are the prefill's rows of those positions.
    L = 203
    full = packed_problem([L], [L], seed=41)
    pre = orc.hybrid_queries(full)
    for nq in (1, 7, 64):
        s = dict(full)
        s["cu_q"] = np.array([0, nq])
        s["qI"] = full["qI"][L - nq:]
        s["q"] = full["q"][L - nq:]
        got = orc.hybrid_queries(s)
        for key in ("idx", "oC", "lseC", "oH", "lseH"):
            assert np.array_equal(got[key], pre[key][L - nq:]), (nq, key)


def test_decode_position_against_library_attention(orc):
    # m_C = m_H = 1 and k >= L: both branches are dense causal MQA, so a decode
    # query (n_q = 1) over a packed batch equals the last row of causal SDPA (a
    # library routine) on its own sequence; a chunked query set the last rows.
    lengths, n_q = [37, 50, 23], [1, 5, 1]
    p = packed_problem(lengths, n_q, d=8, H=2, mC=1, mH=1, k=64, seed=42)
    out = orc.hybrid_queries(p)
    full = packed_problem(lengths, lengths, d=8, H=2, mC=1, mH=1, k=64, seed=42)
    row = 0
    for b, (L, nq) in enumerate(zip(lengths, n_q)):
        kv = full["kv"][full["cu_kv"][b]:full["cu_kv"][b + 1]]
        q = np.concatenate([full["q"][full["cu_q"][b]:full["cu_q"][b + 1] - nq], p["q"][row:row + nq]])
        ref = sdpa_causal(q, kv, p["scale"])[L - nq:]
        assert np.allclose(out["oC"][row:row + nq], ref, atol=1e-12), b
        assert np.allclose(out["oH"][row:row + nq], ref, atol=1e-12), b
        row += nq


def test_compress_packed_and_selected_equal_the_single_sequence_compressor(orc):
    # compress_packed writes sequence b's entries at rows cu[b] ..; compress_selected
    # finds the owner of a global entry row; both must give the single-sequence
    # compressor's entries (pinned above to closed forms) bit for bit.
    lengths = [9, 130, 3, 64, 257]
    for m in (4, 16):
        p = packed_problem(lengths, [1] * len(lengths), d=8, mC=m, mH=128, seed=43 + m)
        cu = p["cu_csa"]
        packed = orc.compress_packed(p["cu_kv"], cu, p["kv"], p["gate"], m)
        for b, L in enumerate(lengths):
            kv0 = p["cu_kv"][b]
            alone = orc.compress(p["kv"][kv0:kv0 + L], p["gate"][kv0:kv0 + L], m)
            assert np.array_equal(packed[cu[b]:cu[b + 1]], alone), (m, b)
        rng = np.random.default_rng(m)
        rows = np.concatenate([[0, cu[-1] - 1], cu[1:-1], cu[1:-1] - 1, rng.integers(0, cu[-1], 20)])
        rows = rows[(rows >= 0) & (rows < cu[-1])]
        sel = orc.compress_selected(p["cu_kv"], cu, p["kv"], p["gate"], m, rows)
        assert np.array_equal(sel, packed[rows]), m


# ----------------------------------------------------------------------------
# sliding-window attention over the raw tokens (bjdmk.com.cn DeepSeek-V4
# walkthrough, §3.2 SWA; window of a token at t: positions t - w + 1 .. t)
# ----------------------------------------------------------------------------

def sdpa_band(q_bits, kv_bits, scale, w):
    """MQA over a causal band of width w through torch's library routine
    (boolean mask: key j visible to query i iff i - w < j <= i), fp64 on the CPU."""
    q = torch.from_numpy(f(q_bits)).permute(1, 0, 2)[None]          # [1, H, L, d]
    L = q.shape[2]
    kv = torch.from_numpy(f(kv_bits))[None, None].expand(1, q.shape[1], -1, -1)
    i = torch.arange(L)[:, None]
    j = torch.arange(L)[None, :]
    mask = (j <= i) & (j > i - w)
    o = torch.nn.functional.scaled_dot_product_attention(q, kv, kv, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2).numpy()                             # [L, H, d]


def test_swa_matches_library_attention_with_a_band_mask(orc):
    # every window from one token to more than the sequence, on a prefill
    p = packed_problem([47], [47], d=8, H=3, seed=60)
    for w in (1, 2, 5, 16, 46, 47, 48, 1000):
        o, lse = orc.swa_queries(p["cu_kv"], p["cu_q"], p["kv"], p["q"], w, p["scale"])
        assert np.allclose(o, sdpa_band(p["q"], p["kv"], p["scale"], w), atol=1e-12), w


def test_swa_window_one_returns_the_token_itself(orc):
    # a single key: its weight is 1, the output is the token's row and the
    # log-sum-exp is the one logit, scale * q_h . c_t
    p = packed_problem([19, 5], [19, 5], d=8, H=2, seed=61)
    o, lse = orc.swa_queries(p["cu_kv"], p["cu_q"], p["kv"], p["q"], 1, p["scale"])
    kv, q = f(p["kv"]), f(p["q"])
    assert np.array_equal(o, np.broadcast_to(kv[:, None, :], o.shape))
    assert np.allclose(lse, p["scale"] * np.einsum("qhd,qd->qh", q, kv), atol=1e-12)


def test_swa_reads_exactly_the_window(orc):
    # changing a token outside t - w + 1 .. t leaves query t's result bit for
    # bit; changing the window's first or last token changes it
    L, w, t = 60, 9, 40
    p = packed_problem([L], [L], d=8, H=2, seed=62)
    base_o, base_l = orc.swa_queries(p["cu_kv"], p["cu_q"], p["kv"], p["q"], w, p["scale"], eval_q=[t])
    for u, inside in ((t - w, False), (t + 1, False), (t - w + 1, True), (t, True), (0, False), (L - 1, False)):
        kv = p["kv"].copy()
        kv[u] = bf(f(kv[u]) * -2.0 + 0.25)
        o, l = orc.swa_queries(p["cu_kv"], p["cu_q"], kv, p["q"], w, p["scale"], eval_q=[t])
        assert np.array_equal(o, base_o) != inside, u
        assert np.array_equal(l, base_l) != inside, u


def test_swa_packed_batch_and_decode_layout(orc):
    # A packed batch (prefill, decode and chunked sequences, one without
    # queries) equals each sequence alone, and a decode / chunked query equals
    # the same position of that sequence's prefill, bit for bit.
    lengths, n_q, w = [70, 1, 45, 130, 9], [70, 1, 0, 12, 1], 13
    p = packed_problem(lengths, n_q, seed=63)
    o, lse = orc.swa_queries(p["cu_kv"], p["cu_q"], p["kv"], p["q"], w, p["scale"])
    full = packed_problem(lengths, lengths, seed=63)
    row = 0
    for b, (L, nq) in enumerate(zip(lengths, n_q)):
        if nq == 0:
            continue
        s = one_sequence(p, b)
        oa, la = orc.swa_queries(s["cu_kv"], s["cu_q"], s["kv"], s["q"], w, p["scale"])
        assert np.array_equal(o[row:row + nq], oa) and np.array_equal(lse[row:row + nq], la), b
        # the same tokens as a prefill whose last nq query rows are these
        fs = one_sequence(full, b)
        q = np.concatenate([fs["q"][:L - nq], p["q"][row:row + nq]])
        op, lp = orc.swa_queries(fs["cu_kv"], fs["cu_q"], fs["kv"], q, w, p["scale"])
        assert np.array_equal(op[L - nq:], oa) and np.array_equal(lp[L - nq:], la), b
        row += nq
    assert row == o.shape[0]


# ----------------------------------------------------------------------------
# inverse-RoPE correction of the attention output ("DeepSeek V4's architecture
# debt chain", Constraint 1 -> Innovation 1; convention readings P1-P4, which
# the pages do not fix: parity partly unpinned)
# ----------------------------------------------------------------------------

def _rope_problem(lengths, n_q, H=3, d=16, seed=70):
    rng = np.random.default_rng(seed)
    cu_kv = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    cu_q = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int64)
    o = rng.standard_normal((int(cu_q[-1]), H, d))
    return cu_kv, cu_q, o


def test_inverse_rope_position_zero_and_other_dims_unchanged(orc):
    cu_kv, cu_q, o = _rope_problem([40, 7], [40, 7])
    for d_rope in (2, 8, 16):
        out = orc.inverse_rope(cu_kv, cu_q, o, d_rope, 10000.0)
        assert np.array_equal(out[:, :, :16 - d_rope], o[:, :, :16 - d_rope])   # untouched dims
        assert np.array_equal(out[0], o[0]) and np.array_equal(out[40], o[40])   # t = 0 of each sequence
        pairs_in = o[:, :, 16 - d_rope:].reshape(len(o), 3, -1, 2)
        pairs_out = out[:, :, 16 - d_rope:].reshape(len(o), 3, -1, 2)
        assert np.allclose(np.hypot(*np.moveaxis(pairs_out, -1, 0)), np.hypot(*np.moveaxis(pairs_in, -1, 0)),
                           rtol=1e-13)


def test_inverse_rope_undoes_the_forward_rotary_embedding(orc):
    # Rotary position embedding (RoFormer): the pair (x, y) of frequency theta_i
    # at position t is the complex number x + iy times e^{i t theta_i}; numpy's
    # complex exponential applies it, and the correction must give x + iy back
    # (a correction that turned the other way, or paired other dims, fails)
    cu_kv, cu_q, o = _rope_problem([300, 1], [300, 1], d=16)
    d_rope, base = 8, 500.0
    t = np.concatenate([np.arange(300), [0]]).astype(np.float64)
    theta = base ** (-2.0 * np.arange(d_rope // 2) / d_rope)
    z = o[:, :, 16 - d_rope::2] + 1j * o[:, :, 16 - d_rope + 1::2]
    zr = z * np.exp(1j * t[:, None, None] * theta[None, None, :])
    fwd = o.copy()
    fwd[:, :, 16 - d_rope::2], fwd[:, :, 16 - d_rope + 1::2] = zr.real, zr.imag
    assert np.allclose(orc.inverse_rope(cu_kv, cu_q, fwd, d_rope, base), o, atol=1e-12)


def test_inverse_rope_composes_over_positions(orc):
    # the correction for position a followed by that for b is the one for
    # a + b: the angle is linear in the query position t = L - n_q + i
    rng = np.random.default_rng(71)
    o = rng.standard_normal((1, 2, 12))
    one = lambda L, x: orc.inverse_rope(np.array([0, L]), np.array([0, 1]), x, 12, 10000.0)
    for a, b in ((3, 5), (100, 1), (4095, 4096), (70000, 12345)):
        assert np.allclose(one(b + 1, one(a + 1, o)), one(a + b + 1, o), atol=1e-9), (a, b)
