"""Host logic of bench.py: the algorithmic bytes and flops that the roofline
divides by, checked against their closed forms (no GPU)."""
import importlib.util
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def shape(lengths, n_q, H=64, d=512, HI=4, dI=64, k=512, mC=4, mH=128):
    return dict(lengths=lengths, n_q=n_q, H=H, d=d, HI=HI, dI=dI, top_k=k, mC=mC, mH=mH)


def test_decode_64k_index_bytes_closed_form():
    # 16 queries at t = 65535: n_C = 16384 visible keys of d_I = 64 bf16 each,
    # the query's 4 x 64 bf16 indexer heads, and 512 output indices
    b = _bench()
    p = shape([65536] * 16, [1] * 16)
    w, fl = b.step_work(p)
    assert w["index_topk"] == 16 * (2 * 4 * 64 + 16384 * 2 * 64 + 4 * 512) == 33_595_392
    w8, _ = b.step_work(p, fp8=True)
    assert w8["index_topk"] == 16 * (2 * 4 * 64 + 16384 * (64 + 4) + 4 * 512) == 17_866_752
    # the other calls do not depend on the key format
    assert {k: v for k, v in w.items() if k != "index_topk"} == {k: v for k, v in w8.items() if k != "index_topk"}
    # sparse: 512 selected entries (t + 1 is a multiple of 4: no raw tail), q in and o out
    assert w["sparse_attend"] == 16 * (2 * (512 * 512 + 2 * 64 * 512) + 4 * 512 + 4 * 64)
    # dense: 512 HCA entries, no tail
    assert w["dense_attend"] == 16 * (2 * (512 * 512 + 2 * 64 * 512) + 4 * 64)
    assert fl["index"] == 16 * 2 * 64 * 16384
    assert fl["sparse"] == 16 * 4 * 64 * 512 * 512


def test_compress_bytes_count_closed_blocks_only():
    b = _bench()
    # one decode query at t = 4095 closes one CSA block (4 tokens) and one HCA block (128 tokens)
    w, _ = b.step_work(shape([4096], [1], d=512))
    tok = 128
    assert w["compress"] == 2 * 512 * tok + 4 * tok + 2 * 512 * 2
    # at t = 4096 no block closes: nothing to compress
    w, _ = b.step_work(shape([4097], [1], d=512))
    assert w["compress"] == 0


def test_fast_count_equals_the_per_position_count():
    b = _bench()
    for fp8 in (False, True):
        p = shape([5003, 130], [5003, 130], H=8, d=128, HI=2, dI=32, k=64)   # > 4096 queries: closed form
        slow = b.step_work(p, fp8)
        fast = b.step_work_fast(p, fp8)
        assert slow == fast


def test_job_value_counts_every_rank():
    b = _bench()
    assert b.job_value(16, 4, 0.5) == 16 * 4 / 0.5e-3


def test_swa_flops_closed_form_equals_the_per_position_count():
    # 4 H d flops per key per query (scores and weighted sum), min(t + 1, w)
    # keys for the query at position t
    for lengths, n_q, w in (([100], [100], 7), ([100], [3], 7), ([5, 300, 64], [5, 1, 30], 64),
                            ([4097, 10], [4097, 1], 4096), ([50], [50], 1000), ([1], [1], 1)):
        per_pos = sum(min(t + 1, w) for L, nq in zip(lengths, n_q) for t in range(L - nq, L))
        assert _bench().swa_flops(lengths, n_q, 2, 3, w) == 4 * 2 * 3 * per_pos


def test_rope_bytes_count_the_rope_slices_read_and_written():
    assert _bench().rope_bytes(32768, 64, 64) == 2 * 32768 * 64 * 64 * 2
