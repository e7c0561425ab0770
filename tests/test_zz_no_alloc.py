"""lightning_index_topk_static: the indexer + top-k for callers that cannot
allocate device memory.

Some callers (a plug-in host that gives a custom operation only its input and
output buffers, or a latency-critical loop that may not call cudaMalloc) have
no way to provide the workspace that lightning_index_topk takes.  The
scratch-free entry point uses a library-owned device array instead.  These
tests check that it gives exactly the results of the workspace entry point,
on two calls in a row and across problems of different shapes (so that what
one call leaves in the shared array cannot leak into the next), and that a
problem too large for the array is refused on the host.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from compressed_sparse_attention_21_b300 import _lib as csa
from compressed_sparse_attention_21_b300 import build as csa_build
from compressed_sparse_attention_21_b300 import workloads as wl

CSA_ERR_WORKSPACE = 3


def _problem(lengths, n_q, HI, dI, k, seed):
    w = wl.Workload("no_alloc", len(lengths), list(lengths), False, H=8, d=128, HI=HI, dI=dI, top_k=k,
                    seed=seed)
    return wl.make_problem(w, n_q=n_q)


def _run_both(p, k, repeats=2):
    dev = torch.device("cuda")
    layout = csa.Layout(p["lengths"], p["n_q"], p["mC"], p["mH"], device=dev)
    qI, kI = p["qI"].to(dev), p["kI"].to(dev)
    ref_idx, ref_score = csa.lightning_index_topk(layout, qI, kI, k)
    torch.cuda.synchronize()
    for _ in range(repeats):
        idx = torch.full_like(ref_idx, 12345)
        score = torch.full_like(ref_score, 7.0)
        csa.lightning_index_topk_static(layout, qI, kI, k, idx_out=idx, score_out=score)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        # same kernels and arithmetic: the scores match bit for bit
        assert torch.equal(score.view(torch.int32), ref_score.view(torch.int32))
    assert csa.check_device_error() == 0


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    csa_build.build()
    csa.load()
    # decode-shaped: the multi-CTA path, which uses the scratch
    lengths = [1, 5, 100, 4096, 5001, 20000, 70001]
    _run_both(_problem(lengths, [1] * len(lengths), HI=4, dI=64, k=512, seed=41), 512)
    # a different shape right after: more queries, longer rows, another k
    lengths = [131071, 65537, 99999, 40000, 3, 250000]
    _run_both(_problem(lengths, [2, 1, 3, 1, 1, 1], HI=2, dI=32, k=1024, seed=42), 1024)
    # and back to a small one
    _run_both(_problem([9000, 300], [1, 1], HI=1, dI=128, k=7, seed=43), 7)


@pytest.mark.gpu
def test_static_scratch_prefill_sized_batch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    csa_build.build()
    csa.load()
    # 2200 queries at top-k 64 over at most 375 entries: the prefill block
    # path.  Its full workspace holds one 512 KiB candidate slot for each of
    # the 138 query blocks (on 148 SMs); the 32 MiB array holds 64 slots, so
    # the scratch-free call runs fewer persistent CTAs than the workspace call.
    lengths = [1500, 700]
    p = _problem(lengths, lengths, HI=2, dI=32, k=64, seed=44)
    full_ws = csa.index_workspace_size(csa.Layout(lengths, lengths, 4, 128, device="cuda"), 2, 32, 64)
    assert full_ws > csa.STATIC_SCRATCH_BYTES
    _run_both(p, 64)


def test_static_scratch_rejects_oversized_problem_on_host():
    csa_build.build()
    lib = csa.load()
    fake = 256   # non-null and 16-byte aligned; a refused call dereferences nothing
    # one decode query over 2^25 entries needs far more than the 32 MiB array
    L = csa.csa_layout(batch=1, max_kv_len=1 << 27, max_q_len=1, reserved=0, cu_kv=fake, cu_q=fake, cu_csa=fake,
                       cu_hca=fake, total_kv=1 << 27, total_q=1, total_csa=1 << 25, total_hca=0)
    need = ctypes.c_size_t(0)
    assert lib.csa_index_workspace_size(ctypes.byref(L), 4, 64, 4, 1024, ctypes.byref(need)) == 0
    assert need.value > csa.STATIC_SCRATCH_BYTES
    rc = lib.lightning_index_topk_static(ctypes.byref(L), fake, fake, 4, 64, 4, 1024, fake, None, None)
    assert rc == CSA_ERR_WORKSPACE
