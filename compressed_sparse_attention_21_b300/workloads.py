"""Seeded synthetic workloads for the CSA + HCA hybrid attention.

This module only draws random inputs and describes their shapes; it holds
none of the method's arithmetic.  The tests, the benchmark and the oracle
checks all take their inputs from here, so the CUDA path and the oracle see
the same bytes.

Recipe (per workload, all on the CPU):

* ragged lengths (only the ragged-decode workload): ``torch.randint(lo, hi+1)``
  from ``torch.Generator().manual_seed(seed)``, one draw per sequence,
  redrawn while the length is a multiple of 128;
* then, in this order, per-token KV ``c [ΣL, d]``, gate logits ``z [ΣL]``,
  indexer queries ``qI [ΣQ, HI, dI]``, indexer keys ``kI [ΣE_C, dI]`` (one
  per compressed entry) and attention queries ``q [ΣQ, H, d]``.  Each tensor
  is drawn as standard normal fp32 in fixed chunks of ``CHUNK`` elements;
  chunk ``i`` of tensor number ``n`` uses its own generator seeded with
  ``seed * 1_000_003 + n * 10_007 + i`` (so chunks can be drawn in parallel),
  multiplied by the tensor's standard deviation, and cast to bf16 (``z``
  stays fp32).

Queries of sequence b are its last ``n_q`` positions (``n_q = L`` for
prefill, 1 for decode).
"""
from __future__ import annotations

import concurrent.futures as _fut
import dataclasses
import math
from typing import Optional, Sequence

import torch

CHUNK = 1 << 24  # elements per generator chunk


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    lengths: Optional[Sequence[int]]  # None -> drawn (ragged)
    decode: bool                      # True: one query per sequence; False: every position
    H: int
    d: int
    HI: int
    dI: int
    top_k: int
    mC: int = 4
    mH: int = 128
    gate_std: float = 1.0
    seed: int = 0
    ragged_range: Optional[tuple] = None

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads: a 4K causal prefill for correctness, 64K decode,
# 128K long prefill, ragged 32K-128K decode and 1M-token decode.
WORKLOADS = {
    "prefill_4k": Workload("prefill_4k", 1, [4096], False, H=8, d=128, HI=2, dI=32, top_k=64,
                           gate_std=1.0, seed=0),
    "decode_64k": Workload("decode_64k", 16, [65536] * 16, True, H=64, d=512, HI=4, dI=64,
                           top_k=512, gate_std=2.0, seed=1),
    "prefill_128k": Workload("prefill_128k", 1, [131072], False, H=64, d=512, HI=4, dI=64,
                             top_k=1024, gate_std=1.0, seed=2),
    "ragged_decode": Workload("ragged_decode", 64, None, True, H=64, d=512, HI=4, dI=64,
                              top_k=1024, gate_std=1.0, seed=3, ragged_range=(32768, 131072)),
    "decode_1m": Workload("decode_1m", 4, [1 << 20] * 4, True, H=128, d=512, HI=4, dI=64,
                          top_k=1024, gate_std=1.0, seed=4),
}


def draw_lengths(w: Workload) -> list:
    if w.lengths is not None:
        return list(w.lengths)
    g = torch.Generator().manual_seed(w.seed)
    lo, hi = w.ragged_range
    out = []
    for _ in range(w.batch):
        L = int(torch.randint(lo, hi + 1, (1,), generator=g))
        while L % 128 == 0:
            L = int(torch.randint(lo, hi + 1, (1,), generator=g))
        out.append(L)
    return out


def _prefix(xs) -> torch.Tensor:
    out = torch.zeros(len(xs) + 1, dtype=torch.int64)
    if len(xs):
        out[1:] = torch.cumsum(torch.tensor(xs, dtype=torch.int64), 0)
    return out


def _chunk(seed: int, tensor_no: int, i: int, n: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed * 1_000_003 + tensor_no * 10_007 + i)
    return torch.randn(n, generator=g)


def randn(seed: int, tensor_no: int, shape, std: float = 1.0, dtype=torch.bfloat16,
          threads: int = 8) -> torch.Tensor:
    """Chunked, seeded standard-normal draw (see the module recipe)."""
    numel = 1
    for s in shape:
        numel *= int(s)
    out = torch.empty(numel, dtype=dtype)
    n_chunks = (numel + CHUNK - 1) // CHUNK

    def fill(i):
        lo = i * CHUNK
        n = min(CHUNK, numel - lo)
        x = _chunk(seed, tensor_no, i, n)
        if std != 1.0:
            x.mul_(std)
        out[lo:lo + n] = x.to(dtype)

    if n_chunks <= 1:
        for i in range(n_chunks):
            fill(i)
    else:
        with _fut.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.view(*[int(s) for s in shape])


def make_problem(w: Workload, lengths=None, n_q=None, seed=None) -> dict:
    """Draw one problem.  Returns CPU tensors and the packed layout.

    ``lengths``/``n_q``/``seed`` override the workload (for small test cases);
    ``n_q`` may be an int or a per-sequence list.
    """
    seed = w.seed if seed is None else seed
    Ls = list(lengths) if lengths is not None else draw_lengths(w)
    if n_q is None:
        nqs = [1 if w.decode else L for L in Ls]
    elif isinstance(n_q, int):
        nqs = [min(n_q, L) for L in Ls]
    else:
        nqs = list(n_q)
    E_C = [L // w.mC for L in Ls]
    E_H = [L // w.mH for L in Ls]
    total_kv, total_q = sum(Ls), sum(nqs)
    kv = randn(seed, 0, (total_kv, w.d))
    gate = randn(seed, 1, (total_kv,), std=w.gate_std, dtype=torch.float32)
    qI = randn(seed, 2, (total_q, w.HI, w.dI))
    kI = randn(seed, 3, (sum(E_C), w.dI))
    q = randn(seed, 4, (total_q, w.H, w.d))
    return dict(workload=w.name, lengths=Ls, n_q=nqs,
                cu_kv=_prefix(Ls), cu_q=_prefix(nqs), cu_csa=_prefix(E_C), cu_hca=_prefix(E_H),
                kv=kv, gate=gate, qI=qI, kI=kI, q=q,
                H=w.H, d=w.d, HI=w.HI, dI=w.dI, top_k=w.top_k, mC=w.mC, mH=w.mH,
                scale=w.scale)


def bits(t: torch.Tensor):
    """A bf16 tensor's raw bit patterns as a numpy uint16 array (no copy)."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def to_numpy(p: dict) -> dict:
    """The problem in the oracle's numpy form (bf16 as uint16 bit patterns)."""
    return dict(cu_kv=p["cu_kv"].numpy(), cu_q=p["cu_q"].numpy(), cu_csa=p["cu_csa"].numpy(),
                cu_hca=p["cu_hca"].numpy(), kv=bits(p["kv"]), gate=p["gate"].numpy(),
                qI=bits(p["qI"]), kI=bits(p["kI"]), q=bits(p["q"]), mC=p["mC"], mH=p["mH"],
                top_k=p["top_k"], scale=p["scale"])
