"""fp64 CPU oracle for the CSA + HCA hybrid compressed attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package.  The CUDA library
never links, loads or calls it, and this package never touches the CUDA
library: the two meet only in the tests, on the same seeded inputs.

The arithmetic lives in ``csa_oracle.c`` (plain C, double precision, plain
loops; OpenMP only over independent queries and blocks).  This module only
builds that file with gcc and marshals numpy arrays through ctypes.

bf16 tensors are passed as their raw bit patterns (``numpy.uint16``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``csa_oracle.c`` into ``liboracle.so`` (gcc -O2, no fast-math)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                                   "-Wall", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        D = ctypes.c_double
        lib.orc_num_threads.restype = I
        lib.orc_compress.argtypes = [P, P, I64, I, I, P]
        lib.orc_index_scores.argtypes = [P, P, I64, I, I, P]
        lib.orc_topk.argtypes = [P, I64, I, P]
        lib.orc_attend.argtypes = [P, I, I, P, I64, D, P, P]
        lib.orc_hybrid_queries.argtypes = [I, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, D,
                                           P, I64, P, P, I, I, P, P, P, P, P]
        lib.orc_compress_packed.argtypes = [I, P, P, P, P, I, I, P]
        lib.orc_compress_selected.argtypes = [I, P, P, P, P, I, I, I64, P, P]
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_decode.restype = D
        lib.orc_e4m3_encode.argtypes = [D]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_quantize_index_keys.argtypes = [P, I64, I, P, P]
        lib.orc_index_scores_fp8.argtypes = [P, P, P, I64, I, I, P]
        lib.orc_swa_queries.argtypes = [I, P, P, P, P, I, I, I64, D, I64, P, P, P]
        lib.orc_inverse_rope.argtypes = [I, P, P, I, I, I, D, P, P]
        for f in ("orc_compress", "orc_index_scores", "orc_topk", "orc_attend",
                  "orc_hybrid_queries", "orc_compress_packed", "orc_compress_selected",
                  "orc_quantize_index_keys", "orc_index_scores_fp8", "orc_swa_queries",
                  "orc_inverse_rope"):
            getattr(lib, f).restype = I
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def num_threads() -> int:
    return int(_load().orc_num_threads())


def compress(c_bits, z, m):
    """Entries of all complete m-token blocks of ONE sequence: [L//m, d] fp64."""
    c_bits = _c(c_bits, np.uint16)
    z = _c(z, np.float32)
    L, d = c_bits.shape
    out = np.empty((L // m, d), np.float64)
    _check(_load().orc_compress(_ptr(c_bits), _ptr(z), L, d, m, _ptr(out)), "compress")
    return out


def compress_packed(cu_kv, cu_out, kv_bits, gate, m):
    cu_kv = _c(cu_kv, np.int64)
    cu_out = _c(cu_out, np.int64)
    kv_bits = _c(kv_bits, np.uint16)
    gate = _c(gate, np.float32)
    d = kv_bits.shape[1]
    out = np.empty((int(cu_out[-1]), d), np.float64)
    _check(_load().orc_compress_packed(len(cu_kv) - 1, _ptr(cu_kv), _ptr(cu_out), _ptr(kv_bits),
                                       _ptr(gate), d, m, _ptr(out)), "compress_packed")
    return out


def compress_selected(cu_kv, cu_out, kv_bits, gate, m, entries):
    cu_kv = _c(cu_kv, np.int64)
    cu_out = _c(cu_out, np.int64)
    kv_bits = _c(kv_bits, np.uint16)
    gate = _c(gate, np.float32)
    entries = _c(entries, np.int64)
    d = kv_bits.shape[1]
    out = np.empty((len(entries), d), np.float64)
    _check(_load().orc_compress_selected(len(cu_kv) - 1, _ptr(cu_kv), _ptr(cu_out), _ptr(kv_bits),
                                         _ptr(gate), d, m, len(entries), _ptr(entries), _ptr(out)),
           "compress_selected")
    return out


def index_scores(qI_bits, kI_bits):
    """qI: [HI, dI]; kI: [n, dI] -> s[n] fp64."""
    qI_bits = _c(qI_bits, np.uint16)
    kI_bits = _c(kI_bits, np.uint16)
    HI, dI = qI_bits.shape
    n = kI_bits.shape[0]
    s = np.empty(n, np.float64)
    _check(_load().orc_index_scores(_ptr(qI_bits), _ptr(kI_bits), n, HI, dI, _ptr(s)), "index_scores")
    return s


def e4m3_decode(code: int) -> float:
    """Value of one FP8 E4M3 code (NaN for 0x7f / 0xff)."""
    return float(_load().orc_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    """Nearest E4M3 code, ties to even, saturating at +-448, sign kept."""
    return int(_load().orc_e4m3_encode(float(x)))


def quantize_index_keys(kI_bits):
    """kI: [n, dI] bf16 bits -> (codes [n, dI] uint8, scale [n] float32)."""
    kI_bits = _c(kI_bits, np.uint16)
    n, dI = kI_bits.shape
    codes = np.empty((n, dI), np.uint8)
    scale = np.empty(n, np.float32)
    _check(_load().orc_quantize_index_keys(_ptr(kI_bits), n, dI, _ptr(codes), _ptr(scale)),
           "quantize_index_keys")
    return codes, scale


def index_scores_fp8(qI_bits, codes, scale):
    """qI: [HI, dI] bf16 bits; codes [n, dI]; scale [n] -> s[n] fp64."""
    qI_bits = _c(qI_bits, np.uint16)
    codes = _c(codes, np.uint8)
    scale = _c(scale, np.float32)
    HI, dI = qI_bits.shape
    n = codes.shape[0]
    s = np.empty(n, np.float64)
    _check(_load().orc_index_scores_fp8(_ptr(qI_bits), _ptr(codes), _ptr(scale), n, HI, dI, _ptr(s)),
           "index_scores_fp8")
    return s


def topk(s, k):
    s = _c(s, np.float64)
    idx = np.empty(k, np.int32)
    _check(_load().orc_topk(_ptr(s), len(s), k, _ptr(idx)), "topk")
    return idx


def attend(q_bits, keys, scale):
    """q: [H, d] bf16 bits; keys: [nk, d] fp64 -> (o [H, d], lse [H])."""
    q_bits = _c(q_bits, np.uint16)
    keys = _c(keys, np.float64)
    H, d = q_bits.shape
    o = np.empty((H, d), np.float64)
    lse = np.empty(H, np.float64)
    _check(_load().orc_attend(_ptr(q_bits), H, d, _ptr(keys), keys.shape[0], float(scale),
                              _ptr(o), _ptr(lse)), "attend")
    return o, lse


def hybrid_queries(inp, eval_q=None, given_idx=None, do_csa=True, do_hca=True,
                   hca_entries=None):
    """Evaluate whole queries of a packed problem.

    ``inp`` is a mapping with numpy arrays: cu_kv, cu_q, cu_csa, cu_hca (int64),
    kv (uint16 [ΣL, d]), gate (f32 [ΣL]), qI (uint16 [ΣQ, HI, dI]), kI (uint16
    [ΣE_C, dI]), q (uint16 [ΣQ, H, d]) and ints mC, mH, top_k, plus float scale.
    Returns a dict with idx [n, k] int32, oC/oH [n, H, d] fp64 and lseC/lseH [n, H].
    """
    lib = _load()
    cu_kv = _c(inp["cu_kv"], np.int64)
    cu_q = _c(inp["cu_q"], np.int64)
    cu_csa = _c(inp["cu_csa"], np.int64)
    cu_hca = _c(inp["cu_hca"], np.int64)
    kv = _c(inp["kv"], np.uint16)
    gate = _c(inp["gate"], np.float32)
    qI = _c(inp["qI"], np.uint16)
    kI = _c(inp["kI"], np.uint16)
    q = _c(inp["q"], np.uint16)
    B = len(cu_kv) - 1
    d = kv.shape[1]
    H = q.shape[1]
    HI, dI = qI.shape[1], qI.shape[2]
    mC, mH, k = int(inp["mC"]), int(inp["mH"]), int(inp["top_k"])
    scale = float(inp["scale"])
    if eval_q is None:
        eval_q = np.arange(int(cu_q[-1]), dtype=np.int64)
    eval_q = _c(eval_q, np.int64)
    n = len(eval_q)
    if do_hca and hca_entries is None:
        hca_entries = compress_packed(cu_kv, cu_hca, kv, gate, mH)
    hca_entries = _c(hca_entries, np.float64) if do_hca else None
    if given_idx is not None:
        given_idx = _c(given_idx, np.int32)
        assert given_idx.shape == (n, k)
    out = dict(idx=np.full((n, k), -1, np.int32),
               oC=np.zeros((n, H, d)) if do_csa else None,
               lseC=np.zeros((n, H)) if do_csa else None,
               oH=np.zeros((n, H, d)) if do_hca else None,
               lseH=np.zeros((n, H)) if do_hca else None)
    rc = lib.orc_hybrid_queries(B, _ptr(cu_kv), _ptr(cu_q), _ptr(cu_csa), _ptr(cu_hca), _ptr(kv),
                                _ptr(gate), _ptr(qI), _ptr(kI), _ptr(q), d, H, HI, dI, mC, mH, k,
                                scale, _ptr(hca_entries), n, _ptr(eval_q), _ptr(given_idx),
                                int(bool(do_csa)), int(bool(do_hca)), _ptr(out["idx"]),
                                _ptr(out["oC"]), _ptr(out["lseC"]), _ptr(out["oH"]),
                                _ptr(out["lseH"]))
    _check(rc, "hybrid_queries")
    return out


def swa_queries(cu_kv, cu_q, kv_bits, q_bits, window, scale, eval_q=None):
    """Sliding-window attention of whole queries of a packed problem: each
    query over its own raw token and the window - 1 tokens before it.
    kv_bits [ΣL, d] and q_bits [ΣQ, H, d] are bf16 bit patterns.  Returns
    (o [n, H, d] fp64, lse [n, H] fp64)."""
    cu_kv = _c(cu_kv, np.int64)
    cu_q = _c(cu_q, np.int64)
    kv = _c(kv_bits, np.uint16)
    q = _c(q_bits, np.uint16)
    B = len(cu_kv) - 1
    d = kv.shape[1]
    H = q.shape[1]
    if eval_q is None:
        eval_q = np.arange(int(cu_q[-1]), dtype=np.int64)
    eval_q = _c(eval_q, np.int64)
    n = len(eval_q)
    o = np.zeros((n, H, d))
    lse = np.zeros((n, H))
    _check(_load().orc_swa_queries(B, _ptr(cu_kv), _ptr(cu_q), _ptr(kv), _ptr(q), d, H, int(window), float(scale),
                                   n, _ptr(eval_q), _ptr(o), _ptr(lse)), "swa_queries")
    return o, lse


def inverse_rope(cu_kv, cu_q, o, d_rope, base):
    """Inverse-RoPE correction of attention outputs o [ΣQ, H, d] (fp64): each
    query's last d_rope dims of every head, pairs (2i, 2i+1), turned by
    -t * base^(-2i/d_rope) for the query's position t.  Returns a new array."""
    cu_kv = _c(cu_kv, np.int64)
    cu_q = _c(cu_q, np.int64)
    o = _c(o, np.float64)
    out = np.empty_like(o)
    H, d = o.shape[1], o.shape[2]
    _check(_load().orc_inverse_rope(len(cu_kv) - 1, _ptr(cu_kv), _ptr(cu_q), H, d, int(d_rope), float(base),
                                    _ptr(o), _ptr(out)), "inverse_rope")
    return out
