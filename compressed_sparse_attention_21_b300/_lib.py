"""ctypes binding of ``libcsa.so``: argument marshalling only.

Every function here forwards device pointers, sizes and the current torch
CUDA stream to one C-ABI call of ``include/csa.h``; all arithmetic runs in the
library's sm_103a kernels.  There is no fallback: a missing library or a
non-CUDA tensor raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")
_lib = None

CSA_SKIP_COMPRESS = 0x1
CSA_INDEX_FP8 = 0x2
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported size", 3: "workspace missing or too small",
          4: "CUDA error", 5: "device wait timed out", 6: "device-side layout or index error"}


class CsaError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = int(status)
        super().__init__(f"{what}: {STATUS.get(self.status, 'unknown')} (status {self.status})")


class csa_layout(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_kv_len", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("cu_kv", ctypes.c_void_p), ("cu_q", ctypes.c_void_p),
                ("cu_csa", ctypes.c_void_p), ("cu_hca", ctypes.c_void_p), ("total_kv", ctypes.c_int64),
                ("total_q", ctypes.c_int64), ("total_csa", ctypes.c_int64), ("total_hca", ctypes.c_int64)]


class csa_hybrid_params(ctypes.Structure):
    _fields_ = [("layout", csa_layout), ("d", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_heads_idx", ctypes.c_int32), ("d_idx", ctypes.c_int32), ("ratio_csa", ctypes.c_int32),
                ("ratio_hca", ctypes.c_int32), ("top_k", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("scale", ctypes.c_float), ("reserved", ctypes.c_int32), ("kv", ctypes.c_void_p),
                ("gate", ctypes.c_void_p), ("q_idx", ctypes.c_void_p), ("k_idx", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("csa_cache", ctypes.c_void_p), ("hca_cache", ctypes.c_void_p),
                ("idx_out", ctypes.c_void_p), ("score_out", ctypes.c_void_p), ("o_csa", ctypes.c_void_p),
                ("lse_csa", ctypes.c_void_p), ("o_hca", ctypes.c_void_p), ("lse_hca", ctypes.c_void_p),
                ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t), ("k_idx_fp8", ctypes.c_void_p),
                ("k_idx_scale", ctypes.c_void_p)]


# Every symbol include/csa.h declares (checked by the CPU test suite).
EXPORTS = ("csa_compress", "hca_compress", "lightning_index_topk", "csa_index_workspace_size",
           "lightning_index_topk_static", "csa_quantize_index_keys", "csa_quantize_index_keys_closed",
           "lightning_index_topk_fp8",
           "csa_index_fp8_workspace_size",
           "sparse_mqa_attend", "hca_dense_attend", "csa_attend_workspace_size", "swa_attend",
           "swa_workspace_size", "csa_inverse_rope", "hybrid_attend",
           "csa_workspace_size", "csa_workspace_init", "csa_status_string", "csa_check_device_error",
           "csa_version", "csa_timing_enable", "csa_timing_read", "csa_timing_reset")


def load():
    """Load libcsa.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libcsa.so not built ({LIB_PATH}); run "
                           "`python -m compressed_sparse_attention_21_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    LP = ctypes.POINTER(csa_layout)
    lib.csa_compress.argtypes = [LP, P, P, I, I, P, P]
    lib.hca_compress.argtypes = [LP, P, P, I, I, P, P]
    lib.lightning_index_topk.argtypes = [LP, P, P, I, I, I, I, P, P, P, Z, P]
    lib.csa_index_workspace_size.argtypes = [LP, I, I, I, I, ctypes.POINTER(Z)]
    lib.lightning_index_topk_static.argtypes = [LP, P, P, I, I, I, I, P, P, P]
    lib.csa_quantize_index_keys.argtypes = [LP, P, I, P, P, P]
    lib.csa_quantize_index_keys_closed.argtypes = [LP, P, I, I, P, P, P]
    lib.lightning_index_topk_fp8.argtypes = [LP, P, P, P, I, I, I, I, P, P, P, Z, P]
    lib.csa_index_fp8_workspace_size.argtypes = [LP, I, I, I, I, ctypes.POINTER(Z)]
    lib.sparse_mqa_attend.argtypes = [LP, P, P, P, P, I, I, I, I, F, P, P, P, Z, P]
    lib.hca_dense_attend.argtypes = [LP, P, P, P, I, I, I, F, P, P, P, Z, P]
    lib.csa_attend_workspace_size.argtypes = [LP, I, I, I, I, ctypes.POINTER(Z)]
    lib.swa_attend.argtypes = [LP, P, P, I, I, I, F, P, P, P, Z, P]
    lib.swa_workspace_size.argtypes = [LP, I, I, I, ctypes.POINTER(Z)]
    lib.csa_inverse_rope.argtypes = [LP, P, I, I, I, F, P]
    lib.hybrid_attend.argtypes = [ctypes.POINTER(csa_hybrid_params), P]
    lib.csa_workspace_size.argtypes = [ctypes.POINTER(csa_hybrid_params), ctypes.POINTER(Z)]
    lib.csa_workspace_init.argtypes = [P, Z, P]
    lib.csa_status_string.argtypes = [I]
    lib.csa_status_string.restype = ctypes.c_char_p
    lib.csa_check_device_error.argtypes = [P, ctypes.POINTER(I)]
    lib.csa_version.restype = I
    lib.csa_timing_enable.argtypes = [I]
    lib.csa_timing_read.argtypes = [I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_int64),
                                    ctypes.POINTER(ctypes.c_double)]
    lib.csa_timing_read.restype = I
    lib.csa_timing_reset.restype = None
    for f in ("csa_compress", "hca_compress", "lightning_index_topk", "csa_index_workspace_size",
              "lightning_index_topk_static", "csa_quantize_index_keys", "csa_quantize_index_keys_closed",
              "lightning_index_topk_fp8", "csa_index_fp8_workspace_size", "sparse_mqa_attend", "hca_dense_attend", "csa_attend_workspace_size",
              "swa_attend", "swa_workspace_size", "csa_inverse_rope", "hybrid_attend",
              "csa_workspace_size", "csa_workspace_init", "csa_check_device_error", "csa_timing_enable"):
        getattr(lib, f).restype = I
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libcsa must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libcsa must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, what):
    if status != 0:
        raise CsaError(status, what)


class Layout:
    """Packed variable-length batch (host copies + device cu arrays).

    Sequence b has ``lengths[b]`` tokens; its queries are its last ``n_q[b]``
    positions.  Entry counts per sequence are floor(L / ratio).
    """

    def __init__(self, lengths, n_q, ratio_csa=4, ratio_hca=128, device="cuda"):
        lengths = [int(x) for x in lengths]
        n_q = [int(x) for x in n_q]
        if len(lengths) != len(n_q) or not lengths:
            raise ValueError("lengths and n_q must be non-empty lists of equal length")
        if any(q < 0 or q > L for q, L in zip(n_q, lengths)):
            raise ValueError("0 <= n_q[b] <= lengths[b] must hold")
        self.lengths, self.n_q = lengths, n_q
        self.ratio_csa, self.ratio_hca = int(ratio_csa), int(ratio_hca)
        self.batch = len(lengths)
        self.max_kv_len = max(lengths)
        self.max_q_len = max(n_q)
        self.host = {
            "cu_kv": prefix(lengths),
            "cu_q": prefix(n_q),
            "cu_csa": prefix([L // self.ratio_csa for L in lengths]),
            "cu_hca": prefix([L // self.ratio_hca for L in lengths]),
        }
        self.total_kv = int(self.host["cu_kv"][-1])
        self.total_q = int(self.host["cu_q"][-1])
        self.total_csa = int(self.host["cu_csa"][-1])
        self.total_hca = int(self.host["cu_hca"][-1])
        self.device = device
        self.dev = {k: torch.tensor(v, dtype=torch.int64, device=device) for k, v in self.host.items()}
        self._c = csa_layout(self.batch, self.max_kv_len, self.max_q_len, 0,
                             self.dev["cu_kv"].data_ptr(), self.dev["cu_q"].data_ptr(),
                             self.dev["cu_csa"].data_ptr(), self.dev["cu_hca"].data_ptr(),
                             self.total_kv, self.total_q, self.total_csa, self.total_hca)

    @property
    def c(self):
        return self._c


def prefix(xs):
    out = [0]
    for x in xs:
        out.append(out[-1] + int(x))
    return out


def _ws(bytes_, device, ws):
    if bytes_ == 0:
        return None, 0
    if ws is None or ws.numel() < bytes_:
        ws = torch.zeros(bytes_, dtype=torch.uint8, device=device)   # zero-filled as the ABI requires
    return ws, bytes_


def csa_compress(layout, kv, gate, out, ratio=None, stream=None):
    ratio = layout.ratio_csa if ratio is None else ratio
    _check(load().csa_compress(ctypes.byref(layout.c), _ptr(kv), _ptr(gate), kv.shape[-1], ratio, _ptr(out),
                               _stream(stream)), "csa_compress")
    return out


def hca_compress(layout, kv, gate, out, ratio=None, stream=None):
    ratio = layout.ratio_hca if ratio is None else ratio
    _check(load().hca_compress(ctypes.byref(layout.c), _ptr(kv), _ptr(gate), kv.shape[-1], ratio, _ptr(out),
                               _stream(stream)), "hca_compress")
    return out


def index_workspace_size(layout, n_heads_idx, d_idx, top_k, ratio=None):
    n = ctypes.c_size_t(0)
    _check(load().csa_index_workspace_size(ctypes.byref(layout.c), n_heads_idx, d_idx,
                                           layout.ratio_csa if ratio is None else ratio, top_k, ctypes.byref(n)),
           "csa_index_workspace_size")
    return n.value


def lightning_index_topk(layout, q_idx, k_idx, top_k, idx_out=None, score_out=None, ws=None, ratio=None,
                         stream=None, with_scores=True):
    ratio = layout.ratio_csa if ratio is None else ratio
    dev = q_idx.device
    if idx_out is None:
        idx_out = torch.empty((layout.total_q, top_k), dtype=torch.int32, device=dev)
    if score_out is None and with_scores:
        score_out = torch.empty((layout.total_q, top_k), dtype=torch.float32, device=dev)
    HI, dI = q_idx.shape[-2], q_idx.shape[-1]
    ws, nb = _ws(index_workspace_size(layout, HI, dI, top_k, ratio), dev, ws)
    _check(load().lightning_index_topk(ctypes.byref(layout.c), _ptr(q_idx), _ptr(k_idx), HI, dI, ratio, top_k,
                                       _ptr(idx_out), _ptr(score_out), _ptr(ws), nb, _stream(stream)),
           "lightning_index_topk")
    return idx_out, score_out


def quantize_index_keys(layout, k_idx, k_fp8=None, k_scale=None, stream=None):
    """E4M3 codes [total_csa, d_idx] (uint8) and per-row fp32 scales of the indexer keys."""
    dev = k_idx.device
    dI = k_idx.shape[-1]
    if k_fp8 is None:
        k_fp8 = torch.empty((layout.total_csa, dI), dtype=torch.uint8, device=dev)
    if k_scale is None:
        k_scale = torch.empty((layout.total_csa,), dtype=torch.float32, device=dev)
    _check(load().csa_quantize_index_keys(ctypes.byref(layout.c), _ptr(k_idx), dI, _ptr(k_fp8), _ptr(k_scale),
                                          _stream(stream)), "csa_quantize_index_keys")
    return k_fp8, k_scale


def quantize_closed_index_keys(layout, k_idx, k_fp8, k_scale, ratio=None, stream=None):
    """Update k_fp8 / k_scale in place for the entries the layout's query positions close."""
    ratio = layout.ratio_csa if ratio is None else ratio
    _check(load().csa_quantize_index_keys_closed(ctypes.byref(layout.c), _ptr(k_idx), k_idx.shape[-1], ratio,
                                                 _ptr(k_fp8), _ptr(k_scale), _stream(stream)),
           "csa_quantize_index_keys_closed")
    return k_fp8, k_scale


def index_fp8_workspace_size(layout, n_heads_idx, d_idx, top_k, ratio=None):
    ratio = layout.ratio_csa if ratio is None else ratio
    n = ctypes.c_size_t(0)
    _check(load().csa_index_fp8_workspace_size(ctypes.byref(layout.c), n_heads_idx, d_idx, ratio, top_k,
                                               ctypes.byref(n)), "csa_index_fp8_workspace_size")
    return n.value


def lightning_index_topk_fp8(layout, q_idx, k_fp8, k_scale, top_k, idx_out=None, score_out=None, ws=None,
                             ratio=None, stream=None, with_scores=True):
    """lightning_index_topk on E4M3 keys (see quantize_index_keys)."""
    ratio = layout.ratio_csa if ratio is None else ratio
    dev = q_idx.device
    if idx_out is None:
        idx_out = torch.empty((layout.total_q, top_k), dtype=torch.int32, device=dev)
    if score_out is None and with_scores:
        score_out = torch.empty((layout.total_q, top_k), dtype=torch.float32, device=dev)
    HI, dI = q_idx.shape[-2], q_idx.shape[-1]
    ws, nb = _ws(index_fp8_workspace_size(layout, HI, dI, top_k, ratio), dev, ws)
    _check(load().lightning_index_topk_fp8(ctypes.byref(layout.c), _ptr(q_idx), _ptr(k_fp8), _ptr(k_scale), HI, dI,
                                           ratio, top_k, _ptr(idx_out), _ptr(score_out), _ptr(ws), nb,
                                           _stream(stream)), "lightning_index_topk_fp8")
    return idx_out, score_out


STATIC_SCRATCH_BYTES = 32 << 20   # CSA_INDEX_STATIC_SCRATCH_BYTES


def lightning_index_topk_static(layout, q_idx, k_idx, top_k, idx_out=None, score_out=None, ratio=None, stream=None,
                                with_scores=True):
    """lightning_index_topk for callers that cannot allocate device memory.

    The library takes the scratch from its own fixed device array, so no
    workspace is passed or allocated for the call itself; only the outputs
    are created here when the caller does not pass them.
    """
    ratio = layout.ratio_csa if ratio is None else ratio
    dev = q_idx.device
    if idx_out is None:
        idx_out = torch.empty((layout.total_q, top_k), dtype=torch.int32, device=dev)
    if score_out is None and with_scores:
        score_out = torch.empty((layout.total_q, top_k), dtype=torch.float32, device=dev)
    HI, dI = q_idx.shape[-2], q_idx.shape[-1]
    _check(load().lightning_index_topk_static(ctypes.byref(layout.c), _ptr(q_idx), _ptr(k_idx), HI, dI, ratio,
                                              top_k, _ptr(idx_out), _ptr(score_out), _stream(stream)),
           "lightning_index_topk_static")
    return idx_out, score_out


def attend_workspace_size(layout, n_heads, d, ratio, top_k):
    n = ctypes.c_size_t(0)
    _check(load().csa_attend_workspace_size(ctypes.byref(layout.c), n_heads, d, ratio, top_k, ctypes.byref(n)),
           "csa_attend_workspace_size")
    return n.value


def sparse_mqa_attend(layout, q, csa_entries, kv, idx, top_k, scale, out=None, lse=None, ws=None, ratio=None,
                      stream=None):
    ratio = layout.ratio_csa if ratio is None else ratio
    H, d = q.shape[-2], q.shape[-1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((layout.total_q, H), dtype=torch.float32, device=q.device)
    ws, nb = _ws(attend_workspace_size(layout, H, d, ratio, top_k), q.device, ws)
    _check(load().sparse_mqa_attend(ctypes.byref(layout.c), _ptr(q), _ptr(csa_entries), _ptr(kv), _ptr(idx), H, d,
                                    ratio, top_k, float(scale), _ptr(out), _ptr(lse), _ptr(ws), nb,
                                    _stream(stream)), "sparse_mqa_attend")
    return out, lse


def hca_dense_attend(layout, q, hca_entries, kv, scale, out=None, lse=None, ws=None, ratio=None, stream=None):
    ratio = layout.ratio_hca if ratio is None else ratio
    H, d = q.shape[-2], q.shape[-1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((layout.total_q, H), dtype=torch.float32, device=q.device)
    ws, nb = _ws(attend_workspace_size(layout, H, d, ratio, 0), q.device, ws)
    _check(load().hca_dense_attend(ctypes.byref(layout.c), _ptr(q), _ptr(hca_entries), _ptr(kv), H, d, ratio,
                                   float(scale), _ptr(out), _ptr(lse), _ptr(ws), nb, _stream(stream)),
           "hca_dense_attend")
    return out, lse


def swa_workspace_size(layout, n_heads, d, window):
    n = ctypes.c_size_t(0)
    _check(load().swa_workspace_size(ctypes.byref(layout.c), n_heads, d, window, ctypes.byref(n)),
           "swa_workspace_size")
    return n.value


def swa_attend(layout, q, kv, window, scale, out=None, lse=None, ws=None, stream=None):
    """Sliding-window attention of each query over its own raw token and the
    window - 1 tokens before it (all heads share the tokens as keys and values)."""
    H, d = q.shape[-2], q.shape[-1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((layout.total_q, H), dtype=torch.float32, device=q.device)
    ws, nb = _ws(swa_workspace_size(layout, H, d, window), q.device, ws)
    _check(load().swa_attend(ctypes.byref(layout.c), _ptr(q), _ptr(kv), H, d, int(window), float(scale), _ptr(out),
                             _ptr(lse), _ptr(ws), nb, _stream(stream)), "swa_attend")
    return out, lse


def inverse_rope(layout, out, d_rope, base=10000.0, stream=None):
    """Inverse-RoPE correction of an attention output [total_q, H, d] in place:
    each query's last d_rope dims of every head, pairs (2i, 2i+1), turned by
    -t * base^(-2i/d_rope) for the query's position t."""
    H, d = out.shape[-2], out.shape[-1]
    _check(load().csa_inverse_rope(ctypes.byref(layout.c), _ptr(out), H, d, int(d_rope), float(base),
                                   _stream(stream)), "csa_inverse_rope")
    return out


class Hybrid:
    """One hybrid_attend problem: owns the parameter block and its buffers."""

    def __init__(self, layout, kv, gate, q_idx, k_idx, q, top_k, scale, csa_cache=None, hca_cache=None,
                 skip_compress=False, with_scores=False, ws=None, k_idx_fp8=None, outputs=None):
        """outputs: optional (o_csa, o_hca, lse_csa, lse_hca) device tensors to write into
        (e.g. views of one buffer that a single copy moves to the host)."""
        dev = q.device
        H, d = q.shape[-2], q.shape[-1]
        self.layout = layout
        self.kv, self.gate, self.q_idx, self.k_idx, self.q = kv, gate, q_idx, k_idx, q
        self.csa_cache = csa_cache if csa_cache is not None else \
            torch.empty((layout.total_csa, d), dtype=torch.bfloat16, device=dev)
        self.hca_cache = hca_cache if hca_cache is not None else \
            torch.empty((layout.total_hca, d), dtype=torch.bfloat16, device=dev)
        self.idx = torch.empty((layout.total_q, top_k), dtype=torch.int32, device=dev)
        self.score = torch.empty((layout.total_q, top_k), dtype=torch.float32, device=dev) if with_scores else None
        if outputs is not None:
            self.o_csa, self.o_hca, self.lse_csa, self.lse_hca = outputs
        else:
            self.o_csa = torch.empty_like(q)
            self.o_hca = torch.empty_like(q)
            self.lse_csa = torch.empty((layout.total_q, H), dtype=torch.float32, device=dev)
            self.lse_hca = torch.empty((layout.total_q, H), dtype=torch.float32, device=dev)
        p = csa_hybrid_params()
        p.layout = layout.c
        p.d, p.n_heads, p.n_heads_idx, p.d_idx = d, H, q_idx.shape[-2], q_idx.shape[-1]
        p.ratio_csa, p.ratio_hca, p.top_k = layout.ratio_csa, layout.ratio_hca, top_k
        # k_idx_fp8: (codes, scales) from quantize_index_keys; the indexer then reads them
        self.k_idx_fp8 = k_idx_fp8
        self._fp8 = CSA_INDEX_FP8 if k_idx_fp8 is not None else 0
        p.flags = (CSA_SKIP_COMPRESS if skip_compress else 0) | self._fp8
        p.scale = float(scale)
        if k_idx_fp8 is not None:
            p.k_idx_fp8 = _ptr(k_idx_fp8[0]).value
            p.k_idx_scale = _ptr(k_idx_fp8[1]).value
        for name, t in (("kv", kv), ("gate", gate), ("q_idx", q_idx), ("k_idx", k_idx), ("q", q),
                        ("csa_cache", self.csa_cache), ("hca_cache", self.hca_cache), ("idx_out", self.idx),
                        ("score_out", self.score), ("o_csa", self.o_csa), ("lse_csa", self.lse_csa),
                        ("o_hca", self.o_hca), ("lse_hca", self.lse_hca)):
            setattr(p, name, None if t is None else _ptr(t).value)
        n = ctypes.c_size_t(0)
        _check(load().csa_workspace_size(ctypes.byref(p), ctypes.byref(n)), "csa_workspace_size")
        self.ws, nb = _ws(n.value, dev, ws)
        p.ws = None if self.ws is None else self.ws.data_ptr()
        p.ws_bytes = nb
        self.params = p

    def set_flags(self, skip_compress):
        self.params.flags = (CSA_SKIP_COMPRESS if skip_compress else 0) | self._fp8

    def __call__(self, stream=None):
        _check(load().hybrid_attend(ctypes.byref(self.params), _stream(stream)), "hybrid_attend")
        return self


def check_device_error(stream=None):
    st = ctypes.c_int(0)
    _check(load().csa_check_device_error(_stream(stream), ctypes.byref(st)), "csa_check_device_error")
    return st.value


def timing_enable(on=True):
    load().csa_timing_enable(1 if on else 0)


def timing_reset():
    load().csa_timing_reset()


def timing_read():
    lib = load()
    n = lib.csa_timing_read(0, None, None, None)
    names = (ctypes.c_char_p * max(n, 1))()
    launches = (ctypes.c_int64 * max(n, 1))()
    ms = (ctypes.c_double * max(n, 1))()
    n = lib.csa_timing_read(n, names, launches, ms)
    return {names[i].decode(): (int(launches[i]), float(ms[i])) for i in range(n)}
