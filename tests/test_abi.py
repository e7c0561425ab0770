"""CPU checks of the C-ABI library: it builds for sm_103a, loads, exports every
symbol include/csa.h declares, and rejects bad arguments on the host before
any CUDA call (no GPU needed for any of these)."""
import ctypes
import os
import re

import pytest

from compressed_sparse_attention_21_b300 import _lib
from compressed_sparse_attention_21_b300 import build as csa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


@pytest.fixture(scope="module")
def lib():
    csa_build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "return", "sizeof")))


def test_header_declarations_match_binding_list():
    assert sorted(_lib.EXPORTS) == declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.csa_version() == 130
    assert lib.csa_status_string(0) == b"ok"
    assert lib.csa_status_string(3) == b"workspace missing or too small"


def layout(**kw):
    fake = 256  # any non-null, 16-aligned value: host checks never dereference it
    base = dict(batch=1, max_kv_len=16, max_q_len=1, reserved=0, cu_kv=fake, cu_q=fake, cu_csa=fake,
                cu_hca=fake, total_kv=16, total_q=1, total_csa=4, total_hca=0)
    base.update(kw)
    return _lib.csa_layout(**base)


BAD_LAYOUTS = [dict(batch=0), dict(reserved=1), dict(cu_kv=None), dict(max_kv_len=0),
               dict(max_q_len=17), dict(total_q=2), dict(total_kv=17), dict(total_kv=-1)]


@pytest.mark.parametrize("bad", BAD_LAYOUTS)
def test_bad_layout_rejected_on_host(lib, bad):
    L = layout(**bad)
    rc = lib.csa_compress(ctypes.byref(L), 256, 256, 128, 4, 256, None)
    assert rc == 1
    rc = lib.lightning_index_topk(ctypes.byref(L), 256, 256, 2, 32, 4, 8, 256, None, None, 0, None)
    assert rc == 1


def test_unsupported_sizes_rejected_on_host(lib):
    L = layout()
    assert lib.csa_compress(ctypes.byref(L), 256, 256, 96, 4, 256, None) == 2        # d
    assert lib.csa_compress(ctypes.byref(L), 256, 256, 128, 3, 256, None) == 2       # ratio
    assert lib.lightning_index_topk(ctypes.byref(L), 256, 256, 2, 48, 4, 8, 256, None, None, 0, None) == 2
    assert lib.lightning_index_topk(ctypes.byref(L), 256, 256, 2, 32, 4, 4096, 256, None, None, 0, None) == 2
    assert lib.sparse_mqa_attend(ctypes.byref(L), 256, 256, 256, 256, 32, 128, 4, 8, 1.0, 256, None, None, 0,
                                 None) == 2                                            # 32 heads
    assert lib.hca_dense_attend(ctypes.byref(L), 256, 256, 256, 8, 256, 128, 1.0, 256, None, None, 0,
                                None) == 2                                             # d = 256


def test_misaligned_or_null_pointers_rejected(lib):
    L = layout()
    assert lib.csa_compress(ctypes.byref(L), 258, 256, 128, 4, 256, None) == 1       # kv misaligned
    assert lib.csa_compress(ctypes.byref(L), 256, None, 128, 4, 256, None) == 1      # gate missing
    assert lib.sparse_mqa_attend(ctypes.byref(L), 256, 256, 256, None, 8, 128, 4, 8, 1.0, 256, None, None, 0,
                                 None) == 1                                            # idx missing
    assert lib.csa_workspace_init(None, 16, None) == 1


def test_layout_helper_host_logic():
    pytest.importorskip("torch")
    assert _lib.prefix([3, 0, 5]) == [0, 3, 3, 8]
    with pytest.raises(ValueError):
        _lib.Layout([4, 5], [5, 1], device="cpu")
    L = _lib.Layout([10, 300, 7], [10, 1, 2], ratio_csa=4, ratio_hca=128, device="cpu")
    assert L.host["cu_csa"] == [0, 2, 77, 78]
    assert L.host["cu_hca"] == [0, 0, 2, 2]
    assert (L.total_q, L.max_kv_len, L.max_q_len) == (13, 300, 10)


def test_ops_refuse_cpu_tensors():
    torch = pytest.importorskip("torch")
    L = _lib.Layout([8], [8], device="cpu")
    kv = torch.zeros(8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        _lib.csa_compress(L, kv, torch.zeros(8), torch.zeros(2, 128, dtype=torch.bfloat16))


def test_fp8_index_entry_points_check_arguments_on_host(lib):
    L = layout()
    n = ctypes.c_size_t(0)
    # quantiser: unsupported width, missing codes, misaligned or missing scales
    assert lib.csa_quantize_index_keys(ctypes.byref(L), 256, 48, 256, 256, None) == 2
    assert lib.csa_quantize_index_keys(ctypes.byref(L), 256, 64, None, 256, None) == 1
    assert lib.csa_quantize_index_keys(ctypes.byref(L), 256, 64, 256, 258, None) == 1
    assert lib.csa_quantize_index_keys(ctypes.byref(L), 256, 64, 256, None, None) == 1
    # the closed-rows form: bad ratio, unsupported width, misaligned scales
    assert lib.csa_quantize_index_keys_closed(ctypes.byref(L), 256, 64, 0, 256, 256, None) == 1
    assert lib.csa_quantize_index_keys_closed(ctypes.byref(L), 256, 48, 4, 256, 256, None) == 2
    assert lib.csa_quantize_index_keys_closed(ctypes.byref(L), 256, 64, 4, 256, 258, None) == 1
    assert lib.csa_quantize_index_keys_closed(ctypes.byref(L), None, 64, 4, 256, 256, None) == 1
    # FP8 indexer: missing or misaligned scales, missing codes, unsupported sizes
    assert lib.lightning_index_topk_fp8(ctypes.byref(L), 256, 256, None, 2, 32, 4, 8, 256, None, None, 0,
                                        None) == 1
    assert lib.lightning_index_topk_fp8(ctypes.byref(L), 256, 256, 258, 2, 32, 4, 8, 256, None, None, 0,
                                        None) == 1
    assert lib.lightning_index_topk_fp8(ctypes.byref(L), 256, None, 256, 2, 32, 4, 8, 256, None, None, 0,
                                        None) == 1
    assert lib.lightning_index_topk_fp8(ctypes.byref(L), 256, 256, 256, 2, 48, 4, 8, 256, None, None, 0,
                                        None) == 2
    assert lib.csa_index_fp8_workspace_size(ctypes.byref(L), 2, 32, 4, 8, None) == 1
    assert lib.csa_index_fp8_workspace_size(ctypes.byref(L), 2, 32, 4, 8, ctypes.byref(n)) == 0
    # rows longer than the FP8 select holds (262144 entries at ratio 4) are refused
    long_L = layout(max_kv_len=4 * 262144 + 4, total_kv=4 * 262144 + 4, total_csa=262145)
    assert lib.csa_index_fp8_workspace_size(ctypes.byref(long_L), 2, 32, 4, 8, ctypes.byref(n)) == 2
    assert lib.lightning_index_topk_fp8(ctypes.byref(long_L), 256, 256, 256, 2, 32, 4, 8, 256, None, None, 0,
                                        None) == 2


def test_hybrid_flags_checked_on_host(lib):
    p = _lib.csa_hybrid_params()
    p.layout = layout()
    p.d, p.n_heads, p.n_heads_idx, p.d_idx, p.ratio_csa, p.ratio_hca, p.top_k = 128, 8, 2, 32, 4, 128, 8
    p.scale = 1.0
    for name in ("kv", "gate", "q_idx", "k_idx", "q", "csa_cache", "hca_cache", "idx_out", "o_csa", "o_hca"):
        setattr(p, name, 256)
    p.flags = 0x4                                            # no such flag
    assert lib.hybrid_attend(ctypes.byref(p), None) == 1
    p.flags = _lib.CSA_INDEX_FP8                             # FP8 keys named but not given
    assert lib.hybrid_attend(ctypes.byref(p), None) == 1
    p.k_idx_fp8 = 256
    p.k_idx_scale = 258                                      # scales misaligned
    assert lib.hybrid_attend(ctypes.byref(p), None) == 1
    # with valid arguments the host checks pass and, without a GPU, the call
    # stops at the device (status 4).  Where a GPU is present these fake
    # pointers must never reach a launch, so the control runs only without one.
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        p.k_idx_scale = 256
        assert lib.hybrid_attend(ctypes.byref(p), None) == 4
        assert lib.csa_quantize_index_keys(ctypes.byref(layout()), 256, 64, 256, 256, None) == 4


def test_swa_arguments_checked_on_host(lib):
    # swa_attend reads only cu_kv and cu_q of the layout; a window below one,
    # an unsupported head count or d, a missing or misaligned pointer and a
    # bad layout are refused before anything runs
    L = layout(cu_csa=None, cu_hca=None)
    need = ctypes.c_size_t(0)
    for bad_window in (0, -5):
        assert lib.swa_attend(ctypes.byref(L), 256, 256, 8, 128, bad_window, 1.0, 256, None, None, 0, None) == 1
        assert lib.swa_workspace_size(ctypes.byref(L), 8, 128, bad_window, ctypes.byref(need)) == 1
    assert lib.swa_attend(ctypes.byref(L), 256, 256, 32, 128, 64, 1.0, 256, None, None, 0, None) == 2   # 32 heads
    assert lib.swa_attend(ctypes.byref(L), 256, 256, 8, 256, 64, 1.0, 256, None, None, 0, None) == 2   # d = 256
    assert lib.swa_attend(ctypes.byref(L), None, 256, 8, 128, 64, 1.0, 256, None, None, 0, None) == 1  # q
    assert lib.swa_attend(ctypes.byref(L), 256, 264, 8, 128, 64, 1.0, 256, None, None, 0, None) == 1   # kv
    assert lib.swa_attend(ctypes.byref(L), 256, 256, 8, 128, 64, 1.0, 256, 258, None, 0, None) == 1    # lse
    assert lib.swa_workspace_size(ctypes.byref(L), 8, 128, 64, None) == 1
    for bad in BAD_LAYOUTS:
        B = layout(**bad)
        assert lib.swa_attend(ctypes.byref(B), 256, 256, 8, 128, 64, 1.0, 256, None, None, 0, None) == 1, bad


def test_inverse_rope_arguments_checked_on_host(lib):
    L = layout(cu_csa=None, cu_hca=None)
    assert lib.csa_inverse_rope(ctypes.byref(L), 256, 8, 128, 12, 10000.0, None) == 2     # d_rope not a multiple of 8
    assert lib.csa_inverse_rope(ctypes.byref(L), 256, 8, 128, 136, 10000.0, None) == 2    # d_rope > d
    assert lib.csa_inverse_rope(ctypes.byref(L), 256, 8, 100, 64, 10000.0, None) == 2     # d not a multiple of 8
    assert lib.csa_inverse_rope(ctypes.byref(L), 256, 8, 1024, 1024, 10000.0, None) == 2  # d_rope > 512
    assert lib.csa_inverse_rope(ctypes.byref(L), 256, 0, 128, 64, 10000.0, None) == 1     # heads
    assert lib.csa_inverse_rope(ctypes.byref(L), 256, 8, 128, 64, 0.0, None) == 1         # base
    assert lib.csa_inverse_rope(ctypes.byref(L), 256, 8, 128, 64, float("inf"), None) == 1
    assert lib.csa_inverse_rope(ctypes.byref(L), None, 8, 128, 64, 10000.0, None) == 1    # out
    assert lib.csa_inverse_rope(ctypes.byref(L), 264, 8, 128, 64, 10000.0, None) == 1     # misaligned
    for bad in BAD_LAYOUTS:
        B = layout(**bad)
        assert lib.csa_inverse_rope(ctypes.byref(B), 256, 8, 128, 64, 10000.0, None) == 1, bad
