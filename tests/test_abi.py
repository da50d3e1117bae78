"""The C ABI loads and behaves on the host (no GPU needed).

Checks that librpa.so exports every function include/rpa.h declares, that
workspace sizing works, and that host-checkable argument errors are refused
before anything touches the GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from ragged_paged_attention_kv_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(rpa_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("rpa_forward", "rpa_update_cache", "rpa_workspace_size", "rpa_get_status",
                 "rpa_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


class _Ptr:
    """Stands in for a device tensor: only its address reaches the host checks."""

    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def _params(**over):
    from ragged_paged_attention_kv_gb300 import make_params
    kw = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, num_pages=80000,
              pages_per_seq=256, max_num_seqs=256, total_tokens=256)
    kw.update(over)
    return make_params(**kw)


def test_q_scale_accepted_with_an_fp8_cache(lib):
    n = ctypes.c_size_t(0)
    p = _params(kv_fp8=True, q_scale=0.05)
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0 and n.value > 0


def test_workspace_size_host_only(lib):
    from ragged_paged_attention_kv_gb300 import workspace_size
    n = workspace_size(_params())
    assert 0 < n < 1 << 30
    assert workspace_size(_params(total_tokens=65536, max_num_seqs=2)) > 0


@pytest.mark.parametrize("head_dim", [64, 96, 128, 192, 256])
def test_supported_head_dims(lib, head_dim):
    n = ctypes.c_size_t(0)
    p = _params(head_dim=head_dim)
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0 and n.value > 0


@pytest.mark.parametrize("over,code", [
    (dict(head_dim=80), 2),
    (dict(head_dim=160), 2),
    (dict(head_dim=512), 2),
    (dict(kv_fp8=True, head_dim=96, page_size=1), 2),  # 96-byte fp8 rows need 2-row pages
    (dict(num_q_heads=24, num_kv_heads=8), 2),
    (dict(num_q_heads=30, num_kv_heads=8), 2),
    (dict(page_size=24), 2),
    (dict(num_pages=0), 1),
    (dict(sliding_window=-1), 1),
    (dict(k_scale=0.5), 1),              # bf16 cache needs unit scales
    (dict(kv_fp8=True, k_scale=0.0), 1),
    (dict(logits_soft_cap=-1.0), 1),
    (dict(softmax_scale=0.0), 1),
    (dict(softmax_scale=-0.5), 1),
    (dict(k_scale_heads=_Ptr(256)), 1),           # per-head scales need an fp8 cache
    (dict(kv_fp8=True, v_scale_heads=_Ptr(258)), 1),  # misaligned per-head scales
    (dict(q_scale=0.05), 1),                      # quantised queries need an fp8 cache
    (dict(kv_fp8=True, q_scale=-0.05), 1),
    (dict(kv_fp8=True, q_scale=float("inf")), 1),
    (dict(kv_fp8=True, q_scale=float("nan")), 1),
])
def test_invalid_params_are_refused(lib, over, code):
    n = ctypes.c_size_t(0)
    p = _params(**over)
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == code
    # rpa_forward refuses the same params before touching any pointer or the GPU
    z = ctypes.c_void_p(16)
    assert lib.rpa_forward(ctypes.byref(p), z, z, z, z, z, z, z, z, None, z, z, 1 << 40, None) == code


def test_null_pointers_and_workspace_are_refused(lib):
    p = _params()
    z = ctypes.c_void_p(256)
    assert lib.rpa_forward(ctypes.byref(p), None, z, z, z, z, z, z, z, None, z, z, 1 << 40, None) == 1
    n = ctypes.c_size_t(0)
    lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n))
    # too small, misaligned, null
    assert lib.rpa_forward(ctypes.byref(p), z, z, z, z, z, z, z, z, None, z, z, n.value - 1, None) == 3
    assert lib.rpa_forward(ctypes.byref(p), z, z, z, z, z, z, z, z, None, z,
                           ctypes.c_void_p(257), n.value, None) == 3
    assert lib.rpa_forward(ctypes.byref(p), z, z, z, z, z, z, z, z, None, z, None, n.value, None) == 3
    assert lib.rpa_update_cache(ctypes.byref(p), None, z, z, z, z, z, z, z, n.value, None) == 1
    assert lib.rpa_get_status(None, None, None) == 1


def test_status_strings(lib):
    for code in range(5):
        assert lib.rpa_status_string(code)
    assert lib.rpa_status_string(99) == b"unknown code"


def test_binding_raises_without_library(monkeypatch, tmp_path):
    from ragged_paged_attention_kv_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.load()


@pytest.mark.parametrize("which", ["queries", "keys", "values", "kv_cache", "out", "kv_lens",
                                   "block_tables", "query_start_loc", "distribution", "sink"])
def test_misaligned_pointers_are_refused_before_any_gpu_work(lib, which):
    """Valid params with one misaligned pointer: refused on the host
    (checked before the workspace and before any CUDA call)."""
    p = _params()
    ptrs = {k: ctypes.c_void_p(1 << 20) for k in ("queries", "keys", "values", "kv_cache", "out",
                                                  "kv_lens", "block_tables", "query_start_loc",
                                                  "distribution", "sink")}
    ptrs[which] = ctypes.c_void_p((1 << 20) + (8 if which in ("queries", "keys", "values",
                                                              "kv_cache", "out") else 2))
    ws = ctypes.c_void_p(1 << 21)
    rc = lib.rpa_forward(ctypes.byref(p), ptrs["queries"], ptrs["keys"], ptrs["values"],
                         ptrs["kv_cache"], ptrs["kv_lens"], ptrs["block_tables"],
                         ptrs["query_start_loc"], ptrs["distribution"], ptrs["sink"],
                         ptrs["out"], ws, 1 << 40, None)
    assert rc == 1
    if which in ("keys", "values", "kv_cache", "kv_lens", "block_tables", "query_start_loc",
                 "distribution"):
        rc = lib.rpa_update_cache(ctypes.byref(p), ptrs["keys"], ptrs["values"], ptrs["kv_cache"],
                                  ptrs["kv_lens"], ptrs["block_tables"], ptrs["query_start_loc"],
                                  ptrs["distribution"], ws, 1 << 40, None)
        assert rc == 1


def test_binding_rejects_mismatched_head_dims():
    import torch
    import ragged_paged_attention_kv_gb300 as rpa
    T, S = 4, 2
    q = torch.zeros(T, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(T, 2, 32, dtype=torch.bfloat16)
    cache = torch.zeros(4, 16, 4, 32, dtype=torch.bfloat16)
    i32 = lambda n: torch.zeros(n, dtype=torch.int32)  # noqa: E731
    with pytest.raises(ValueError):
        rpa.forward(q, k, k.clone(), cache, i32(S), i32(S * 4), i32(S + 1), i32(3))
