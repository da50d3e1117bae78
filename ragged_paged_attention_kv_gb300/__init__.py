"""Ragged paged attention for GB300 (sm_103a): Python binding of librpa.so.

The functions here only check tensors and pass their device pointers to the C
ABI declared in ``include/rpa.h``; every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  If librpa.so is missing, the first call raises -- there is no
fallback.

    out = forward(queries, keys, values, kv_cache, kv_lens, block_tables,
                  query_start_loc, distribution, attention_sink=None,
                  softmax_scale=..., sliding_window=None, logits_soft_cap=None,
                  k_scale=None, v_scale=None, q_scale=None)

``k_scale`` / ``v_scale`` are numbers, or (fp8 caches) float32 device tensors
of num_kv_heads entries for one scale per kv head; ``q_scale`` (fp8 caches)
quantises the queries to e4m3 as well (w8a8).  The argument list follows the ejkernel ``ragged_page_attention_v3``
interface; ``kv_cache`` is updated in place (the new keys/values are written
into their pages) instead of being returned.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import RpaError, RpaParams  # noqa: F401

__all__ = ["make_params", "workspace_size", "alloc_workspace", "forward", "update_cache",
           "get_status", "RpaError", "RpaParams"]


def make_params(*, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, pages_per_seq,
                max_num_seqs, total_tokens, kv_fp8=False, sliding_window=None,
                softmax_scale=1.0, logits_soft_cap=None, k_scale=None, v_scale=None,
                k_scale_heads=None, v_scale_heads=None, q_scale=None) -> RpaParams:
    """``k_scale_heads`` / ``v_scale_heads``: optional float32 device tensors of
    num_kv_heads per-head scales (fp8 caches); they must outlive the calls
    that use these params.  ``q_scale`` (fp8 caches): quantise the queries to
    e4m3 with this scale (None or 0 = off)."""
    return RpaParams(int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size),
                     int(num_pages), int(pages_per_seq), int(max_num_seqs), int(total_tokens),
                     _lib.RPA_KV_FP8_E4M3 if kv_fp8 else _lib.RPA_KV_BF16,
                     int(sliding_window or 0), float(softmax_scale), float(logits_soft_cap or 0.0),
                     float(1.0 if k_scale is None else k_scale),
                     float(1.0 if v_scale is None else v_scale),
                     None if k_scale_heads is None else k_scale_heads.data_ptr(),
                     None if v_scale_heads is None else v_scale_heads.data_ptr(),
                     float(q_scale or 0.0))


def workspace_size(params: RpaParams) -> int:
    n = ctypes.c_size_t(0)
    _lib.check("rpa_workspace_size", _lib.load().rpa_workspace_size(ctypes.byref(params), ctypes.byref(n)))
    return int(n.value)


def alloc_workspace(params: RpaParams, device=None) -> torch.Tensor:
    """A device byte buffer large enough for ``params`` (torch allocations are
    at least 256-byte aligned)."""
    return torch.empty(workspace_size(params), dtype=torch.uint8, device=device or "cuda")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtypes, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


_FP8_TYPES = (torch.uint8, torch.float8_e4m3fn)


def _scale_arg(x, name, Hkv, device):
    """(scalar, per-head tensor or None) for a k_scale / v_scale argument."""
    if isinstance(x, torch.Tensor):
        _need(x, name, (torch.float32,), device)
        if x.numel() != Hkv:
            raise ValueError(f"{name} as a tensor must have num_kv_heads entries")
        return 1.0, x
    return x, None


def _params_from(queries_or_none, keys, kv_cache, kv_lens, block_tables, softmax_scale,
                 sliding_window, logits_soft_cap, k_scale, v_scale, num_q_heads=None,
                 q_scale=None):
    T, Hkv, D = keys.shape
    k_scale, k_heads = _scale_arg(k_scale, "k_scale", Hkv, keys.device)
    v_scale, v_heads = _scale_arg(v_scale, "v_scale", Hkv, keys.device)
    num_pages, P, C, D2 = kv_cache.shape
    if C != 2 * Hkv or D2 != D:
        raise ValueError("kv_cache must be [num_pages, page_size, 2*num_kv_heads, head_dim]")
    fp8 = kv_cache.dtype in _FP8_TYPES
    max_num_seqs = kv_lens.numel()
    if block_tables.numel() % max_num_seqs:
        raise ValueError("block_tables must hold max_num_seqs * pages_per_seq entries")
    Hq = queries_or_none.shape[1] if queries_or_none is not None else (num_q_heads or Hkv)
    return make_params(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
                       num_pages=num_pages, pages_per_seq=block_tables.numel() // max_num_seqs,
                       max_num_seqs=max_num_seqs, total_tokens=T, kv_fp8=fp8,
                       sliding_window=sliding_window, softmax_scale=softmax_scale,
                       logits_soft_cap=logits_soft_cap, k_scale=k_scale, v_scale=v_scale,
                       k_scale_heads=k_heads, v_scale_heads=v_heads, q_scale=q_scale)


def forward(queries, keys, values, kv_cache, kv_lens, block_tables, query_start_loc,
            distribution, attention_sink=None, *, softmax_scale=1.0, sliding_window=None,
            logits_soft_cap=None, k_scale=None, v_scale=None, q_scale=None, out=None,
            workspace=None, stream=None, events=None) -> torch.Tensor:
    """Writes the new keys/values into ``kv_cache`` and returns the attention
    output [total_tokens, num_q_heads, head_dim] (bf16).  Asynchronous on the
    current (or given) stream; data-dependent problems are reported through
    ``get_status(workspace)``.  ``events`` (four timing-enabled
    torch.cuda.Event, already recorded once) selects rpa_forward_timed, which
    records them around the planner, decode and prefill kernels."""
    dev = queries.device
    _need(queries, "queries", (torch.bfloat16,), dev)
    _need(keys, "keys", (torch.bfloat16,), dev)
    _need(values, "values", (torch.bfloat16,), dev)
    _need(kv_cache, "kv_cache", (torch.bfloat16,) + _FP8_TYPES, dev)
    for name, t in (("kv_lens", kv_lens), ("block_tables", block_tables),
                    ("query_start_loc", query_start_loc), ("distribution", distribution)):
        _need(t, name, (torch.int32,), dev)
    if attention_sink is not None:
        _need(attention_sink, "attention_sink", (torch.float32,), dev)
    if (queries.dim() != 3 or keys.dim() != 3 or keys.shape != values.shape or
            keys.shape[0] != queries.shape[0] or keys.shape[2] != queries.shape[2]):
        raise ValueError("queries [T,Hq,D], keys/values [T,Hkv,D] expected")
    if query_start_loc.numel() != kv_lens.numel() + 1 or distribution.numel() != 3:
        raise ValueError("query_start_loc must have max_num_seqs+1 entries, distribution 3")
    params = _params_from(queries, keys, kv_cache, kv_lens, block_tables, softmax_scale,
                          sliding_window, logits_soft_cap, k_scale, v_scale, q_scale=q_scale)
    if attention_sink is not None and attention_sink.numel() != params.num_q_heads:
        raise ValueError("attention_sink must have num_q_heads entries")
    if out is None:
        out = torch.empty_like(queries)
    else:
        _need(out, "out", (torch.bfloat16,), dev)
        if out.shape != queries.shape:
            raise ValueError("out must have the shape of queries")
    if workspace is None:
        workspace = alloc_workspace(params, dev)
    _need(workspace, "workspace", (torch.uint8,), dev)
    args = (ctypes.byref(params), _ptr(queries), _ptr(keys), _ptr(values), _ptr(kv_cache),
            _ptr(kv_lens), _ptr(block_tables), _ptr(query_start_loc), _ptr(distribution),
            _ptr(attention_sink), _ptr(out), _ptr(workspace), workspace.numel(),
            _stream(stream, dev))
    if events is None:
        _lib.check("rpa_forward", _lib.load().rpa_forward(*args))
    else:
        handles = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
        _lib.check("rpa_forward_timed", _lib.load().rpa_forward_timed(*args, handles))
    return out


def update_cache(keys, values, kv_cache, kv_lens, block_tables, query_start_loc, distribution,
                 *, k_scale=None, v_scale=None, workspace=None, stream=None, num_q_heads=None):
    """The page write alone (bf16 copy or fp8 quantisation of the new keys/values)."""
    dev = keys.device
    _need(keys, "keys", (torch.bfloat16,), dev)
    _need(values, "values", (torch.bfloat16,), dev)
    _need(kv_cache, "kv_cache", (torch.bfloat16,) + _FP8_TYPES, dev)
    for name, t in (("kv_lens", kv_lens), ("block_tables", block_tables),
                    ("query_start_loc", query_start_loc), ("distribution", distribution)):
        _need(t, name, (torch.int32,), dev)
    params = _params_from(None, keys, kv_cache, kv_lens, block_tables, 1.0, None, None,
                          k_scale, v_scale, num_q_heads=num_q_heads)
    if workspace is None:
        workspace = alloc_workspace(params, dev)
    rc = _lib.load().rpa_update_cache(
        ctypes.byref(params), _ptr(keys), _ptr(values), _ptr(kv_cache), _ptr(kv_lens),
        _ptr(block_tables), _ptr(query_start_loc), _ptr(distribution), _ptr(workspace),
        workspace.numel(), _stream(stream, dev))
    _lib.check("rpa_update_cache", rc)
    return kv_cache


def get_status(workspace: torch.Tensor, stream=None) -> int:
    """The device status word of the last call on ``workspace`` (syncs the stream)."""
    st = ctypes.c_int32(0)
    rc = _lib.load().rpa_get_status(_ptr(workspace), _stream(stream, workspace.device),
                                    ctypes.byref(st))
    _lib.check("rpa_get_status", rc)
    return int(st.value)
