"""CPU oracle for ragged paged attention -- TEST INFRASTRUCTURE ONLY.

The slow, plain fp64 definition (``rpa_oracle.c``) that the CUDA library is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library itself
never does, and the two share no code.

The C source is compiled on first use with the host's gcc (``build()``); the
functions here only marshal numpy arrays to it.  Every function states what it
follows; the numeric definitions live in ``rpa_oracle.c``:

* ``update_cache`` -- new-KV page write (tpu-inference 0.12.0 RPA v3
  kernel.py, ``_update_kv_cache``; positions from vLLM 0.10.2
  differential_flash_attn.py metadata, seq_len = context_len + query_len).
* ``attention`` / ``attention_rows`` -- exact softmax attention with GQA,
  causal mask, sliding window, soft cap, sink, fp8 scales (RPA v3 kernel's
  ``flash_attention_step1_qk_softmax`` / ``step2_pv`` reach the same value;
  options from the ejkernel ``ragged_page_attention_v3`` interface).
* ``e4m3_encode`` / ``e4m3_decode`` / ``quantize`` -- the fp8 KV format
  (tpu-inference 0.11.1rc3 layers/vllm/attention.py, ``quantize_kv``);
  with ``q_scale`` the queries are quantised the same way (w8a8: the
  ejkernel interface's ``q_scale``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rpa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "librpa_oracle.so")
_lock = threading.Lock()
_lib = None


class OracleParams(ctypes.Structure):
    _fields_ = [
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("pages_per_seq", ctypes.c_int32),
        ("max_num_seqs", ctypes.c_int32),
        ("total_tokens", ctypes.c_int32),
        ("kv_fp8", ctypes.c_int32),
        ("sliding_window", ctypes.c_int32),
        ("softmax_scale", ctypes.c_double),
        ("logits_soft_cap", ctypes.c_double),
        ("k_scale", ctypes.c_double),
        ("v_scale", ctypes.c_double),
        ("k_scale_heads", ctypes.POINTER(ctypes.c_double)),
        ("v_scale_heads", ctypes.POINTER(ctypes.c_double)),
        ("q_scale", ctypes.c_double),
    ]


ORACLE_OK, ORACLE_BAD_ARG, ORACLE_BAD_METADATA, ORACLE_BAD_PAGE = 0, 1, 2, 3


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__(f"oracle rejected the call (code {code})")
        self.code = code


def build(force: bool = False) -> str:
    """Compile ``rpa_oracle.c`` into ``_build/librpa_oracle.so`` with gcc."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        vp = ctypes.c_void_p
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quantize.argtypes = [ctypes.c_uint16, ctypes.c_double]
        lib.oracle_quantize.restype = ctypes.c_uint8
        lib.oracle_check_distribution.argtypes = [P(OracleParams), vp, vp]
        lib.oracle_check_distribution.restype = ctypes.c_int
        lib.oracle_update_cache.argtypes = [P(OracleParams), vp, vp, vp, vp, vp,
                                            vp, ctypes.c_int32]
        lib.oracle_update_cache.restype = ctypes.c_int
        lib.oracle_attention_rows.argtypes = [
            P(OracleParams), vp, vp, vp, vp, vp, ctypes.c_int32, vp, vp,
            ctypes.c_int32, vp, ctypes.c_int32]
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_forward.argtypes = [P(OracleParams), vp, vp, vp, vp, vp, vp,
                                       vp, ctypes.c_int32, vp, vp,
                                       ctypes.c_int32]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def make_params(*, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                pages_per_seq, max_num_seqs, total_tokens, kv_fp8=False,
                sliding_window=0, softmax_scale=1.0, logits_soft_cap=0.0,
                k_scale=1.0, v_scale=1.0, k_scale_heads=None, v_scale_heads=None,
                q_scale=None) -> OracleParams:
    """Scales are fp32 numbers in the interface; they are rounded to fp32 here.
    ``k_scale_heads`` / ``v_scale_heads``: optional per-kv-head scales (fp8).
    ``q_scale``: fp8 only, quantises the queries (None or 0 = off)."""
    f32 = lambda x: float(np.float32(x))

    def heads(x):
        if x is None:
            return None, None
        a = np.asarray(x, dtype=np.float32).astype(np.float64)
        if a.shape != (int(num_kv_heads),):
            raise ValueError("per-head scales need num_kv_heads entries")
        a = np.ascontiguousarray(a)
        return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))

    kh, kp = heads(k_scale_heads)
    vh, vp = heads(v_scale_heads)
    p = OracleParams(int(num_q_heads), int(num_kv_heads), int(head_dim),
                     int(page_size), int(num_pages), int(pages_per_seq),
                     int(max_num_seqs), int(total_tokens), int(bool(kv_fp8)),
                     int(sliding_window or 0), f32(softmax_scale),
                     f32(logits_soft_cap or 0.0), f32(k_scale), f32(v_scale), kp, vp,
                     f32(q_scale or 0.0))
    p._keep = (kh, vh)  # the arrays must live as long as the params
    return p


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits16(x):
    """bf16 data as uint16 bit patterns (accepts uint16 or a torch bf16 tensor)."""
    if hasattr(x, "dtype") and str(getattr(x, "dtype", "")) == "torch.bfloat16":
        x = x.contiguous().view(dtype=__import__("torch").int16).numpy().view(np.uint16)
    return _c(x, np.uint16)


def _cache_bytes(cache):
    if hasattr(cache, "numpy"):  # torch tensor (bf16 or fp8 or uint8)
        import torch
        cache = cache.contiguous().view(torch.uint8).numpy()
    return np.ascontiguousarray(cache).view(np.uint8)


def check_distribution(p: OracleParams, distribution, query_start_loc) -> int:
    d = _c(distribution, np.int32)
    q = _c(query_start_loc, np.int32)
    return int(_load().oracle_check_distribution(ctypes.byref(p), _ptr(d), _ptr(q)))


def update_cache(p: OracleParams, keys, values, kv_cache, kv_lens, block_tables,
                 query_start_loc, num_seqs):
    """Writes the new keys/values into ``kv_cache`` (a uint8 byte view of the
    pool, modified in place; the same memory is returned)."""
    k, v = _bits16(keys), _bits16(values)
    cache = _cache_bytes(kv_cache)
    if not cache.flags.writeable:
        raise ValueError("kv_cache must be writeable")
    kl = _c(kv_lens, np.int32)
    bt = _c(block_tables, np.int32)
    qsl = _c(query_start_loc, np.int32)
    rc = _load().oracle_update_cache(ctypes.byref(p), _ptr(k), _ptr(v), _ptr(cache),
                                     _ptr(kl), _ptr(bt), _ptr(qsl), int(num_seqs))
    if rc:
        raise OracleError(rc)
    return cache


def attention_rows(p: OracleParams, queries, kv_cache, kv_lens, block_tables,
                   query_start_loc, num_seqs, tokens, attention_sink=None,
                   nthreads=0):
    """fp64 attention for the query tokens in ``tokens`` (all q-heads);
    keys/values come from the (already updated) pool."""
    q = _bits16(queries)
    cache = _cache_bytes(kv_cache)
    kl = _c(kv_lens, np.int32)
    bt = _c(block_tables, np.int32)
    qsl = _c(query_start_loc, np.int32)
    toks = _c(np.asarray(tokens, dtype=np.int32), np.int32)
    sink = None if attention_sink is None else _c(np.asarray(attention_sink, np.float32), np.float32)
    out = np.zeros((len(toks), p.num_q_heads, p.head_dim), dtype=np.float64)
    rc = _load().oracle_attention_rows(ctypes.byref(p), _ptr(q), _ptr(cache), _ptr(kl),
                                       _ptr(bt), _ptr(qsl), int(num_seqs), _ptr(sink),
                                       _ptr(toks), len(toks), _ptr(out), int(nthreads))
    if rc:
        raise OracleError(rc)
    return out


def forward(p: OracleParams, queries, keys, values, kv_cache, kv_lens,
            block_tables, query_start_loc, num_seqs, attention_sink=None,
            nthreads=0):
    """Whole call: page write (in place on ``kv_cache``) then attention of all
    ``query_start_loc[num_seqs]`` tokens.  Returns (out fp64, cache bytes)."""
    q, k, v = _bits16(queries), _bits16(keys), _bits16(values)
    cache = _cache_bytes(kv_cache)
    kl = _c(kv_lens, np.int32)
    bt = _c(block_tables, np.int32)
    qsl = _c(query_start_loc, np.int32)
    sink = None if attention_sink is None else _c(np.asarray(attention_sink, np.float32), np.float32)
    n = int(qsl[num_seqs])
    out = np.zeros((n, p.num_q_heads, p.head_dim), dtype=np.float64)
    rc = _load().oracle_forward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(cache),
                                _ptr(kl), _ptr(bt), _ptr(qsl), int(num_seqs), _ptr(sink),
                                _ptr(out), int(nthreads))
    if rc:
        raise OracleError(rc)
    return out, cache


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_decode(int(x)) for x in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    lib = _load()
    a = np.asarray(x, dtype=np.float32)
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in a.ravel()],
                    dtype=np.uint8).reshape(a.shape)


def quantize(bf16_bits, scale) -> np.ndarray:
    lib = _load()
    b = _bits16(bf16_bits)
    s = float(np.float32(scale))
    return np.array([lib.oracle_quantize(int(x), s) for x in b.ravel()],
                    dtype=np.uint8).reshape(b.shape)


def bf16_to_double(bits) -> np.ndarray:
    lib = _load()
    b = _bits16(bits)
    return np.array([lib.oracle_bf16_to_double(int(x)) for x in b.ravel()],
                    dtype=np.float64).reshape(b.shape)
