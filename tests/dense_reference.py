"""Dense brute-force attention used to pin the CPU oracle (tests only).

It is written independently of the oracle: it reads each sequence's keys and
values back out of the pool through the flat slot index
``slot = block_tables[s][pos // P] * P + pos % P`` (the slot_mapping
arithmetic of vLLM 0.10.2 differential_flash_attn.py's metadata builder),
takes the new tokens from the inputs (quantised through torch's own
float8_e4m3fn cast for fp8 caches, and the queries too when q_scale is
set), and evaluates
``softmax(scale * Q K^T + mask) V`` as whole numpy matrices in fp64 with a
dense causal/window mask and an extra sink column.
"""
from __future__ import annotations

import numpy as np
import torch


def flat_slots(w, s: int, positions) -> np.ndarray:
    positions = np.asarray(positions, dtype=np.int64)
    pages = w.block_tables[s * w.pages_per_seq + positions // w.page_size].astype(np.int64)
    return pages * w.page_size + positions % w.page_size


def fp8_roundtrip(x_bf16: torch.Tensor, scale: float) -> np.ndarray:
    """bf16 -> (x / scale in fp32) -> e4m3 (torch cast) -> value * scale, fp64."""
    q = (x_bf16.float() / torch.tensor(np.float32(scale))).to(torch.float8_e4m3fn)
    return q.to(torch.float64).numpy() * float(np.float32(scale))


def head_scales(w, kind: str) -> np.ndarray:
    """[Hkv] fp64 values of the fp32 key ("k") or value ("v") scales: the
    per-head ones when the workload has them, else the scalar repeated."""
    per_head = w.k_scale_heads if kind == "k" else w.v_scale_heads
    scalar = w.k_scale if kind == "k" else w.v_scale
    if per_head is None:
        return np.full(w.num_kv_heads, float(np.float32(scalar)))
    return np.asarray(per_head, np.float32).astype(np.float64)


def pool_values(w, pool: torch.Tensor) -> np.ndarray:
    """The pool as fp64 numbers [num_pages*P, 2Hkv, D] (fp8 codes dequantised
    with torch's float8_e4m3fn, channel 2h by head h's key scale and 2h+1 by
    its value scale)."""
    shape = (w.num_pages * w.page_size, 2 * w.num_kv_heads, w.head_dim)
    if w.kv_dtype == "fp8":
        vals = pool.view(torch.float8_e4m3fn).to(torch.float64).numpy().reshape(shape)
        chan = np.empty(2 * w.num_kv_heads)
        chan[0::2] = head_scales(w, "k")
        chan[1::2] = head_scales(w, "v")
        return vals * chan[None, :, None]
    return pool.to(torch.float64).numpy().reshape(shape)


def logical_kv(w, pool_before: torch.Tensor, keys, values, s: int):
    """K, V of sequence s as [kv_len, Hkv, D] fp64: context from the pool
    (before the call), new tokens from the inputs."""
    qsl = w.query_start_loc
    q0, q1 = int(qsl[s]), int(qsl[s + 1])
    q_len = q1 - q0
    kv_len = int(w.kv_lens_valid[s])
    ctx = kv_len - q_len
    Hkv = w.num_kv_heads
    vals = pool_values(w, pool_before)
    slots = flat_slots(w, s, np.arange(ctx))
    K = np.empty((kv_len, Hkv, w.head_dim))
    V = np.empty((kv_len, Hkv, w.head_dim))
    K[:ctx] = vals[slots][:, 0::2, :]
    V[:ctx] = vals[slots][:, 1::2, :]
    if w.kv_dtype == "fp8":
        ks, vs = head_scales(w, "k"), head_scales(w, "v")
        for h in range(Hkv):
            K[ctx:, h] = fp8_roundtrip(keys[q0:q1, h], ks[h])
            V[ctx:, h] = fp8_roundtrip(values[q0:q1, h], vs[h])
    else:
        K[ctx:] = keys[q0:q1].to(torch.float64).numpy()
        V[ctx:] = values[q0:q1].to(torch.float64).numpy()
    return K, V


def dense_attention(w, queries, keys, values, pool_before, sink=None) -> np.ndarray:
    """[num_query_tokens, Hq, D] fp64."""
    qsl = w.query_start_loc
    g = w.group
    out = np.zeros((w.num_query_tokens, w.num_q_heads, w.head_dim))
    sc = float(np.float32(w.softmax_scale))
    cap = float(np.float32(w.logits_soft_cap))
    for s in range(w.num_seqs):
        q0, q1 = int(qsl[s]), int(qsl[s + 1])
        if q1 == q0:
            continue
        K, V = logical_kv(w, pool_before, keys, values, s)
        kv_len = K.shape[0]
        ctx = kv_len - (q1 - q0)
        pos = ctx + np.arange(q1 - q0)[:, None]
        j = np.arange(kv_len)[None, :]
        allowed = j <= pos
        if w.sliding_window:
            allowed &= (pos - j) < w.sliding_window
        if getattr(w, "q_scale", 0.0):
            Q = fp8_roundtrip(queries[q0:q1], w.q_scale)
        else:
            Q = queries[q0:q1].to(torch.float64).numpy()
        for hq in range(w.num_q_heads):
            h = hq // g
            S = sc * (Q[:, hq, :] @ K[:, h, :].T)
            if cap > 0:
                S = cap * np.tanh(S / cap)
            S = np.where(allowed, S, -np.inf)
            if sink is not None:
                S = np.concatenate([S, np.full((S.shape[0], 1), float(sink[hq]))], axis=1)
            S = S - S.max(axis=1, keepdims=True)
            E = np.exp(S)
            Pm = E / E.sum(axis=1, keepdims=True)
            out[q0:q1, hq, :] = Pm[:, :kv_len] @ V[:, h, :]
    return out


def expected_pool_after(w, pool_before: torch.Tensor, keys, values) -> torch.Tensor:
    """The pool after the page write, by flat slot index (torch's fp8 cast)."""
    pool = pool_before.clone()
    flat = pool.view(w.num_pages * w.page_size, 2 * w.num_kv_heads, w.head_dim)
    qsl = w.query_start_loc
    for s in range(w.num_seqs):
        q0, q1 = int(qsl[s]), int(qsl[s + 1])
        ctx = int(w.kv_lens_valid[s]) - (q1 - q0)
        slots = torch.as_tensor(flat_slots(w, s, ctx + np.arange(q1 - q0)))
        if len(slots) == 0:
            continue
        k, v = keys[q0:q1], values[q0:q1]
        if w.kv_dtype == "fp8":
            ks = torch.tensor(head_scales(w, "k").astype(np.float32))[None, :, None]
            vs = torch.tensor(head_scales(w, "v").astype(np.float32))[None, :, None]
            k = (k.float() / ks).to(torch.float8_e4m3fn).view(torch.uint8)
            v = (v.float() / vs).to(torch.float8_e4m3fn).view(torch.uint8)
        flat[slots, 0::2, :] = k
        flat[slots, 1::2, :] = v
    return pool
