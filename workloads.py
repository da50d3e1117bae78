"""Seeded synthetic inputs for ragged paged attention.

This module only draws inputs: sequence lengths, page assignments, query /
key / value tensors, sinks and the prior contents of the page pool.  It holds
none of the attention arithmetic, so both the CUDA library's tests and the CPU
oracle can take their inputs from it.

Shapes follow the ejkernel ``ragged_page_attention_v3`` interface:
queries [T, Hq, D], keys/values [T, Hkv, D], kv_cache
[num_pages, page_size, 2*Hkv, D] (key head h in channel 2h, value head h in
channel 2h+1), kv_lens [max_num_seqs], block_tables
[max_num_seqs * pages_per_seq], query_start_loc [max_num_seqs + 1] and a
3-entry ``distribution`` (cumulative ends of the decode-only, chunked-prefill
and mixed classes).  ``kv_lens`` counts the new tokens too (vLLM 0.10.2
differential_flash_attn.py metadata: seq_len = context_len + query_len).

Named workloads (all q/k/v ~ N(0,1) in bf16; workload k draws everything
from ``torch.Generator().manual_seed(1000 + k)`` on the CPU):

  tiny     3 seqs (q,kv) = (1,17),(24,24),(5,40); Hq4/Hkv2/D64/P16;
           16-page pool, pages from a seeded permutation; scale 1/8.
  decode   256 seqs q=1, kv ~ U[512,4096]; Hq32/Hkv8/D128/P16; 80000-page
           pool, tables from a seeded shuffle; scale 1/sqrt(128).
  mixed    128 decode (kv ~ U[1024,8192]) + 8 chunks of 512 (prior kv ~
           U[0,4096]) + 2 fresh prefills of 1536; Hq64/Hkv8/D128/P32;
           distribution [128,136,138]; pool = pages used + 10%.
  long     2 seqs q = kv = 32768 causal; Hq32/Hkv8/D128/P64; 2048 pages;
           ``long_w4096`` adds sliding_window 4096.
  fp8      512 decode (kv ~ U[256,16384]) + 8 chunks of 256 (prior kv ~
           U[0,8192]); Hq64/Hkv8/D64/P16; fp8 e4m3 cache, k/v scale 0.05,
           soft cap 30, sinks ~ N(0,1), sliding_window 128, scale 1/8.
  decode_d256, long_d256
           head_dim 256 (Gemma-2-9B attention shape): 256 decode seqs with
           window 4096 and cap 50; 2 x 8192 causal prefill.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    pages_per_seq: int
    max_num_seqs: int
    kv_dtype: str                      # "bf16" or "fp8"
    softmax_scale: float
    sliding_window: int                # 0 = none
    logits_soft_cap: float             # 0 = none
    k_scale: float
    v_scale: float
    has_sink: bool
    q_lens: np.ndarray                 # [num_seqs] int32
    kv_lens_valid: np.ndarray          # [num_seqs] int32
    block_tables: np.ndarray           # [max_num_seqs * pages_per_seq] int32
    distribution: np.ndarray           # [3] int32
    total_tokens: int                  # rows of queries/keys/values/out
    # optional per-kv-head fp8 scales [num_kv_heads] (fp32 numbers); they
    # replace k_scale / v_scale head by head
    k_scale_heads: Optional[np.ndarray] = None
    v_scale_heads: Optional[np.ndarray] = None
    # fp8 caches: > 0 quantises the queries to e4m3 with this scale (w8a8)
    q_scale: float = 0.0

    # ------------------------------------------------------------- metadata
    @property
    def num_seqs(self) -> int:
        return int(len(self.q_lens))

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def query_start_loc(self) -> np.ndarray:
        qsl = np.zeros(self.max_num_seqs + 1, dtype=np.int32)
        qsl[1:self.num_seqs + 1] = np.cumsum(self.q_lens, dtype=np.int64)
        qsl[self.num_seqs + 1:] = qsl[self.num_seqs]
        return qsl

    @property
    def kv_lens(self) -> np.ndarray:
        kl = np.zeros(self.max_num_seqs, dtype=np.int32)
        kl[:self.num_seqs] = self.kv_lens_valid
        return kl

    @property
    def num_query_tokens(self) -> int:
        return int(self.q_lens.sum())

    @property
    def elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "fp8" else 2

    @property
    def pool_shape(self):
        return (self.num_pages, self.page_size, 2 * self.num_kv_heads, self.head_dim)

    @property
    def pool_bytes(self) -> int:
        return int(np.prod(self.pool_shape)) * self.elem_bytes

    def pages_of(self, s: int) -> np.ndarray:
        n = -(-int(self.kv_lens_valid[s]) // self.page_size)
        return self.block_tables[s * self.pages_per_seq: s * self.pages_per_seq + n]

    def params(self) -> dict:
        return dict(num_q_heads=self.num_q_heads, num_kv_heads=self.num_kv_heads,
                    head_dim=self.head_dim, page_size=self.page_size,
                    num_pages=self.num_pages, pages_per_seq=self.pages_per_seq,
                    max_num_seqs=self.max_num_seqs, total_tokens=self.total_tokens,
                    kv_fp8=self.kv_dtype == "fp8", sliding_window=self.sliding_window,
                    softmax_scale=self.softmax_scale,
                    logits_soft_cap=self.logits_soft_cap,
                    k_scale=self.k_scale, v_scale=self.v_scale,
                    **({} if self.k_scale_heads is None else {"k_scale_heads": self.k_scale_heads}),
                    **({} if self.v_scale_heads is None else {"v_scale_heads": self.v_scale_heads}),
                    **({} if not self.q_scale else {"q_scale": self.q_scale}))

    # --------------------------------------------------------------- tensors
    def _gen(self, stream: int) -> torch.Generator:
        return torch.Generator().manual_seed(self.seed * 16 + stream)

    def make_qkv(self):
        """(queries, keys, values) as CPU bf16 tensors, ~N(0,1)."""
        g = self._gen(1)
        T = self.total_tokens
        q = torch.randn(T, self.num_q_heads, self.head_dim, generator=g).to(torch.bfloat16)
        k = torch.randn(T, self.num_kv_heads, self.head_dim, generator=g).to(torch.bfloat16)
        v = torch.randn(T, self.num_kv_heads, self.head_dim, generator=g).to(torch.bfloat16)
        return q, k, v

    def make_sink(self) -> Optional[torch.Tensor]:
        if not self.has_sink:
            return None
        return torch.randn(self.num_q_heads, generator=self._gen(2)).to(torch.float32)

    def make_pool(self, device="cpu") -> torch.Tensor:
        """Prior pool contents: every slot (used or not) holds seeded data, so
        stray writes show up in a whole-pool compare.  bf16 pools hold
        N(0,1); fp8 pools hold the e4m3 codes of N(0,1)/k_scale (torch's own
        cast) as uint8."""
        device = torch.device(device)
        if device.type == "cuda":
            g = torch.Generator(device=device).manual_seed(self.seed * 16 + 3)
        else:
            g = self._gen(3)
        shape = self.pool_shape
        if self.kv_dtype == "bf16":
            pool = torch.empty(shape, dtype=torch.bfloat16, device=device)
            flat = pool.view(-1)
            step = 1 << 28
            for i in range(0, flat.numel(), step):
                n = min(step, flat.numel() - i)
                flat[i:i + n] = torch.randn(n, generator=g, device=device).to(torch.bfloat16)
            return pool
        pool = torch.empty(shape, dtype=torch.uint8, device=device)
        flat = pool.view(-1)
        step = 1 << 28
        for i in range(0, flat.numel(), step):
            n = min(step, flat.numel() - i)
            x = torch.randn(n, generator=g, device=device) * (1.0 / self.k_scale)
            flat[i:i + n] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        return pool

    # -------------------------------------------------------------- subsets
    def subset(self, seq_ids: Sequence[int], pool_before: Optional[torch.Tensor],
               slack_pages: int = 2):
        """A compact copy of the listed sequences for CPU checks.

        Returns (sub_workload, sub_pool_cpu, token_map) where the sub-workload
        keeps the same options, its pool holds only the pages those sequences
        use (copied from ``pool_before``, plus ``slack_pages`` spare pages)
        with the block tables renumbered, and token_map[i] is the row of the
        full batch that sub-batch row i came from.  With pool_before=None the
        compact pool is filled with fresh seeded data instead (for timing runs
        that never compare values)."""
        seq_ids = [int(s) for s in seq_ids]
        pages = [self.pages_of(s) for s in seq_ids]
        n_used = int(sum(len(p) for p in pages))
        n_pool = n_used + slack_pages
        pps = max(1, max(len(p) for p in pages))
        bt = np.zeros(len(seq_ids) * pps, dtype=np.int32)
        src = np.concatenate(pages).astype(np.int64) if n_used else np.zeros(0, np.int64)
        c = 0
        for i, p in enumerate(pages):
            bt[i * pps: i * pps + len(p)] = np.arange(c, c + len(p))
            c += len(p)
        if pool_before is None:
            tmp = dataclasses.replace(self, num_pages=n_pool)
            sub_pool = tmp.make_pool("cpu")
        else:
            idx = torch.as_tensor(src, device=pool_before.device)
            sub_pool = torch.empty((n_pool,) + tuple(pool_before.shape[1:]),
                                   dtype=pool_before.dtype)
            if n_used:
                sub_pool[:n_used] = pool_before.index_select(0, idx).cpu()
            if slack_pages:
                sub_pool[n_used:] = pool_before[:slack_pages].cpu()
        qsl = self.query_start_loc
        token_map = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seq_ids]).astype(np.int64) \
            if seq_ids else np.zeros(0, np.int64)
        sub = dataclasses.replace(
            self, name=f"{self.name}[subset]", num_pages=n_pool, pages_per_seq=pps,
            max_num_seqs=len(seq_ids), q_lens=self.q_lens[seq_ids].copy(),
            kv_lens_valid=self.kv_lens_valid[seq_ids].copy(), block_tables=bt,
            distribution=np.array([len(seq_ids)] * 3, np.int32),
            total_tokens=int(len(token_map)))
        return sub, sub_pool, token_map


# ------------------------------------------------------------------ builders
def _assign_pages(kv_lens: np.ndarray, page_size: int, num_pages: int,
                  max_num_seqs: int, pages_per_seq: int, g: torch.Generator):
    need = [-(-int(k) // page_size) for k in kv_lens]
    if sum(need) > num_pages:
        raise ValueError("pool too small")
    perm = torch.randperm(num_pages, generator=g).numpy().astype(np.int32)
    bt = np.zeros(max_num_seqs * pages_per_seq, dtype=np.int32)
    c = 0
    for s, n in enumerate(need):
        bt[s * pages_per_seq: s * pages_per_seq + n] = perm[c:c + n]
        c += n
    return bt


def make_custom(name: str, seed: int, q_lens, kv_lens, *, num_q_heads, num_kv_heads,
                head_dim, page_size, num_pages=None, pool_slack=0.1, pages_per_seq=None,
                max_num_seqs=None, kv_dtype="bf16", softmax_scale=None,
                sliding_window=0, logits_soft_cap=0.0, k_scale=1.0, v_scale=1.0,
                has_sink=False, distribution=None, extra_tokens=0, k_scale_heads=None,
                v_scale_heads=None, q_scale=0.0) -> Workload:
    """A workload from explicit per-sequence (q_len, kv_len) lists."""
    q_lens = np.asarray(q_lens, dtype=np.int32)
    kv_lens = np.asarray(kv_lens, dtype=np.int32)
    assert q_lens.shape == kv_lens.shape and np.all(kv_lens >= q_lens)
    S = len(q_lens)
    need = int(sum(-(-int(k) // page_size) for k in kv_lens))
    if num_pages is None:
        num_pages = max(1, int(math.ceil(need * (1.0 + pool_slack))) + 1)
    if pages_per_seq is None:
        pages_per_seq = max(1, max((-(-int(k) // page_size) for k in kv_lens), default=1))
    if max_num_seqs is None:
        max_num_seqs = max(S, 1)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(head_dim)
    if distribution is None:
        n_dec = 0
        while n_dec < S and q_lens[n_dec] == 1:
            n_dec += 1
        distribution = [n_dec, n_dec, S]
    g = torch.Generator().manual_seed(seed * 16)
    bt = _assign_pages(kv_lens, page_size, num_pages, max_num_seqs, pages_per_seq, g)
    return Workload(name=name, seed=seed, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                    head_dim=head_dim, page_size=page_size, num_pages=num_pages,
                    pages_per_seq=pages_per_seq, max_num_seqs=max_num_seqs, kv_dtype=kv_dtype,
                    softmax_scale=float(softmax_scale), sliding_window=int(sliding_window or 0),
                    logits_soft_cap=float(logits_soft_cap or 0.0), k_scale=float(k_scale),
                    v_scale=float(v_scale), has_sink=bool(has_sink), q_lens=q_lens,
                    kv_lens_valid=kv_lens, block_tables=bt,
                    distribution=np.asarray(distribution, dtype=np.int32),
                    total_tokens=int(q_lens.sum()) + int(extra_tokens),
                    k_scale_heads=None if k_scale_heads is None
                    else np.asarray(k_scale_heads, np.float32),
                    v_scale_heads=None if v_scale_heads is None
                    else np.asarray(v_scale_heads, np.float32),
                    q_scale=float(q_scale or 0.0))


def _randint(g, lo, hi, n):
    """n integers uniform on [lo, hi] inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=g).numpy().astype(np.int32)


def tiny() -> Workload:
    seed = 1001
    q_lens = np.array([1, 24, 5], np.int32)
    kv_lens = np.array([17, 24, 40], np.int32)
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(16, generator=g).numpy().astype(np.int32)
    pps = 3
    bt = np.zeros(3 * pps, np.int32)
    c = 0
    for s, k in enumerate(kv_lens):
        n = -(-int(k) // 16)
        bt[s * pps: s * pps + n] = perm[c:c + n]
        c += n
    return Workload(name="tiny", seed=seed, num_q_heads=4, num_kv_heads=2, head_dim=64,
                    page_size=16, num_pages=16, pages_per_seq=pps, max_num_seqs=3,
                    kv_dtype="bf16", softmax_scale=1.0 / 8.0, sliding_window=0,
                    logits_soft_cap=0.0, k_scale=1.0, v_scale=1.0, has_sink=False,
                    q_lens=q_lens, kv_lens_valid=kv_lens, block_tables=bt,
                    distribution=np.array([1, 2, 3], np.int32), total_tokens=30)


def decode() -> Workload:
    seed = 1002
    g = torch.Generator().manual_seed(seed)
    S, P = 256, 16
    kv = _randint(g, 512, 4096, S)
    q = np.ones(S, np.int32)
    pps = 4096 // P
    bt = _assign_pages(kv, P, 80000, S, pps, g)
    return Workload(name="decode", seed=seed, num_q_heads=32, num_kv_heads=8, head_dim=128,
                    page_size=P, num_pages=80000, pages_per_seq=pps, max_num_seqs=S,
                    kv_dtype="bf16", softmax_scale=1.0 / math.sqrt(128), sliding_window=0,
                    logits_soft_cap=0.0, k_scale=1.0, v_scale=1.0, has_sink=False,
                    q_lens=q, kv_lens_valid=kv, block_tables=bt,
                    distribution=np.array([S, S, S], np.int32), total_tokens=S)


def decode_d256(S: int = 256, name: str = "decode_d256") -> Workload:
    """Decode with Gemma-2-9B's attention shape (head_dim 256): Hq16/Hkv8,
    sliding window 4096, logit soft cap 50, softmax scale 1/16; S sequences of
    one new token each with kv_len ~ U[512, 4096], bf16 cache, page_size 16."""
    seed = 1009
    g = torch.Generator().manual_seed(seed)
    P = 16
    kv = _randint(g, 512, 4096, S)
    q = np.ones(S, np.int32)
    pps = 4096 // P
    need = int(sum(-(-int(k) // P) for k in kv))
    num_pages = int(need * 1.1) + 1
    bt = _assign_pages(kv, P, num_pages, S, pps, g)
    return Workload(name=name, seed=seed, num_q_heads=16, num_kv_heads=8, head_dim=256,
                    page_size=P, num_pages=num_pages, pages_per_seq=pps, max_num_seqs=S,
                    kv_dtype="bf16", softmax_scale=1.0 / 16.0, sliding_window=4096,
                    logits_soft_cap=50.0, k_scale=1.0, v_scale=1.0, has_sink=False,
                    q_lens=q, kv_lens_valid=kv, block_tables=bt,
                    distribution=np.array([S, S, S], np.int32), total_tokens=S)


def decode_small() -> Workload:
    """The decode workload's shape and length mix at a quarter of the batch
    (64 sequences) with a pool of the pages used + 10%: small enough for a
    many-pass profiler capture, still far above L2."""
    seed = 1012
    g = torch.Generator().manual_seed(seed)
    S, P = 64, 16
    kv = _randint(g, 512, 4096, S)
    q = np.ones(S, np.int32)
    pps = 4096 // P
    need = int(sum(-(-int(k) // P) for k in kv))
    num_pages = int(math.ceil(need * 1.1))
    bt = _assign_pages(kv, P, num_pages, S, pps, g)
    return Workload(name="decode_small", seed=seed, num_q_heads=32, num_kv_heads=8,
                    head_dim=128, page_size=P, num_pages=num_pages, pages_per_seq=pps,
                    max_num_seqs=S, kv_dtype="bf16", softmax_scale=1.0 / math.sqrt(128),
                    sliding_window=0, logits_soft_cap=0.0, k_scale=1.0, v_scale=1.0,
                    has_sink=False, q_lens=q, kv_lens_valid=kv, block_tables=bt,
                    distribution=np.array([S, S, S], np.int32), total_tokens=S)


def mixed() -> Workload:
    seed = 1003
    g = torch.Generator().manual_seed(seed)
    P = 32
    dec_kv = _randint(g, 1024, 8192, 128)
    chunk_ctx = _randint(g, 0, 4096, 8)
    q = np.concatenate([np.ones(128, np.int32), np.full(8, 512, np.int32),
                        np.full(2, 1536, np.int32)])
    kv = np.concatenate([dec_kv, chunk_ctx + 512, np.full(2, 1536, np.int32)]).astype(np.int32)
    need = int(sum(-(-int(k) // P) for k in kv))
    num_pages = int(math.ceil(need * 1.1))
    pps = -(-8192 // P)
    bt = _assign_pages(kv, P, num_pages, len(q), pps, g)
    return Workload(name="mixed", seed=seed, num_q_heads=64, num_kv_heads=8, head_dim=128,
                    page_size=P, num_pages=num_pages, pages_per_seq=pps, max_num_seqs=len(q),
                    kv_dtype="bf16", softmax_scale=1.0 / math.sqrt(128), sliding_window=0,
                    logits_soft_cap=0.0, k_scale=1.0, v_scale=1.0, has_sink=False,
                    q_lens=q, kv_lens_valid=kv, block_tables=bt,
                    distribution=np.array([128, 136, 138], np.int32),
                    total_tokens=int(q.sum()))


def long(sliding_window: int = 0) -> Workload:
    seed = 1004
    g = torch.Generator().manual_seed(seed)
    P, L = 64, 32768
    q = np.full(2, L, np.int32)
    kv = np.full(2, L, np.int32)
    pps = L // P
    bt = _assign_pages(kv, P, 2048, 2, pps, g)
    return Workload(name="long" if not sliding_window else f"long_w{sliding_window}",
                    seed=seed, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=P,
                    num_pages=2048, pages_per_seq=pps, max_num_seqs=2, kv_dtype="bf16",
                    softmax_scale=1.0 / math.sqrt(128), sliding_window=sliding_window,
                    logits_soft_cap=0.0, k_scale=1.0, v_scale=1.0, has_sink=False,
                    q_lens=q, kv_lens_valid=kv, block_tables=bt,
                    distribution=np.array([0, 0, 2], np.int32), total_tokens=2 * L)


def long_d256() -> Workload:
    """Long causal prefill at head_dim 256 (Gemma-2-9B attention shape
    without its window and cap): 2 seqs q = kv = 8192, Hq16/Hkv8/D256, bf16
    cache, page_size 64, scale 1/16."""
    seed = 1016
    g = torch.Generator().manual_seed(seed)
    P, L = 64, 8192
    q = np.full(2, L, np.int32)
    kv = np.full(2, L, np.int32)
    pps = L // P
    need = 2 * pps
    num_pages = int(need * 1.1) + 1
    bt = _assign_pages(kv, P, num_pages, 2, pps, g)
    return Workload(name="long_d256", seed=seed, num_q_heads=16, num_kv_heads=8, head_dim=256,
                    page_size=P, num_pages=num_pages, pages_per_seq=pps, max_num_seqs=2,
                    kv_dtype="bf16", softmax_scale=1.0 / 16.0, sliding_window=0,
                    logits_soft_cap=0.0, k_scale=1.0, v_scale=1.0, has_sink=False,
                    q_lens=q, kv_lens_valid=kv, block_tables=bt,
                    distribution=np.array([0, 0, 2], np.int32), total_tokens=2 * L)


def long_small(kv_dtype: str = "bf16", name: str = "long_small", q_scale: float = 0.0) -> Workload:
    """The long-context shape at one sequence of 8192 tokens (profiling size);
    with kv_dtype "fp8" the same prefill into an e4m3 cache (k/v scale 0.05),
    and with q_scale > 0 its queries quantised as well."""
    seed = 1014
    g = torch.Generator().manual_seed(seed)
    P, L = 64, 8192
    q = np.full(1, L, np.int32)
    kv = np.full(1, L, np.int32)
    pps = L // P
    bt = _assign_pages(kv, P, 256, 1, pps, g)
    fp8 = kv_dtype == "fp8"
    return Workload(name=name, seed=seed, num_q_heads=32, num_kv_heads=8, head_dim=128,
                    page_size=P, num_pages=256, pages_per_seq=pps, max_num_seqs=1,
                    kv_dtype=kv_dtype, softmax_scale=1.0 / math.sqrt(128), sliding_window=0,
                    logits_soft_cap=0.0, k_scale=0.05 if fp8 else 1.0,
                    v_scale=0.05 if fp8 else 1.0, has_sink=False,
                    q_lens=q, kv_lens_valid=kv, block_tables=bt,
                    distribution=np.array([0, 0, 1], np.int32), total_tokens=L, q_scale=q_scale)


def fp8(q_scale: float = 0.0, name: str = "fp8") -> Workload:
    """The fp8 e4m3 cache configuration; with q_scale > 0 the same batch in
    the w8a8 mode (queries quantised to e4m3 with that scale)."""
    seed = 1005
    g = torch.Generator().manual_seed(seed)
    P = 16
    dec_kv = _randint(g, 256, 16384, 512)
    chunk_ctx = _randint(g, 0, 8192, 8)
    q = np.concatenate([np.ones(512, np.int32), np.full(8, 256, np.int32)])
    kv = np.concatenate([dec_kv, chunk_ctx + 256]).astype(np.int32)
    need = int(sum(-(-int(k) // P) for k in kv))
    num_pages = int(math.ceil(need * 1.1))
    pps = -(-max(16384, 8192 + 256) // P)
    bt = _assign_pages(kv, P, num_pages, len(q), pps, g)
    return Workload(name=name, seed=seed, num_q_heads=64, num_kv_heads=8, head_dim=64,
                    page_size=P, num_pages=num_pages, pages_per_seq=pps, max_num_seqs=len(q),
                    kv_dtype="fp8", softmax_scale=1.0 / 8.0, sliding_window=128,
                    logits_soft_cap=30.0, k_scale=0.05, v_scale=0.05, has_sink=True,
                    q_lens=q, kv_lens_valid=kv, block_tables=bt,
                    distribution=np.array([512, 520, 520], np.int32),
                    total_tokens=int(q.sum()), q_scale=q_scale)


def fp8_small() -> Workload:
    """The fp8 workload's shape and options with 64 decode sequences (profiling size)."""
    seed = 1015
    g = torch.Generator().manual_seed(seed)
    P = 16
    dec_kv = _randint(g, 256, 16384, 64)
    chunk_ctx = _randint(g, 0, 8192, 8)
    q = np.concatenate([np.ones(64, np.int32), np.full(8, 256, np.int32)])
    kv = np.concatenate([dec_kv, chunk_ctx + 256]).astype(np.int32)
    need = int(sum(-(-int(k) // P) for k in kv))
    num_pages = int(math.ceil(need * 1.1))
    pps = -(-max(16384, 8192 + 256) // P)
    bt = _assign_pages(kv, P, num_pages, len(q), pps, g)
    return Workload(name="fp8_small", seed=seed, num_q_heads=64, num_kv_heads=8, head_dim=64,
                    page_size=P, num_pages=num_pages, pages_per_seq=pps, max_num_seqs=len(q),
                    kv_dtype="fp8", softmax_scale=1.0 / 8.0, sliding_window=128,
                    logits_soft_cap=30.0, k_scale=0.05, v_scale=0.05, has_sink=True,
                    q_lens=q, kv_lens_valid=kv, block_tables=bt,
                    distribution=np.array([64, 72, 72], np.int32),
                    total_tokens=int(q.sum()))


WORKLOADS = {
    "tiny": tiny,
    "decode": decode,
    "decode_small": decode_small,
    "mixed": mixed,
    "long": lambda: long(0),
    "long_w4096": lambda: long(4096),
    "long_small": long_small,
    "long_small_fp8": lambda: long_small("fp8", "long_small_fp8"),
    "long_small_fp8_w8a8": lambda: long_small("fp8", "long_small_fp8_w8a8", 0.02),
    "fp8": fp8,
    # the fp8 batch with quantised queries: |q| of N(0,1) samples stays far
    # below 448 * 0.02, so no query code saturates
    "fp8_w8a8": lambda: fp8(0.02, "fp8_w8a8"),
    "fp8_small": fp8_small,
    "decode_d256": decode_d256,
    "decode_d256_small": lambda: decode_d256(64, "decode_d256_small"),
    "long_d256": long_d256,
}


def get(name: str) -> Workload:
    return WORKLOADS[name]()
