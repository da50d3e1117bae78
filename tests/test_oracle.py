"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: torch's
own float8_e4m3fn codec, the dense numpy brute force in dense_reference.py,
closed forms of special cases, invariances the definition implies, and the
worked example the pages print.  Every test is chosen so that a plausible
slip in the oracle (a dropped sink term, a swapped K/V channel, a wrong GQA
index, an off-by-one window, a wrong soft-cap sign) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from dense_reference import dense_attention, expected_pool_after, fp8_roundtrip
from helpers import pool_bytes, run_oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- fp8 codec
def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(mine[~nan], ref[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_e4m3_midpoints_round_to_even():
    pos = np.arange(0, 0x7E, dtype=np.uint8)  # adjacent positive pairs c, c+1
    lo = oracle.e4m3_decode(pos)
    hi = oracle.e4m3_decode(pos + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)  # exact in fp32
    got = oracle.e4m3_encode(mid)
    want = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.e4m3_encode(-mid), want | 0x80)


def test_e4m3_saturates():
    big = np.array([448.0, 449.0, 464.0, 480.0, 1e6, np.inf], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)


def test_e4m3_encode_matches_torch_random():
    g = torch.Generator().manual_seed(7)
    x = torch.cat([torch.randn(20000, generator=g) * 40,
                   torch.randn(5000, generator=g) * 2.0 ** -7,
                   (torch.rand(5000, generator=g) * 2 - 1) * 463]).float()
    mine = oracle.e4m3_encode(x.numpy())
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_quantize_is_fp32_divide_then_encode():
    g = torch.Generator().manual_seed(8)
    x = torch.randn(4000, generator=g).to(torch.bfloat16)
    for scale in (0.05, 0.3, 1.0, 7.5):
        mine = oracle.quantize(x, scale)
        ref = (x.float() / torch.tensor(np.float32(scale))).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(mine, ref), scale


def test_bf16_decode():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F], dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.bf16_to_double(bits), ref)


# ------------------------------------------------------------------ golden
def test_query_start_loc_golden_example():
    rows = {}
    with open(os.path.join(GOLDEN, "query_start_loc_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                rows[k] = [int(x) for x in v]
    w = wl.make_custom("golden", 1, rows["q_lens"], rows["q_lens"], num_q_heads=2,
                       num_kv_heads=1, head_dim=8, page_size=4)
    assert list(w.query_start_loc) == rows["query_start_loc"]


# ---------------------------------------------------------------- workloads
def _small(name, seed, q_lens, kv_lens, **kw):
    base = dict(num_q_heads=4, num_kv_heads=2, head_dim=16, page_size=8)
    base.update(kw)
    return wl.make_custom(name, seed, q_lens, kv_lens, **base)


def _inputs(w):
    q, k, v = w.make_qkv()
    return q, k, v, w.make_pool("cpu"), w.make_sink()


SMALL_CASES = [
    ("tiny", lambda: wl.tiny()),
    ("mha_decode", lambda: _small("a", 11, [1, 1, 1], [1, 9, 30], num_q_heads=2, num_kv_heads=2)),
    ("gqa8_mixed", lambda: _small("b", 12, [1, 7, 16, 3], [20, 7, 33, 3], num_q_heads=16, num_kv_heads=2)),
    ("window", lambda: _small("c", 13, [1, 12, 5], [40, 25, 9], sliding_window=6)),
    ("softcap_sink", lambda: _small("d", 14, [1, 10], [18, 10], logits_soft_cap=2.5, has_sink=True,
                                   softmax_scale=0.9)),
    ("fp8_all", lambda: _small("e", 15, [1, 9, 4], [31, 17, 4], kv_dtype="fp8", k_scale=0.05,
                              v_scale=0.08, logits_soft_cap=30.0, has_sink=True, sliding_window=5,
                              num_q_heads=8, num_kv_heads=2, page_size=4)),
    ("page32", lambda: _small("f", 16, [3, 1], [70, 45], page_size=32, head_dim=32)),
    ("fp8_per_head", lambda: _small("pf", 18, [1, 6, 3], [27, 14, 3], kv_dtype="fp8",
                                    num_q_heads=6, num_kv_heads=3,
                                    k_scale_heads=[0.02, 0.09, 0.3],
                                    v_scale_heads=[0.15, 0.04, 0.011], has_sink=True)),
    ("q_len0", lambda: _small("g", 17, [0, 4, 0], [5, 4, 11])),
    ("d256", lambda: _small("h", 19, [1, 6, 2], [23, 6, 9], head_dim=256, num_q_heads=4,
                            num_kv_heads=2, logits_soft_cap=50.0, sliding_window=8)),
    ("d96_fp8", lambda: _small("i", 20, [1, 5], [17, 5], head_dim=96, kv_dtype="fp8",
                               k_scale=0.05, v_scale=0.07)),
    # q_scale: the queries quantised to e4m3 too (the dense reference uses
    # torch's own float8_e4m3fn cast of q / q_scale)
    ("fp8_q_scale_all", lambda: _small("j", 21, [1, 9, 4], [31, 17, 4], kv_dtype="fp8",
                                       k_scale=0.05, v_scale=0.08, q_scale=0.03,
                                       logits_soft_cap=30.0, has_sink=True, sliding_window=5,
                                       num_q_heads=8, num_kv_heads=2, page_size=4)),
    ("fp8_q_scale_per_head_d256", lambda: _small("k", 22, [1, 6, 2], [23, 6, 9], head_dim=256,
                                                 kv_dtype="fp8", q_scale=0.011,
                                                 k_scale_heads=[0.04, 0.1],
                                                 v_scale_heads=[0.06, 0.02])),
]


@pytest.mark.parametrize("name,make", SMALL_CASES, ids=[c[0] for c in SMALL_CASES])
def test_oracle_matches_dense_brute_force(name, make):
    w = make()
    q, k, v, pool, sink = _inputs(w)
    out, _ = run_oracle(w, q, k, v, pool, sink)
    ref = dense_attention(w, q, k, v, pool, sink)
    assert out.shape == ref.shape
    assert np.max(np.abs(out - ref)) < 1e-10


@pytest.mark.parametrize("name,make", SMALL_CASES, ids=[c[0] for c in SMALL_CASES])
def test_oracle_cache_write_matches_slot_mapping(name, make):
    w = make()
    q, k, v, pool, sink = _inputs(w)
    _, cache = run_oracle(w, q, k, v, pool, sink)
    want = pool_bytes(expected_pool_after(w, pool, k, v))
    assert np.array_equal(cache, want)


# -------------------------------------------------------------- closed forms
def test_single_key_gives_v():
    for kv_dtype in ("bf16", "fp8"):
        w = _small("h", 21, [1, 1], [1, 1], kv_dtype=kv_dtype, k_scale=0.05, v_scale=0.07)
        q, k, v, pool, _ = _inputs(w)
        out, _ = run_oracle(w, q, k, v, pool)
        if kv_dtype == "fp8":
            vv = fp8_roundtrip(v, w.v_scale)
        else:
            vv = v.double().numpy()
        want = np.repeat(vv, w.group, axis=1)
        assert np.max(np.abs(out - want)) < 1e-12


def test_sink_single_key_closed_form():
    w = _small("i", 22, [1], [1], has_sink=True, softmax_scale=0.37)
    q, k, v, pool, sink = _inputs(w)
    out, _ = run_oracle(w, q, k, v, pool, sink)
    for hq in range(w.num_q_heads):
        h = hq // w.group
        s = float(np.float32(0.37)) * float(q[0, hq].double() @ k[0, h].double())
        sig = 1.0 / (1.0 + math.exp(-(s - float(sink[hq]))))
        assert np.allclose(out[0, hq], sig * v[0, h].double().numpy(), atol=1e-12, rtol=0)


def test_window_one_gives_own_value():
    w = _small("j", 23, [6, 1], [6, 13], sliding_window=1)
    q, k, v, pool, _ = _inputs(w)
    out, _ = run_oracle(w, q, k, v, pool)
    want = np.repeat(v.double().numpy(), w.group, axis=1)
    assert np.max(np.abs(out - want)) < 1e-12


def test_window_at_least_kv_len_is_no_window():
    base = dict(q_lens=[1, 9], kv_lens=[25, 30])
    w0 = _small("k", 24, **base)
    w1 = _small("k", 24, **base, sliding_window=30)
    q, k, v, pool, _ = _inputs(w0)
    o0, _ = run_oracle(w0, q, k, v, pool)
    o1, _ = run_oracle(w1, q, k, v, pool)
    assert np.array_equal(o0, o1)
    w2 = _small("k", 24, **base, sliding_window=29)  # one key fewer for the last rows
    o2, _ = run_oracle(w2, q, k, v, pool)
    assert not np.array_equal(o0, o2)


def test_rows_sum_to_one_and_sink_mass():
    w = _small("l", 25, [1, 8], [19, 12], logits_soft_cap=5.0)
    q, k, _, pool, _ = _inputs(w)
    ones = torch.ones(w.total_tokens, w.num_kv_heads, w.head_dim, dtype=torch.bfloat16)
    vpool = pool.clone()
    vpool[:, :, 1::2, :] = 1.0
    out, _ = run_oracle(w, q, k, ones, vpool)
    assert np.max(np.abs(out - 1.0)) < 1e-12
    # with a sink the weights of the keys sum to 1 - sigma-share of the sink
    w_s = _small("l", 25, [1, 8], [19, 12], logits_soft_cap=5.0, has_sink=True)
    sink = torch.full((w_s.num_q_heads,), 0.75)
    out_s, _ = run_oracle(w_s, q, k, ones, vpool, sink)
    # every logit is capped to (-5, 5); so the key mass lies strictly inside (0, 1)
    assert np.all(out_s < 1.0) and np.all(out_s > 0.0)
    # single-key row: mass of the key = sigmoid(s - sink)
    w1 = _small("l1", 26, [1], [1], logits_soft_cap=5.0, has_sink=True)
    q1, k1, _, pool1, _ = _inputs(w1)
    ones1 = torch.ones(1, w1.num_kv_heads, w1.head_dim, dtype=torch.bfloat16)
    o1, _ = run_oracle(w1, q1, k1, ones1, pool1, sink)
    for hq in range(w1.num_q_heads):
        s = float(np.float32(w1.softmax_scale)) * float(q1[0, hq].double() @ k1[0, hq // w1.group].double())
        s = 5.0 * math.tanh(s / 5.0)
        assert abs(o1[0, hq, 0] - 1.0 / (1.0 + math.exp(0.75 - s))) < 1e-12


def test_soft_cap_two_key_closed_form_and_limit():
    D = 16
    w = _small("m", 27, [2], [2], num_q_heads=1, num_kv_heads=1, head_dim=D,
               softmax_scale=1.0, logits_soft_cap=3.0)
    q = torch.zeros(2, 1, D, dtype=torch.bfloat16)
    k = torch.zeros(2, 1, D, dtype=torch.bfloat16)
    v = torch.zeros(2, 1, D, dtype=torch.bfloat16)
    q[1, 0, 0] = 4.0
    k[0, 0, 0] = 1.0
    k[1, 0, 0] = -1.0
    v[0, 0, :] = 1.0
    v[1, 0, :] = -2.0
    pool = w.make_pool("cpu")
    out, _ = run_oracle(w, q, k, v, pool)
    s1, s2 = 3.0 * math.tanh(4.0 / 3.0), 3.0 * math.tanh(-4.0 / 3.0)
    p1 = math.exp(s1) / (math.exp(s1) + math.exp(s2))
    assert abs(out[1, 0, 0] - (p1 * 1.0 + (1 - p1) * -2.0)) < 1e-12
    assert abs(out[0, 0, 3] - 1.0) < 1e-12  # first row sees only key 0
    # cap -> infinity is no cap
    w_inf = _small("m", 27, [2], [2], num_q_heads=1, num_kv_heads=1, head_dim=D,
                   softmax_scale=1.0, logits_soft_cap=1e7)
    w_none = _small("m", 27, [2], [2], num_q_heads=1, num_kv_heads=1, head_dim=D, softmax_scale=1.0)
    o_inf, _ = run_oracle(w_inf, q, k, v, pool)
    o_none, _ = run_oracle(w_none, q, k, v, pool)
    assert np.max(np.abs(o_inf - o_none)) < 1e-9
    e = math.exp(4.0) / (math.exp(4.0) + math.exp(-4.0))
    assert abs(o_none[1, 0, 0] - (e - 2 * (1 - e))) < 1e-12


# ---------------------------------------------------------------- invariances
def test_page_permutation_invariance():
    w = _small("n", 31, [1, 11, 4], [29, 11, 21])
    q, k, v, pool, _ = _inputs(w)
    out, cache = run_oracle(w, q, k, v, pool)
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(3))
    inv = torch.argsort(perm)
    # physical page p moves to slot inv[p]; tables follow
    pool2 = pool[perm]
    w2 = _small("n", 31, [1, 11, 4], [29, 11, 21])
    w2.block_tables = inv.numpy()[w.block_tables].astype(np.int32)
    out2, cache2 = run_oracle(w2, q, k, v, pool2)
    assert np.array_equal(out, out2)
    c1 = torch.from_numpy(cache).view(w.pool_shape[0], -1)
    c2 = torch.from_numpy(cache2).view(w.pool_shape[0], -1)
    assert torch.equal(c1[perm], c2)


def test_page_size_invariance():
    q_lens, kv_lens = [1, 13, 2], [37, 20, 64]
    outs = []
    for P in (4, 16, 32):
        w = _small("o", 32, q_lens, kv_lens, page_size=P)
        q, k, v, _, _ = _inputs(w)
        # same logical context in every layout
        gen = torch.Generator().manual_seed(99)
        ctx_vals = [torch.randn(kl, 2 * w.num_kv_heads, w.head_dim, generator=gen).to(torch.bfloat16)
                    for kl in kv_lens]
        pool = w.make_pool("cpu")
        flat = pool.view(-1, 2 * w.num_kv_heads, w.head_dim)
        for s, kl in enumerate(kv_lens):
            pos = np.arange(kl)
            slots = w.block_tables[s * w.pages_per_seq + pos // P].astype(np.int64) * P + pos % P
            flat[torch.as_tensor(slots)] = ctx_vals[s]
        o, _ = run_oracle(w, q, k, v, pool)
        outs.append(o)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_decode_equals_last_row_of_prefill():
    L = 23
    wp = _small("p", 33, [L], [L])
    q, k, v, pool, _ = _inputs(wp)
    out_p, cache_p = run_oracle(wp, q, k, v, pool)
    # same sequence: first L-1 tokens already cached, last token decoded
    wd = _small("p", 33, [1], [L])
    wd.block_tables = wp.block_tables.copy()
    pool_d = torch.from_numpy(cache_p.copy()).view(pool.dtype).view(pool.shape).clone()
    out_d, _ = run_oracle(wd, q[L - 1:], k[L - 1:], v[L - 1:], pool_d)
    assert np.array_equal(out_d[0], out_p[L - 1])


def test_chunked_prefill_equals_one_call():
    L, L1 = 30, 12
    w = _small("q", 34, [L], [L], sliding_window=9, logits_soft_cap=4.0, has_sink=True)
    q, k, v, pool, sink = _inputs(w)
    out, cache = run_oracle(w, q, k, v, pool, sink)
    w1 = _small("q", 34, [L1], [L1], sliding_window=9, logits_soft_cap=4.0, has_sink=True)
    w1.block_tables = w.block_tables.copy()
    w1.num_pages = w.num_pages
    o1, c1 = run_oracle(w1, q[:L1], k[:L1], v[:L1], pool, sink)
    w2 = _small("q", 34, [L - L1], [L], sliding_window=9, logits_soft_cap=4.0, has_sink=True)
    w2.block_tables = w.block_tables.copy()
    pool1 = torch.from_numpy(c1.copy()).view(pool.dtype).view(pool.shape).clone()
    o2, c2 = run_oracle(w2, q[L1:], k[L1:], v[L1:], pool1, sink)
    assert np.array_equal(np.concatenate([o1, o2]), out)
    assert np.array_equal(c2, cache)


def test_gqa_equals_mha_with_replicated_kv():
    q_lens, kv_lens = [1, 6], [14, 9]
    wg = _small("r", 35, q_lens, kv_lens, num_q_heads=8, num_kv_heads=2)
    q, k, v, pool, _ = _inputs(wg)
    og, _ = run_oracle(wg, q, k, v, pool)
    wm = _small("r", 35, q_lens, kv_lens, num_q_heads=8, num_kv_heads=8)
    wm.block_tables = wg.block_tables.copy()
    # replicate every kv head to its 4 q-heads, in the inputs and in the pool
    rep = torch.arange(8) // 4
    pool_m = torch.empty(wm.pool_shape, dtype=pool.dtype)
    pool_m[:, :, 0::2] = pool[:, :, 0::2][:, :, rep]
    pool_m[:, :, 1::2] = pool[:, :, 1::2][:, :, rep]
    om, _ = run_oracle(wm, q, k[:, rep], v[:, rep], pool_m)
    assert np.array_equal(og, om)


def test_result_ignores_distribution_and_padding():
    w = _small("s", 36, [1, 1, 5], [9, 3, 12], max_num_seqs=6, extra_tokens=4)
    q, k, v, pool, _ = _inputs(w)
    out, cache = run_oracle(w, q, k, v, pool)
    assert out.shape[0] == 7  # padded token rows are not attended
    w.distribution = np.array([0, 0, 3], np.int32)
    out2, cache2 = run_oracle(w, q, k, v, pool)
    assert np.array_equal(out, out2) and np.array_equal(cache, cache2)


# ---------------------------------------------------------------- validation
def test_oracle_rejects_bad_metadata():
    w = _small("t", 37, [1, 4], [9, 4])
    q, k, v, pool, _ = _inputs(w)
    p = oracle.make_params(**w.params())
    bt = w.block_tables.copy()
    bt[0] = w.num_pages  # out of range page
    with pytest.raises(oracle.OracleError) as e:
        oracle.forward(p, q, k, v, pool_bytes(pool), w.kv_lens, bt, w.query_start_loc, w.num_seqs)
    assert e.value.code == oracle.ORACLE_BAD_PAGE
    kl = w.kv_lens.copy()
    kl[1] = 3  # kv_len < q_len
    with pytest.raises(oracle.OracleError):
        oracle.forward(p, q, k, v, pool_bytes(pool), kl, w.block_tables, w.query_start_loc, w.num_seqs)
    assert oracle.check_distribution(p, np.array([1, 2, 2], np.int32), w.query_start_loc) == 0
    assert oracle.check_distribution(p, np.array([2, 2, 2], np.int32), w.query_start_loc) != 0
    assert oracle.check_distribution(p, np.array([1, 0, 2], np.int32), w.query_start_loc) != 0


def test_equal_per_head_scales_are_the_scalar_scales():
    """Per-kv-head scales that all equal the scalar ones give the same cache
    bytes and outputs; one head's scale changed moves only that head's
    channels and outputs."""
    kw = dict(kv_dtype="fp8", num_q_heads=8, num_kv_heads=4, k_scale=0.05, v_scale=0.07)
    base = _small("ph", 19, [1, 5], [23, 9], **kw)
    same = _small("ph", 19, [1, 5], [23, 9], k_scale_heads=[0.05] * 4, v_scale_heads=[0.07] * 4,
                  **kw)
    one = _small("ph", 19, [1, 5], [23, 9], k_scale_heads=[0.05, 0.05, 0.2, 0.05],
                 v_scale_heads=[0.07, 0.07, 0.02, 0.07], **kw)
    q, k, v, pool, sink = _inputs(base)
    o0, c0 = run_oracle(base, q, k, v, pool, sink)
    o1, c1 = run_oracle(same, q, k, v, pool, sink)
    o2, c2 = run_oracle(one, q, k, v, pool, sink)
    assert np.array_equal(c0, c1) and np.array_equal(o0, o1)
    # head 2 (q-heads 4, 5; pool channels 4, 5) differs, every other head is unchanged
    assert not np.array_equal(o0[:, 4:6], o2[:, 4:6])
    assert np.array_equal(np.delete(o0, [4, 5], axis=1), np.delete(o2, [4, 5], axis=1))
    shape = (base.num_pages * base.page_size, 2 * base.num_kv_heads, base.head_dim)
    d = (c0 != c2).reshape(shape).any(axis=(0, 2))
    assert d[4] and d[5] and not d[[0, 1, 2, 3, 6, 7]].any()


# ------------------------------------------------------------ random sweep
def _random_case(i):
    """A seeded random small call: shapes, ragged lengths (some q_len = 0),
    every option on or off, fp8 with scalar or per-head scales and with or
    without quantised queries."""
    rng = np.random.default_rng(1000 + i)
    Hkv = int(rng.integers(1, 4))
    G = int(rng.choice([1, 2, 4]))
    D = int(rng.choice([8, 16, 24]))
    P = int(rng.choice([1, 2, 4, 8]))
    S = int(rng.integers(1, 5))
    q_lens = [int(x) for x in rng.integers(0, 7, size=S)]
    kv_lens = [q + int(rng.integers(0, 21)) for q in q_lens]
    kv_lens = [max(kv, 1) for kv in kv_lens]
    kw = dict(num_q_heads=Hkv * G, num_kv_heads=Hkv, head_dim=D, page_size=P,
              softmax_scale=float(rng.uniform(0.2, 1.2)),
              sliding_window=int(rng.choice([0, 0, 1, 3, 7])),
              logits_soft_cap=float(rng.choice([0.0, 0.0, 2.5, 20.0])),
              has_sink=bool(rng.integers(0, 2)))
    if rng.integers(0, 2):
        kw["kv_dtype"] = "fp8"
        if rng.integers(0, 2):
            kw["k_scale_heads"] = [float(x) for x in rng.uniform(0.01, 0.3, Hkv)]
            kw["v_scale_heads"] = [float(x) for x in rng.uniform(0.01, 0.3, Hkv)]
        else:
            kw["k_scale"], kw["v_scale"] = float(rng.uniform(0.02, 0.2)), float(rng.uniform(0.02, 0.2))
        if rng.integers(0, 2):
            kw["q_scale"] = float(rng.uniform(0.005, 0.05))
    # decode class: a prefix of the one-token sequences
    d0 = 0
    while d0 < S and q_lens[d0] == 1:
        d0 += 1
    d0 = int(rng.integers(0, d0 + 1))
    d1 = int(rng.integers(d0, S + 1))
    kw["distribution"] = [d0, d1, S]
    return wl.make_custom(f"r{i}", 2000 + i, q_lens, kv_lens, **kw)


@pytest.mark.parametrize("i", range(40))
def test_oracle_matches_dense_brute_force_random(i):
    w = _random_case(i)
    q, k, v, pool, sink = _inputs(w)
    out, cache = run_oracle(w, q, k, v, pool, sink)
    ref = dense_attention(w, q, k, v, pool, sink)
    assert out.shape == ref.shape
    assert np.max(np.abs(out - ref), initial=0.0) < 1e-10
    assert np.array_equal(cache, pool_bytes(expected_pool_after(w, pool, k, v)))


# ------------------------------------------------- unread slots, tolerance
@pytest.mark.parametrize("kind", ["bf16_window", "bf16", "fp8_window_options"])
def test_oracle_reads_no_slot_outside_the_band(kind):
    """Slots outside [window start, ctx) of every sequence -- rows past
    kv_len, rows before the window, the new tokens' slots before the write,
    unused pages -- filled with NaN / Inf change nothing: the outputs equal
    those on the clean pool bit for bit and the poisoned bytes pass through
    the page write untouched.  This also checks the GPU tests' read_slots."""
    from helpers import poison_unread_slots, read_slots
    extra = {"bf16_window": dict(sliding_window=37),
             "bf16": {},
             "fp8_window_options": dict(kv_dtype="fp8", k_scale=0.05, v_scale=0.07,
                                        logits_soft_cap=30.0, has_sink=True,
                                        sliding_window=20)}[kind]
    w = wl.make_custom("poison", 77, [1, 1, 40, 9, 0], [300, 5, 140, 9, 12], num_q_heads=8,
                       num_kv_heads=2, head_dim=64, page_size=16, **extra)
    q, k, v = w.make_qkv()
    pool = w.make_pool("cpu")
    sink = w.make_sink()
    bad = poison_unread_slots(w, pool)
    out_clean, cache_clean = run_oracle(w, q, k, v, pool, sink)
    out_bad, cache_bad = run_oracle(w, q, k, v, bad, sink)
    assert np.all(np.isfinite(out_bad))
    assert np.array_equal(out_bad, out_clean)
    # every slot is either read (identical bytes) or carries its poison,
    # except the new tokens' slots, which both writes fill identically
    rows = w.num_pages * w.page_size
    cb = cache_bad.reshape(rows, -1)
    cc = cache_clean.reshape(rows, -1)
    written = np.zeros(rows, bool)
    for s in range(w.num_seqs):
        ctx = int(w.kv_lens_valid[s]) - int(w.q_lens[s])
        pos = np.arange(ctx, int(w.kv_lens_valid[s]))
        written[w.block_tables[s * w.pages_per_seq + pos // w.page_size] * w.page_size
                + pos % w.page_size] = True
    assert np.array_equal(cb[written | read_slots(w)], cc[written | read_slots(w)])
    assert np.array_equal(cb[~(written | read_slots(w))],
                          pool_bytes(bad).reshape(rows, -1)[~(written | read_slots(w))])


def test_tolerance_rule_is_the_stated_bound_where_attainable():
    """max |err| <= 1e-2 wherever |exact| < 4 (the correctly rounded bf16
    output is always within half an ulp <= 2^-7 there); from |exact| = 4 on,
    the bound adds the output's own rounding, half an ulp >= 2^-6."""
    from helpers import assert_close, max_abs_bound, output_errors
    exact = np.array([0.0, 0.3, 1.5, 3.99, 4.0, 7.9, 8.0, 100.0])
    b = max_abs_bound(exact)
    assert np.all(b[:4] == 1e-2)
    assert b[4] == 2.0 ** -6 + 1e-2 and b[5] == 2.0 ** -6 + 1e-2
    assert b[6] == 2.0 ** -5 + 1e-2 and b[7] == 2.0 ** -2 + 1e-2
    # the correctly rounded bf16 value always meets the max rule, at any
    # magnitude (the mean rule is a property of the data, checked separately)
    x = np.random.default_rng(0).normal(0, 30, 20000)
    rounded = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert output_errors(rounded, x)[0] <= 1.0
    # an error of 0.011 at |exact| = 2 (where half an ulp is 2^-8) fails
    y = np.full(1000, 2.0)
    y_got = y.copy()
    y_got[0] += 0.011
    with pytest.raises(AssertionError):
        assert_close(y_got, y, "one element off by 0.011")


# --------------------------------------------------------------- q_scale
def _q_scale_case(q_scale, **kw):
    base = dict(num_q_heads=8, num_kv_heads=2, head_dim=16, page_size=4, kv_dtype="fp8",
                k_scale=0.05, v_scale=0.07, has_sink=True, logits_soft_cap=20.0)
    base.update(kw)
    return wl.make_custom("qs", 23, [1, 7, 3], [25, 12, 3], q_scale=q_scale, **base)


def test_q_scale_exact_codes_equal_plain_queries():
    """Queries that are e4m3 values times a power-of-two q_scale quantise
    exactly, so the w8a8 path must give the plain path's outputs bit for
    bit (a dropped or doubled q_scale, or quantising with another scale,
    changes them)."""
    w8 = _q_scale_case(2.0 ** -4)
    plain = _q_scale_case(0.0)
    q, k, v, pool, sink = _inputs(plain)
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 0x7F, size=q.numel()).astype(np.uint8)  # finite, positive
    codes |= (rng.integers(0, 2, size=q.numel()) << 7).astype(np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float() * 2.0 ** -4
    qx = vals.reshape(q.shape).to(torch.bfloat16)
    assert torch.equal(qx.float(), vals.reshape(q.shape))  # exact in bf16
    o8, c8 = run_oracle(w8, qx, k, v, pool, sink)
    op, cp = run_oracle(plain, qx, k, v, pool, sink)
    assert np.array_equal(o8, op) and np.array_equal(c8, cp)
    # and with another q_scale the same queries do change the outputs
    o9, _ = run_oracle(_q_scale_case(0.3), qx, k, v, pool, sink)
    assert not np.array_equal(o9, op)


def test_q_scale_saturates_queries():
    """|q| / q_scale beyond 448 saturates to the largest code: equal to the
    plain path on queries clamped to +-448 * q_scale."""
    qs = 2.0 ** -6
    w8 = _q_scale_case(qs)
    plain = _q_scale_case(0.0)
    q, k, v, pool, sink = _inputs(plain)
    big = (q.float() * 40.0).to(torch.bfloat16)            # |q| up to ~160 >> 448 * 2^-6 = 7
    clamped = big.float().clamp(-448 * qs, 448 * qs)
    # inside the range the codes must be exact too: keep the clamped values
    # and the in-range ones on e4m3 points by snapping through torch's cast
    snapped = (clamped / qs).to(torch.float8_e4m3fn).float() * qs
    o8, _ = run_oracle(w8, big, k, v, pool, sink)
    op, _ = run_oracle(plain, snapped.to(torch.bfloat16), k, v, pool, sink)
    assert np.max(np.abs(o8 - op)) < 1e-12
    assert (big.float().abs() > 448 * qs).any()


def test_q_scale_needs_an_fp8_cache():
    w = _small("qb", 24, [1, 3], [9, 3])
    p = oracle.make_params(**w.params(), q_scale=0.05)
    q, k, v, pool, sink = _inputs(w)
    with pytest.raises(oracle.OracleError):
        oracle.forward(p, q, k, v, pool_bytes(pool), w.kv_lens, w.block_tables,
                       w.query_start_loc, w.num_seqs)
