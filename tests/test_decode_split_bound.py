"""The decode workspace bound against the planner's split rule (CPU only).

The planner splits each decode (sequence, kv head) key range [lo, kv_len)
into chunks on 64-key stage boundaries: chunk = the 64-multiple at or above
ceil(total keys * Hkv / target), at least 256 keys, and a sequence takes
ceil((kv_len - (lo & ~63)) / chunk) splits per kv head.  The workspace holds
target + 2 * max_num_seqs * Hkv decode units.  These checks search adversarial
and random batches (window starts one key short of a stage boundary, many
one-key sequences, long and short mixes) for a batch that needs more.
"""
import numpy as np
import pytest

TARGET, CHUNK_MIN, STAGE = 512, 256, 64


def planned_units(kv_lens, lo, hkv):
    keys = int(np.sum(kv_lens - lo))
    want = -(-keys * hkv // TARGET)
    chunk = max(CHUNK_MIN, -(-want // STAGE) * STAGE)
    stage0 = lo & ~(STAGE - 1)
    nsplit = -(-(kv_lens - stage0) // chunk)
    return int(nsplit.sum()) * hkv


def bound(S, hkv):
    return TARGET + 2 * S * hkv


def test_the_construction_that_exceeded_the_old_bound():
    S, hkv = 65, 8
    kv = np.array([1063 + 64 * (s % 4) for s in range(S)], np.int64)
    lo = kv - 1000
    units = planned_units(kv, lo, hkv)
    assert units == 1040 > TARGET + S * hkv  # the old bound: target + S * Hkv
    assert units <= bound(S, hkv)


@pytest.mark.parametrize("hkv", [1, 2, 8, 16])
def test_window_starts_just_short_of_a_stage(hkv):
    worst = 0.0
    for S in (1, 2, 7, 33, 65, 128, 256, 600):
        for base in range(960, 2200, 37):
            kv = np.array([base + 64 * (s % 5) for s in range(S)], np.int64)
            for window in (1000, 999, 961, 256, 193):
                lo = np.maximum(kv - window, 0)
                units = planned_units(kv, lo, hkv)
                assert units <= bound(S, hkv), (S, base, window, units)
                worst = max(worst, (units - TARGET) / (S * hkv))
    assert worst <= 2.0


@pytest.mark.parametrize("seed", range(20))
def test_random_batches(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        S = int(rng.integers(1, 700))
        hkv = int(rng.choice([1, 2, 4, 8, 16]))
        kv = rng.integers(1, int(rng.choice([64, 1000, 20000])), size=S).astype(np.int64)
        window = int(rng.choice([0, 1, 63, 64, 65, 1000, 4096]))
        lo = np.maximum(kv - window, 0) if window else np.zeros(S, np.int64)
        assert planned_units(kv, lo, hkv) <= bound(S, hkv)


def test_one_key_sequences_take_one_split_each():
    for S in (1, 100, 700):
        kv = np.ones(S, np.int64)
        assert planned_units(kv, np.zeros(S, np.int64), 8) == S * 8 <= bound(S, 8)
