"""Pins for the scheduling-metadata oracle: the pages' worked numbers, a
second independent formulation by brute force, and tiling invariants."""
import os
import random

import pytest

from oracle.sched_ref import CHUNK, auto_num_parts, ceil_div, part_segments, sched_ref, split_token_ranges

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_metax_shape_fixed_split_ranges():
    rows = []
    with open(os.path.join(GOLDEN, "metax_split8_ranges.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                rows.append(tuple(int(x) for x in ln.split()))
    ref = sched_ref([1536] * 8, H_kv=4, splits=8, num_sms=152)
    assert ref.num_parts == 64 and ref.total_splits == 64
    ranges = split_token_ranges(ref, [1536] * 8)
    for b in range(8):
        for (s, c0, c1, t0, t1) in rows:
            assert ref.parts[b * 8 + s] == (b, s, 24 * b + c0, 24 * b + c1)
            assert ranges[b][s] == (t0, t1)


def test_fixed_split_hand_example_with_empty_split():
    # n_b = 5 chunks over S = 4 splits: per = 2 -> [0,2) [2,4) [4,5) [5,5)
    ref = sched_ref([5 * CHUNK - 3], H_kv=1, splits=4, num_sms=8)
    assert [p[2:] for p in ref.parts] == [(0, 2), (2, 4), (4, 5), (5, 5)]
    assert split_token_ranges(ref, [5 * CHUNK - 3])[0][3] == (5 * CHUNK - 3, 5 * CHUNK - 3)


def test_auto_part_counts_for_the_workloads():
    assert auto_num_parts(152, 8, 1) == 19
    assert auto_num_parts(148, 8, 1) == 18
    assert auto_num_parts(152, 4, 1) == 38
    assert auto_num_parts(152, 1, 2) == 76
    assert auto_num_parts(4, 8, 1) == 1


def _brute_auto(seqlens, num_parts):
    """Independent formulation: label every chunk with its part, then read the
    splits off the labels."""
    labels = []          # (b, local chunk)
    for b, L in enumerate(seqlens):
        labels += [(b, c) for c in range(ceil_div(L, CHUNK))]
    total = len(labels)
    per = max(1, ceil_div(total, num_parts))
    owner = [i // per for i in range(total)]
    splits = []
    for b in range(len(seqlens)):
        ps = sorted({owner[i] for i, (bb, _) in enumerate(labels) if bb == b})
        splits.append(ps)
    return total, per, owner, splits


@pytest.mark.parametrize("seed", range(40))
def test_auto_mode_matches_brute_force(seed):
    rnd = random.Random(seed)
    B = rnd.randint(1, 12)
    seqlens = [rnd.choice([0, 1, 63, 64, 65, rnd.randint(0, 3000)]) for _ in range(B)]
    num_sms = rnd.randint(1, 40)
    H_kv = rnd.randint(1, 4)
    ref = sched_ref(seqlens, H_kv, 0, num_sms)
    num_parts = max(1, num_sms // H_kv)
    total, per, owner, splits = _brute_auto(seqlens, num_parts)
    assert ref.num_parts == num_parts and ref.per == per and ref.total_chunks == total
    assert ref.num_splits == [len(s) for s in splits]
    assert ref.split_offset[-1] == ref.total_splits == sum(len(s) for s in splits)
    # every part covers exactly the chunks labelled with it, in order
    covered = []
    for p in range(ref.num_parts):
        b0, s0, c0, c1 = ref.parts[p]
        assert c1 - c0 <= per
        assert [i for i in range(total) if owner[i] == p] == list(range(c0, c1))
        for (b, s, lc0, lc1) in part_segments(ref, p):
            assert splits[b][s] == p
            covered += [(b, c) for c in range(lc0, lc1)]
    labels = [(b, c) for b, L in enumerate(seqlens) for c in range(ceil_div(L, CHUNK))]
    assert covered == labels
    # the split token ranges of each request tile [0, L_b)
    ranges = split_token_ranges(ref, seqlens)
    for b, L in enumerate(seqlens):
        pos = 0
        for (t0, t1) in ranges[b]:
            assert t0 == pos and t1 > t0
            pos = t1
        assert pos == L


@pytest.mark.parametrize("seed", range(20))
def test_fixed_mode_tiles_each_request(seed):
    rnd = random.Random(100 + seed)
    B = rnd.randint(1, 6)
    S = rnd.randint(1, 9)
    seqlens = [rnd.choice([0, 1, 64, 65, rnd.randint(0, 2000)]) for _ in range(B)]
    ref = sched_ref(seqlens, 2, S, 100)
    assert ref.num_parts == B * S and ref.total_splits == B * S
    ranges = split_token_ranges(ref, seqlens)
    for b, L in enumerate(seqlens):
        assert len(ranges[b]) == S
        pos = 0
        per = ceil_div(ceil_div(L, CHUNK), S)
        for s, (t0, t1) in enumerate(ranges[b]):
            assert t0 == pos and t1 >= t0 and (t1 - t0) <= per * CHUNK
            pos = t1
        assert pos == L


@pytest.mark.parametrize("seed", range(20))
def test_window_chunks_are_exactly_the_read_ones(seed):
    """With a sliding window, a request's chunks are exactly the 64-token
    chunks that hold a token some query token sees (brute force over tokens),
    and the splits' token ranges tile [first visible token, L)."""
    rng = random.Random(500 + seed)
    B = rng.randint(1, 9)
    s_q = rng.choice([1, 2, 4])
    W = rng.choice([1, 5, 64, 100, 1000])
    lengths = [rng.choice([0, 1, 3, 63, 64, 65, 200, rng.randint(0, 3000)]) for _ in range(B)]
    splits = rng.choice([0, 1, 3])
    ref = sched_ref(lengths, H_kv=2, splits=splits, num_sms=rng.choice([16, 152]), window=W, s_q=s_q)
    for b, L in enumerate(lengths):
        seen = set()
        for j in range(s_q):
            pos = L - s_q + j
            for t in range(max(0, pos - W + 1), pos + 1):
                seen.add(t // CHUNK)
        n = ref.chunk_offset[b + 1] - ref.chunk_offset[b]
        if not seen:
            assert n == 0
            continue
        assert n == max(seen) - min(seen) + 1 == len(seen)
    ranges = split_token_ranges(ref, lengths, window=W, s_q=s_q)
    for b, L in enumerate(lengths):
        start = max(0, L - s_q + 1 - W)
        toks = [t for (t0, t1) in ranges[b] for t in range(t0, t1)]
        assert toks == list(range(start, L)) if L > 0 else toks == []


def test_sparse_schedule_counts_topk_slots():
    ref = sched_ref([0, 5, 10000, 64], H_kv=1, splits=0, num_sms=152, cpc=2, topk=100)
    assert ref.chunk_offset == [0, 2, 4, 6, 8]
    ref = sched_ref([0, 5, 10000, 64], H_kv=1, splits=3, num_sms=152, cpc=2, topk=2048)
    assert ref.chunk_offset == [0, 32, 64, 96, 128] and len(ref.parts) == 12
