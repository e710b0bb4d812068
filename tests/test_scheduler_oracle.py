"""Pins for the scheduler oracle (the split-KV work partition is this project's design;
what the pages fix is that it must cover every KV block exactly once, keep each
sequence's splits contiguous and ordered, and balance work across the parts)."""
import numpy as np
import pytest

from oracle import scheduler as sch

FIXED = 5


def check_partition(seqlens, parts, fixed):
    meta, num_splits = sch.schedule(seqlens, parts, fixed)
    b = len(seqlens)
    assert len(meta) == parts and len(num_splits) == b + 1
    assert num_splits[0] == 0 and all(x < y for x, y in zip(num_splits, num_splits[1:]))
    covered = [np.zeros(sch.num_blocks(L), dtype=int) for L in seqlens]
    touched = [0] * b
    split_ids = []
    prev_end = (0, 0)
    costs = []
    for row in meta:
        assert (row[0], row[1]) == prev_end  # parts are contiguous and ordered
        prev_end = (row[2], row[3])
        cost = 0
        for (i, lo, hi, sid) in sch.segments_of_part(row, seqlens):
            assert 0 <= lo <= hi <= sch.num_blocks(seqlens[i])
            assert lo < hi or sch.num_blocks(seqlens[i]) == 0
            covered[i][lo:hi] += 1
            touched[i] += 1
            split_ids.append((sid, i, lo))
            cost += hi - lo + fixed
        costs.append(cost)
    assert prev_end == (b, 0)
    for i in range(b):
        assert (covered[i] == 1).all()            # every block exactly once
        assert touched[i] == num_splits[i + 1] - num_splits[i]
    # split ids are 0..S-1 in (sequence, block) order, each sequence's ids contiguous
    split_ids.sort()
    assert [s for s, _, _ in split_ids] == list(range(num_splits[b]))
    assert [(i, lo) for _, i, lo in split_ids] == sorted((i, lo) for _, i, lo in split_ids)
    for s, i, _ in split_ids:
        assert num_splits[i] <= s < num_splits[i + 1]
    # balance: no part exceeds its share by more than a block plus two fixed costs
    total = sum(sch.num_blocks(L) + fixed for L in seqlens)
    assert max(costs) <= total / parts + 2 * fixed + 1
    return meta, num_splits


@pytest.mark.parametrize("seed", range(40))
def test_random_partitions(seed):
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 300))
    kind = seed % 4
    if kind == 0:
        lens = rng.integers(0, 20000, size=b)
    elif kind == 1:
        lens = np.full(b, int(rng.integers(1, 9000)))
    elif kind == 2:
        lens = rng.integers(0, 130, size=b)
    else:
        lens = np.where(rng.random(b) < 0.3, 0, rng.integers(1, 70000, size=b))
    parts = int(rng.integers(1, 160))
    check_partition([int(x) for x in lens], parts, FIXED if seed % 5 else 0)


def test_config_shapes():
    # the paged / split / mqa decode workloads on 76 SM pairs
    for b, L in ((64, 4096), (128, 8192), (256, 32768), (2, 256)):
        meta, ns = check_partition([L] * b, 76, FIXED)
    # one part: every sequence in one split (num_split = 1)
    meta, ns = check_partition([4096] * 64, 1, FIXED)
    assert ns == list(range(65))


def test_more_parts_than_work():
    meta, ns = check_partition([1, 0, 64], 150, FIXED)
    assert ns[-1] >= 3


def test_hand_example():
    """Three sequences of 2, 0 and 3 blocks, F = 1, two parts: TOTAL = 8, cut at 4,
    which lands in sequence 1's fixed cost... sequence 0 spans [0,3), 1 spans [3,4),
    2 spans [4,8): position 4 is sequence 2's fixed unit -> cut (2, 0)."""
    meta, ns = sch.schedule([128, 0, 150], 2, 1)
    assert meta[0][:5] == [0, 0, 2, 0, 0]
    assert meta[1][:5] == [2, 0, 3, 0, 2]
    assert ns == [0, 1, 2, 3]
    # with three parts: cuts at floor(8/3)=2 -> seq 0 block 1, floor(16/3)=5 -> seq 2 block 0
    meta, ns = sch.schedule([128, 0, 150], 3, 1)
    assert [m[:5] for m in meta] == [[0, 0, 0, 1, 0], [0, 1, 2, 0, 1], [2, 0, 3, 0, 3]]
    assert ns == [0, 2, 3, 4]


# ---- choosing the part count ----------------------------------------------------------

def test_part_costs_count_segments_and_blocks():
    # two sequences of 3 and 2 blocks, cut inside the first: part 0 holds one
    # segment of 2 blocks, part 1 two segments (1 + 2 blocks)
    meta, _ = sch.schedule([192, 128], 2, 0)
    assert [r[:4] for r in meta] == [[0, 0, 0, 2], [0, 2, 2, 0]]
    assert sch.part_costs(meta, [192, 128], 10) == [10 + 2, 20 + 3]


def test_candidate_parts():
    assert sch.candidate_parts(64, 76) == [76, 64]
    assert sch.candidate_parts(128, 76) == [76, 64]
    assert sch.candidate_parts(20, 76) == [76, 60, 40]
    assert sch.candidate_parts(1, 76) == [76, 75, 74, 73, 72, 71, 70, 69]
    assert sch.candidate_parts(7, 1) == [1]
    assert sch.candidate_parts(5, 10) == [10, 5]


def splits_any_sequence(lens, parts):
    """Brute force: some sequence is touched by more than one part."""
    touched = [0] * len(lens)
    for row in sch.schedule(lens, parts, FIXED)[0]:
        for (i, _, _, _) in sch.segments_of_part(row, lens):
            touched[i] += 1
    return any(t > 1 for t in touched)


@pytest.mark.parametrize("seed", range(25))
def test_choose_parts_is_the_cheapest_score(seed):
    """Brute force over the candidate counts: the chosen one has the lowest score
    (most expensive part, plus S if some sequence is split, counted by walking
    the parts), and no larger candidate ties with it."""
    rng = np.random.default_rng(1000 + seed)
    b = int(rng.integers(1, 120))
    lens = [int(x) for x in rng.integers(0, 9000, size=b)]
    if seed % 3 == 0:
        lens = [int(rng.integers(1, 9000))] * b       # equal sequences
    max_parts = int(rng.integers(1, 90))
    G = int(rng.choice([0, 4, 16, 40]))
    S = int(rng.choice([0, 10, 100]))
    p = sch.choose_parts(lens, max_parts, FIXED, G, S)
    cands = sch.candidate_parts(b, max_parts)
    assert p in cands and (max_parts + 1) // 2 <= p <= max_parts
    score = {q: max(sch.part_costs(sch.schedule(lens, q, FIXED)[0], lens, G))
             + (S if splits_any_sequence(lens, q) else 0) for q in cands}
    assert score[p] == min(score.values())
    assert all(score[q] > score[p] for q in cands if q > p)


def test_split_cost_decides_only_close_calls():
    # 128 sequences of 64 blocks on up to 76 parts: 76 parts (most expensive part
    # 155, 68 sequences split) against 64 parts of two whole sequences (160): the
    # combine pass of the split schedule tips it to 64
    lens = [4096] * 128
    assert sch.choose_parts(lens, 76, FIXED, 16, 0) == 76
    assert sch.choose_parts(lens, 76, FIXED, 16, 10) == 64
    # 8192-token sequences: 262 against 288, far apart: still 76 parts
    assert sch.choose_parts([8192] * 128, 76, FIXED, 16, 10) == 76
    # a schedule that splits nothing pays no split cost: 64 equal sequences
    assert sch.choose_parts([4096] * 64, 76, FIXED, 16, 10 ** 6) == 64
    # every candidate splits (one sequence): the cost shifts all scores alike
    assert sch.choose_parts([100000], 76, FIXED, 16, 10) == sch.choose_parts([100000], 76, FIXED, 16, 0)


def test_equal_sequences_get_one_part_each_when_segments_are_dear():
    # 64 sequences of 64 blocks on up to 76 parts: 76 parts cut most sequences in
    # two (two segments in most parts); 64 parts give each part one whole sequence
    lens = [4096] * 64
    assert sch.choose_parts(lens, 76, FIXED, 16, 0) == 64
    # with free segments the largest count wins
    assert sch.choose_parts(lens, 76, FIXED, 0, 0) == 76


@pytest.mark.parametrize("seed", range(10))
def test_schedule_auto_pads_with_empty_parts(seed):
    rng = np.random.default_rng(2000 + seed)
    b = int(rng.integers(1, 100))
    lens = [int(x) for x in rng.integers(0, 20000, size=b)]
    max_parts = int(rng.integers(2, 80))
    meta, ns, p = sch.schedule_auto(lens, max_parts, FIXED, 16, 10)
    assert len(meta) == max_parts
    ref_meta, ref_ns = check_partition(lens, p, FIXED)
    assert meta[:p] == ref_meta and ns == ref_ns
    for row in meta[p:]:
        assert row == [b, 0, b, 0, ns[b], 0, 0, 0]
        assert sch.segments_of_part(row, lens) == []


def test_binding_constants_match_the_header():
    import os
    import re
    import mla_decode_gb300 as mla
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "mla_decode.h")).read()
    for name in ("SCHED_FIXED_COST", "SCHED_SEGMENT_COST", "SCHED_SPLIT_COST", "BLOCK_N",
                 "META_STRIDE", "MAX_NUM_SM"):
        m = re.search(r"#define MLA_%s (\d+)" % name, hdr)
        assert m and int(m.group(1)) == getattr(mla, name), name


# (part count, split sequences) the scheduler gives each named workload on one GB300
# (152 SMs: 76 SM pairs, halved per extra 128-row tile); the measured tables and the
# benchmark's combine choice (fused exactly when nothing is split) rest on these
WORKLOAD_SCHEDULES = {
    "tiny": (76, 6), "paged": (64, 0), "split": (76, 72), "paged_8k": (76, 72),
    "varlen": (76, 75), "mqa": (76, 72), "mtp": (32, 0), "paged_fp8": (64, 0),
    "tl_example": (76, 72), "tl_bench_1024": (64, 0), "tl_bench_2048": (64, 0),
    "tl_bench_4096": (64, 0), "tl_bench_8192": (76, 72), "tl_bench_16384": (76, 72),
    "tl_bench_32768": (76, 72),
}


@pytest.mark.parametrize("name", sorted(WORKLOAD_SCHEDULES))
def test_workload_schedules(name):
    import mla_decode_gb300 as mla
    import workloads
    w = workloads.get(name)
    max_parts = 76 // ((w.rows + 127) // 128)
    meta, ns, p = sch.schedule_auto([int(x) for x in w.seqlens], max_parts, mla.SCHED_FIXED_COST,
                                    mla.SCHED_SEGMENT_COST, mla.SCHED_SPLIT_COST)
    assert (p, ns[-1] - w.batch) == WORKLOAD_SCHEDULES[name]
