"""Tile-scheduler oracle: plain-Python restatement of the split-KV work partition.

TEST INFRASTRUCTURE ONLY (imported by tests, the smoke check and the CPU
baseline leg of the benchmark; never by the product path).

The pages name the scheduler's inputs and outputs but not its algorithm:
  "DeepSeek开源周第一天：FlashMLA 深度分析", section 内存访问优化
  (Flash_fwd_mla_params: tile_scheduler_metadata_ptr, num_sm_parts,
  num_splits_ptr), and the TileLang MLA guide ("用 TileLang 编写高性能
  DeepSeek MLA 内核…完整实战指南"), section 6. Split-KV (per-sequence
  blocks_per_split / remaining_blocks from cache_seqlens).  So the partition
  below is this project's design; this file states it as plainly as possible
  and the GPU metadata kernel must reproduce it bit for bit.

The partition
-------------
Each sequence i has nblk_i = ceil(L_i / 64) KV blocks of 64 tokens and a fixed
per-segment cost F (query load, epilogue, combine), counted in blocks.  Lay the
sequences end to end on a cost axis: sequence i occupies
[C_i, C_i + F + nblk_i), where C_i is the sum of (F + nblk_j) over j < i, and
the F units come first.  With TOTAL = C_b, part k (of P) starts at the cost
position x_k = floor(k * TOTAL / P).  A position x inside sequence i maps to
the cut (i, blk) with blk = max(0, x - C_i - F); position TOTAL maps to (b, 0).
Part k covers the block range [cut_k, cut_{k+1}) in (sequence, block)
lexicographic order.  Every sequence, including an empty one, yields one
segment per part that touches it; segments are numbered globally in
(sequence, block) order, which is also the order of their partial outputs.

Outputs (the layout the C ABI documents):
  metadata[k] = [begin_seq, begin_blk, end_seq, end_blk, first_split, 0, 0, 0]
  num_splits  = prefix sums, num_splits[i+1] - num_splits[i] = segments of i

How many parts
--------------
A segment costs far more than the F of the cost axis suggests once it is run
(loading the query, filling and draining the pipeline, writing its output), so
cutting a sequence into more segments can lose more than the extra parts gain.
`schedule_auto` therefore tries a few part counts, charges each part G per
segment plus one per block, scores a count by its most expensive part plus S
when its partition splits some sequence (a split sequence needs the combine
pass, a cost outside every part), and keeps the count with the lowest score
(the larger count on a tie).  The counts tried are P_max and, from
P_max - 1 down to ceil(P_max / 2), the first seven that divide b or are a
multiple of it: on a batch of equal sequences those are the counts whose cuts
fall on sequence boundaries or split every sequence alike.  Parts P..P_max-1
are left empty: [b, 0, b, 0, num_splits[b], 0, 0, 0].
"""

BLOCK_N = 64
META_STRIDE = 8


def num_blocks(seqlen):
    return 0 if seqlen <= 0 else (seqlen + BLOCK_N - 1) // BLOCK_N


def schedule(seqlens, num_parts, fixed_cost):
    """Return (metadata rows, num_splits prefix list) for the given lengths."""
    b = len(seqlens)
    nblk = [num_blocks(int(L)) for L in seqlens]
    start = []  # C_i
    acc = 0
    for n in nblk:
        start.append(acc)
        acc += fixed_cost + n
    total = acc

    def cut_at(x):
        if x >= total:
            return (b, 0)
        i = 0
        while i + 1 < b and start[i + 1] <= x:
            i += 1
        return (i, max(0, x - start[i] - fixed_cost))

    cuts = [cut_at((k * total) // num_parts) for k in range(num_parts)] + [(b, 0)]

    # Segment starts inside each sequence: block 0, plus every distinct cut
    # that falls strictly inside the sequence's block range.
    inner = [set() for _ in range(b)]
    for (i, blk) in cuts:
        if i < b and blk > 0:
            inner[i].add(blk)
    num_splits = [0]
    for i in range(b):
        num_splits.append(num_splits[-1] + 1 + len(inner[i]))

    meta = []
    for k in range(num_parts):
        (bi, bb), (ei, eb) = cuts[k], cuts[k + 1]
        if bi < b:
            first = num_splits[bi] + sum(1 for c in inner[bi] if c <= bb)
        else:
            first = num_splits[b]
        meta.append([bi, bb, ei, eb, first, 0, 0, 0])
    return meta, num_splits


def part_costs(meta, seqlens, segment_cost):
    """Cost of each part: `segment_cost` per segment it holds plus one per block."""
    return [sum(segment_cost + (hi - lo) for (_, lo, hi, _) in segments_of_part(row, seqlens))
            for row in meta]


MAX_CANDIDATES = 8


def candidate_parts(b, max_parts):
    """max_parts, then the first MAX_CANDIDATES - 1 counts below it, down to
    ceil(max_parts / 2), that divide b or are a multiple of b (descending)."""
    out = [max_parts]
    for p in range(max_parts - 1, (max_parts + 1) // 2 - 1, -1):
        if len(out) == MAX_CANDIDATES:
            break
        if b % p == 0 or p % b == 0:
            out.append(p)
    return out


def choose_parts(seqlens, max_parts, fixed_cost, segment_cost, split_cost):
    """Among candidate_parts(), the count with the lowest score: its most
    expensive part, plus split_cost when some sequence gets more than one
    segment; ties go to the larger count."""
    b = len(seqlens)
    best, best_p = None, max_parts
    for p in candidate_parts(b, max_parts):
        meta, num_splits = schedule(seqlens, p, fixed_cost)
        t = max(part_costs(meta, seqlens, segment_cost))
        if num_splits[b] > b:
            t += split_cost
        if best is None or t < best:
            best, best_p = t, p
    return best_p


def schedule_auto(seqlens, max_parts, fixed_cost, segment_cost, split_cost):
    """schedule() with the part count chosen by choose_parts(); the metadata has
    max_parts rows, the ones past the chosen count empty.  Returns (metadata rows,
    num_splits prefix list, parts used)."""
    b = len(seqlens)
    p = choose_parts(seqlens, max_parts, fixed_cost, segment_cost, split_cost)
    meta, num_splits = schedule(seqlens, p, fixed_cost)
    meta = meta + [[b, 0, b, 0, num_splits[b], 0, 0, 0] for _ in range(max_parts - p)]
    return meta, num_splits, p


def segments_of_part(meta_row, seqlens):
    """Enumerate (seq, blk_begin, blk_end, split_id) for one part, in order."""
    bi, bb, ei, eb, split = meta_row[:5]
    out = []
    i, blk = bi, bb
    while (i, blk) < (ei, eb):
        end = num_blocks(int(seqlens[i])) if i < ei else eb
        out.append((i, blk, end, split))
        split += 1
        i, blk = i + 1, 0
    return out
