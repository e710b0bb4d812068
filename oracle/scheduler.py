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
