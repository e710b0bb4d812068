// Tile-scheduler metadata kernel.
//
// Inputs and outputs follow FlashMLA's scheduling fields ("DeepSeek开源周第一天：
// FlashMLA 深度分析", section 内存访问优化: tile_scheduler_metadata_ptr,
// num_sm_parts, num_splits_ptr); per-sequence split sizing from cache_seqlens
// follows the paged variant of the TileLang MLA guide (section 6. Split-KV).
// The partition itself is this library's design:
//
//   sequence i costs F + ceil(L_i / 64) units and occupies [C_i, C_i + F + n_i)
//   on a cost axis (the F units first).  Part k starts at position
//   x_k = floor(k * TOTAL / P), mapped to the cut (i, max(0, x_k - C_i - F))
//   with i the last sequence whose start C_i <= x_k; x >= TOTAL maps to (b, 0).
//   Segments are numbered in (sequence, block) order; the number of segments
//   before cut k is cut_seq + (distinct interior cuts among cuts[0..k]).
//
// How many parts: a few counts P are tried: P_max and, from P_max - 1 down to
// ceil(P_max / 2), the first seven that divide b or are a multiple of b (on a
// batch of equal sequences, the counts whose cuts fall on sequence boundaries or
// split every sequence alike).  Part k of P costs G per segment it holds plus one
// per block; P scores its most expensive part, plus S when it splits some
// sequence (a partition with an interior cut needs the combine pass), and the
// lowest score wins (the larger P on a tie).  A segment costs more to run than F
// suggests (query load, pipeline fill and drain, output), so on a batch of equal
// sequences one part per sequence can beat more, split, parts.  Parts
// P..P_max-1 are left empty.
//
// One CTA; block scans in shared memory, no serial pass over the batch.
#include <stdint.h>

#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

constexpr int kMetaThreads = 512;
constexpr int kMetaWarps = kMetaThreads / 32;
constexpr int kCachedSeqs = 4096;  // per-sequence costs kept in shared memory up to this batch
constexpr int kMaxCand = 8;        // part counts tried

__device__ __forceinline__ int cost_of(const int32_t *seqlens, int i, int fixed) {
  const int L = seqlens[i];
  return fixed + (L > 0 ? (L + 63) / 64 : 0);
}

// floor(k * total / p) for 0 <= k <= p, in 32-bit arithmetic when p * total fits
// (a 64-bit division is a long instruction sequence).
__device__ __forceinline__ int64_t cost_position(int k, int64_t total, int p) {
  if ((uint64_t)p * (uint64_t)total < (1ull << 32)) return (int64_t)((uint32_t)k * (uint32_t)total / (uint32_t)p);
  return ((int64_t)k * total) / p;
}

// Exclusive prefix of v over the block (all threads call it); *total gets the sum.
__device__ int64_t block_exclusive_scan(int64_t v, int64_t *warp_sums, int64_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < kMetaWarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kMetaWarps) warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const int64_t excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  *total = warp_sums[kMetaWarps - 1];
  __syncthreads();  // warp_sums is reused by the next call
  return excl;
}

// The cut of cost position x: the last sequence ci whose start C_ci <= x (the
// last chunk whose start is <= x, then a walk inside it) and the block
// max(0, x - C_ci - F); x >= total maps to (b, 0).  *cstart gets C_ci (total
// for ci = b).  `cost` holds the sequences' costs when the batch fits the cache,
// else it is NULL and they are read from `seqlens`.
__device__ void cut_of(int64_t x, const int64_t *chunk_start, int nchunks, int per, int b,
                       int64_t total, const int32_t *seqlens, const int32_t *cost, int fixed,
                       int *ci, int *cb, int64_t *cstart) {
  if (x >= total) {
    *ci = b;
    *cb = 0;
    *cstart = total;
    return;
  }
  int lo_t = 0, hi_t = nchunks - 1;
  while (lo_t < hi_t) {
    const int mid = (lo_t + hi_t + 1) >> 1;
    if (chunk_start[mid] <= x) lo_t = mid; else hi_t = mid - 1;
  }
  int i = lo_t * per;
  const int end = min(b, i + per);
  int64_t start = chunk_start[lo_t];
  while (i + 1 < end) {  // (no walk when a chunk is one sequence)
    const int64_t next = start + (cost ? cost[i] : cost_of(seqlens, i, fixed));
    if (next > x) break;
    start = next;
    ++i;
  }
  *ci = i;
  const int64_t off = x - start - fixed;
  *cb = off > 0 ? (int)off : 0;
  *cstart = start;
}

__global__ void __launch_bounds__(kMetaThreads)
metadata_kernel(const int32_t *__restrict__ seqlens, int b, int max_parts, int fixed, int seg_cost,
                int split_cost, int32_t *__restrict__ meta, int32_t *__restrict__ num_splits) {
  extern __shared__ int32_t sh[];
  int32_t *cut_seq = sh;                        // [max_parts + 1]
  int32_t *cut_blk = cut_seq + max_parts + 1;   // [max_parts + 1]
  int32_t *rank = cut_blk + max_parts + 1;      // [max_parts + 1]
  int32_t *cost = b <= kCachedSeqs ? rank + max_parts + 1 : nullptr;  // [b] when cached
  __shared__ int64_t chunk_start[kMetaThreads];
  __shared__ int64_t warp_sums[kMetaWarps];
  __shared__ unsigned int worst[kMaxCand];  // per candidate part count (saturated at 2^31 - 1)
  __shared__ unsigned int splits[kMaxCand];  // per candidate: some cut falls inside a sequence
  __shared__ int cand[kMaxCand], ncand_sh, chosen;
  const int tid = threadIdx.x;
  // launched with programmatic stream serialisation: cache_seqlens may have been
  // written, and meta / num_splits still be read, by the kernels before this one
  sm100::grid_dependency_wait();
  sm100::launch_dependents();

  // Phase 1: thread t owns sequences [t per, (t + 1) per); the block scan of the
  // chunk costs gives each chunk's start on the cost axis, and TOTAL.
  const int per = (b + kMetaThreads - 1) / kMetaThreads;
  const int nchunks = (b + per - 1) / per;
  const int lo = min(b, tid * per), hi = min(b, lo + per);
  int64_t s = 0;
  for (int i = lo; i < hi; ++i) {
    const int ci = cost_of(seqlens, i, fixed);
    if (cost) cost[i] = ci;
    s += ci;
  }
  int64_t total = 0;
  chunk_start[tid] = block_exclusive_scan(s, warp_sums, &total);

  // Phase 1b: the part count.  Pairs (candidate c, part k < P_c) are spread over
  // the threads; part k of P costs seg_cost per segment plus its blocks (the
  // blocks before cut (i, blk) are C_i - F i + blk).
  if (tid < 32) {  // warp 0 scans the counts below max_parts 32 at a time, in order
    int n = 1;
    if (tid == 0) cand[0] = max_parts;
    const int p_lo = (max_parts + 1) / 2;
    for (int base = max_parts - 1; base >= p_lo && n < kMaxCand; base -= 32) {
      const int p = base - tid;
      const bool ok = p >= p_lo && (b % p == 0 || p % b == 0);
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      const int before = __popc(m & ((1u << tid) - 1u));
      if (ok && n + before < kMaxCand) cand[n + before] = p;
      n += __popc(m);
    }
    if (tid == 0) ncand_sh = min(n, kMaxCand);
  }
  if (tid < kMaxCand) {
    worst[tid] = 0u;
    splits[tid] = 0u;
  }
  __syncthreads();
  const int ncand = ncand_sh;
  {
    int64_t npairs = 0;
    for (int c = 0; c < ncand; ++c) npairs += cand[c];
    int c = 0;  // candidate c holds pairs [off, off + cand[c]); j only grows
    int64_t off = 0;
    for (int64_t j = tid; j < npairs; j += kMetaThreads) {
      while (j >= off + cand[c]) {
        off += cand[c];
        ++c;
      }
      const int P = cand[c], k = (int)(j - off);
      const int64_t x0 = cost_position(k, total, P);
      const int64_t x1 = cost_position(k + 1, total, P);
      int i0, b0, i1, b1;
      int64_t c0, c1;
      cut_of(x0, chunk_start, nchunks, per, b, total, seqlens, cost, fixed, &i0, &b0, &c0);
      cut_of(x1, chunk_start, nchunks, per, b, total, seqlens, cost, fixed, &i1, &b1, &c1);
      const int64_t blocks = (c1 - (int64_t)fixed * i1 + b1) - (c0 - (int64_t)fixed * i0 + b0);
      const int64_t segs = i0 < i1 ? (int64_t)(i1 - i0) + (b1 > 0 ? 1 : 0) : (b1 > b0 ? 1 : 0);
      const int64_t cst = segs * seg_cost + blocks;
      atomicMax(&worst[c], (unsigned int)(cst < 0x7fffffff ? cst : 0x7fffffff));
      if (b0 > 0) atomicOr(&splits[c], 1u);  // cut k lies inside sequence i0's blocks
    }
  }
  __syncthreads();
  if (tid == 0) {
    auto score = [&](int c) { return (int64_t)worst[c] + (splits[c] ? split_cost : 0); };
    int best = 0;  // candidates are in descending order: ties keep the larger count
    for (int c = 1; c < ncand; ++c)
      if (score(c) < score(best)) best = c;
    chosen = cand[best];
  }
  __syncthreads();
  const int parts = chosen;

  // Phase 2: the cut of each part.
  for (int k = tid; k <= parts; k += kMetaThreads) {
    const int64_t x = cost_position(k, total, parts);
    int ci, cb;
    int64_t cs;
    cut_of(x, chunk_start, nchunks, per, b, total, seqlens, cost, fixed, &ci, &cb, &cs);
    cut_seq[k] = ci;
    cut_blk[k] = cb;
  }
  __syncthreads();

  // Phase 3: running count of distinct interior cuts (a block scan per 512 cuts).
  int64_t carry = 0;
  for (int base = 0; base <= parts; base += kMetaThreads) {
    const int k = base + tid;
    int inner = 0;
    if (k <= parts)
      inner = cut_blk[k] > 0 &&
              (k == 0 || cut_seq[k] != cut_seq[k - 1] || cut_blk[k] != cut_blk[k - 1]);
    int64_t sum = 0;
    const int64_t excl = block_exclusive_scan(inner, warp_sums, &sum);
    if (k <= parts) rank[k] = (int32_t)(carry + excl + inner);
    carry += sum;
  }
  __syncthreads();

  // Phase 4: split prefix per sequence, and the metadata rows.
  for (int i = tid; i <= b; i += kMetaThreads) {
    int lo_k = 0, hi_k = parts + 1;  // first k with cut_seq[k] >= i
    while (lo_k < hi_k) {
      const int mid = (lo_k + hi_k) >> 1;
      if (cut_seq[mid] < i) lo_k = mid + 1; else hi_k = mid;
    }
    num_splits[i] = i + (lo_k > 0 ? rank[lo_k - 1] : 0);
  }
  for (int k = tid; k < max_parts; k += kMetaThreads) {
    int32_t *row = meta + (int64_t)k * MLA_META_STRIDE;  // (4-byte alignment only)
    if (k < parts) {
      row[0] = cut_seq[k];
      row[1] = cut_blk[k];
      row[2] = cut_seq[k + 1];
      row[3] = cut_blk[k + 1];
      row[4] = cut_seq[k] + rank[k];
    } else {  // unused part: an empty range at the end
      row[0] = b;
      row[1] = 0;
      row[2] = b;
      row[3] = 0;
      row[4] = b + rank[parts];
    }
    row[5] = 0;
    row[6] = 0;
    row[7] = 0;
  }
}

}  // namespace

cudaError_t launch_metadata(const int32_t *seqlens, int b, int parts, int fixed, int seg_cost,
                            int32_t *meta, int32_t *num_splits, cudaStream_t s) {
  size_t smem = sizeof(int32_t) * (3 * (size_t)(parts + 1) + (b <= kCachedSeqs ? (size_t)b : 0));
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(metadata_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(kMetaThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, metadata_kernel, seqlens, b, parts, fixed, seg_cost,
                            (int)MLA_SCHED_SPLIT_COST, meta, num_splits);
}

}  // namespace mla
