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
// One CTA; block scans in shared memory, no serial pass over the batch.
#include <stdint.h>

#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

constexpr int kMetaThreads = 512;
constexpr int kMetaWarps = kMetaThreads / 32;

__device__ __forceinline__ int cost_of(const int32_t *seqlens, int i, int fixed) {
  const int L = seqlens[i];
  return fixed + (L > 0 ? (L + 63) / 64 : 0);
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

__global__ void __launch_bounds__(kMetaThreads)
metadata_kernel(const int32_t *__restrict__ seqlens, int b, int parts, int fixed,
                int32_t *__restrict__ meta, int32_t *__restrict__ num_splits) {
  extern __shared__ int32_t sh[];
  int32_t *cut_seq = sh;                    // [parts + 1]
  int32_t *cut_blk = cut_seq + parts + 1;   // [parts + 1]
  int32_t *rank = cut_blk + parts + 1;      // [parts + 1]
  __shared__ int64_t chunk_start[kMetaThreads];
  __shared__ int64_t warp_sums[kMetaWarps];
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
  for (int i = lo; i < hi; ++i) s += cost_of(seqlens, i, fixed);
  int64_t total = 0;
  chunk_start[tid] = block_exclusive_scan(s, warp_sums, &total);
  __syncthreads();

  // Phase 2: the cut of each part.  The sequence is the last one whose start is
  // <= x: the last chunk whose start is <= x, then a walk inside it.
  for (int k = tid; k <= parts; k += kMetaThreads) {
    const int64_t x = (k == parts) ? total : ((int64_t)k * total) / parts;
    int ci, cb;
    if (x >= total) {
      ci = b;
      cb = 0;
    } else {
      int lo_t = 0, hi_t = nchunks - 1;
      while (lo_t < hi_t) {
        const int mid = (lo_t + hi_t + 1) >> 1;
        if (chunk_start[mid] <= x) lo_t = mid; else hi_t = mid - 1;
      }
      int i = lo_t * per;
      const int end = min(b, i + per);
      int64_t start = chunk_start[lo_t];
      for (;;) {
        const int64_t next = start + cost_of(seqlens, i, fixed);
        if (i + 1 >= end || next > x) break;
        start = next;
        ++i;
      }
      ci = i;
      const int64_t off = x - start - fixed;
      cb = off > 0 ? (int)off : 0;
    }
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
  for (int k = tid; k < parts; k += kMetaThreads) {
    int32_t *row = meta + (int64_t)k * MLA_META_STRIDE;  // (4-byte alignment only)
    row[0] = cut_seq[k];
    row[1] = cut_blk[k];
    row[2] = cut_seq[k + 1];
    row[3] = cut_blk[k + 1];
    row[4] = cut_seq[k] + rank[k];
    row[5] = 0;
    row[6] = 0;
    row[7] = 0;
  }
}

}  // namespace

cudaError_t launch_metadata(const int32_t *seqlens, int b, int parts, int fixed,
                            int32_t *meta, int32_t *num_splits, cudaStream_t s) {
  size_t smem = sizeof(int32_t) * 3 * (size_t)(parts + 1);
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
  return cudaLaunchKernelEx(&cfg, metadata_kernel, seqlens, b, parts, fixed, meta, num_splits);
}

}  // namespace mla
