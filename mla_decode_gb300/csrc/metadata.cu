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
// One CTA; every phase is a simple loop, so the kernel costs a few us.
#include <stdint.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kMetaThreads = 512;

__global__ void __launch_bounds__(kMetaThreads)
metadata_kernel(const int32_t *__restrict__ seqlens, int b, int parts, int fixed,
                int32_t *__restrict__ meta, int32_t *__restrict__ num_splits) {
  extern __shared__ int32_t sh[];
  int32_t *cut_seq = sh;                    // [parts + 1]
  int32_t *cut_blk = cut_seq + parts + 1;   // [parts + 1]
  int32_t *rank = cut_blk + parts + 1;      // [parts + 1]
  __shared__ int64_t chunk_sum[kMetaThreads];
  const int tid = threadIdx.x;

  // Phase 1: exclusive prefix of per-sequence cost, kept in num_splits[0..b-1]
  // for the moment; TOTAL in num_splits[b].
  const int per = (b + kMetaThreads - 1) / kMetaThreads;
  const int lo = min(b, tid * per), hi = min(b, lo + per);
  int64_t s = 0;
  for (int i = lo; i < hi; ++i) {
    int L = seqlens[i];
    s += fixed + (L > 0 ? (L + 63) / 64 : 0);
  }
  chunk_sum[tid] = s;
  __syncthreads();
  if (tid == 0) {
    int64_t acc = 0;
    for (int t = 0; t < kMetaThreads; ++t) {
      int64_t v = chunk_sum[t];
      chunk_sum[t] = acc;
      acc += v;
    }
    num_splits[b] = (int32_t)acc;
  }
  __syncthreads();
  {
    int64_t acc = chunk_sum[tid];
    for (int i = lo; i < hi; ++i) {
      num_splits[i] = (int32_t)acc;
      int L = seqlens[i];
      acc += fixed + (L > 0 ? (L + 63) / 64 : 0);
    }
  }
  __syncthreads();
  const int64_t total = num_splits[b];

  // Phase 2: the cut of each part.
  for (int k = tid; k <= parts; k += kMetaThreads) {
    int64_t x = (k == parts) ? total : ((int64_t)k * total) / parts;
    int ci, cb;
    if (x >= total) {
      ci = b;
      cb = 0;
    } else {
      int lo_i = 0, hi_i = b - 1;  // last i with start_i <= x
      while (lo_i < hi_i) {
        int mid = (lo_i + hi_i + 1) >> 1;
        if ((int64_t)num_splits[mid] <= x) lo_i = mid; else hi_i = mid - 1;
      }
      ci = lo_i;
      int64_t off = x - (int64_t)num_splits[ci] - fixed;
      cb = off > 0 ? (int)off : 0;
    }
    cut_seq[k] = ci;
    cut_blk[k] = cb;
  }
  __syncthreads();

  // Phase 3: running count of distinct interior cuts.
  if (tid == 0) {
    int r = 0;
    for (int k = 0; k <= parts; ++k) {
      bool inner = cut_blk[k] > 0 &&
                   (k == 0 || cut_seq[k] != cut_seq[k - 1] || cut_blk[k] != cut_blk[k - 1]);
      r += inner ? 1 : 0;
      rank[k] = r;
    }
  }
  __syncthreads();

  // Phase 4: split prefix per sequence, and the metadata rows.
  for (int i = tid; i <= b; i += kMetaThreads) {
    int lo_k = 0, hi_k = parts + 1;  // first k with cut_seq[k] >= i
    while (lo_k < hi_k) {
      int mid = (lo_k + hi_k) >> 1;
      if (cut_seq[mid] < i) lo_k = mid + 1; else hi_k = mid;
    }
    num_splits[i] = i + (lo_k > 0 ? rank[lo_k - 1] : 0);
  }
  for (int k = tid; k < parts; k += kMetaThreads) {
    int32_t *row = meta + (int64_t)k * MLA_META_STRIDE;
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
  metadata_kernel<<<1, kMetaThreads, smem, s>>>(seqlens, b, parts, fixed, meta, num_splits);
  return cudaGetLastError();
}

}  // namespace mla
