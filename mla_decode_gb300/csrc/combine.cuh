// The split-KV combine of one 32-row x 32-column block ("用 TileLang 编写高性能
// DeepSeek MLA 内核…", section Combine Kernel): for a sequence with n > 1 splits
// and each query row,
//   lse_max = max_k lse_k
//   lse     = log2(sum_k 2^(lse_k - lse_max)) + lse_max
//   out     = sum_k 2^(lse_k - lse) * O_k
// with lse_k the base-2 LSE of split k (scale folded in) and O_k its normalised
// partial output.  One warp: lane = query row head0 + lane, columns
// [4 c0, 4 c0 + 32).  Used by the combine kernel and by the split kernel's own
// combine phase, so both give the same bits.
//
// The partials are stored [split][128 column chunks][h rows][4 floats], so the
// warp reads 512 contiguous bytes per chunk.  The 16-bit results pass through the
// warp's swizzled 2 KB shared-memory tile so that every output row is written as
// 64-byte pieces.
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace mla {

constexpr int kCombineChunks = 8;  // 4-column chunks per warp block: 32 columns
constexpr int kCombineLse = 8;     // splits whose LSEs are held in registers

template <typename T>
__device__ __forceinline__ void combine_block(const FwdArgs &a, int seq, int s0, int n, int head0, int c0,
                                              uint4 (*tile)[4], int lane) {
  const int head = head0 + lane;  // this lane's query row
  const bool hv = head < a.h;
  // the first two splits' partial rows do not depend on the LSE reduction: their
  // loads are in flight while it runs
  const float4 *base = reinterpret_cast<const float4 *>(a.oaccum) + (int64_t)c0 * a.h + head;
  const int64_t split_stride = (int64_t)128 * a.h;  // float4s between splits
  // each partial row is read once: its L2 lines go first (the split kernel wrote
  // them with evict_last)
  const uint64_t drop = sm100::l2_policy_evict_first();
  auto load = [&](int k, float4 (&v)[kCombineChunks]) {
    const float4 *src = base + (int64_t)(s0 + k) * split_stride;
#pragma unroll
    for (int c = 0; c < kCombineChunks; ++c)
      v[c] = hv ? sm100::ld_global_v4_hint(src + (int64_t)c * a.h, drop) : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  // the LSEs of the first kCombineLse splits are loaded together with the first
  // two partial rows (one memory round trip for the common case)
  const float *lrow = a.lseaccum + (int64_t)s0 * a.h + head;
  float lk[kCombineLse];
#pragma unroll
  for (int k = 0; k < kCombineLse; ++k) lk[k] = (hv && k < n) ? lrow[(int64_t)k * a.h] : -INFINITY;
  auto lse_of = [&](int k) { return k < kCombineLse ? lk[k] : lrow[(int64_t)k * a.h]; };
  float4 v0[kCombineChunks], v1[kCombineChunks];
  load(0, v0);
  load(1, v1);

  float mx = -INFINITY;
  if (hv) {
#pragma unroll
    for (int k = 0; k < kCombineLse; ++k)
      if (k < n) mx = fmaxf(mx, lk[k]);
    for (int k = kCombineLse; k < n; ++k) mx = fmaxf(mx, lrow[(int64_t)k * a.h]);
  }
  const float mref = (mx == -INFINITY) ? 0.f : mx;
  float sum = 0.f;
  if (hv) {
#pragma unroll
    for (int k = 0; k < kCombineLse; ++k)
      if (k < n) sum += fast_exp2(lk[k] - mref);
    for (int k = kCombineLse; k < n; ++k) sum += fast_exp2(lrow[(int64_t)k * a.h] - mref);
  }
  const float lse = sum > 0.f ? fast_log2(sum) + mref : -INFINITY;
  auto weight = [&](int k) { return (!hv || lse == -INFINITY) ? 0.f : fast_exp2(lse_of(k) - lse); };

  float4 acc[kCombineChunks];
  {
    const float w0 = weight(0), w1 = weight(1);
#pragma unroll
    for (int c = 0; c < kCombineChunks; ++c)
      acc[c] = make_float4(fmaf(w1, v1[c].x, w0 * v0[c].x), fmaf(w1, v1[c].y, w0 * v0[c].y),
                           fmaf(w1, v1[c].z, w0 * v0[c].z), fmaf(w1, v1[c].w, w0 * v0[c].w));
  }
  for (int k = 2; k < n; ++k) {
    load(k, v0);
    const float w = weight(k);
#pragma unroll
    for (int c = 0; c < kCombineChunks; ++c) {
      acc[c].x = fmaf(w, v0[c].x, acc[c].x);
      acc[c].y = fmaf(w, v0[c].y, acc[c].y);
      acc[c].z = fmaf(w, v0[c].z, acc[c].z);
      acc[c].w = fmaf(w, v0[c].w, acc[c].w);
    }
  }

  // my row's 32 columns as 16-bit values: four 16-byte pieces, piece j stored at
  // position j ^ ((row >> 1) & 3), which spreads 8 consecutive rows over all 32
  // banks (no conflicts on the write or the read below)
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 &x = acc[2 * j], &y = acc[2 * j + 1];
    T q8[8] = {Elem<T>::from_f(x.x), Elem<T>::from_f(x.y), Elem<T>::from_f(x.z), Elem<T>::from_f(x.w),
               Elem<T>::from_f(y.x), Elem<T>::from_f(y.y), Elem<T>::from_f(y.z), Elem<T>::from_f(y.w)};
    tile[lane][j ^ ((lane >> 1) & 3)] = *reinterpret_cast<const uint4 *>(q8);
  }
  __syncwarp();
  // eight rows x 64 bytes per store instruction
  T *out = reinterpret_cast<T *>(a.out) + (int64_t)seq * a.o_batch_stride + 4 * c0;
#pragma unroll
  for (int r0 = 0; r0 < 32; r0 += 8) {
    const int row = r0 + (lane >> 2), j = lane & 3;
    if (head0 + row < a.h)
      *reinterpret_cast<uint4 *>(out + (int64_t)(head0 + row) * a.o_head_stride + 8 * j) =
          tile[row][j ^ ((row >> 1) & 3)];
  }
  __syncwarp();  // the tile is reused by the warp's next block
  if (c0 == 0 && hv) a.lse[seq * a.lse_stride + head] = lse * kLn2;
}

}  // namespace mla
