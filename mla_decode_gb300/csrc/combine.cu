// Split-KV combine kernel ("用 TileLang 编写高性能 DeepSeek MLA 内核…", section
// Combine Kernel): for a sequence with S > 1 splits and each query row,
//   lse_max = max_k lse_k
//   lse     = log2(sum_k 2^(lse_k - lse_max)) + lse_max
//   out     = sum_k 2^(lse_k - lse) * O_k
// with lse_k the base-2 LSE of split k (scale folded in) and O_k its
// normalised partial output.  Sequences with one split were finished by the
// split kernel and are skipped.
//
// The partials are stored [split][128 column chunks][h rows][4 floats], so a
// warp whose lanes are 32 consecutive rows reads 512 contiguous bytes per chunk.
// Grid (b, ceil(h / 32), 2): one CTA per sequence, 32-row group and half of the
// 512 columns; 4 warps of 64 columns (16 chunks) each.  The 16-bit results go
// through a swizzled shared-memory tile so that every output row is written as
// 128-byte pieces.
#include <stdint.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 4;
constexpr int kChunks = 16;  // 4-column chunks per warp

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(FwdArgs a) {
  const int seq = blockIdx.x;
  const int s0 = a.num_splits[seq];
  const int n = a.num_splits[seq + 1] - s0;
  if (n <= 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head0 = blockIdx.y * 32;
  const int head = head0 + lane;  // this lane's query row
  const bool hv = head < a.h;
  const int c0 = 64 * blockIdx.z + kChunks * warp;  // first column chunk of this warp
  __shared__ uint4 tile[kWarps][32][8];             // [warp][row][16-B piece ^ (row & 7)]

  // the first split's partial rows do not depend on the LSE reduction: their loads
  // are in flight while it runs
  const float4 *base = reinterpret_cast<const float4 *>(a.oaccum) + (int64_t)c0 * a.h + head;
  const int64_t split_stride = (int64_t)128 * a.h;  // float4s between splits
  float4 v[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; ++c)
    v[c] = hv ? base[(int64_t)s0 * split_stride + (int64_t)c * a.h] : make_float4(0.f, 0.f, 0.f, 0.f);

  float mx = -INFINITY;
  if (hv)
    for (int k = 0; k < n; ++k) mx = fmaxf(mx, a.lseaccum[(int64_t)(s0 + k) * a.h + head]);
  const float mref = (mx == -INFINITY) ? 0.f : mx;
  float sum = 0.f;
  if (hv)
    for (int k = 0; k < n; ++k) sum += fast_exp2(a.lseaccum[(int64_t)(s0 + k) * a.h + head] - mref);
  const float lse = sum > 0.f ? fast_log2(sum) + mref : -INFINITY;
  auto weight = [&](int k) {
    return (!hv || lse == -INFINITY) ? 0.f
                                     : fast_exp2(a.lseaccum[(int64_t)(s0 + k) * a.h + head] - lse);
  };

  float4 acc[kChunks];
  {
    const float w = weight(0);
#pragma unroll
    for (int c = 0; c < kChunks; ++c)
      acc[c] = make_float4(w * v[c].x, w * v[c].y, w * v[c].z, w * v[c].w);
  }
  for (int k = 1; k < n; ++k) {
#pragma unroll
    for (int c = 0; c < kChunks; ++c)
      v[c] = hv ? base[(int64_t)(s0 + k) * split_stride + (int64_t)c * a.h]
                : make_float4(0.f, 0.f, 0.f, 0.f);
    const float w = weight(k);
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      acc[c].x = fmaf(w, v[c].x, acc[c].x);
      acc[c].y = fmaf(w, v[c].y, acc[c].y);
      acc[c].z = fmaf(w, v[c].z, acc[c].z);
      acc[c].w = fmaf(w, v[c].w, acc[c].w);
    }
  }

  // my row's 64 columns as 16-bit values: eight 16-byte pieces, piece j stored at
  // position j ^ (row & 7) (no bank conflicts on the write or the read below)
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 &x = acc[2 * j], &y = acc[2 * j + 1];
    T q8[8] = {Elem<T>::from_f(x.x), Elem<T>::from_f(x.y), Elem<T>::from_f(x.z), Elem<T>::from_f(x.w),
               Elem<T>::from_f(y.x), Elem<T>::from_f(y.y), Elem<T>::from_f(y.z), Elem<T>::from_f(y.w)};
    tile[warp][lane][j ^ (lane & 7)] = *reinterpret_cast<const uint4 *>(q8);
  }
  __syncwarp();
  // four rows x 128 bytes per store instruction
  T *out = reinterpret_cast<T *>(a.out) + (int64_t)seq * a.o_batch_stride + 4 * c0;
#pragma unroll
  for (int r0 = 0; r0 < 32; r0 += 4) {
    const int row = r0 + (lane >> 3), j = lane & 7;
    if (head0 + row < a.h)
      *reinterpret_cast<uint4 *>(out + (int64_t)(head0 + row) * a.o_head_stride + 8 * j) =
          tile[warp][row][j ^ (row & 7)];
  }
  if (blockIdx.z == 0 && warp == 0 && hv) a.lse[seq * a.lse_stride + head] = lse * kLn2;
}

}  // namespace

cudaError_t launch_combine(const FwdArgs &a, cudaStream_t s) {
  dim3 grid(a.b, (a.h + 31) / 32, 2);
  if (a.dtype == MLA_DTYPE_BF16)
    combine_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, s>>>(a);
  else
    combine_kernel<__half><<<grid, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
