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
// Grid (b, ceil(h / 32), 4): one CTA per sequence, 32-row group and quarter of
// the 512 columns; 4 warps of 32 columns (8 chunks) each.  The 16-bit results go
// through a swizzled shared-memory tile so that every output row is written as
// 64-byte pieces.
#include <stdint.h>

#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

constexpr int kWarps = 4;
constexpr int kChunks = 8;  // 4-column chunks per warp: 32 columns

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(FwdArgs a) {
  // launched with programmatic stream serialisation: the split kernel's partials
  // are read only once it has completed
  sm100::grid_dependency_wait();
  sm100::launch_dependents();
  const int seq = blockIdx.x;
  const int s0 = a.num_splits[seq];
  const int n = a.num_splits[seq + 1] - s0;
  if (n <= 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head0 = blockIdx.y * 32;
  const int head = head0 + lane;  // this lane's query row
  const bool hv = head < a.h;
  const int c0 = 32 * blockIdx.z + kChunks * warp;  // first column chunk of this warp
  __shared__ uint4 tile[kWarps][32][4];             // [warp][row][16-B piece, swizzled]

  // the first two splits' partial rows do not depend on the LSE reduction: their
  // loads are in flight while it runs
  const float4 *base = reinterpret_cast<const float4 *>(a.oaccum) + (int64_t)c0 * a.h + head;
  const int64_t split_stride = (int64_t)128 * a.h;  // float4s between splits
  auto load = [&](int k, float4 (&v)[kChunks]) {
    const float4 *src = base + (int64_t)(s0 + k) * split_stride;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) v[c] = hv ? src[(int64_t)c * a.h] : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  float4 v0[kChunks], v1[kChunks];
  load(0, v0);
  load(1, v1);

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
    const float w0 = weight(0), w1 = weight(1);
#pragma unroll
    for (int c = 0; c < kChunks; ++c)
      acc[c] = make_float4(fmaf(w1, v1[c].x, w0 * v0[c].x), fmaf(w1, v1[c].y, w0 * v0[c].y),
                           fmaf(w1, v1[c].z, w0 * v0[c].z), fmaf(w1, v1[c].w, w0 * v0[c].w));
  }
  for (int k = 2; k < n; ++k) {
    load(k, v0);
    const float w = weight(k);
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
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
    tile[warp][lane][j ^ ((lane >> 1) & 3)] = *reinterpret_cast<const uint4 *>(q8);
  }
  __syncwarp();
  // eight rows x 64 bytes per store instruction
  T *out = reinterpret_cast<T *>(a.out) + (int64_t)seq * a.o_batch_stride + 4 * c0;
#pragma unroll
  for (int r0 = 0; r0 < 32; r0 += 8) {
    const int row = r0 + (lane >> 2), j = lane & 3;
    if (head0 + row < a.h)
      *reinterpret_cast<uint4 *>(out + (int64_t)(head0 + row) * a.o_head_stride + 8 * j) =
          tile[warp][row][j ^ ((row >> 1) & 3)];
  }
  if (blockIdx.z == 0 && warp == 0 && hv) a.lse[seq * a.lse_stride + head] = lse * kLn2;
}

}  // namespace

cudaError_t launch_combine(const FwdArgs &a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.b, (a.h + 31) / 32, 4);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // e4m3 inputs give bf16 outputs
  return a.dtype == MLA_DTYPE_FP16 ? cudaLaunchKernelEx(&cfg, combine_kernel<__half>, a)
                                   : cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16>, a);
}

}  // namespace mla
