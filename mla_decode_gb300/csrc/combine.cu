// Split-KV combine kernel ("用 TileLang 编写高性能 DeepSeek MLA 内核…", section
// Combine Kernel): for a sequence with S > 1 splits and each head,
//   lse_max = max_k lse_k
//   lse     = log2(sum_k 2^(lse_k - lse_max)) + lse_max
//   out     = sum_k 2^(lse_k - lse) * O_k
// with lse_k the base-2 LSE of split k (scale folded in) and O_k its
// normalised partial output.  Sequences with one split were finished by the
// split kernel and are skipped.
//
// Grid (b, ceil(h / 8)); one warp per head; lane j owns columns
// 4j + 128c + {0..3}, c = 0..3, so every partial row is read as four fully
// coalesced 512-byte warp loads.
#include <stdint.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(FwdArgs a) {
  const int seq = blockIdx.x;
  const int s0 = a.num_splits[seq];
  const int n = a.num_splits[seq + 1] - s0;
  if (n <= 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.y * kWarps + warp;
  if (head >= a.h) return;

  const int64_t base = (int64_t)s0 * a.h + head;
  float4 acc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  auto load_row = [&](int64_t sp, float4 (&v)[4]) {
    const float4 *src = reinterpret_cast<const float4 *>(a.oaccum + sp * MLA_HEAD_DIM_V);
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = src[lane + 32 * c];
  };
  auto add = [&](float w, const float4 (&v)[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      acc[c].x = fmaf(w, v[c].x, acc[c].x);
      acc[c].y = fmaf(w, v[c].y, acc[c].y);
      acc[c].z = fmaf(w, v[c].z, acc[c].z);
      acc[c].w = fmaf(w, v[c].w, acc[c].w);
    }
  };
  // the first two partial rows (n >= 2 here) do not depend on the LSE reduction:
  // their loads are in flight while it runs
  float4 v0[4], v1[4];
  load_row(base, v0);
  load_row(base + a.h, v1);

  // lane k keeps split k's LSE (k < 32) for the sum and the weights
  float mine = -INFINITY, mx = -INFINITY;
  for (int k = lane; k < n; k += 32) {
    const float l = a.lseaccum[base + (int64_t)k * a.h];
    if (k == lane) mine = l;
    mx = fmaxf(mx, l);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float mref = (mx == -INFINITY) ? 0.f : mx;
  float sum = 0.f;
  for (int k = lane; k < n; k += 32)
    sum += fast_exp2((k == lane ? mine : a.lseaccum[base + (int64_t)k * a.h]) - mref);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float lse = sum > 0.f ? fast_log2(sum) + mref : -INFINITY;
  auto weight = [&](int k) {
    const float l = k < 32 ? __shfl_sync(0xffffffffu, mine, k) : a.lseaccum[base + (int64_t)k * a.h];
    return lse == -INFINITY ? 0.f : fast_exp2(l - lse);
  };

  add(weight(0), v0);
  add(weight(1), v1);
  // the rest two at a time, both rows' loads issued before either is used
  int k = 2;
  for (; k + 1 < n; k += 2) {
    load_row(base + (int64_t)k * a.h, v0);
    load_row(base + (int64_t)(k + 1) * a.h, v1);
    add(weight(k), v0);
    add(weight(k + 1), v1);
  }
  if (k < n) {
    load_row(base + (int64_t)k * a.h, v0);
    add(weight(k), v0);
  }
  // four consecutive 16-bit outputs per lane and column group: one 8-byte store
  T *o = reinterpret_cast<T *>(a.out) + seq * a.o_batch_stride + (int64_t)head * a.o_head_stride;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int d = 4 * lane + 128 * c;
    T q4[4] = {Elem<T>::from_f(acc[c].x), Elem<T>::from_f(acc[c].y), Elem<T>::from_f(acc[c].z),
               Elem<T>::from_f(acc[c].w)};
    *reinterpret_cast<uint2 *>(o + d) = *reinterpret_cast<const uint2 *>(q4);
  }
  if (lane == 0) a.lse[seq * a.lse_stride + head] = lse * kLn2;
}

}  // namespace

cudaError_t launch_combine(const FwdArgs &a, cudaStream_t s) {
  dim3 grid(a.b, (a.h + kWarps - 1) / kWarps);
  if (a.dtype == MLA_DTYPE_BF16)
    combine_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, s>>>(a);
  else
    combine_kernel<__half><<<grid, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
