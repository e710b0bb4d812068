// Correctness-first split kernel on the CUDA cores (no tensor cores).
//
// Same contract as the tensor-core split kernel: one CTA per (metadata part,
// 16-head tile) walks the part's segments; per 64-token block it forms the
// 576-wide scores, runs the exp2 online-softmax update and accumulates the
// 512-wide value sum in fp32 ("用 TileLang 编写高性能 DeepSeek MLA 内核…",
// sections 先看核心难点 and Split Kernel; FlashMLA analysis, section Softmax
// 计算优化 for the -inf guard and the exp2/FFMA form).  A sequence with one
// split writes out/lse directly; otherwise the normalised partial and its
// base-2 LSE go to the workspace for the combine kernel.
#include <stdint.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kHT = 16;          // heads per CTA
constexpr int kThreads = 256;
constexpr int kRow = 578;        // padded smem row (elements): odd word stride
constexpr int kBlockN = 64;

template <typename T>
__global__ void __launch_bounds__(kThreads)
split_simt_kernel(FwdArgs a) {
  extern __shared__ float smem_f[];
  float *q_s = smem_f;                                   // [16][576] fp32
  float *p_s = q_s + kHT * MLA_HEAD_DIM;                 // [16][64]
  uint16_t *kv_s = reinterpret_cast<uint16_t *>(p_s + kHT * kBlockN);  // [64][578]

  const int tid = threadIdx.x;
  const int part = blockIdx.x;
  const int head0 = blockIdx.y * kHT;
  const int hh = tid >> 4;   // head within the tile
  const int g = tid & 15;    // lane within the head group
  const int head = head0 + hh;
  const bool head_ok = head < a.h;

  const int32_t *row = a.meta + (int64_t)part * MLA_META_STRIDE;
  int seq = row[0], blk0 = row[1];
  const int end_seq = row[2], end_blk = row[3];
  int split = row[4];

  const T *q = reinterpret_cast<const T *>(a.q);
  const uint16_t *kv = reinterpret_cast<const uint16_t *>(a.kv);

  while (seq < end_seq || (seq == end_seq && blk0 < end_blk)) {
    const int L = max(0, a.seqlens[seq]);
    const int nblk = (L + kBlockN - 1) / kBlockN;
    const int blk1 = seq < end_seq ? nblk : end_blk;

    __syncthreads();
    for (int idx = tid; idx < kHT * MLA_HEAD_DIM; idx += kThreads) {
      int r = idx / MLA_HEAD_DIM, c = idx % MLA_HEAD_DIM;
      float v = 0.f;
      if (head0 + r < a.h)
        v = Elem<T>::to_f(q[seq * a.q_batch_stride + (int64_t)(head0 + r) * a.q_head_stride + c]);
      q_s[idx] = v;
    }

    float m = -INFINITY, l = 0.f;
    float acc[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] = 0.f;

    for (int blk = blk0; blk < blk1; ++blk) {
      const int tok0 = blk * kBlockN;
      const int nvalid = min(kBlockN, L - tok0);
      const int lblk = tok0 / a.page_size;
      int page = a.block_table[seq * a.bt_stride + lblk];
      if (page < 0 || page >= a.num_pages || lblk >= a.max_blocks) {
        report_error(a.err, MLA_ERR_DEVICE_BOUNDS, seq);
        page = 0;
      }
      const int row0 = tok0 % a.page_size;
      __syncthreads();
      // copy the valid rows (32-bit words; padded rows keep 4-byte alignment)
      for (int idx = tid; idx < nvalid * (MLA_HEAD_DIM / 2); idx += kThreads) {
        int r = idx / (MLA_HEAD_DIM / 2), w = idx % (MLA_HEAD_DIM / 2);
        const uint32_t *src = reinterpret_cast<const uint32_t *>(
            kv + (int64_t)page * a.kv_page_stride + (int64_t)(row0 + r) * a.kv_row_stride);
        reinterpret_cast<uint32_t *>(kv_s + r * kRow)[w] = src[w];
      }
      __syncthreads();

      // scores for tokens g, g+16, g+32, g+48 (base-2 units)
      float s[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int t = g + 16 * j;
        float dot = 0.f;
        if (t < nvalid) {
          const float *qr = q_s + hh * MLA_HEAD_DIM;
          const uint16_t *kr = kv_s + t * kRow;
          for (int c = 0; c < MLA_HEAD_DIM; ++c) dot = fmaf(qr[c], Elem<T>::bits_to_f(kr[c]), dot);
          s[j] = dot * a.scale_log2;
        } else {
          s[j] = -INFINITY;  // masked: token at or beyond cache_seqlens
        }
      }
      float mb = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      const float m_new = fmaxf(m, mb);
      // guard: an all -inf row keeps a finite reference (never NaN)
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = fast_exp2(m - m_use);
      float ps = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // the row sum takes the fp32 weight; the value product takes it rounded
        // to the input dtype (the split kernel's reduce_sum over acc_s precedes
        // its cast to acc_s_cast)
        const float p = fast_exp2(s[j] - m_use);
        p_s[hh * kBlockN + g + 16 * j] = round_to<T>(p);
        ps += p;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l = l * alpha + ps;
      m = m_new;
      __syncthreads();

      // O = O * alpha + P V over the valid tokens; this thread owns columns
      // d = 2g + 32k + {0, 1}, k = 0..15
#pragma unroll
      for (int k = 0; k < 32; ++k) acc[k] *= alpha;
      for (int t = 0; t < nvalid; ++t) {
        const float p = p_s[hh * kBlockN + t];
        const uint32_t *vr = reinterpret_cast<const uint32_t *>(kv_s + t * kRow);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          uint32_t w = vr[g + 16 * k];
          acc[2 * k] = fmaf(p, Elem<T>::bits_to_f((uint16_t)(w & 0xffffu)), acc[2 * k]);
          acc[2 * k + 1] = fmaf(p, Elem<T>::bits_to_f((uint16_t)(w >> 16)), acc[2 * k + 1]);
        }
      }
    }

    // epilogue
    const int nsplit = a.num_splits[seq + 1] - a.num_splits[seq];
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    const float lse2 = l > 0.f ? m + fast_log2(l) : -INFINITY;  // base-2 units
    if (head_ok) {
      if (nsplit == 1) {
        T *o = reinterpret_cast<T *>(a.out) + seq * a.o_batch_stride + (int64_t)head * a.o_head_stride;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          o[2 * g + 32 * k] = Elem<T>::from_f(acc[2 * k] * inv_l);
          o[2 * g + 32 * k + 1] = Elem<T>::from_f(acc[2 * k + 1] * inv_l);
        }
        if (g == 0) a.lse[seq * a.lse_stride + head] = lse2 * kLn2;
      } else {
        float *o = a.oaccum + ((int64_t)split * a.h + head) * MLA_HEAD_DIM_V;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          o[2 * g + 32 * k] = acc[2 * k] * inv_l;
          o[2 * g + 32 * k + 1] = acc[2 * k + 1] * inv_l;
        }
        if (g == 0) a.lseaccum[(int64_t)split * a.h + head] = lse2;
      }
    }
    ++split;
    ++seq;
    blk0 = 0;
  }
}

}  // namespace

cudaError_t launch_split_simt(const FwdArgs &a, cudaStream_t s) {
  const size_t smem = sizeof(float) * (kHT * MLA_HEAD_DIM + kHT * kBlockN) +
                      sizeof(uint16_t) * kBlockN * kRow;
  dim3 grid(a.num_parts, (a.h + kHT - 1) / kHT);
  cudaError_t e;
  if (a.dtype == MLA_DTYPE_BF16) {
    e = cudaFuncSetAttribute(split_simt_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    split_simt_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(split_simt_kernel<__half>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    split_simt_kernel<__half><<<grid, kThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace mla

