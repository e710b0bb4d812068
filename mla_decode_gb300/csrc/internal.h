// Internal declarations shared by the library's translation units (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla_decode.h"

namespace mla {

// Everything a split / combine kernel needs, resolved and validated on the host.
struct FwdArgs {
  int b, h, dtype;   // h: query rows per sequence (seqlen_q * heads, token-major)
  int q_len;         // query tokens per sequence
  int heads;         // query heads per token (rows q_len * heads)
  int causal;        // token qi sees the cached tokens t < L - (q_len - 1 - qi)
  float scale_log2;  // softmax_scale * log2(e) (times q_scale * kv_scale for e4m3):
                     // scores are kept in base-2 units
  float o_scale;     // multiplies the normalised output: kv_scale for e4m3, else 1
  const void *q;
  int64_t q_batch_stride, q_head_stride;
  const void *kv;
  int64_t kv_page_stride, kv_row_stride;
  // RoPE columns: separate tensors, or columns 512..575 of q / kv (resolved on
  // the host, so the kernels see one layout)
  const void *q_pe;
  int64_t q_pe_batch_stride, q_pe_head_stride;
  const void *k_pe;
  int64_t k_pe_page_stride, k_pe_row_stride;
  int k_fused;       // the RoPE columns are columns 512..575 of each kv_cache row
  int num_pages, page_size;
  const int32_t *block_table;
  int64_t bt_stride;
  int max_blocks;
  const int32_t *seqlens;
  void *out;
  int64_t o_batch_stride, o_head_stride;
  float *lse;
  int64_t lse_stride;
  const int32_t *meta;
  const int32_t *num_splits;
  int num_parts;
  float *oaccum;    // [max_splits][128 column chunks][h][4] (rows interleaved per chunk)
  float *lseaccum;  // [max_splits][h], base-2 units
  int max_splits;
  int *err;         // device error word (two ints: code, detail)
  int forced_timeout;  // test hook: load warps idle, the K wait gives up after 1 ms
  int fused_combine;   // the split kernel combines split sequences after a grid barrier
  uint32_t token;      // this call's tag for the barrier counters (never 0)
  unsigned long long *grid_bar;  // workspace: {arrivals, departures}, tag in the high half
};

int max_splits_for(int b, int num_parts);
size_t workspace_bytes_for(int b, int h, int num_parts);

// device error word of the current device
int *device_error_word();

cudaError_t launch_metadata(const int32_t *seqlens, int b, int parts, int fixed, int seg_cost,
                            int32_t *meta, int32_t *num_splits, cudaStream_t s);
cudaError_t launch_split_tc(const FwdArgs &a, cudaStream_t s);
cudaError_t split_tc_num_sm(int device, int *num_sm);
cudaError_t launch_combine(const FwdArgs &a, cudaStream_t s);

}  // namespace mla
