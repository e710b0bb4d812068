// C ABI of the MLA decode library: argument validation, workspace layout,
// scheduler shape and the launch sequence (metadata -> split -> combine).
#include <cuda_runtime.h>
#include <math.h>
#include <atomic>
#include <mutex>
#include <stdint.h>

#include "internal.h"

namespace mla {

// Device error word: {code, detail}.  One instance per device context.
__device__ int g_error_word[2];

// Scratch for mla_decode_fwd_static: oaccum and lseaccum of one call.  One
// instance per device context; never cleared (nothing in it is read before the
// same call writes it).  Host code must not pass this name to a kernel: it
// stands for the array only on the device; static_workspace() gives the
// device address.
static __device__ __align__(256) unsigned char g_static_workspace[MLA_STATIC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_err_ptr[kMaxDevices] = {nullptr};
int g_num_sm[kMaxDevices] = {0};
void *g_static_ws_ptr[kMaxDevices] = {nullptr};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int head_tiles(int h) { return (h + 127) / 128; }
}  // namespace

int *device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int *>(p);
  }
  return g_err_ptr[dev];
}

// Device address of g_static_workspace on the current device, looked up once.
void *static_workspace() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_static_ws_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess) return nullptr;
    g_static_ws_ptr[dev] = p;
  }
  return g_static_ws_ptr[dev];
}

int max_splits_for(int b, int num_parts) { return b + num_parts; }

// [oaccum][lseaccum, padded to 256 B][grid barrier: 256 B]
size_t workspace_bytes_for(int b, int h, int num_parts) {
  size_t splits = (size_t)max_splits_for(b, num_parts);
  size_t o = splits * (size_t)h * MLA_HEAD_DIM_V * sizeof(float);
  size_t l = splits * (size_t)h * sizeof(float);
  return o + ((l + 255) & ~(size_t)255) + 256;
}

// A tag per call for the fused combine's barrier counters, never 0.
static uint32_t next_token() {
  static std::atomic<uint32_t> counter{0};
  uint32_t t;
  do {
    t = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  } while (t == 0);
  return t;
}

}  // namespace mla

using namespace mla;

extern "C" {

int mla_abi_version(void) { return MLA_ABI_VERSION; }

size_t mla_fwd_params_size(void) { return sizeof(mla_fwd_params); }

const char *mla_status_string(int s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_NULL: return "a required pointer is NULL";
    case MLA_ERR_SHAPE: return "unsupported or inconsistent shape";
    case MLA_ERR_DTYPE:
      return "dtype must be fp16, bf16 or e4m3 (e4m3: fused layout, finite positive scales)";
    case MLA_ERR_ALIGN: return "pointer or stride is not 16-byte aligned";
    case MLA_ERR_PAGE: return "page_block_size must be a positive multiple of 64";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_CUDA: return "CUDA runtime error";
    case MLA_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    case MLA_ERR_DEVICE_BOUNDS: return "block table entry or sequence length out of range";
    case MLA_ERR_ARCH: return "device is not sm_103 (GB300)";
    default: return "unknown status";
  }
}

int mla_device_num_sm(int device, int *num_sm) {
  if (!num_sm) return MLA_ERR_NULL;
  if (device < 0 || device >= kMaxDevices) return MLA_ERR_SHAPE;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_num_sm[device] > 0) {
      *num_sm = g_num_sm[device];
      return MLA_OK;
    }
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MLA_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return MLA_ERR_ARCH;
  int n = 0;
  if (split_tc_num_sm(device, &n) != cudaSuccess || n < 2) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  g_num_sm[device] = n;
  *num_sm = n;
  return MLA_OK;
}

int mla_metadata_shape(int b, int h, int num_sm, int *num_sm_parts, int *meta_stride) {
  if (!num_sm_parts || !meta_stride) return MLA_ERR_NULL;
  if (b < 1 || h < 1 || h > 1024 || num_sm < 1 || num_sm > MLA_MAX_NUM_SM) return MLA_ERR_SHAPE;
  int parts = (num_sm / 2) / head_tiles(h);
  *num_sm_parts = parts < 1 ? 1 : parts;
  *meta_stride = MLA_META_STRIDE;
  return MLA_OK;
}

int mla_get_metadata(const int32_t *cache_seqlens, int b, int h, int num_sm,
                     int32_t *tile_scheduler_metadata, int32_t *num_splits, void *stream) {
  if (!cache_seqlens || !tile_scheduler_metadata || !num_splits) return MLA_ERR_NULL;
  int parts = 0, stride = 0;
  int rc = mla_metadata_shape(b, h, num_sm, &parts, &stride);
  if (rc != MLA_OK) return rc;
  cudaError_t e = launch_metadata(cache_seqlens, b, parts, MLA_SCHED_FIXED_COST,
                                  MLA_SCHED_SEGMENT_COST, tile_scheduler_metadata, num_splits,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_workspace_size(int b, int h, int num_sm_parts, size_t *bytes) {
  if (!bytes) return MLA_ERR_NULL;
  if (b < 1 || h < 1 || h > 1024 || num_sm_parts < 1) return MLA_ERR_SHAPE;
  *bytes = workspace_bytes_for(b, h, num_sm_parts);
  return MLA_OK;
}

int mla_decode_fwd(const mla_fwd_params *p, void *stream) {
  return mla_decode_fwd_timed(p, stream, nullptr, nullptr);
}

int mla_decode_fwd_static(const mla_fwd_params *p, void *stream) {
  if (!p) return MLA_ERR_NULL;
  if (p->b < 1 || p->h < 1 || p->h > 1024 || p->seqlen_q < 1 || p->seqlen_q > 1024 ||
      p->seqlen_q * p->h > 1024 || p->num_sm_parts < 1)
    return MLA_ERR_SHAPE;
  if (workspace_bytes_for(p->b, p->seqlen_q * p->h, p->num_sm_parts) >
      (size_t)MLA_STATIC_WORKSPACE_BYTES)
    return MLA_ERR_WORKSPACE;
  void *ws = static_workspace();
  if (!ws) return MLA_ERR_CUDA;
  mla_fwd_params with_ws = *p;
  with_ws.workspace = ws;
  with_ws.workspace_bytes = MLA_STATIC_WORKSPACE_BYTES;
  return mla_decode_fwd(&with_ws, stream);
}

}  // extern "C"

namespace {

// Validates *p on the host and resolves it into the kernels' arguments.
int resolve_args(const mla_fwd_params *p, FwdArgs &a) {
  if (!p) return MLA_ERR_NULL;
  if (!p->q || !p->kv_cache || !p->block_table || !p->cache_seqlens || !p->out || !p->lse ||
      !p->tile_scheduler_metadata || !p->num_splits || !p->workspace)
    return MLA_ERR_NULL;
  if (p->b < 1 || p->seqlen_q < 1 || p->seqlen_q > 1024 || p->h < 1 || p->h > 1024 ||
      p->h_k != 1 || p->d != MLA_HEAD_DIM || p->d_v != MLA_HEAD_DIM_V)
    return MLA_ERR_SHAPE;
  const int rows = p->seqlen_q * p->h;  // query rows per sequence, token-major
  if (rows > 1024) return MLA_ERR_SHAPE;
  if (p->dtype != MLA_DTYPE_FP16 && p->dtype != MLA_DTYPE_BF16 && p->dtype != MLA_DTYPE_E4M3)
    return MLA_ERR_DTYPE;
  const bool f8 = p->dtype == MLA_DTYPE_E4M3;
  const bool sep_q = p->q_pe != nullptr, sep_k = p->k_pe != nullptr;
  if (f8 && (sep_q || sep_k || !(isfinite(p->q_scale) && p->q_scale > 0.f) ||
             !(isfinite(p->kv_scale) && p->kv_scale > 0.f)))
    return MLA_ERR_DTYPE;
  if (p->page_block_size <= 0 || p->page_block_size % MLA_BLOCK_N != 0) return MLA_ERR_PAGE;
  const int kv_cols = sep_k ? MLA_HEAD_DIM_V : MLA_HEAD_DIM;
  if (p->num_pages < 1 || p->max_blocks_per_seq < 1 || p->num_sm_parts < 1 ||
      p->q_head_stride < 1 || p->q_batch_stride < 1 || p->kv_row_stride < kv_cols ||
      p->kv_page_stride < (int64_t)p->page_block_size * p->kv_row_stride ||
      p->o_head_stride < 1 || p->o_batch_stride < 1 || p->lse_batch_stride < rows ||
      p->block_table_batch_stride < p->max_blocks_per_seq || !isfinite(p->softmax_scale))
    return MLA_ERR_SHAPE;
  if (sep_q && (p->q_pe_head_stride < 1 || p->q_pe_batch_stride < 1)) return MLA_ERR_SHAPE;
  if (sep_k && (p->k_pe_row_stride < MLA_HEAD_DIM - MLA_HEAD_DIM_V ||
                p->k_pe_page_stride < (int64_t)p->page_block_size * p->k_pe_row_stride))
    return MLA_ERR_SHAPE;
  // TMA strides are multiples of 16 bytes: 8 16-bit elements, 16 e4m3 bytes
  const int64_t in16 = f8 ? 16 : 8;
  if (!aligned16(p->q) || !aligned16(p->kv_cache) || !aligned16(p->out) ||
      !aligned16(p->workspace) || (p->q_batch_stride % in16) || (p->q_head_stride % in16) ||
      (p->kv_page_stride % in16) || (p->kv_row_stride % in16) || (p->o_batch_stride % 8) ||
      (p->o_head_stride % 8))
    return MLA_ERR_ALIGN;
  if (sep_q && (!aligned16(p->q_pe) || (p->q_pe_batch_stride % 8) || (p->q_pe_head_stride % 8)))
    return MLA_ERR_ALIGN;
  if (sep_k && (!aligned16(p->k_pe) || (p->k_pe_page_stride % 8) || (p->k_pe_row_stride % 8)))
    return MLA_ERR_ALIGN;
  if (p->workspace_bytes < workspace_bytes_for(p->b, rows, p->num_sm_parts))
    return MLA_ERR_WORKSPACE;

  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;

  a.b = p->b;
  a.h = rows;
  a.q_len = p->seqlen_q;
  a.heads = p->h;
  a.causal = p->seqlen_q > 1 && p->is_causal != 0;
  a.dtype = p->dtype;
  a.scale_log2 = f8 ? (float)((double)p->softmax_scale * 1.4426950408889634 * p->q_scale * p->kv_scale)
                   : p->softmax_scale * 1.4426950408889634f;
  a.o_scale = f8 ? p->kv_scale : 1.f;
  a.q = p->q;
  a.q_batch_stride = p->q_batch_stride;
  a.q_head_stride = p->q_head_stride;
  a.kv = p->kv_cache;
  a.kv_page_stride = p->kv_page_stride;
  a.kv_row_stride = p->kv_row_stride;
  // fused layout: the RoPE columns are 512 elements into each row
  const int64_t rope_off = MLA_HEAD_DIM_V * (f8 ? 1 : 2);
  a.q_pe = sep_q ? p->q_pe : static_cast<const char *>(p->q) + rope_off;
  a.q_pe_batch_stride = sep_q ? p->q_pe_batch_stride : p->q_batch_stride;
  a.q_pe_head_stride = sep_q ? p->q_pe_head_stride : p->q_head_stride;
  a.k_pe = sep_k ? p->k_pe : static_cast<const char *>(p->kv_cache) + rope_off;
  a.k_pe_page_stride = sep_k ? p->k_pe_page_stride : p->kv_page_stride;
  a.k_pe_row_stride = sep_k ? p->k_pe_row_stride : p->kv_row_stride;
  a.k_fused = sep_k ? 0 : 1;
  a.num_pages = p->num_pages;
  a.page_size = p->page_block_size;
  a.block_table = p->block_table;
  a.bt_stride = p->block_table_batch_stride;
  a.max_blocks = p->max_blocks_per_seq;
  a.seqlens = p->cache_seqlens;
  a.out = p->out;
  a.o_batch_stride = p->o_batch_stride;
  a.o_head_stride = p->o_head_stride;
  a.lse = p->lse;
  a.lse_stride = p->lse_batch_stride;
  a.meta = p->tile_scheduler_metadata;
  a.num_splits = p->num_splits;
  a.num_parts = p->num_sm_parts;
  a.max_splits = max_splits_for(p->b, p->num_sm_parts);
  a.oaccum = static_cast<float *>(p->workspace);
  a.lseaccum = reinterpret_cast<float *>(static_cast<char *>(p->workspace) +
                                         (size_t)a.max_splits * rows * MLA_HEAD_DIM_V * sizeof(float));
  a.err = err;
  a.forced_timeout = 0;
  a.fused_combine = p->fused_combine != 0;
  if (a.fused_combine) {
    // the grid barrier waits for every CTA: the grid must fit on the device at once
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    const int r = mla_device_num_sm(dev, &n);
    if (r != MLA_OK) return r;
    if ((int64_t)p->num_sm_parts * head_tiles(rows) > n / 2) return MLA_ERR_SHAPE;
  }
  a.token = next_token();
  {
    const size_t o = (size_t)a.max_splits * rows * MLA_HEAD_DIM_V * sizeof(float);
    const size_t l = (size_t)a.max_splits * rows * sizeof(float);
    a.grid_bar = reinterpret_cast<unsigned long long *>(static_cast<char *>(p->workspace) + o +
                                                        ((l + 255) & ~(size_t)255));
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_decode_fwd_timed(const mla_fwd_params *p, void *stream, void *split_begin,
                         void *split_end) {
  FwdArgs a;
  const int rc = resolve_args(p, a);
  if (rc != MLA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (split_begin && cudaEventRecord(static_cast<cudaEvent_t>(split_begin), s) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (launch_split_tc(a, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (split_end && cudaEventRecord(static_cast<cudaEvent_t>(split_end), s) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (!a.fused_combine && launch_combine(a, s) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_test_forced_timeout(const mla_fwd_params *p, void *stream) {
  FwdArgs a;
  const int rc = resolve_args(p, a);
  if (rc != MLA_OK) return rc;
  a.forced_timeout = 1;
  return launch_split_tc(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MLA_OK
                                                                               : MLA_ERR_CUDA;
}

int mla_get_device_error(void *stream, int *detail) {
  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  int host[2] = {0, 0};
  if (cudaMemcpy(host, err, sizeof host, cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  if (host[0] != 0) {
    int zero[2] = {0, 0};
    if (cudaMemcpy(err, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return MLA_ERR_CUDA;
  }
  if (detail) *detail = host[1];
  return host[0];
}

}  // extern "C"
