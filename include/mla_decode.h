/*
 * mla_decode.h — C ABI of the GB300 (sm_103a) MLA decode library.
 *
 * DeepSeek Multi-Head Latent Attention, decode phase: one query token per
 * sequence, h query heads sharing ONE latent KV head.  Query and key rows are
 * 576 wide (512 latent + 64 RoPE); the value is the first 512 columns of the
 * same cached row.  The cache is paged: 64-token-aligned pages addressed
 * through a per-sequence block table.
 *
 * Sources (cited by page title and section):
 *   [TL] "用 TileLang 编写高性能 DeepSeek MLA 内核：从 FlashAttention 到 FlashMLA
 *        级性能的完整实战指南" (lmnt.cn/news/253096)
 *   [FM] "DeepSeek开源周第一天：FlashMLA 深度分析" (pxiaoer.blog)
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates no device memory and keeps no state between calls (apart from
 *     a per-device error word and cached device properties).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; no entry point synchronises
 *     except mla_get_device_error.
 *   - Strides are in ELEMENTS.  Element types: q / kv_cache / out (and q_pe /
 *     k_pe) are fp16 or bf16 (the same for all), or q / kv_cache are e4m3 and
 *     out is bf16 (MLA_DTYPE_E4M3, below); lse, the workspace are fp32; tables
 *     int32.
 *   - Argument errors are detected on the host, before any launch, and return
 *     a negative mla_status without touching the GPU.  Launch failures return
 *     MLA_ERR_CUDA.  Faults the kernels detect while running (a block-table
 *     entry outside the cache, a wait that ran out) are recorded in the
 *     device error word and read back with mla_get_device_error.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_ABI_VERSION 5

/* Shape contract [TL §先看核心难点]: 576 = 512 latent + 64 RoPE; v = 512. */
#define MLA_HEAD_DIM 576
#define MLA_HEAD_DIM_V 512
/* KV tokens per scheduling block (pages must be a multiple of it). */
#define MLA_BLOCK_N 64
/* Integers per part in tile_scheduler_metadata. */
#define MLA_META_STRIDE 8
/* Fixed per-sequence cost, in 64-token blocks, on the scheduler's cost axis. */
#define MLA_SCHED_FIXED_COST 5
/* Cost of one segment (a part's share of one sequence), in 64-token blocks, by
 * which the scheduler chooses how many parts to use. */
#define MLA_SCHED_SEGMENT_COST 16
/* Cost, in 64-token blocks, that the scheduler adds to a part count whose
 * partition splits some sequence: the combine pass that such a schedule needs. */
#define MLA_SCHED_SPLIT_COST 10
/* Largest num_sm the scheduler accepts. */
#define MLA_MAX_NUM_SM 2046

typedef enum {
  MLA_OK = 0,
  MLA_ERR_NULL = -1,            /* a required pointer is NULL */
  MLA_ERR_SHAPE = -2,           /* unsupported or inconsistent dimension */
  MLA_ERR_DTYPE = -3,           /* dtype is not fp16 / bf16 / e4m3, or e4m3 with
                                   separate q_pe / k_pe or a non-finite scale */
  MLA_ERR_ALIGN = -4,           /* pointer or stride violates 16-byte alignment */
  MLA_ERR_PAGE = -5,            /* page_block_size not a positive multiple of 64 */
  MLA_ERR_WORKSPACE = -6,       /* workspace missing or too small */
  MLA_ERR_CUDA = -7,            /* a CUDA runtime call or launch failed */
  MLA_ERR_DEVICE_TIMEOUT = -8,  /* (device word) a bounded wait gave up */
  MLA_ERR_DEVICE_BOUNDS = -9,   /* (device word) block table / length out of range */
  MLA_ERR_ARCH = -10            /* the current device is not sm_103 */
} mla_status;

/*
 * MLA_DTYPE_E4M3: an FP8 KV cache [TL §变体内核 names an FP8-cache variant of
 * the decode kernel and fixes no format; this is the library's reading].  q and
 * kv_cache hold OCP e4m3 bytes (1 sign, 4 exponent bits with bias 7, 3 fraction
 * bits, no infinities, S.1111.111 is NaN), each tensor with one fp32
 * dequantisation scale: the decode runs on q_scale * q and kv_scale * kv, i.e.
 * x_t = softmax_scale * q_scale * kv_scale * (q . kv[t]) and
 * out = kv_scale * sum_t softmax_t(x) * kv[t][0:512].  out is bf16.  The
 * softmax weights are rounded to e4m3 before the value product (they are at most
 * 256 there, so none saturates); O is divided by the sum of the rounded weights.
 * Only the fused layout: q_pe and k_pe must be NULL.  Strides count bytes.
 */
enum { MLA_DTYPE_FP16 = 0, MLA_DTYPE_BF16 = 1, MLA_DTYPE_E4M3 = 2 };

/*
 * Detail code of MLA_ERR_DEVICE_TIMEOUT: the split kernel's wait that gave up
 * (every wait is bounded at 1 s).  The score CTA of a 2-CTA cluster streams K and
 * computes the scores and the softmax; the value CTA streams V and accumulates O.
 */
typedef enum {
  MLA_WAIT_K_EMPTY = 1,      /* score: K producer waits for a free ring slot */
  MLA_WAIT_Q_FREE = 2,       /* score: the previous segment's MMAs are done with Q */
  MLA_WAIT_S_FREE = 3,       /* score: the softmax has read an S page buffer */
  MLA_WAIT_K_FULL = 4,       /* score: MMA warp waits for K (or Q) data */
  MLA_WAIT_S_FULL = 5,       /* score: softmax waits for S */
  MLA_WAIT_STAGE_FREE = 6,   /* score: a P staging tile has left for the value CTA */
  MLA_WAIT_HDR_FREE = 7,     /* score: the value CTA has read a rescale header */
  MLA_WAIT_SLOT_FREE = 8,    /* score: a P slot of the value CTA is free */
  MLA_WAIT_V_EMPTY = 9,      /* value: V producer waits for a free ring slot */
  MLA_WAIT_O_FREE = 10,      /* value: the epilogue has read O */
  MLA_WAIT_O_READY = 11,     /* value: O has been rescaled */
  MLA_WAIT_P_FULL = 12,      /* value: a P tile has arrived */
  MLA_WAIT_V_FULL = 13,      /* value: V data has arrived */
  MLA_WAIT_HDR_FULL = 14,    /* value: a rescale header has arrived */
  MLA_WAIT_O_DONE = 15,      /* value: the P.V MMAs of a superblock are done */
  MLA_WAIT_STAGE_READY = 16, /* score: copier waits for staged P tiles */
  MLA_WAIT_GRID = 17         /* any CTA: the grid-wide barrier before the fused combine */
} mla_wait_site;

/*
 * Arguments of one decode call.  Follows the field set of FlashMLA's
 * Flash_fwd_mla_params [FM §内存访问优化], including seqlen_q and is_causal;
 * with one KV head, ngroups (query heads per KV head) is h and h_h_k_ratio
 * is h, so neither is a separate field.
 *
 * Several query tokens per sequence (seqlen_q = s > 1, e.g. speculative or
 * multi-token decoding): the s * h query rows of a sequence are folded into
 * one run of rows, token-major (row r = qi * h + head), and all read the same
 * cache.  q's rows are then addressed as q + i*q_batch_stride + r*q_head_stride
 * (a [b][s][h][576] tensor whose token stride is h * q_head_stride), out's the
 * same way with o_head_stride, and lse is [b][s * h].  The cache already holds
 * the s new tokens: query token qi stands at position L_i - s + qi, and with
 * is_causal it sees the cached tokens t < L_i - (s - 1 - qi) (a row that sees
 * none gives out = 0, lse = -inf); without it every row sees all L_i tokens.
 * Pass h_rows = s * h wherever an entry point below asks for h
 * (mla_metadata_shape, mla_get_metadata, mla_workspace_size).
 *
 * Tensors (device, caller-owned):
 *   q            [b][s][h][576]        strides q_batch_stride, q_head_stride
 *                                      (token stride h * q_head_stride);
 *                                      the 576 columns contiguous.
 *   kv_cache     [num_pages][page_block_size][1][576]
 *                                      strides kv_page_stride, kv_row_stride;
 *                                      columns contiguous.  Token t of sequence
 *                                      i is row t % page_block_size of page
 *                                      block_table[i][t / page_block_size]
 *                                      [TL §变体内核].
 *   q_pe, k_pe   optional split layout [TL §Split Kernel: Q / Q_pe and
 *                KV / K_pe are separate tensors, and the score is
 *                Q.KV^T + Q_pe.K_pe^T].  When q_pe is non-NULL, q holds only
 *                the 512 latent columns ([b][s][h][512], same strides) and
 *                q_pe [b][s][h][64] the RoPE columns (strides
 *                q_pe_batch_stride, q_pe_head_stride).  When k_pe is
 *                non-NULL, kv_cache rows hold only the 512 latent columns
 *                (which are also the value) and k_pe
 *                [num_pages][page_block_size][1][64] the RoPE columns (strides
 *                k_pe_page_stride, k_pe_row_stride; same pages, same block
 *                table).  Either may be given without the other; NULL means
 *                the RoPE columns are columns 512..575 of q / kv_cache, and
 *                the four stride fields of a NULL pointer are ignored.
 *   block_table  int32 [b][max_blocks_per_seq], row stride
 *                block_table_batch_stride.  Only the first
 *                ceil(L_i / page_block_size) entries of row i are read; each
 *                must lie in [0, num_pages).
 *   cache_seqlens int32 [b], 0 <= L_i <= max_blocks_per_seq*page_block_size.
 *   out          [b][s][h][512]        strides o_batch_stride, o_head_stride
 *                                      (token stride h * o_head_stride).
 *   lse          fp32 [b][s * h]       stride lse_batch_stride (rows
 *                contiguous); natural-log log-sum-exp of the scaled scores,
 *                -inf for a row that sees no token (whose out row is zeros).
 *   tile_scheduler_metadata, num_splits: as written by mla_get_metadata for
 *                the same cache_seqlens, b, s * h and num_sm.
 *   workspace    at least mla_workspace_size(b, s * h, num_sm_parts) bytes,
 *                16-byte aligned; holds per-split partial outputs and their
 *                LSEs (the layout is the library's own).
 *
 * Result: out[i][qi][j][:] = sum_t softmax_t(x) * kv[t][0:512] with
 * x_t = softmax_scale * q[i][qi][j][:] . kv[t][:] over the tokens t that query
 * token qi sees (all t < L_i, or t < L_i - (s - 1 - qi) with is_causal), computed with
 * exp2-based online softmax, split-KV partials and a combine pass
 * [TL §Split Kernel, §Combine Kernel].  Accumulation is fp32; the softmax
 * weights are rounded to the input dtype before the value product (for e4m3,
 * see MLA_DTYPE_E4M3 for the scales).
 */
typedef struct mla_fwd_params {
  int32_t b;              /* sequences (>= 1) */
  int32_t seqlen_q;       /* query tokens per sequence, s >= 1 */
  int32_t h;              /* query heads per token; s * h <= 1024 */
  int32_t h_k;            /* KV heads: must be 1 */
  int32_t d;              /* must be MLA_HEAD_DIM */
  int32_t d_v;            /* must be MLA_HEAD_DIM_V */
  int32_t dtype;          /* MLA_DTYPE_FP16, MLA_DTYPE_BF16 or MLA_DTYPE_E4M3 */
  float softmax_scale;    /* multiplies q.k before the softmax */

  const void *q;
  int64_t q_batch_stride, q_head_stride;

  const void *kv_cache;
  int64_t kv_page_stride, kv_row_stride;
  int32_t num_pages;
  int32_t page_block_size;

  const int32_t *block_table;
  int64_t block_table_batch_stride;
  int32_t max_blocks_per_seq;

  const int32_t *cache_seqlens;

  void *out;
  int64_t o_batch_stride, o_head_stride;
  float *lse;
  int64_t lse_batch_stride;

  const int32_t *tile_scheduler_metadata;
  const int32_t *num_splits;
  int32_t num_sm_parts;

  void *workspace;
  size_t workspace_bytes;

  /* split layout (see above); NULL = RoPE columns inside q / kv_cache */
  const void *q_pe;
  int64_t q_pe_batch_stride, q_pe_head_stride;
  const void *k_pe;
  int64_t k_pe_page_stride, k_pe_row_stride;

  /* seqlen_q > 1 only: nonzero = causal mask among the query tokens (above) */
  int32_t is_causal;

  /* MLA_DTYPE_E4M3 only (ignored otherwise): dequantisation scales of q and
   * kv_cache, finite and > 0 */
  float q_scale;
  float kv_scale;

  /* Nonzero: the split kernel combines the sequences it split itself [TL
   * §变体内核, the persistent variant, which synchronises its split and combine
   * phases grid-wide]: once every CTA of its grid has finished its parts and
   * passed a grid-wide barrier, all of them run the combine, and no combine
   * kernel is launched.  Zero: the combine kernel runs after the split kernel.
   * Same results, bit for bit.  The barrier's two counters live in the
   * workspace (mla_workspace_size) and need no initial value: each call tags
   * them with its own number, and the last CTA to leave the barrier resets
   * them for a replay of the same call (a captured CUDA graph).  After a call
   * that reported MLA_ERR_DEVICE_TIMEOUT, re-capture such a graph.  The barrier
   * needs the whole grid resident at once: num_sm_parts * ceil(seqlen_q * h /
   * 128) must not exceed half of mla_device_num_sm (the co-resident clusters),
   * which metadata shaped for at most that num_sm satisfies; otherwise the call
   * returns MLA_ERR_SHAPE before launching anything.  With other kernels on the
   * device the barrier waits until the grid's last CTA has started. */
  int32_t fused_combine;
} mla_fwd_params;

/* ABI version (MLA_ABI_VERSION) and sizeof(mla_fwd_params), for bindings. */
int mla_abi_version(void);
size_t mla_fwd_params_size(void);

/* Static string for an mla_status value (never NULL). */
const char *mla_status_string(int status);

/*
 * How many SMs the split kernel can occupy at once on `device`: twice the
 * number of co-resident 2-CTA clusters of its launch configuration.  Pass it
 * as num_sm below.  Returns MLA_ERR_CUDA / MLA_ERR_ARCH on failure.
 */
int mla_device_num_sm(int device, int *num_sm);

/*
 * Scheduler shape for b sequences and h query rows per sequence (heads, or
 * seqlen_q * heads) on num_sm SMs (host only, no
 * GPU needed): *num_sm_parts = max(1, (num_sm / 2) / ceil(h / 128)) parts (one
 * 2-CTA cluster per part and 128-head tile), *meta_stride = MLA_META_STRIDE.
 */
int mla_metadata_shape(int b, int h, int num_sm, int *num_sm_parts, int *meta_stride);

/*
 * Tile-scheduler metadata [FM §内存访问优化: tile_scheduler_metadata_ptr,
 * num_sm_parts, num_splits_ptr; TL §6. Split-KV: per-sequence split sizing
 * from cache_seqlens].  One small device kernel, no host synchronisation.
 *   cache_seqlens           device int32 [b]
 *   tile_scheduler_metadata device int32 [num_sm_parts][MLA_META_STRIDE]:
 *       {begin_seq, begin_blk, end_seq, end_blk, first_split, 0, 0, 0}; part k
 *       covers the 64-token blocks from (begin_seq, begin_blk) up to, not
 *       including, (end_seq, end_blk) in (sequence, block) order.
 *   num_splits              device int32 [b + 1]: prefix sums; sequence i owns
 *       split slots num_splits[i] .. num_splits[i+1]-1 of the workspace.
 * Partition: sequences are laid end to end on a cost axis, each costing
 * MLA_SCHED_FIXED_COST + ceil(L_i/64) blocks; with P parts, part k starts at
 * cost position floor(k*TOTAL/P).  P is chosen from ceil(num_sm_parts / 2) to
 * num_sm_parts: part k of P costs MLA_SCHED_SEGMENT_COST per segment it holds
 * (a sequence it touches) plus one per block; P scores its most expensive part,
 * plus MLA_SCHED_SPLIT_COST when some cut falls inside a sequence (the schedule
 * then splits that sequence), and the lowest score is used (the larger P on a
 * tie).  Parts P..num_sm_parts-1 are
 * empty: {b, 0, b, 0, num_splits[b], 0, 0, 0}.  Deterministic; the decode
 * result does not depend on it beyond rounding.  num_sm <= MLA_MAX_NUM_SM.
 */
int mla_get_metadata(const int32_t *cache_seqlens, int b, int h, int num_sm,
                     int32_t *tile_scheduler_metadata, int32_t *num_splits,
                     void *stream);

/* Workspace bytes for mla_decode_fwd: fp32 partial outputs and LSEs for up to
 * b + num_sm_parts splits of h query rows (heads, or seqlen_q * heads), then
 * 256 bytes for the fused combine's grid barrier. */
int mla_workspace_size(int b, int h, int num_sm_parts, size_t *bytes);

/*
 * Paged split-KV MLA decode [TL §Split Kernel, §Combine Kernel, §变体内核;
 * FM §内存访问优化, §Softmax 计算优化].  Enqueues the split kernel (a
 * persistent grid of 2-CTA clusters walking the metadata) and, unless
 * params->fused_combine is set, the combine kernel on `stream`.  Alignment: q, kv_cache, out, workspace (and q_pe,
 * k_pe when given) 16-byte aligned; all their strides multiples of 16 bytes
 * (8 elements; 16 for e4m3 q / kv_cache).  Row strides must cover the row: kv_row_stride >= 576 (>= 512
 * with k_pe), k_pe_row_stride >= 64, each page stride >= page_block_size
 * times its row stride.
 */
int mla_decode_fwd(const mla_fwd_params *params, void *stream);

/*
 * mla_decode_fwd plus a measurement hook: records the caller-owned CUDA events
 * `split_begin` and `split_end` (cudaEvent_t as void*, either may be NULL) on
 * `stream` immediately before and after the split kernel, so that its device
 * time can be read with cudaEventElapsedTime.  Same results and errors as
 * mla_decode_fwd.
 */
int mla_decode_fwd_timed(const mla_fwd_params *params, void *stream, void *split_begin,
                         void *split_end);

/*
 * Size of the library's built-in per-device scratch used by
 * mla_decode_fwd_static: 64 MiB, enough for b + num_sm_parts <= 255 at 128 query
 * rows (b = 128 with 76 parts needs 53.6 MB) and <= 127 at 256 rows (two query
 * tokens of 128 heads); see mla_workspace_size.
 */
#define MLA_STATIC_WORKSPACE_BYTES (64u << 20)

/*
 * mla_decode_fwd with no caller workspace and no allocation of any kind.  The
 * source pages have no counterpart: their decode always receives a workspace
 * tensor from the caller.  This entry is for callers that cannot allocate
 * device memory on the decode path: plain C hosts with no device allocator of
 * their own, and runtimes that reserve all device memory up front, for whom a
 * cudaMalloc/cudaFree per step (each of which synchronises the device) would
 * stall the stream.
 *
 * The split kernel's partial outputs and log-sum-exps go to a fixed array of
 * MLA_STATIC_WORKSPACE_BYTES inside the library, one per device, held from
 * the library's first use on that device until the process exits.
 * params->workspace and params->workspace_bytes are ignored; every other field
 * means what it means for mla_decode_fwd, and so do the results and errors.
 * If mla_workspace_size(b, h, num_sm_parts) exceeds
 * MLA_STATIC_WORKSPACE_BYTES, the call returns MLA_ERR_WORKSPACE before
 * touching the device (MLA_ERR_SHAPE if b, h or num_sm_parts is out of range).
 *
 * The first call on a device, made with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and caches it; make that first
 * call before any stream capture.  The cached address (like the device error
 * word's) belongs to that device's primary context: after cudaDeviceReset on
 * the device it is stale, and the library must not be called on that device
 * again in the same process.  Nothing in the array has to start at zero:
 * every partial the combine kernel reads was written by the split kernel
 * earlier in the same call, so what an earlier call left there is never read.
 * All calls on a device share the one array, so calls that overlap on the GPU
 * (on different streams, or unordered calls from several host threads) race
 * on it and give wrong results: order them on one stream or with events.
 */
int mla_decode_fwd_static(const mla_fwd_params *params, void *stream);

/*
 * Test hook for the device-side failure path; not for production use.  The
 * source pages have no counterpart.  Validates `params` exactly as
 * mla_decode_fwd does, then launches only the split kernel with its load warps
 * switched off: no TMA load and no copy between the two CTAs of a cluster is
 * issued, so nothing is in flight, and the score CTA's MMA warp gives up its
 * first wait for K data after about 1 ms (instead of 1 s).  The kernel records
 * MLA_ERR_DEVICE_TIMEOUT with detail MLA_WAIT_K_FULL, every role of every
 * cluster unwinds, and the kernel exits normally; read the error with
 * mla_get_device_error.  out, lse and the workspace are left unspecified, and
 * the context stays usable: the next call computes normally.
 */
int mla_test_forced_timeout(const mla_fwd_params *params, void *stream);

/*
 * Synchronises `stream`, then returns (and clears) the device error word of
 * the current device: MLA_OK, MLA_ERR_DEVICE_BOUNDS or MLA_ERR_DEVICE_TIMEOUT.
 * If `detail` is non-NULL it receives a kernel-specific code (which wait, or
 * the offending sequence index).
 */
int mla_get_device_error(void *stream, int *detail);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
