// Split kernel for sm_103a: tcgen05 tensor cores, TMEM accumulators, TMA loads,
// a 2-CTA cluster per scheduler part.
//
// What it computes (per sequence segment and 128-head tile) is the TileLang
// guide's split kernel ("用 TileLang 编写高性能 DeepSeek MLA 内核…", sections
// 先看核心难点, Split Kernel, 变体内核 (paged), 6. Split-KV) with FlashMLA's
// softmax form ("DeepSeek开源周第一天：FlashMLA 深度分析", section Softmax 计算优化:
// exp2 with log2(e) folded into the scale, the -inf guard):
//   S = Q . K^T over the 576 columns, masked past cache_seqlens; online softmax
//   in base 2; P rounded to the input dtype; O += P . V with V the first 512
//   columns of the same cached rows; at the segment end O / l and the base-2 LSE.
//
// How it is laid out on the GPU (this library's design, not the pages'): the
// fp32 accumulator O[128 heads][512] fills an SM's whole tensor memory, so each
// part is served by a cluster of two CTAs with different roles:
//   * score CTA (cluster rank 0): Q columns 0..511 live in TMEM as the A operand
//     (packed 16-bit pairs), the RoPE columns 512..575 in shared memory.  For a
//     superblock of up to four 64-token pages it issues S = Q K^T as 36 MMAs of
//     M=128 x N=256 x K=16 into a TMEM accumulator, streaming K through a ring of
//     [256 tokens x 64 columns] TMA tiles.  Eight softmax warps read S, keep the
//     running max with a lazy rescale (the reference max only moves when a block
//     exceeds it by more than kTau in log2 units, which is exact in real
//     arithmetic), write P as 16-bit swizzled tiles and bulk-copy them, with the
//     per-head rescale factors, into the value CTA's shared memory.
//   * value CTA (rank 1): O lives in TMEM (two 256-column halves).  Its own TMA
//     stream brings each page's 512 value columns; per page and O half it issues
//     M=128 x N=256 x K=16 MMAs with P (shared memory, K-major) as A and V
//     (shared memory, N-major) as B.  Eight correction warps apply the rescale
//     factors to O when the score CTA moved its reference max, and run the
//     epilogue (O / l to out, or to the split workspace).
// Every wait is bounded; a wait that runs out records MLA_ERR_DEVICE_TIMEOUT
// with the wait site as detail, and the CTA unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kThreads = 352;            // 11 warps (see the role map in the kernel)
constexpr int kSB = 4;                   // pages (64 tokens each) per score superblock
constexpr int kNK = 4;                   // K tiles in flight (score CTA)
#ifndef MLA_NV
#define MLA_NV 5
#endif
constexpr int kNV = MLA_NV;              // V half-page tiles in flight (value CTA)
constexpr int kNPR = 3;                  // P tiles in the value CTA's ring
#ifndef MLA_TAU
#define MLA_TAU 0.0f
#endif
constexpr float kTau = MLA_TAU;          // lazy-rescale threshold, log2 units
constexpr int kChunk = 8192;             // [64 rows][128 B] swizzled TMA box
constexpr int kKSlot = kSB * kChunk;     // 64 columns of 256 tokens
constexpr int kVSlot = 4 * kChunk;       // 256 value columns of one page
constexpr int kPTile = 16384;            // [128 heads][64 tokens] 16-bit, swizzled
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct Header {  // score -> value CTA, one per superblock
  float alpha[128];
  float l[128];
  float m[128];
  uint32_t flags;  // bit 0: rescale O first; bit 1: last superblock of the segment
  uint32_t pad[3];
};
static_assert(sizeof(Header) % 16 == 0, "bulk copies move multiples of 16 bytes");

// shared-memory map (offsets from the 1024-aligned base)
constexpr int kOffQ8 = 0;                                   // score: Q columns 512..575
constexpr int kOffK = kOffQ8 + 16384;                       // score: K ring
constexpr int kOffPStage = kOffK + kNK * kKSlot;            // score: P staging tiles
constexpr int kOffHdrStage = kOffPStage + kSB * kPTile;     // score: 2 staging headers
constexpr int kOffRed = kOffHdrStage + 2 * (int)sizeof(Header);  // score: [2][2][128] floats
constexpr int kOffV = 0;                                    // value: V ring
constexpr int kOffPRing = kOffV + kNV * kVSlot;             // value: P tiles
constexpr int kOffHdr = kOffPRing + kNPR * kPTile;          // value: 2 headers
constexpr int kOffBars = (((kOffRed + 4 * 128 * 4) > (kOffHdr + 2 * (int)sizeof(Header))
                               ? (kOffRed + 4 * 128 * 4)
                               : (kOffHdr + 2 * (int)sizeof(Header))) + 127) & ~127;
static_assert(kOffHdr + 2 * (int)sizeof(Header) <= kOffBars, "value layout overlaps barriers");

struct Bars {
  uint64_t k_full[kNK], k_empty[kNK];  // score
  uint64_t s_full, s_free, q_ready;    // score
  uint64_t stage_ready;                // score: P tiles + header staged (softmax -> copier)
  uint64_t stage_free[kSB];            // score, arrived by the value CTA
  uint64_t slot_free[kNPR];            // score, value-CTA MMA commits (multicast)
  uint64_t hdr_free[2];                // score, arrived by the value CTA
  uint64_t v_full[kNV], v_empty[kNV];  // value
  uint64_t p_full[kNPR];               // value, bulk copies from the score CTA
  uint64_t hdr_full[2];                // value, bulk copies from the score CTA
  uint64_t o_ready[2], o_done[2], o_free;  // value
  uint32_t tmem_base;
  int abort;
};
constexpr int kSmemBytes = kOffBars + (int)sizeof(Bars) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// wait sites (reported as the error detail on a timeout)
enum : int {
  W_K_EMPTY = 1, W_Q_READY, W_S_FREE, W_K_FULL, W_S_FULL, W_STAGE_FREE, W_HDR_FREE, W_SLOT_FREE,
  W_V_EMPTY, W_O_FREE, W_O_READY, W_P_FULL, W_V_FULL, W_HDR_FULL, W_O_DONE, W_STAGE_READY
};

// Optional event trace of part 0 (build with -DMLA_TRACE=1): globaltimer stamps
// per (role, superblock, event), read back with mla_debug_trace().
#if MLA_TRACE
__device__ unsigned long long g_trace[2][256][16];
__device__ unsigned long long g_trace_k[2][256][16];  // per K chunk: [0..8] arrival, [9..] reuse
__device__ unsigned long long g_trace_v[256][16];     // value CTA per page p: p_full, v_full h0/h1, V issue
__device__ unsigned long long g_parts[1024][4];        // per part: start, score end, value end, segments
#define TRACE_V(part, sb, ev)                                                     \
  do {                                                                            \
    if ((part) == 0 && (sb) < 256) g_trace_v[(sb)][(ev)] = globaltimer_ns();      \
  } while (0)
#define TRACE_K(role, part, sb, ev)                                                   \
  do {                                                                                \
    if ((part) == 0 && (sb) < 256) g_trace_k[(role)][(sb)][(ev)] = globaltimer_ns(); \
  } while (0)
#define TRACE(role, part, sb, ev)                                             \
  do {                                                                        \
    if ((part) == 0 && (sb) < 256) g_trace[(role)][(sb)][(ev)] = globaltimer_ns(); \
  } while (0)
#else
#define TRACE(role, part, sb, ev) \
  do {                            \
  } while (0)
#define TRACE_K(role, part, sb, ev) \
  do {                              \
  } while (0)
#define TRACE_V(part, sb, ev) \
  do {                        \
  } while (0)
#endif

#ifndef MLA_LINE_PREFETCH_SB
#define MLA_LINE_PREFETCH_SB 0
#endif
// The value CTA's correction warps prefetch, line by line into L2, the cache rows
// of the superblock this many superblocks ahead of the one they are handling.
constexpr int kLinePrefetchSb = MLA_LINE_PREFETCH_SB;

struct Ctx {
  Bars *bars;
  int *err;
  __device__ bool aborted() const { return *reinterpret_cast<volatile int *>(&bars->abort) != 0; }
};

template <bool kCl>
__device__ __forceinline__ bool wait_bar(const Ctx &c, uint64_t *bar, uint32_t parity, int where) {
  const uint32_t addr = smem_u32(bar);
  if (kCl ? mbar_try_wait_cluster(addr, parity) : mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (kCl ? mbar_try_wait_cluster(addr, parity) : mbar_try_wait(addr, parity)) return true;
    if (*reinterpret_cast<volatile int *>(&c.bars->abort)) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      c.bars->abort = 1;
      const uint32_t peer = map_to_rank(smem_u32(&c.bars->abort), cluster_ctarank() ^ 1);
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer), "r"(1) : "memory");
      report_error(c.err, MLA_ERR_DEVICE_TIMEOUT, where);
      return false;
    }
  }
}

// One sequence's share of a part: blocks [lo, hi) of sequence `seq`.
struct Seg {
  int seq, lo, hi, split, L, nsplit;
};

struct SegWalk {
  int seq, blk, end_seq, end_blk, split;
  __device__ SegWalk(const FwdArgs &a, int part) {
    const int32_t *row = a.meta + (int64_t)part * MLA_META_STRIDE;
    seq = row[0];
    blk = row[1];
    end_seq = row[2];
    end_blk = row[3];
    split = row[4];
  }
  __device__ __forceinline__ bool next(const FwdArgs &a, Seg &s) {
    if (!(seq < end_seq || (seq == end_seq && blk < end_blk))) return false;
    int L = a.seqlens[seq];
    const int cap = a.max_blocks * a.page_size;
    if (L < 0 || L > cap) {
      report_error(a.err, MLA_ERR_DEVICE_BOUNDS, seq);
      L = L < 0 ? 0 : cap;
    }
    const int nblk = (L + 63) >> 6;
    s.seq = seq;
    s.lo = blk;
    s.hi = seq < end_seq ? nblk : min(end_blk, nblk);
    s.split = split;
    s.L = L;
    s.nsplit = a.num_splits[seq + 1] - a.num_splits[seq];
    ++seq;
    blk = 0;
    ++split;
    return true;
  }
};


// Per-tile barrier bookkeeping in registers (arrays indexed by a run-time tile
// number would live in local memory): bit t of `par` is the parity of the number
// of completed uses of tile t, bit t of `used` says whether it was used at all.
struct TileUse {
  uint32_t par = 0, used = 0;
  __device__ __forceinline__ uint32_t parity(int t) const { return (par >> t) & 1u; }
  __device__ __forceinline__ bool was_used(int t) const { return (used >> t) & 1u; }
  __device__ __forceinline__ void advance(int np) {
    const uint32_t m = (1u << np) - 1u;
    par ^= m;
    used |= m;
  }
};

// Physical pages and first rows of the (up to four) pages of a superblock.  The
// block-table loads are issued early (issue) and only consumed later (finish):
// issued right before use they would queue behind this SM's in-flight TMA traffic
// for microseconds.  Out-of-range entries are reported and clamped to page 0.
struct SbPages {
  int page[kSB], row0[kSB];
};
__device__ __forceinline__ void issue_sb_pages(const FwdArgs &a, int seq, int blk0, int np,
                                               SbPages &r) {
#pragma unroll
  for (int p = 0; p < kSB; ++p) {
    const int tok0 = (blk0 + p) << 6;
    const int lb = tok0 / a.page_size;
    r.row0[p] = tok0 - lb * a.page_size;
    r.page[p] = (p < np && lb < a.max_blocks) ? a.block_table[(int64_t)seq * a.bt_stride + lb]
                                              : (p < np ? -1 : 0);
  }
}
__device__ __forceinline__ void finish_sb_pages(const FwdArgs &a, int seq, int np, SbPages &r) {
#pragma unroll
  for (int p = 0; p < kSB; ++p) {
    if (p < np && (r.page[p] < 0 || r.page[p] >= a.num_pages)) {
      report_error(a.err, MLA_ERR_DEVICE_BOUNDS, seq);
      r.page[p] = 0;
    }
  }
}

template <typename T> struct Pack;
template <> struct Pack<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t two(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
  static constexpr bool kBf16 = true;
};
template <> struct Pack<__half> {
  static __device__ __forceinline__ uint32_t two(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
  static constexpr bool kBf16 = false;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Walks this part's non-empty superblocks in order.
struct SbWalk {
  SegWalk w;
  Seg s;
  bool more;
  int sb0;
  __device__ SbWalk(const FwdArgs &a, int part) : w(a, part) {
    more = w.next(a, s);
    sb0 = more ? s.lo : 0;
    skip(a);
  }
  __device__ void skip(const FwdArgs &a) {
    while (more && sb0 >= s.hi) {
      more = w.next(a, s);
      sb0 = more ? s.lo : 0;
    }
  }
  __device__ void advance(const FwdArgs &a) {
    sb0 += kSB;
    skip(a);
  }
};

// A superblock job with its block-table loads in flight (see issue_sb_pages).
struct SbJob {
  int seq, sb0, np;
  SbPages pg;
};
__device__ __forceinline__ void issue_job(const FwdArgs &a, SbWalk &w, SbJob &j) {
  j.seq = w.s.seq;
  j.sb0 = w.sb0;
  j.np = min(kSB, w.s.hi - w.sb0);
  issue_sb_pages(a, j.seq, j.sb0, j.np, j.pg);
  w.advance(a);
}

// ------------------------------------------------------------------------------ score CTA

template <typename T>
__device__ void score_producer(const FwdArgs &a, const CUtensorMap *map, uint8_t *smem,
                               const Ctx &c, int part) {
  Bars *b = c.bars;
  uint32_t kc = 0, tsb = 0;
  // two superblock jobs in flight: the block-table loads of job j + 2 are issued
  // while job j's chunks are being loaded
  SbWalk w(a, part);
  SbJob ja, jb;
  bool ha = w.more, hb = false;
  if (ha) issue_job(a, w, ja);
  hb = w.more;
  if (hb) issue_job(a, w, jb);
  auto run = [&](SbJob &j) -> bool {
    TRACE(0, part, tsb, 8);
    finish_sb_pages(a, j.seq, j.np, j.pg);
    TRACE(0, part, tsb, 10);
    for (int ch = 0; ch < 9; ++ch, ++kc) {
      const uint32_t slot = kc % kNK, use = kc / kNK;
      if (use > 0 && !wait_bar<false>(c, &b->k_empty[slot], (use - 1) & 1, W_K_EMPTY)) return false;
      TRACE_K(1, part, tsb, ch);  // issue time of K chunk ch
      mbar_arrive_expect_tx(&b->k_full[slot], j.np * kChunk);
      uint8_t *dst = smem + kOffK + slot * kKSlot;
#pragma unroll
      for (int p = 0; p < kSB; ++p)
        if (p < j.np)
          tma_load_3d(dst + p * kChunk, map, &b->k_full[slot], 64 * ch, j.pg.row0[p], j.pg.page[p]);
    }
    TRACE(0, part, tsb, 9);
    ++tsb;
    return true;
  };
  while (ha) {
    if (!run(ja)) return;
    ha = w.more;
    if (ha) issue_job(a, w, ja);
    if (!hb) break;
    if (!run(jb)) return;
    hb = w.more;
    if (hb) issue_job(a, w, jb);
  }
}

template <typename T>
__device__ void score_mma(const FwdArgs &a, uint8_t *smem, const Ctx &c, int part, uint32_t tmem) {
  Bars *b = c.bars;
  const uint32_t tQ = tmem, tS = tmem + 256;
  const uint32_t idesc = idesc_f16(128, 256, Pack<T>::kBf16, false, false);
  const uint32_t q8 = smem_u32(smem + kOffQ8);
  uint32_t kc = 0, sb = 0, segn = 0;
  SegWalk walk(a, part);
  Seg s;
  while (walk.next(a, s)) {
    if (s.hi <= s.lo) continue;
    if (!wait_bar<false>(c, &b->q_ready, segn & 1, W_Q_READY)) return;
    tc_fence_after();
    for (int sb0 = s.lo; sb0 < s.hi; sb0 += kSB, ++sb) {
      if (sb > 0) {
        if (!wait_bar<false>(c, &b->s_free, (sb - 1) & 1, W_S_FREE)) return;
        tc_fence_after();
      }
      TRACE(0, part, sb, 0);
      for (int ch = 0; ch < 9; ++ch, ++kc) {
        const uint32_t slot = kc % kNK, use = kc / kNK;
        if (!wait_bar<false>(c, &b->k_full[slot], use & 1, W_K_FULL)) return;
        tc_fence_after();
        if (ch == 0) TRACE(0, part, sb, 1);
        TRACE_K(0, part, sb, ch);
        const uint32_t kb = smem_u32(smem + kOffK + slot * kKSlot);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t bd = desc_kmajor_sw128(kb + 32 * k);
          if (ch < 8)
            mma_ts(tS, tQ + 32 * ch + 8 * k, bd, idesc, (ch | k) != 0);
          else
            mma_ss(tS, desc_kmajor_sw128(q8 + 32 * k), bd, idesc, 1);
        }
        mma_commit(&b->k_empty[slot]);
        if (ch == 5) TRACE(0, part, sb, 11);
      }
      mma_commit(&b->s_full);
      TRACE(0, part, sb, 2);
    }
    ++segn;
  }
}

// Ships each superblock's staged P tiles and header into the value CTA once the
// value CTA has freed the matching ring slots.
__device__ void score_copier(const FwdArgs &a, uint8_t *smem, const Ctx &c, int part) {
  Bars *b = c.bars;
  const uint32_t peer_pring = map_to_rank(smem_u32(smem + kOffPRing), 1);
  const uint32_t peer_hdr = map_to_rank(smem_u32(smem + kOffHdr), 1);
  const uint32_t peer_pfull = map_to_rank(smem_u32(&b->p_full[0]), 1);
  const uint32_t peer_hfull = map_to_rank(smem_u32(&b->hdr_full[0]), 1);
  uint32_t pc = 0;  // P tiles shipped so far (ring slot pc % kNPR)
  uint32_t sb = 0;
  SegWalk walk(a, part);
  Seg s;
  while (walk.next(a, s)) {
    for (int sb0 = s.lo; sb0 < s.hi; sb0 += kSB, ++sb) {
      const int np = min(kSB, s.hi - sb0);
      if (!wait_bar<false>(c, &b->stage_ready, sb & 1, W_STAGE_READY)) return;
      // the header first: the value CTA can prepare O for this superblock while it
      // is still consuming the previous one's tiles
      const int hs = sb & 1;
      bulk_copy_to_peer(peer_hdr + hs * sizeof(Header), smem + kOffHdrStage + hs * sizeof(Header),
                        sizeof(Header), peer_hfull + hs * 8);
      for (int p = 0; p < np; ++p, ++pc) {
        const uint32_t r = pc % kNPR, use = pc / kNPR;
        if (use > 0 && !wait_bar<true>(c, &b->slot_free[r], (use - 1) & 1, W_SLOT_FREE)) return;
        bulk_copy_to_peer(peer_pring + r * kPTile, smem + kOffPStage + p * kPTile, kPTile,
                          peer_pfull + r * 8);
      }
      TRACE(0, part, sb, 7);
    }
  }
}

template <typename T>
__device__ void score_softmax(const FwdArgs &a, uint8_t *smem, const Ctx &c, int part,
                              uint32_t tmem, int head0) {
  Bars *b = c.bars;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sw = warp - 2;             // 0..7
  const int quad = warp & 3;           // TMEM lane quadrant this warp may touch
  const int half = sw >> 2;            // column half of S
  const int r = 32 * quad + lane;      // head row within the tile
  const int head = head0 + r;
  const bool head_ok = head < a.h;
  const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
  const uint32_t tQ = tmem + lane_off, tS = tmem + 256 + lane_off;
  float *red_max = reinterpret_cast<float *>(smem + kOffRed);  // [2][128]
  float *red_sum = red_max + 256;                               // [2][128]
  const T *q = reinterpret_cast<const T *>(a.q);

  const float scale = a.scale_log2;
  uint32_t sb = 0;
  TileUse tu;
  SegWalk walk(a, part);
  Seg s;
  while (walk.next(a, s)) {
    if (s.hi <= s.lo) {  // empty sequence: lse = -inf (its out row is zeroed by the value CTA)
      if (half == 0 && head_ok) {
        if (s.nsplit == 1) a.lse[(int64_t)s.seq * a.lse_stride + head] = -INFINITY;
        else a.lseaccum[(int64_t)s.split * a.h + head] = -INFINITY;
      }
      continue;
    }
    // ---- Q of this sequence: columns 0..511 into TMEM, 512..575 into shared memory
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          q + (int64_t)s.seq * a.q_batch_stride + (int64_t)(head_ok ? head : head0) * a.q_head_stride);
      const int c0 = half * 4;
      for (int ch = c0; ch < c0 + 4; ++ch) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 v = head_ok ? src[ch * 8 + i] : make_uint4(0, 0, 0, 0);
          w[4 * i + 0] = v.x;
          w[4 * i + 1] = v.y;
          w[4 * i + 2] = v.z;
          w[4 * i + 3] = v.w;
        }
        tmem_st32(tQ + 32 * ch, w);
      }
      if (half == 1) {
        const uint32_t row = smem_u32(smem + kOffQ8) + r * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 v = head_ok ? src[64 + i] : make_uint4(0, 0, 0, 0);
          st_shared_v4(row + ((i ^ (r & 7)) << 4), v.x, v.y, v.z, v.w);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&b->q_ready);
    }

    float m_ref = -INFINITY, l = 0.f;
    const int nsb = (s.hi - s.lo + kSB - 1) / kSB;
    for (int j = 0; j < nsb; ++j, ++sb) {
      const int sb0 = s.lo + j * kSB;
      const int np = min(kSB, s.hi - sb0);
      const bool last = j == nsb - 1;
      bool ok = wait_bar<false>(c, &b->s_full, sb & 1, W_S_FULL);
      if (sw == 0 && lane == 0) TRACE(0, part, sb, 3);
      tc_fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int i = 0; i < 4; ++i) tmem_ld32(tS + 128 * half + 32 * i, v[i]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&b->s_free);

      // scale to base-2 units and mask tokens past the sequence / superblock
      // (the valid columns of a superblock are a prefix of length min(64 np, L - 64 sb0))
      const int lim = min(np << 6, s.L - (sb0 << 6)) - 128 * half;
      float mloc = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float x = (32 * i + e < lim) ? __uint_as_float(v[i][e]) * scale : -INFINITY;
          v[i][e] = __float_as_uint(x);
          mloc = fmaxf(mloc, x);
        }
      }
      red_max[half * 128 + r] = mloc;
      if (bar_red_or(1, 256, !ok || c.aborted())) return;  // all softmax threads leave together
      if (sw == 0 && lane == 0) TRACE(0, part, sb, 4);
      const float m_blk = fmaxf(red_max[r], red_max[128 + r]);
      float alpha = 1.f;
      bool resc = false;
      if (m_blk > m_ref + kTau) {  // also the first block (m_ref = -inf)
        alpha = fast_exp2(m_ref - m_blk);
        m_ref = m_blk;
        resc = true;
      }
      // my two staging tiles must have left for the value CTA
#pragma unroll
      for (int t2 = 0; t2 < 2; ++t2) {
        const int t = 2 * half + t2;
        if (ok && t < np && tu.was_used(t))
          ok = wait_bar<true>(c, &b->stage_free[t], tu.parity(t) ^ 1u, W_STAGE_FREE);
      }
      float psum = 0.f;
#pragma unroll
      for (int t2 = 0; t2 < 2; ++t2) {
        const int t = 2 * half + t2;
        const bool write = t < np && ok;
        const uint32_t row = smem_u32(smem + kOffPStage + t * kPTile) + r * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          float p[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            p[e] = fast_exp2(__uint_as_float(v[2 * t2 + (ch >> 2)][(ch & 3) * 8 + e]) - m_ref);
            psum += p[e];
          }
          if (write)
            st_shared_v4(row + ((ch ^ (r & 7)) << 4), Pack<T>::two(p[0], p[1]),
                         Pack<T>::two(p[2], p[3]), Pack<T>::two(p[4], p[5]),
                         Pack<T>::two(p[6], p[7]));
        }
      }
      red_sum[half * 128 + r] = psum;
      if (sw == 0 && lane == 0) TRACE(0, part, sb, 5);
      const int hs = sb & 1;
      Header *hdr = reinterpret_cast<Header *>(smem + kOffHdrStage + hs * sizeof(Header));
      if (ok && half == 0 && sb >= 2)
        ok = wait_bar<true>(c, &b->hdr_free[hs], ((sb >> 1) - 1) & 1, W_HDR_FREE);
      const bool any_resc = bar_red_or(1, 256, resc);
      if (bar_red_or(1, 256, !ok || c.aborted())) return;
      l = l * alpha + (red_sum[r] + red_sum[128 + r]);
      if (half == 0) {
        hdr->alpha[r] = alpha;
        if (last) {
          hdr->l[r] = l;
          hdr->m[r] = m_ref;
          if (head_ok) {
            const float lse2 = m_ref + fast_log2(l);
            if (s.nsplit == 1) a.lse[(int64_t)s.seq * a.lse_stride + head] = lse2 * kLn2;
            else a.lseaccum[(int64_t)s.split * a.h + head] = lse2;
          }
        }
      }
      if (sw == 0 && lane == 0) hdr->flags = ((any_resc && j > 0) ? 1u : 0u) | (last ? 2u : 0u);
      fence_proxy_async_smem();
      mbar_arrive(&b->stage_ready);  // the copier thread ships the tiles and the header
      if (sw == 0 && lane == 0) TRACE(0, part, sb, 6);
      tu.advance(np);
    }
  }
}

// ------------------------------------------------------------------------------ value CTA

template <typename T>
__device__ void value_producer(const FwdArgs &a, const CUtensorMap *map, uint8_t *smem,
                               const Ctx &c, int part) {
  Bars *b = c.bars;
  uint32_t vc = 0, tsb = 0;
  SbWalk w(a, part);
  SbJob ja, jb;
  bool ha = w.more, hb = false;
  if (ha) issue_job(a, w, ja);
  hb = w.more;
  if (hb) issue_job(a, w, jb);
  auto run = [&](SbJob &j) -> bool {
    TRACE(1, part, tsb, 8);
    finish_sb_pages(a, j.seq, j.np, j.pg);
#pragma unroll
    for (int p = 0; p < kSB; ++p) {
      if (p >= j.np) break;
      for (int hv = 0; hv < 2; ++hv, ++vc) {
        const uint32_t slot = vc % kNV, use = vc / kNV;
        if (use > 0 && !wait_bar<false>(c, &b->v_empty[slot], (use - 1) & 1, W_V_EMPTY)) return false;
        if (hv == 0) TRACE_V(part, tsb, 12 + p);
        mbar_arrive_expect_tx(&b->v_full[slot], kVSlot);
        uint8_t *dst = smem + kOffV + slot * kVSlot;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          tma_load_3d(dst + i * kChunk, map, &b->v_full[slot], 64 * (4 * hv + i), j.pg.row0[p],
                      j.pg.page[p]);
      }
    }
    TRACE(1, part, tsb, 9);
    ++tsb;
    return true;
  };
  while (ha) {
    if (!run(ja)) return;
    ha = w.more;
    if (ha) issue_job(a, w, ja);
    if (!hb) break;
    if (!run(jb)) return;
    hb = w.more;
    if (hb) issue_job(a, w, jb);
  }
}

template <typename T>
__device__ void value_mma(const FwdArgs &a, uint8_t *smem, const Ctx &c, int part, uint32_t tmem) {
  Bars *b = c.bars;
  const int lane = threadIdx.x & 31;
  const uint32_t idesc = idesc_f16(128, 256, Pack<T>::kBf16, false, true);
  uint32_t vc = 0, sb = 0, segn = 0;
  uint32_t pc = 0;  // P tiles consumed (ring slot pc % kNPR)
  SegWalk walk(a, part);
  Seg s;
  while (walk.next(a, s)) {
    if (s.hi <= s.lo) continue;
    if (segn > 0) {
      const bool ok = wait_bar<false>(c, &b->o_free, (segn - 1) & 1, W_O_FREE);
      if (__any_sync(0xffffffffu, !ok || c.aborted())) return;
    }
    uint32_t first = 3u;  // bit hv: next MMA into O half hv starts the accumulation
    const int nsb = (s.hi - s.lo + kSB - 1) / kSB;
    for (int j = 0; j < nsb; ++j, ++sb) {
      const int sb0 = s.lo + j * kSB;
      const int np = min(kSB, s.hi - sb0);
      {
        const bool ok = wait_bar<false>(c, &b->o_ready[sb & 1], (sb >> 1) & 1, W_O_READY);
        if (__any_sync(0xffffffffu, !ok || c.aborted())) return;
      }
      if (lane == 0) TRACE(1, part, sb, 0);
      tc_fence_after();
      for (int p = 0; p < np; ++p, ++pc) {
        const uint32_t r = pc % kNPR;
        const int valid = min(64, s.L - ((sb0 + p) << 6));
        const int ksteps = (valid + 15) >> 4;
        {
          const bool ok = wait_bar<true>(c, &b->p_full[r], (pc / kNPR) & 1, W_P_FULL);
          if (__any_sync(0xffffffffu, !ok || c.aborted())) return;
        }
        if (lane == 0) TRACE_V(part, sb, p);
        if (lane == 0 && p == 0) TRACE(1, part, sb, 1);
        const uint32_t pt = smem_u32(smem + kOffPRing + r * kPTile);
        for (int hv = 0; hv < 2; ++hv, ++vc) {
          const uint32_t slot = vc % kNV, use = vc / kNV;
          {
            const bool ok = wait_bar<false>(c, &b->v_full[slot], use & 1, W_V_FULL);
            if (__any_sync(0xffffffffu, !ok || c.aborted())) return;
          }
          if (lane == 0) TRACE_V(part, sb, 4 + 2 * p + hv);
          if (lane == 0 && p == 0 && hv == 0) TRACE(1, part, sb, 3);
          uint8_t *vs = smem + kOffV + slot * kVSlot;
          if (valid & 15) {  // rows past the sequence inside the last K step: make them 0
            const int r0 = valid, r1 = ksteps * 16;
            for (int idx = lane; idx < (r1 - r0) * 4 * 8; idx += 32) {
              const int row = r0 + idx / 32, i = (idx / 8) & 3, ch = idx & 7;
              st_shared_v4(smem_u32(vs + i * kChunk + row * 128 + ch * 16), 0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t vb = smem_u32(vs);
            for (int k = 0; k < ksteps; ++k) {
              mma_ss(tmem + 256 * hv, desc_kmajor_sw128(pt + 32 * k),
                     desc_mnmajor_sw128(vb + 2048 * k, 8192, 1024), idesc,
                     (((first >> hv) & 1u) && k == 0) ? 0u : 1u);
            }
            first &= ~(1u << hv);
            mma_commit(&b->v_empty[slot]);
          }
          __syncwarp();
        }
        if (lane == 0) mma_commit_multicast(&b->slot_free[r], 1);

      }
      if (lane == 0) mma_commit(&b->o_done[sb & 1]);
      if (lane == 0) TRACE(1, part, sb, 2);
      __syncwarp();
    }
    ++segn;
  }
}

// 256 threads bring the four pages of superblock `w` (all 576 columns) into L2.
__device__ __forceinline__ void prefetch_sb_lines(const FwdArgs &a, const SbWalk &w, int tid) {
  if (!w.more) return;
  const int np = min(kSB, w.s.hi - w.sb0);
  SbPages pg;
  issue_sb_pages(a, w.s.seq, w.sb0, np, pg);
  finish_sb_pages(a, w.s.seq, np, pg);
  const char *kv = reinterpret_cast<const char *>(a.kv);
  constexpr int kLinesPerPage = 64 * 9;  // 64 rows x 1152 bytes
#pragma unroll
  for (int k = 0; k < (kSB * kLinesPerPage) / 256; ++k) {
    const int line = tid + 256 * k;
    const int p = line / kLinesPerPage;
    if (p < np) {
      const int rem = line - p * kLinesPerPage;
      const int row = rem / 9, col = rem - row * 9;
      const char *addr = kv + ((int64_t)pg.page[p] * a.kv_page_stride +
                               (int64_t)(pg.row0[p] + row) * a.kv_row_stride) * 2 + col * 128;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(addr));
    }
  }
}

// Arms each incoming P tile's barrier and tells the score CTA as soon as the copy
// has landed, so it can reuse the staging tile.
__device__ void value_receiver(const FwdArgs &a, const Ctx &c, int part) {
  Bars *b = c.bars;
  uint32_t pc = 0;
  SbWalk w(a, part);
  while (w.more) {
    const int np = min(kSB, w.s.hi - w.sb0);
    for (int t = 0; t < np; ++t, ++pc) {
      const uint32_t r = pc % kNPR;
      mbar_arrive_expect_tx(&b->p_full[r], kPTile);
      if (!wait_bar<true>(c, &b->p_full[r], (pc / kNPR) & 1, W_P_FULL)) return;
      mbar_arrive_cluster(&b->stage_free[t], 0);
    }
    w.advance(a);
  }
}

template <typename T>
__device__ void value_correction(const FwdArgs &a, uint8_t *smem, const Ctx &c, int part,
                                 uint32_t tmem, int head0) {
  Bars *b = c.bars;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sw = warp - 2;
  const int quad = warp & 3;
  const int half = sw >> 2;  // O columns [256 * half, 256 * half + 256)
  const int r = 32 * quad + lane;
  const int head = head0 + r;
  const bool head_ok = head < a.h;
  const uint32_t tO = tmem + ((uint32_t)(32 * quad) << 16) + 256 * half;
  uint32_t sb = 0;
  int observed = -1;  // last o_done phase (superblock index) waited on
  SbWalk pf(a, part);
  for (int i = 0; i < kLinePrefetchSb; ++i) {
    prefetch_sb_lines(a, pf, threadIdx.x - 64);
    pf.advance(a);
  }
  auto wait_done = [&](int k) -> bool {
    while (observed < k) {
      const int n = observed + 1;
      if (!wait_bar<false>(c, &b->o_done[n & 1], (n >> 1) & 1, W_O_DONE)) return false;
      observed = n;
    }
    return true;
  };
  SegWalk walk(a, part);
  Seg s;
  while (walk.next(a, s)) {
    if (s.hi <= s.lo) {  // empty sequence: its output row is zero
      if (head_ok && s.nsplit == 1) {
        uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(a.out) +
                                             (int64_t)s.seq * a.o_batch_stride +
                                             (int64_t)head * a.o_head_stride + 256 * half);
        for (int i = 0; i < 32; ++i) o[i] = make_uint4(0, 0, 0, 0);
      } else if (head_ok) {
        float4 *o = reinterpret_cast<float4 *>(a.oaccum + ((int64_t)s.split * a.h + head) * 512 +
                                               256 * half);
        for (int i = 0; i < 64; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      continue;
    }
    const int nsb = (s.hi - s.lo + kSB - 1) / kSB;
    for (int j = 0; j < nsb; ++j, ++sb) {
      const int hs = sb & 1;
      if (kLinePrefetchSb > 0) {
        prefetch_sb_lines(a, pf, threadIdx.x - 64);
        pf.advance(a);
      }
      if (sw == 0 && lane == 0) mbar_arrive_expect_tx(&b->hdr_full[hs], sizeof(Header));
      bool ok = wait_bar<true>(c, &b->hdr_full[hs], (sb >> 1) & 1, W_HDR_FULL);
      if (sw == 0 && lane == 0) TRACE(1, part, sb, 4);
      const Header *hdr = reinterpret_cast<const Header *>(smem + kOffHdr + hs * sizeof(Header));
      const uint32_t flags = hdr->flags;
      const float alpha = hdr->alpha[r];
      const float lrow = hdr->l[r];
      if (bar_red_or(2, 256, !ok || c.aborted())) return;
      if (sw == 0 && lane == 0) mbar_arrive_cluster(&b->hdr_free[hs], 0);
      // O_done(sb - 2) keeps the o_ready barriers from running two phases ahead
      if ((int)sb >= 2) ok = wait_done((int)sb - 2);
      if (ok && (flags & 1u)) ok = wait_done((int)sb - 1);
      if (bar_red_or(2, 256, !ok || c.aborted())) return;
      // only warps with a head whose reference max moved touch O
      if ((flags & 1u) && __any_sync(0xffffffffu, alpha != 1.f)) {
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {
          uint32_t w[32];
          tmem_ld32(tO + 32 * i, w);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * alpha);
          tmem_st32(tO + 32 * i, w);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      mbar_arrive(&b->o_ready[sb & 1]);
      if (sw == 0 && lane == 0) TRACE(1, part, sb, 5);
      if (flags & 2u) {  // epilogue
        ok = wait_done((int)sb);
        if (bar_red_or(2, 256, !ok || c.aborted())) return;
        tc_fence_after();
        const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {
          uint32_t w[32];
          tmem_ld32(tO + 32 * i, w);
          tmem_wait_ld();
          if (!head_ok) continue;
          if (s.nsplit == 1) {
            uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(a.out) +
                                                 (int64_t)s.seq * a.o_batch_stride +
                                                 (int64_t)head * a.o_head_stride + 256 * half +
                                                 32 * i);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float *f = reinterpret_cast<const float *>(&w[8 * k]);
              o[k] = make_uint4(Pack<T>::two(f[0] * inv, f[1] * inv), Pack<T>::two(f[2] * inv, f[3] * inv),
                                Pack<T>::two(f[4] * inv, f[5] * inv), Pack<T>::two(f[6] * inv, f[7] * inv));
            }
          } else {
            float4 *o = reinterpret_cast<float4 *>(a.oaccum + ((int64_t)s.split * a.h + head) * 512 +
                                                   256 * half + 32 * i);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o[k] = make_float4(__uint_as_float(w[4 * k]) * inv, __uint_as_float(w[4 * k + 1]) * inv,
                                 __uint_as_float(w[4 * k + 2]) * inv, __uint_as_float(w[4 * k + 3]) * inv);
          }
        }
        tc_fence_before();
        mbar_arrive(&b->o_free);
        if (sw == 0 && lane == 0) TRACE(1, part, sb, 6);
      }
    }
  }
}

// ------------------------------------------------------------------------------ kernel

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
split_tc_kernel(const __grid_constant__ CUtensorMap kv_map, const FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  Bars *b = reinterpret_cast<Bars *>(smem + kOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t role = cluster_ctarank();  // 0: score CTA, 1: value CTA
  const int part = blockIdx.x >> 1;
  const int head0 = blockIdx.y * 128;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNK; ++i) {
      mbar_init(&b->k_full[i], 1);
      mbar_init(&b->k_empty[i], 1);
    }
    mbar_init(&b->s_full, 1);
    mbar_init(&b->s_free, 256);
    mbar_init(&b->q_ready, 256);
    mbar_init(&b->stage_ready, 256);
    for (int i = 0; i < kSB; ++i) mbar_init(&b->stage_free[i], 1);
    for (int i = 0; i < kNPR; ++i) {
      mbar_init(&b->slot_free[i], 1);
      mbar_init(&b->p_full[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b->hdr_free[i], 1);
      mbar_init(&b->hdr_full[i], 1);
      mbar_init(&b->o_ready[i], 256);
      mbar_init(&b->o_done[i], 1);
    }
    for (int i = 0; i < kNV; ++i) {
      mbar_init(&b->v_full[i], 1);
      mbar_init(&b->v_empty[i], 1);
    }
    mbar_init(&b->o_free, 256);
    b->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&kv_map);
  if (warp == 1) {
    tmem_alloc(&b->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // peer barriers initialised before any remote arrive or copy
  const uint32_t tmem = b->tmem_base;
  const Ctx c{b, a.err};
#if MLA_TRACE
  if (threadIdx.x == 0 && role == 0 && part < 1024 && blockIdx.y == 0) g_parts[part][0] = globaltimer_ns();
#endif

  if (role == 0) {
    // warp 0: K producer, 1: MMA, 2-9: softmax, 10: P/header copier.  Spinning roles
    // never share a warp (a diverged spin loop starves the other lanes' path).
    if (warp == 0) {
      if (lane == 0) score_producer<T>(a, &kv_map, smem, c, part);
    } else if (warp == 1) {
      if (lane == 0) score_mma<T>(a, smem, c, part, tmem);
    } else if (warp < 10) {
      score_softmax<T>(a, smem, c, part, tmem, head0);
    } else {
      if (lane == 0) score_copier(a, smem, c, part);
    }
  } else {
    // warp 0: V producer, 1: MMA, 2-9: correction / epilogue, 10: P-tile receiver
    if (warp == 0) {
      if (lane == 0) value_producer<T>(a, &kv_map, smem, c, part);
    } else if (warp == 1) {
      value_mma<T>(a, smem, c, part, tmem);
    } else if (warp < 10) {
      value_correction<T>(a, smem, c, part, tmem, head0);
    } else {
      if (lane == 0) value_receiver(a, c, part);
    }
  }

  tc_fence_before();
  __syncthreads();
#if MLA_TRACE
  if (threadIdx.x == 0 && part < 1024 && blockIdx.y == 0) g_parts[part][1 + role] = globaltimer_ns();
#endif
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

template <typename T>
cudaError_t launch_typed(const FwdArgs &a, cudaStream_t s) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  cuuint64_t dims[3] = {(cuuint64_t)MLA_HEAD_DIM, (cuuint64_t)a.page_size, (cuuint64_t)a.num_pages};
  cuuint64_t strides[2] = {(cuuint64_t)a.kv_row_stride * 2, (cuuint64_t)a.kv_page_stride * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(&map, Pack<T>::kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   3, const_cast<void *>(a.kv), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(split_tc_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a.num_parts, (a.h + 127) / 128, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_tc_kernel<T>, map, a);
}

}  // namespace

#if MLA_TRACE
extern "C" int mla_debug_trace(void *dst, size_t bytes) {
  if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
  return cudaMemcpyFromSymbol(dst, g_trace, bytes) == cudaSuccess ? 0 : -7;
}
extern "C" int mla_debug_trace_clear(void) {
  static unsigned long long zero[2 * 256 * 16];
  if (cudaMemcpyToSymbol(g_trace_k, zero, sizeof(zero)) != cudaSuccess) return -7;
  if (cudaMemcpyToSymbol(g_trace_v, zero, sizeof(g_trace_v)) != cudaSuccess) return -7;
  return cudaMemcpyToSymbol(g_trace, zero, sizeof(zero)) == cudaSuccess ? 0 : -7;
}
extern "C" int mla_debug_parts(void *dst, size_t bytes) {
  if (bytes > sizeof(g_parts)) bytes = sizeof(g_parts);
  return cudaMemcpyFromSymbol(dst, g_parts, bytes) == cudaSuccess ? 0 : -7;
}
extern "C" int mla_debug_trace_v(void *dst, size_t bytes) {
  if (bytes > sizeof(g_trace_v)) bytes = sizeof(g_trace_v);
  return cudaMemcpyFromSymbol(dst, g_trace_v, bytes) == cudaSuccess ? 0 : -7;
}
extern "C" int mla_debug_trace_k(void *dst, size_t bytes) {
  if (bytes > sizeof(g_trace_k)) bytes = sizeof(g_trace_k);
  return cudaMemcpyFromSymbol(dst, g_trace_k, bytes) == cudaSuccess ? 0 : -7;
}
#endif

cudaError_t launch_split_tc(const FwdArgs &a, cudaStream_t s) {
  return a.dtype == MLA_DTYPE_BF16 ? launch_typed<__nv_bfloat16>(a, s) : launch_typed<__half>(a, s);
}

cudaError_t split_tc_num_sm(int device, int *num_sm) {
  cudaError_t e = cudaFuncSetAttribute(split_tc_kernel<__nv_bfloat16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  int prev = 0;
  cudaGetDevice(&prev);
  if (prev != device) cudaSetDevice(device);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 256, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, split_tc_kernel<__nv_bfloat16>, &cfg);
  if (prev != device) cudaSetDevice(prev);
  if (e != cudaSuccess) return e;
  *num_sm = 2 * clusters;
  return cudaSuccess;
}

}  // namespace mla
