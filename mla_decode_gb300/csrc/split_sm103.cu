// Split kernel for sm_103a: tcgen05 tensor cores, TMEM accumulators, TMA loads,
// a 2-CTA cluster per scheduler part.  One template serves bf16 / fp16 inputs
// (kind::f16 MMAs) and an e4m3 cache with per-tensor scales (kind::f8f6f4, bf16
// out; the geometry differences are in Geo below).
//
// What it computes (per sequence segment and 128-row tile of query rows: heads,
// or seqlen_q x heads token-major) is the TileLang
// guide's split kernel ("用 TileLang 编写高性能 DeepSeek MLA 内核…", sections
// 先看核心难点, Split Kernel, 变体内核 (paged), 6. Split-KV) with FlashMLA's
// softmax form ("DeepSeek开源周第一天：FlashMLA 深度分析", section Softmax 计算优化:
// exp2 with log2(e) folded into the scale, the -inf guard):
//   S = Q . K^T over the 576 columns (latent and RoPE columns through their own
//   tensor maps, so Q / Q_pe and KV / K_pe may be separate tensors), masked past
//   each row's visible length (cache_seqlens, less the later query tokens under
//   the causal mask); online softmax
//   in base 2; P rounded to the input dtype; O += P . V with V the first 512
//   columns of the same cached rows; at the segment end O / l and the base-2 LSE.
//
// How it is laid out on the GPU (this library's design, not the pages'): the
// fp32 accumulator O[128 heads][512] fills an SM's whole tensor memory, so each
// part is served by a cluster of two CTAs with different roles:
//   * score CTA (cluster rank 0): all 576 Q columns live in TMEM as the A operand
//     (packed 16-bit pairs, columns 0..287).  K streams through a ring of whole
//     pages (64 rows x 576 columns as nine swizzled 64-column atoms, in two TMA
//     requests, atoms 0..3 and 4..8, each part filled and released on its own),
//     and per page S = Q K^T is 36 MMAs of M=128 x N=64 x K=16
//     into one of three page accumulators in TMEM (so the MMAs run a superblock
//     ahead of the softmax).  A superblock is two pages.  Eight softmax warps (one
//     64-token page each per head row) keep a lazy running max (the reference max
//     moves only when a block exceeds it by more than 2^8, so P <= 256 and O is
//     rarely rescaled; exact in real arithmetic), write P as 16-bit swizzled tiles into a
//     double-buffered staging area, and a copier warp bulk-copies them, with the
//     per-head rescale factors, into the value CTA.  Two row sums are kept: of the
//     fp32 weights (for the LSE) and of the weights as rounded to 16 bits (the
//     ones P . V used), by which O is divided, so that O is a convex combination
//     of the value rows with exactly the weights the MMAs applied.
//   * value CTA (rank 1): O lives in TMEM as two 256-column halves.  Its own TMA
//     stream brings each page's value columns (one 4-D box of four atoms per
//     256 columns); per superblock one MMA warp per O half issues that half's
//     M=128 x N=256 x K=16 MMAs (P from shared memory, K-major, as A; V from
//     shared memory, N-major, as B).  Two groups of
//     four correction warps, one per half, rescale their half of O when the
//     score CTA moved its reference max, so one half is rescaled while the
//     other half's MMAs still run, and write the epilogue: O / l to out as
//     32-byte row stores (at a part's last segment through the idle V ring and
//     TMA stores), or to the split workspace, whose rows are interleaved per
//     4-column chunk so that a warp writes 512 contiguous bytes.
// Every wait is bounded; a wait that runs out records MLA_ERR_DEVICE_TIMEOUT
// with the wait site as detail, and the CTA unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include <cuda_fp8.h>

#include "combine.cuh"
#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kThreads = 384;            // 12 warps (see the role map in the kernel)
constexpr int kSB = 2;                   // pages (64 tokens each) per superblock
constexpr int kNStageMax = 4;            // superblock staging slots in the score CTA (at most)
constexpr int kSBufs = 3;                // S accumulators in the score CTA's TMEM, one page each
// score CTA TMEM columns: Q (latent, then RoPE), then the S page accumulators
// (64 columns each) from kTS0
constexpr uint32_t kTS0 = 320;
static_assert(kTS0 + 64 * kSBufs <= 512, "score TMEM budget");
constexpr int kChunk = 8192;             // [64 rows][128 B] swizzled atom
constexpr int kQBox = 2 * kChunk;        // [128 rows][128 B] box of Q (16 KB)
constexpr float kTau = 8.f;              // lazy rescale: the reference max moves only when a
                                         // block exceeds it by more than this (log2 units)
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // every wait: 1 s
constexpr uint64_t kForcedWaitNs = 1000000ull;     // the forced-timeout test's K wait: 1 ms

struct Header {  // score -> value CTA, one per superblock
  float alpha[128];  // O rescale factor per row
  float l[128];      // last superblock: row sum of the rounded weights (divides O)
  uint32_t flags;    // bit 1: last superblock of the segment
  uint32_t pad[3];
};
static_assert(sizeof(Header) % 16 == 0, "bulk copies move multiples of 16 bytes");

constexpr int kNKMax = 5, kNVMax = 8, kNPSBMax = 4;  // deepest K / V / P rings (e4m3)

struct Bars {
  uint64_t k_full[2 * kNKMax], k_empty[2 * kNKMax];  // score, [entry][part]
  uint64_t s_full[kSBufs], s_free[kSBufs];  // score, per S page buffer
  uint64_t q_free;                      // score: MMAs of a segment done with Q (MMA commit)
  uint64_t qs_full;                     // score: first segment's Q columns 0..255 in staging
  uint64_t stage_ready[kNStageMax];     // score: a superblock's P tiles + header staged
  uint64_t stage_free[kNStageMax];      // score: a staging slot's copy landed (value CTA)
  uint64_t slot_free[kNPSBMax];         // score, value-CTA MMA commits (multicast)
  uint64_t v_full[kNVMax], v_empty[kNVMax];  // value
  uint64_t p_full[kNPSBMax];            // value, bulk copies from the score CTA
  uint64_t o_ready[2][2], o_done[2][2]; // value, [O half][superblock parity]
  uint64_t o_free;                      // value
  uint32_t tmem_base;
  int abort;
};

// Geometry per element width.  Both widths keep a page's scores in one M=128 x
// N=64 accumulator and feed the tensor cores 32 bytes of each row per MMA (K = 16
// 16-bit or K = 32 8-bit elements).
//  16-bit (kind::f16): a K ring entry is one page's 576 columns as nine swizzled
//    [64 rows x 64 columns] atoms (72 KB, 128-byte swizzle); Q takes TMEM columns
//    0..255 (latent) and 256..287 (RoPE); P tiles are [128 heads x 64 tokens]
//    16-bit with the 128-byte swizzle; a V tile is one O half of one page, four
//    [64 x 64] atoms (32 KB).
//  e4m3 (kind::f8f6f4): a K ring entry is nine [64 rows x 64 B] atoms with the
//    64-byte swizzle (36 KB, two TMA requests), and the ring holds four pages; Q
//    takes TMEM columns 0..127 and 128..143; P tiles are [128 x 64] bytes with the
//    64-byte swizzle (8 KB); a V tile is two [64 rows x 128 B] atoms (16 KB).
template <bool kF8>
struct Geo {
  static constexpr int kKEntry = kF8 ? 9 * 4096 : 9 * kChunk;
  static constexpr int kNK = kF8 ? 4 : 2;             // K ring entries, one page each
  // an entry fills and drains as two parts with barriers of their own, atoms 0..3
  // (A) and atoms 4..8 (B): the next page's A half loads while this page's B
  // half is still in use, and a page's MMAs start once A is in
  static constexpr int kKParts = 2;
  static constexpr int kKAtomsA = 4;
  static constexpr int kKAtom = kF8 ? 4096 : kChunk;  // bytes of one [64 rows x 64 columns] atom
  static constexpr int kNStage = kF8 ? 4 : 2;         // superblock staging slots (score CTA)
  static constexpr int kPTile = kF8 ? 8192 : 16384;
  static constexpr int kVSlot = kF8 ? 2 * kChunk : 4 * kChunk;
  static constexpr int kNV = kF8 ? 8 : 4;             // V tiles in flight
  static constexpr int kVAtoms = kF8 ? 2 : 4;         // [64 rows x 128 B] atoms per V tile
  static constexpr int kQHalf = kF8 ? 2 : 4;          // Q boxes per 256 latent columns
  static constexpr int kQBoxCols = kF8 ? 128 : 64;    // Q columns per box
  // A superblock's P as it travels to the value CTA: [P tile of page 0 | P tile of
  // page 1 | header], one bulk copy (a DSMEM copy costs ~0.25 us plus its bytes)
  static constexpr int kSBBytes = 2 * kPTile + (int)sizeof(Header);
  static constexpr int kSBSlot = (kSBBytes + 1023) & ~1023;
  static constexpr int kNPSB = kF8 ? 4 : 2;           // superblock slots in the value CTA
  static constexpr uint32_t kTQhalf = kF8 ? 64 : 128; // TMEM columns per 256 latent columns
  static constexpr uint32_t kTQpe = 2 * kTQhalf;      // Q's RoPE columns in TMEM
  static constexpr int kRopeCps = kF8 ? 2 : 4;        // 32-byte TMEM copies of a row's RoPE part
  static constexpr int kKStep = kF8 ? 32 : 16;        // K (tokens) per P.V MMA
  // shared-memory map (offsets from the 1024-aligned base)
  static constexpr int kOffK = 0;                                      // score: K ring
  static constexpr int kOffPStage = kOffK + kNK * kKEntry;             // score: superblock staging
  static constexpr int kOffRed = kOffPStage + kNStage * kSBSlot;       // score: [4][2][128] floats
  static constexpr int kScoreEnd = kOffRed + 8 * 128 * 4;
  static constexpr int kOffV = 0;                                      // value: V ring
  static constexpr int kOffPRing = kOffV + kNV * kVSlot;               // value: superblock slots
  static constexpr int kValueEnd = kOffPRing + kNPSB * kSBSlot;
  // the epilogue of a part's last segment stages `out` in the (then idle) V ring:
  // 16 KB per correction warp
  static_assert(kNV * kVSlot >= 8 * 16384, "epilogue staging in the V ring");
  static constexpr int kOffBars = ((kScoreEnd > kValueEnd ? kScoreEnd : kValueEnd) + 127) & ~127;
  static constexpr int kSmemBytes = kOffBars + (int)sizeof(Bars) + 1024;  // + alignment slack
  static_assert(kNK <= kNKMax && kNV <= kNVMax && kNPSB <= kNPSBMax && kNStage <= kNStageMax,
                "ring barriers");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kOffPStage % 1024 == 0 && kKEntry % 1024 == 0 && kOffPRing % 1024 == 0 &&
                kVSlot % 1024 == 0 && kPTile % 1024 == 0, "swizzle atoms");
  static_assert(kQHalf * kQBox <= kKEntry && kQHalf * kQBox <= kNStage * kSBSlot,
                "half of Q's latent columns fit a ring entry and the staging slots");
};

// wait sites, reported as the error detail on a timeout (mla_wait_site)
enum : int {
  W_K_EMPTY = MLA_WAIT_K_EMPTY, W_Q_FREE = MLA_WAIT_Q_FREE, W_S_FREE = MLA_WAIT_S_FREE,
  W_K_FULL = MLA_WAIT_K_FULL, W_S_FULL = MLA_WAIT_S_FULL, W_STAGE_FREE = MLA_WAIT_STAGE_FREE,
  W_HDR_FREE = MLA_WAIT_HDR_FREE, W_SLOT_FREE = MLA_WAIT_SLOT_FREE, W_V_EMPTY = MLA_WAIT_V_EMPTY,
  W_O_FREE = MLA_WAIT_O_FREE, W_O_READY = MLA_WAIT_O_READY, W_P_FULL = MLA_WAIT_P_FULL,
  W_V_FULL = MLA_WAIT_V_FULL, W_HDR_FULL = MLA_WAIT_HDR_FULL, W_O_DONE = MLA_WAIT_O_DONE,
  W_STAGE_READY = MLA_WAIT_STAGE_READY
};

struct Ctx {
  Bars *bars;
  int *err;
  uint64_t limit_ns;  // how long a wait may take before it gives up
  __device__ bool aborted() const { return *reinterpret_cast<volatile int *>(&bars->abort) != 0; }
};

// Bounded wait on an mbarrier phase.  The fast path (the phase already
// completed) is one try_wait inline; the spin, its time limit and the abort
// protocol live out of line so that issue loops stay short.  On timeout the
// CTA and its peer are flagged to unwind and MLA_ERR_DEVICE_TIMEOUT is
// recorded with the wait site.
template <bool kCl>
__device__ __noinline__ bool wait_bar_slow(const Ctx &c, uint32_t addr, uint32_t parity, int where) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (kCl ? mbar_try_wait_cluster(addr, parity) : mbar_try_wait(addr, parity)) return true;
    if (*reinterpret_cast<volatile int *>(&c.bars->abort)) return false;
    if (globaltimer_ns() - t0 > c.limit_ns) {
      c.bars->abort = 1;
      const uint32_t peer = map_to_rank(smem_u32(&c.bars->abort), cluster_ctarank() ^ 1);
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer), "r"(1) : "memory");
      report_error(c.err, MLA_ERR_DEVICE_TIMEOUT, where);
      return false;
    }
  }
}

template <bool kCl>
__device__ __forceinline__ bool wait_addr(const Ctx &c, uint32_t addr, uint32_t parity, int where) {
  if (kCl ? mbar_try_wait_cluster(addr, parity) : mbar_try_wait(addr, parity)) return true;
  return wait_bar_slow<kCl>(c, addr, parity, where);
}

template <bool kCl>
__device__ __forceinline__ bool wait_bar(const Ctx &c, uint64_t *bar, uint32_t parity, int where) {
  return wait_addr<kCl>(c, smem_u32(bar), parity, where);
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
  __device__ __noinline__ bool next(const FwdArgs &a, Seg &s) {
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
  // no segment follows the one next() returned last
  __device__ bool done() const { return !(seq < end_seq || (seq == end_seq && blk < end_blk)); }
};


// Physical pages and first rows of the (up to kSB) pages of a superblock.  The
// block-table loads are issued early (issue) and only consumed later (finish):
// issued right before use they would queue behind this SM's in-flight TMA traffic
// for microseconds.  Out-of-range entries are reported and clamped to page 0.
struct SbPages {
  int page[kSB], row0[kSB];
};
__device__ __forceinline__ void issue_sb_pages(const FwdArgs &a, int seq, int blk0, int np,
                                               SbPages &r) {
  const int tok0 = blk0 << 6;
  int lb = tok0 / a.page_size;
  int row = tok0 - lb * a.page_size;
#pragma unroll
  for (int p = 0; p < kSB; ++p) {
    r.row0[p] = row;
    r.page[p] = (p < np && lb < a.max_blocks) ? a.block_table[(int64_t)seq * a.bt_stride + lb]
                                              : (p < np ? -1 : 0);
    row += 64;
    if (row == a.page_size) {
      row = 0;
      ++lb;
    }
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
// two(lo, hi): a packed pair of 16-bit values; unpack(u): the pair as floats (the
// values the MMA reads).
template <> struct Pack<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t two(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  }
  static constexpr bool kBf16 = true;
};
template <> struct Pack<__half> {
  static __device__ __forceinline__ uint32_t two(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&u));
  }
  static constexpr bool kBf16 = false;
};

// Per element type: the geometry, the type of `out`, and the MMA kind.  e4m3
// inputs give bf16 outputs.
template <typename T>
constexpr bool kIsF8 = std::is_same<T, __nv_fp8_e4m3>::value;
template <typename T>
using GeoOf = Geo<kIsF8<T>>;
template <typename T>
using OutT = typename std::conditional<kIsF8<T>, __nv_bfloat16, T>::type;

// The instruction descriptor's A / B format bits: 0 is f16 for kind::f16 and
// e4m3 for kind::f8f6f4, 1 is bf16.
template <typename T>
constexpr bool kFmtBit = std::is_same<T, __nv_bfloat16>::value;

template <typename T>
__device__ __forceinline__ void mma_ts_t(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
  if constexpr (kIsF8<T>) mma_ts_f8(d, a, b, idesc, acc);
  else mma_ts(d, a, b, idesc, acc);
}
template <typename T>
__device__ __forceinline__ void mma_ss_t(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
  if constexpr (kIsF8<T>) mma_ss_f8(d, a, b, idesc, acc);
  else mma_ss(d, a, b, idesc, acc);
}

// Four weights as e4m3 bytes, the first in the lowest byte (rounded to nearest
// even; the weights are finite and at most 256, so nothing saturates).
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}
// The largest (kMax) or smallest of 64 raw scores held as fp32 bit patterns,
// with three-input max / min: 32 dependent-free pairs folded into 4 chains.
template <bool kMax>
__device__ __forceinline__ float extreme3(const uint32_t (&v)[2][32]) {
  float m[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) m[c] = kMax ? -INFINITY : INFINITY;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float &acc = m[(e >> 1) & 3];
      const float a = __uint_as_float(v[i][e]), b = __uint_as_float(v[i][e + 1]);
      if (kMax) asm("max.f32 %0, %0, %1, %2;" : "+f"(acc) : "f"(a), "f"(b));
      else asm("min.f32 %0, %0, %1, %2;" : "+f"(acc) : "f"(a), "f"(b));
    }
  return kMax ? fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])) : fminf(fminf(m[0], m[1]), fminf(m[2], m[3]));
}

// A 32-byte global store (one L2 sector); `p` must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                             uint32_t e, uint32_t f, uint32_t g, uint32_t h) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d), "r"(e), "r"(f), "r"(g), "r"(h)
               : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
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
  bool first;  // first superblock of its segment
  SbPages pg;
};
__device__ __forceinline__ void issue_job(const FwdArgs &a, SbWalk &w, SbJob &j) {
  j.seq = w.s.seq;
  j.sb0 = w.sb0;
  j.np = min(kSB, w.s.hi - w.sb0);
  j.first = w.sb0 == w.s.lo;
  issue_sb_pages(a, j.seq, j.sb0, j.np, j.pg);
  w.advance(a);
}

// ------------------------------------------------------------------------------ score CTA

// K producer.  A 64-token page of K lands as nine swizzled [64 rows x 64 columns]
// atoms back to back (72 KB, or 36 KB in e4m3: one ring entry), in large 4-D TMA
// requests: a request carries a fixed cost of a few hundred nanoseconds, so one
// SM streams whole pages at 80-90 GB/s where [64 x 64] boxes (8 KB) reach about
// 24.  Two requests per page, atoms 0..3 and atoms 4..8 (with Q_pe / K_pe
// separate, latent atoms 4..7 plus the K_pe box), each part with its own
// barriers, so the next page's first part streams in while this page's second
// part is still being multiplied.  At a segment start the ring first carries
// that sequence's Q, which the MMA warp moves into TMEM: the 512 latent columns
// as eight [128 heads x 64] boxes, four per entry, then the 64 RoPE columns.
// Heads past h read as zeros.  The part's first segment starts from an empty
// pipeline, and its P staging tiles are still free: latent columns 0..255 land
// there while the RoPE columns and columns 256..511 take two ring entries, so
// all of Q is in flight at once and the first K page follows the small RoPE box.
template <typename T>
__device__ void score_producer(const FwdArgs &a, const CUtensorMap *kmap, const CUtensorMap *qmap,
                               const CUtensorMap *pemap, const CUtensorMap *qpemap, const CUtensorMap *map4,
                               uint8_t *smem, const Ctx &c, int part, int head0) {
  using G = GeoOf<T>;
  // the RoPE box of Q: the separate 64-column map (16-bit), or the 128-byte box at
  // column 512 of the 576-byte rows, zero-filled past column 575 (e4m3)
  constexpr int kRopeX = kIsF8<T> ? MLA_HEAD_DIM_V : 0;
  Bars *b = c.bars;
  uint32_t kc = 0;      // ring entries filled so far
  bool first_seg = true;  // the part's first (non-empty) segment
  const bool leader = elect_one();
  SbWalk w(a, part);
  SbJob cur{}, nxt{};
  bool hc = false, hn = false;
  // the next ring entry; part h of it is free once the MMAs of its previous use
  // are done with that part
  uint32_t kuse = 0;
  auto next_entry = [&](uint32_t &slot) {
    slot = kc % G::kNK;
    kuse = kc / G::kNK;
    ++kc;
  };
  auto part_free = [&](uint32_t slot, int h) -> bool {
    return kuse == 0 || wait_bar<false>(c, &b->k_empty[2 * slot + h], (kuse - 1) & 1, W_K_EMPTY);
  };
  auto run = [&](SbJob &j) -> bool {
    if (j.first) {
      // ring uses: first segment: RoPE box, latent 256..511 (latent 0..255 go to the
      // staging tiles); later segments: latent 0..255, latent 256..511, RoPE box
      if (first_seg && leader) {
        mbar_arrive_expect_tx(&b->qs_full, G::kQHalf * kQBox);
#pragma unroll
        for (int bx = 0; bx < G::kQHalf; ++bx)
          tma_load_3d(smem + G::kOffPStage + bx * kQBox, qmap, &b->qs_full, G::kQBoxCols * bx, head0,
                      j.seq);
      }
      for (int i = first_seg ? 1 : 0; i < 3; ++i) {
        const int what = first_seg ? (i == 1 ? 2 : 1) : i;  // 0, 1: latent halves; 2: RoPE
        uint32_t slot;
        next_entry(slot);
        // Q takes the whole entry: part A's barrier carries the bytes, part B's
        // completes by a plain arrival
        for (int h = 0; h < G::kKParts; ++h)
          if (!part_free(slot, h)) return false;
        if (leader) {
          uint8_t *dst = smem + G::kOffK + slot * G::kKEntry;
          uint64_t *full = &b->k_full[2 * slot];
          if (what < 2) {
            mbar_arrive_expect_tx(full, G::kQHalf * kQBox);
#pragma unroll
            for (int bx = 0; bx < G::kQHalf; ++bx)
              tma_load_3d(dst + bx * kQBox, qmap, full, G::kQBoxCols * (G::kQHalf * what + bx), head0, j.seq);
          } else {
            mbar_arrive_expect_tx(full, kQBox);
            tma_load_3d(dst, qpemap, full, kRopeX, head0, j.seq);
          }
          if (G::kKParts == 2) mbar_arrive(&b->k_full[2 * slot + 1]);
        }
      }
      first_seg = false;
    }
    finish_sb_pages(a, j.seq, j.np, j.pg);
#pragma unroll
    for (int p = 0; p < kSB; ++p) {
      if (p >= j.np) break;
      uint32_t slot;
      next_entry(slot);
      uint8_t *dst = smem + G::kOffK + slot * G::kKEntry;
      if constexpr (kIsF8<T>) {
        // part A: atoms 0..3 (16 KB, the four-block map `kmap`), part B: atoms 4..8
        // (20 KB, the five-block map `pemap`)
        if (!part_free(slot, 0)) return false;
        if (leader) {
          mbar_arrive_expect_tx(&b->k_full[2 * slot], G::kKAtomsA * G::kKAtom);
          tma_load_4d(dst, kmap, &b->k_full[2 * slot], 0, j.pg.row0[p], 0, j.pg.page[p]);
        }
        if (!part_free(slot, 1)) return false;
        if (leader) {
          mbar_arrive_expect_tx(&b->k_full[2 * slot + 1], (9 - G::kKAtomsA) * G::kKAtom);
          tma_load_4d(dst + G::kKAtomsA * G::kKAtom, pemap, &b->k_full[2 * slot + 1], 0, j.pg.row0[p],
                      G::kKAtomsA, j.pg.page[p]);
        }
      } else {
        // part A: latent atoms 0..3 (the four-block map); part B: atoms 4..8, as
        // five blocks of the 576-column rows or as latent atoms 4..7 plus the
        // K_pe box
        if (!part_free(slot, 0)) return false;
        if (leader) {
          mbar_arrive_expect_tx(&b->k_full[2 * slot], G::kKAtomsA * kChunk);
          tma_load_4d(dst, map4, &b->k_full[2 * slot], 0, j.pg.row0[p], 0, j.pg.page[p]);
        }
        if (!part_free(slot, 1)) return false;
        if (leader) {
          uint64_t *full = &b->k_full[2 * slot + 1];
          uint8_t *dstb = dst + G::kKAtomsA * kChunk;
          mbar_arrive_expect_tx(full, (9 - G::kKAtomsA) * kChunk);
          if (a.k_fused) {
            tma_load_4d(dstb, kmap, full, 0, j.pg.row0[p], G::kKAtomsA, j.pg.page[p]);
          } else {
            tma_load_4d(dstb, map4, full, 0, j.pg.row0[p], G::kKAtomsA, j.pg.page[p]);
            tma_load_3d(dst + 8 * kChunk, pemap, full, 0, j.pg.row0[p], j.pg.page[p]);
          }
        }
      }
    }
    return true;
  };
  // one superblock of block-table lookahead: job j + 1's loads are issued
  // before job j's tiles are requested
  while (true) {
    cur = nxt;
    hc = hn;
    hn = w.more;
    if (hn) issue_job(a, w, nxt);
    if (!hc) {
      if (!hn) break;
      continue;
    }
    if (!run(cur)) return;
  }
}

// Per page, 36 MMAs of M=128 x N=64 x K=16 with A (Q) from TMEM: 32 over the
// latent atoms, 4 over the RoPE atom, into one of the three page accumulators.
// That is a budget of 32 tensor-core cycles per MMA, so the whole warp runs the
// loop, which keeps its counters and descriptors warp-uniform, one elected lane
// issues the MMAs and commits, and the unrolled page body only adds immediate
// offsets to precomputed descriptors.  No warp-collective call sits in the loop:
// a lane that leaves on a failed wait cannot block the others.
template <typename T>
__device__ void score_mma(const FwdArgs &a, uint8_t *smem, const Ctx &c, int part, uint32_t tmem) {
  using G = GeoOf<T>;
  Bars *b = c.bars;
  const uint32_t tQ = tmem;
  const uint32_t idesc = idesc_f16(128, 64, kFmtBit<T>, false, false);
  const uint64_t kdesc = kIsF8<T> ? desc_kmajor_sw64(smem_u32(smem + G::kOffK))
                                  : desc_kmajor_sw128(smem_u32(smem + G::kOffK));
  const uint32_t kfull = smem_u32(&b->k_full[0]), kempty = smem_u32(&b->k_empty[0]);
  uint32_t slot = 0, phase = 0;  // ring position of the next entry and its k_full parity
  uint32_t pgc = 0, segn = 0;    // pages issued (S page buffer pgc % kSBufs), segments
  const bool leader = elect_one();
  auto advance = [&]() {
    if (++slot == G::kNK) {
      slot = 0;
      phase ^= 1u;
    }
  };
  SegWalk walk(a, part);
  Seg s;
  while (walk.next(a, s)) {
    if (s.hi <= s.lo) continue;
    // this segment's Q: the previous segment's MMAs must be done reading it, then
    // the eight latent boxes and the RoPE box go from the ring into TMEM (32 bytes
    // of each row per copy)
    if (segn > 0) {
      if (!wait_bar<false>(c, &b->q_free, (segn - 1) & 1, W_Q_FREE)) return;
      tc_fence_after();
    }
    // the order the producer filled them in (see score_producer)
#pragma unroll 1
    for (int i = 0; i < 3; ++i) {
      // 0, 1: latent columns 0..255 / 256..511 from the ring, 2: RoPE columns from
      // the ring, 3: latent columns 0..255 from the staging tiles
      const int what = segn == 0 ? (i == 0 ? 2 : (i == 1 ? 3 : 1)) : i;
      uint64_t bd;
      if (what == 3) {  // latent 0..255 in the staging tiles (first segment)
        if (!wait_bar<false>(c, &b->qs_full, 0, W_K_FULL)) return;
        tc_fence_after();
        bd = desc_kmajor_sw128(smem_u32(smem + G::kOffPStage));
      } else {
        if (!wait_addr<false>(c, kfull + 16 * slot, phase, W_K_FULL)) return;
        tc_fence_after();
        // Q boxes use the 128-byte swizzle in either width
        bd = desc_kmajor_sw128(smem_u32(smem + G::kOffK + slot * G::kKEntry));
      }
      if (leader) {
        if (what != 2) {
          const uint32_t t0 = tQ + (what == 1 ? G::kTQhalf : 0);
#pragma unroll
          for (int bx = 0; bx < G::kQHalf; ++bx)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tmem_cp_128x256b(t0 + 32 * bx + 8 * k, bd + (uint64_t)(bx * (kQBox >> 4) + 2 * k));
        } else {
#pragma unroll
          for (int k = 0; k < G::kRopeCps; ++k)
            tmem_cp_128x256b(tQ + G::kTQpe + 8 * k, bd + (uint64_t)(2 * k));
        }
        if (what != 3) {
          mma_commit_addr(kempty + 16 * slot);
          if (G::kKParts == 2) mma_commit_addr(kempty + 16 * slot + 8);
        }
      }
      if (what != 3) advance();
    }
#pragma unroll 1
    for (int pg = s.lo; pg < s.hi; ++pg, ++pgc) {
      const uint32_t sbuf = pgc % kSBufs, use = pgc / kSBufs;
      if (use > 0) {  // the softmax has read this buffer's previous page
        if (!wait_bar<false>(c, &b->s_free[sbuf], (use - 1) & 1, W_S_FREE)) return;
        tc_fence_after();
      }
      const uint32_t tS = tmem + kTS0 + 64 * sbuf;
      if (!wait_addr<false>(c, kfull + 16 * slot, phase, W_K_FULL)) return;
      tc_fence_after();
      const uint64_t bd = kdesc + (uint64_t)(slot * (G::kKEntry >> 4));
      if constexpr (kIsF8<T>) {
        // nine [64 x 64 B] atoms, 4 KB apart, two K = 32 steps each (Q's TMEM
        // columns run on through the RoPE part, 16 per atom): part A, its
        // release, then part B
        if (leader) {
#pragma unroll
          for (int blk = 0; blk < G::kKAtomsA; ++blk)
#pragma unroll
            for (int k = 0; k < 2; ++k)
              mma_ts_t<T>(tS, tQ + 16 * blk + 8 * k, bd + (uint64_t)(blk * (4096 >> 4) + 2 * k), idesc,
                          (blk | k) != 0);
          mma_commit_addr(kempty + 16 * slot);
        }
        if (!wait_addr<false>(c, kfull + 16 * slot + 8, phase, W_K_FULL)) return;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int blk = G::kKAtomsA; blk < 9; ++blk)
#pragma unroll
            for (int k = 0; k < 2; ++k)
              mma_ts_t<T>(tS, tQ + 16 * blk + 8 * k, bd + (uint64_t)(blk * (4096 >> 4) + 2 * k), idesc, 1);
          mma_commit_addr(kempty + 16 * slot + 8);
        }
      } else {
        // part A (atoms 0..3), its release, then part B (atoms 4..8; the ninth is
        // the RoPE part, whose Q columns follow the latent ones)
        if (leader) {
#pragma unroll
          for (int blk = 0; blk < G::kKAtomsA; ++blk)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ts_t<T>(tS, tQ + 32 * blk + 8 * k, bd + (uint64_t)(blk * (kChunk >> 4) + 2 * k), idesc,
                          (blk | k) != 0);
          mma_commit_addr(kempty + 16 * slot);
        }
        if (!wait_addr<false>(c, kfull + 16 * slot + 8, phase, W_K_FULL)) return;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int blk = G::kKAtomsA; blk < 9; ++blk)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ts_t<T>(tS, tQ + 32 * blk + 8 * k, bd + (uint64_t)(blk * (kChunk >> 4) + 2 * k), idesc, 1);
          mma_commit_addr(kempty + 16 * slot + 8);
        }
      }
      if (leader) mma_commit(&b->s_full[sbuf]);
      advance();
    }
    if (leader) mma_commit(&b->q_free);
    ++segn;
  }
}

// Ships each superblock's staged P tiles and header into the value CTA, as one
// bulk copy, once the value CTA has freed the matching superblock slot.
template <typename T>
__device__ void score_copier(const FwdArgs &a, uint8_t *smem, const Ctx &c, int part) {
  using G = GeoOf<T>;
  Bars *b = c.bars;
  const uint32_t peer_pring = map_to_rank(smem_u32(smem + G::kOffPRing), 1);
  const uint32_t peer_pfull = map_to_rank(smem_u32(&b->p_full[0]), 1);
  uint32_t sb = 0;
  const bool leader = elect_one();
  SbWalk w(a, part);
  while (w.more) {
    const uint32_t st = sb % G::kNStage, slot = sb % G::kNPSB, use = sb / G::kNPSB;
    if (!wait_bar<false>(c, &b->stage_ready[st], (sb / G::kNStage) & 1, W_STAGE_READY)) return;
    if (use > 0 && !wait_bar<false>(c, &b->slot_free[slot], (use - 1) & 1, W_SLOT_FREE)) return;
    if (leader)
      bulk_copy_to_peer(peer_pring + slot * G::kSBSlot, smem + G::kOffPStage + st * G::kSBSlot, G::kSBBytes,
                        peer_pfull + slot * 8);
    w.advance(a);
    ++sb;
  }
}

template <typename T>
__device__ void score_softmax(const FwdArgs &a, uint8_t *smem, const Ctx &c, int part,
                              uint32_t tmem, int head0) {
  using G = GeoOf<T>;
  Bars *b = c.bars;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sw = warp - 2;             // 0..7
  const int quad = warp & 3;           // TMEM lane quadrant this warp may touch
  const int half = sw >> 2;            // page of the superblock (64 S columns)
  const int r = 32 * quad + lane;      // head row within the tile
  const int head = head0 + r;
  const bool head_ok = head < a.h;
  // several query tokens per sequence (rows token-major): a causal row of token qi
  // sees q_len - 1 - qi fewer cached tokens than the sequence holds
  const int hidden = (a.causal && head_ok) ? a.q_len - 1 - head / a.heads : 0;
  const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
  // [superblock parity][half][128]: a half can be one superblock ahead of the other
  float *red_max = reinterpret_cast<float *>(smem + G::kOffRed);
  float *red_sum = red_max + 512;                               // [half][128] fp32 weights
  float *red_sumr = red_max + 768;                              // [half][128] 16-bit weights
  const float scale = a.scale_log2;
  uint32_t sb = 0;
  uint32_t pgs = 0;  // pages read so far: page p of a superblock is in S buffer (pgs + p) % kSBufs
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
    // l: row sum of the fp32 weights (the LSE); lr: of the weights rounded to the
    // input dtype, which is what P . V summed (O / lr is then exactly a weighted
    // mean of the value rows: a row dominated by one token gives that token's value
    // rather than value * (1 + the rounding error of its weight)).  e4m3: O is
    // divided by l (lr = l), the TileLang kernel's normalisation.
    // Each half keeps the sums of its own pages (rescaled by the common alpha); the
    // two halves' sums meet once, at the segment's last superblock, so a superblock
    // costs one named barrier (the row-max exchange).
    float m_ref = -INFINITY, l = 0.f, lr = 0.f;
    const int nsb = (s.hi - s.lo + kSB - 1) / kSB;
    for (int j = 0; j < nsb; ++j, ++sb) {
      const int sb0 = s.lo + j * kSB;
      const int np = min(kSB, s.hi - sb0);
      const bool last = j == nsb - 1;
      // staging slot of this superblock: [P tile of page 0 | page 1 | header]
      const uint32_t buf = sb % G::kNStage;
      uint8_t *stage = smem + G::kOffPStage + buf * G::kSBSlot;
      bool ok = true;
      uint32_t v[2][32];
      if (half < np) {  // my page's scores (a half without a page sees only -inf)
        const uint32_t pb = (pgs + half) % kSBufs;
        ok = wait_bar<false>(c, &b->s_full[pb], ((pgs + half) / kSBufs) & 1, W_S_FULL);
        tc_fence_after();
        const uint32_t tS = tmem + lane_off + kTS0 + 64 * pb;
        tmem_ld32(tS, v[0]);
        tmem_ld32(tS + 32, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&b->s_free[pb]);
      } else {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int e = 0; e < 32; ++e) v[i][e] = 0u;
      }
      pgs += np;

      // base-2 units; tokens this row does not see (a suffix of my page, all of it
      // when it starts past the row's end) and a page past the segment end (all of
      // it) become -inf after the scale
      const int lim = half < np ? min(64, s.L - hidden - ((sb0 + half) << 6)) : 0;
      float sc = scale;
      if (lim < 64) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            v[i][e] = __float_as_uint(32 * i + e < lim ? __uint_as_float(v[i][e]) * scale : -INFINITY);
        sc = 1.f;
      }
      // eight independent partial maxima (and sums below): 64-long dependent
      // chains would leave the warp waiting on instruction latency
      // the extreme of the raw scores, scaled once (the scale may be negative; a
      // product rounds monotonically, so this is the largest scaled score):
      // three-input max / min, two new scores per instruction
      const float mloc = sc >= 0.f ? sc * extreme3<true>(v) : sc * extreme3<false>(v);
      float *rmax = red_max + (sb & 1) * 256;
      rmax[half * 128 + r] = mloc;
      if (bar_red_or(1, 256, !ok || c.aborted())) return;  // all softmax threads leave together
      const float m_blk = fmaxf(rmax[r], rmax[128 + r]);
      float alpha = 1.f;
      if (m_blk > m_ref + kTau) {  // also the first block (m_ref = -inf)
        alpha = fast_exp2(m_ref - m_blk);
        m_ref = m_blk;
      }
      // the staging slot's previous superblock must have left for the value CTA
      if (ok && sb >= G::kNStage)
        ok = wait_bar<false>(c, &b->stage_free[buf], (sb / G::kNStage - 1) & 1, W_STAGE_FREE);
      float ps[8], pr[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) ps[e] = pr[e] = 0.f;
      const bool write = ok && half < np;
      // a row that has seen no token yet (causal rows only) has m_ref = -inf: its
      // weights are exp2(-inf) = 0, not exp2(-inf + inf)
      const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
      if constexpr (kIsF8<T>) {
        // e4m3 tile: 64 bytes per row, 16-byte piece ch (tokens 16 ch ..) at
        // ch ^ ((row >> 1) & 3) (the 64-byte swizzle).  The weights are at most
        // 2^kTau = 256 < 448, the largest e4m3 value.  Pairs of scores go through
        // the packed fp32x2 FMA / add; O is divided by the sum of the fp32 weights
        // (as the TileLang split kernel sums acc_s before its cast), so the
        // rounded weights are not summed.
        const uint32_t row = smem_u32(stage + half * G::kPTile) + r * 64;
        const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(nm, nm);
        float2 s2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) s2[e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t u[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t *x = &v[ch >> 1][(ch & 1) * 16 + 4 * q];
            float2 a = __ffma2_rn(make_float2(__uint_as_float(x[0]), __uint_as_float(x[1])), sc2, nm2);
            float2 b = __ffma2_rn(make_float2(__uint_as_float(x[2]), __uint_as_float(x[3])), sc2, nm2);
            a = make_float2(fast_exp2(a.x), fast_exp2(a.y));
            b = make_float2(fast_exp2(b.x), fast_exp2(b.y));
            s2[q] = __fadd2_rn(s2[q], __fadd2_rn(a, b));
            u[q] = pack_e4m3x4(a.x, a.y, b.x, b.y);
          }
          if (write) st_shared_v4(row + ((ch ^ ((r >> 1) & 3)) << 4), u[0], u[1], u[2], u[3]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ps[2 * e] = s2[e].x;
          ps[2 * e + 1] = s2[e].y;
        }
      } else {
        // pairs of scores through the packed fp32x2 FMA / add; the rounded weights'
        // sums (what the MMA multiplies) likewise, eight running sums each
        const uint32_t row = smem_u32(stage + half * G::kPTile) + r * 128;
        const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(nm, nm);
        float2 s2[4], r2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) s2[e] = r2[e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t u[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t *x = &v[ch >> 2][(ch & 3) * 8 + 2 * q];
            float2 p = __ffma2_rn(make_float2(__uint_as_float(x[0]), __uint_as_float(x[1])), sc2, nm2);
            p = make_float2(fast_exp2(p.x), fast_exp2(p.y));
            s2[q] = __fadd2_rn(s2[q], p);
            u[q] = Pack<T>::two(p.x, p.y);
            r2[q] = __fadd2_rn(r2[q], Pack<T>::unpack(u[q]));
          }
          if (write) st_shared_v4(row + ((ch ^ (r & 7)) << 4), u[0], u[1], u[2], u[3]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ps[2 * e] = s2[e].x;
          ps[2 * e + 1] = s2[e].y;
          pr[2 * e] = r2[e].x;
          pr[2 * e + 1] = r2[e].y;
        }
      }
      l = l * alpha + (((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7])));
      if constexpr (kIsF8<T>) lr = l;
      else lr = lr * alpha + (((pr[0] + pr[1]) + (pr[2] + pr[3])) + ((pr[4] + pr[5]) + (pr[6] + pr[7])));
      Header *hdr = reinterpret_cast<Header *>(stage + 2 * G::kPTile);
      if (last) {  // the row's totals: both halves' sums
        red_sum[half * 128 + r] = l;
        red_sumr[half * 128 + r] = lr;
        if (bar_red_or(1, 256, !ok || c.aborted())) return;
        l = red_sum[r] + red_sum[128 + r];
        lr = red_sumr[r] + red_sumr[128 + r];
      }
      if (half == 0) {
        // the first superblock of a segment overwrites O: nothing to rescale
        hdr->alpha[r] = j == 0 ? 1.f : alpha;
        if (last) {
          hdr->l[r] = lr;
          if (head_ok) {
            const float lse2 = m_ref + fast_log2(l);
            if (s.nsplit == 1) a.lse[(int64_t)s.seq * a.lse_stride + head] = lse2 * kLn2;
            else a.lseaccum[(int64_t)s.split * a.h + head] = lse2;
          }
        }
      }
      if (sw == 0 && lane == 0) hdr->flags = last ? 2u : 0u;
      fence_proxy_async_smem();
      mbar_arrive(&b->stage_ready[buf]);  // the copier ships the tiles and the header
    }
  }
}

// ------------------------------------------------------------------------------ value CTA

// V producer.  A V tile is one page's 256 value columns of one O half: four
// swizzled [64 rows x 64 columns] atoms, 8 KB apart.  The 4-D map (columns split
// into 64-wide blocks) lands all four in one TMA request.  The rows were fetched
// by the score CTA's K stream just before, so they come from L2.
template <typename T>
__device__ void value_producer(const FwdArgs &a, const CUtensorMap *map4, uint8_t *smem,
                               const Ctx &c, int part) {
  using G = GeoOf<T>;
  Bars *b = c.bars;
  uint32_t vc = 0;
  const bool leader = elect_one();
  SbWalk w(a, part);
  SbJob cur{}, nxt{};
  bool hc = false, hn = false;

  // the MMA warp's order: all pages' O-half-0 columns, then all pages' half-1 columns
  auto run = [&](SbJob &j) -> bool {
    finish_sb_pages(a, j.seq, j.np, j.pg);
    for (int g = 0; g < 2; ++g) {
#pragma unroll
      for (int p = 0; p < kSB; ++p) {
        if (p >= j.np) break;
        const uint32_t slot = vc % G::kNV, use = vc / G::kNV;
        ++vc;
        if (use > 0 && !wait_bar<false>(c, &b->v_empty[slot], (use - 1) & 1, W_V_EMPTY)) return false;
        if (leader) {
          mbar_arrive_expect_tx(&b->v_full[slot], G::kVSlot);
          tma_load_4d(smem + G::kOffV + slot * G::kVSlot, map4, &b->v_full[slot], 0, j.pg.row0[p],
                      G::kVAtoms * g, j.pg.page[p]);
        }
      }
    }
    return true;
  };
  // one superblock of block-table lookahead: job j + 1's loads are issued
  // before job j's tiles are requested
  while (true) {
    cur = nxt;
    hc = hn;
    hn = w.more;
    if (hn) issue_job(a, w, nxt);
    if (!hc) {
      if (!hn) break;
      continue;
    }
    if (!run(cur)) return;
  }
}

// Rows [r0, r1) of a V tile (`atoms` [64 rows x 128 B] boxes) set to zero, for
// the MMA that reads them (once per segment end, so kept out of line).
__device__ __noinline__ void zero_rows(uint8_t *vs, int atoms, int r0, int r1) {
#pragma unroll 1
  for (int row = r0; row < r1; ++row)
#pragma unroll 1
    for (int i = 0; i < atoms; ++i)
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) st_shared_v4(smem_u32(vs + i * kChunk + row * 128 + ch * 16), 0, 0, 0, 0);
  fence_proxy_async_smem();
}

// One warp per O half g (warps 1 and 11): the two halves' MMAs are issued in
// parallel, since a step's waits, issues and commits take ~500 SM clocks of one
// warp's time, longer than the tensor core needs for its two MMAs.  As in the score
// CTA, the whole warp runs the loop and one elected lane issues.
template <typename T>
__device__ void value_mma(const FwdArgs &a, uint8_t *smem, const Ctx &c, int part, uint32_t tmem,
                          int g) {
  using G = GeoOf<T>;
  Bars *b = c.bars;
  const uint32_t idesc = idesc_f16(128, 256, kFmtBit<T>, false, true);
  // P: K-major, 32 bytes of each row per K step in either width; V: N-major,
  // [64 rows x 128 B] atoms 8 KB apart, K step = G::kKStep rows of 128 B
  const uint64_t pdesc = kIsF8<T> ? desc_kmajor_sw64(smem_u32(smem + G::kOffPRing))
                                  : desc_kmajor_sw128(smem_u32(smem + G::kOffPRing));
  const uint64_t vdesc = desc_mnmajor_sw128(smem_u32(smem + G::kOffV), 8192, 1024);
  constexpr int kSteps = 64 / G::kKStep;
  const uint32_t vfull = smem_u32(&b->v_full[0]), vempty = smem_u32(&b->v_empty[0]);
  const uint32_t pfull = smem_u32(&b->p_full[0]), sfree = smem_u32(&b->slot_free[0]);
  const uint32_t tO = tmem + 256 * g;
  uint32_t vc = 0;  // V tiles (both halves) of the superblocks before the current one
  uint32_t sb = 0, segn = 0;
  const bool leader = elect_one();
  SegWalk walk(a, part);
  Seg s;
  while (walk.next(a, s)) {
    if (s.hi <= s.lo) continue;
    if (segn > 0 && !wait_bar<false>(c, &b->o_free, (segn - 1) & 1, W_O_FREE)) return;  // epilogue read O
    uint32_t acc = 0u;  // the segment's first MMA into this half starts the accumulation
    const int nsb = (s.hi - s.lo + kSB - 1) / kSB;
    for (int j = 0; j < nsb; ++j, ++sb) {
      const int sb0 = s.lo + j * kSB;
      const int np = min(kSB, s.hi - sb0);
      const uint32_t r = sb % G::kNPSB;  // this superblock's P slot
      if (!wait_bar<false>(c, &b->o_ready[g][sb & 1], (sb >> 1) & 1, W_O_READY)) return;
      if (!wait_addr<false>(c, pfull + 8 * r, (sb / G::kNPSB) & 1, W_P_FULL)) return;
      tc_fence_after();
#pragma unroll 1
      for (int p = 0; p < np; ++p) {
        // the V stream holds a superblock's tiles as half 0's pages, then half 1's
        const uint32_t t = vc + g * np + p, vslot = t % G::kNV;
        const int valid = min(64, s.L - ((sb0 + p) << 6));
        const int ksteps = (valid + G::kKStep - 1) / G::kKStep;
        if (!wait_addr<false>(c, vfull + 8 * vslot, (t / G::kNV) & 1, W_V_FULL)) return;
        if (leader && (valid % G::kKStep))
          zero_rows(smem + G::kOffV + vslot * G::kVSlot, G::kVAtoms, valid, ksteps * G::kKStep);
        tc_fence_after();
        const uint64_t pd = pdesc + (uint64_t)((r * G::kSBSlot + p * G::kPTile) >> 4);
        const uint64_t vd = vdesc + (uint64_t)(vslot * (G::kVSlot >> 4));
        if (leader) {
#pragma unroll
          for (int k = 0; k < kSteps; ++k)
            if (k < ksteps)
              mma_ss_t<T>(tO, pd + 2 * k, vd + (uint64_t)((G::kKStep * 128 >> 4) * k), idesc, k == 0 ? acc : 1u);
          mma_commit_addr(vempty + 8 * vslot);
          // the P slot is free once both halves' MMAs on it are done (two arrivals)
          if (p == np - 1) mma_commit_multicast_addr(sfree + 8 * r, 1);
        }
        acc = 1u;
      }
      if (leader) mma_commit(&b->o_done[g][sb & 1]);
      vc += 2 * np;
    }
    ++segn;
  }
}

// Arms each incoming superblock's barrier and tells the score CTA as soon as the
// copy has landed, so it can reuse the staging slot.
template <typename T>
__device__ void value_receiver(const FwdArgs &a, const Ctx &c, int part) {
  using G = GeoOf<T>;
  Bars *b = c.bars;
  uint32_t sb = 0;
  const bool leader = elect_one();
  SbWalk w(a, part);
  while (w.more) {
    const uint32_t slot = sb % G::kNPSB;
    if (leader) mbar_arrive_expect_tx(&b->p_full[slot], G::kSBBytes);
    if (!wait_bar<false>(c, &b->p_full[slot], (sb / G::kNPSB) & 1, W_P_FULL)) return;
    if (leader) mbar_arrive_cluster_relaxed(&b->stage_free[sb % G::kNStage], 0);
    w.advance(a);
    ++sb;
  }
}

// Epilogue of one thread's head row and O half: O / l from TMEM to `out` (one
// split) or to the fp32 split workspace.  Once per segment, so out of line.
// `out` (16-bit): with `stage` (a part's last segment) through the warp's 16 KB
// of the idle V ring and four TMA stores, else as the thread's own 32-byte row
// stores.  The workspace holds the partial outputs as [split][128 column chunks][h rows]
// [4 floats]: a warp's 32 consecutive rows write 512 contiguous bytes per chunk.
// (Row-major partials made every warp store touch 32 rows 2 KB apart, and the
// epilogue of one segment took ~10 us at ~26 GB/s.)
template <typename T>
__device__ __noinline__ void write_out(const FwdArgs &a, int seq, int split, int nsplit, int head,
                                       bool head_ok, int g, uint32_t tO, float lrow, uint32_t stage,
                                       const CUtensorMap *omap) {
  using O = OutT<T>;
  // o_scale: the value dequantisation scale (e4m3 caches), 1 otherwise
  const float inv = lrow > 0.f ? a.o_scale / lrow : 0.f;
  const int lane = threadIdx.x & 31;
  const int row0 = head - lane;  // the warp's first row
  if (nsplit != 1) {
    // partials: the next 32 columns' TMEM load is in flight while the current ones
    // are stored
    // kept in L2 (evict_last) until the combine reads them, across the KV stream
    float4 *o = reinterpret_cast<float4 *>(a.oaccum) + ((int64_t)split * 128 + 64 * g) * a.h + head;
    const uint64_t keep = l2_policy_evict_last();
    uint32_t x[2][32];
    tmem_ld32(tO, x[0]);
    tmem_wait_ld_regs(x[0]);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (q < 7) tmem_ld32(tO + 32 * (q + 1), x[(q + 1) & 1]);
      if (head_ok) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t *v = &x[q & 1][4 * k];
          st_global_v4_hint(o + (int64_t)(8 * q + k) * a.h,
                            make_float4(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv,
                                        __uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                            keep);
        }
      }
      if (q < 7) tmem_wait_ld_regs(x[(q + 1) & 1]);
    }
    return;
  }
  if (stage) {
    // the part's last segment (the V ring is free): the warp's 32 rows x 256 columns
    // go to its 16 KB of the ring as four [32 rows x 64 columns] boxes with the
    // 128-byte swizzle (16-byte piece j of row r at j ^ (r & 7): no bank
    // conflicts) and leave as four TMA stores; rows past h are clipped by the map
    uint32_t w[2][32];
    tmem_ld32(tO, w[0]);
    tmem_wait_ld_regs(w[0]);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (q < 7) tmem_ld32(tO + 32 * (q + 1), w[(q + 1) & 1]);
      uint32_t hv[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        hv[e] = Pack<O>::two(__uint_as_float(w[q & 1][2 * e]) * inv, __uint_as_float(w[q & 1][2 * e + 1]) * inv);
      const uint32_t row = stage + (q >> 1) * 4096 + lane * 128;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_shared_v4(row + ((((q & 1) * 4 + k) ^ (lane & 7)) << 4), hv[4 * k], hv[4 * k + 1], hv[4 * k + 2],
                     hv[4 * k + 3]);
      if (q < 7) tmem_wait_ld_regs(w[(q + 1) & 1]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) tma_store_3d(omap, stage + k * 4096, 256 * g + 64 * k, row0, seq);
      bulk_commit_group();
      bulk_wait_all();
    }
    __syncwarp();
    return;
  }
  // one split: each thread writes its own row's 16-bit values, 32 columns (64 B) at a
  // time as two 32-byte stores (whole L2 sectors; 16-byte stores when `out`'s rows
  // are not 32-byte aligned), while the next 32 columns' TMEM load is in flight.
  O *o = reinterpret_cast<O *>(a.out) + (int64_t)seq * a.o_batch_stride + (int64_t)head * a.o_head_stride +
         256 * g;
  const bool v8 = ((reinterpret_cast<uintptr_t>(a.out) | (uintptr_t)(a.o_batch_stride * 2) |
                    (uintptr_t)(a.o_head_stride * 2)) & 31) == 0;
  uint32_t w[2][32];
  tmem_ld32(tO, w[0]);
  tmem_wait_ld_regs(w[0]);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (q < 7) tmem_ld32(tO + 32 * (q + 1), w[(q + 1) & 1]);
    uint32_t hv[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      hv[e] = Pack<O>::two(__uint_as_float(w[q & 1][2 * e]) * inv, __uint_as_float(w[q & 1][2 * e + 1]) * inv);
    if (head_ok) {
      O *dst = o + 32 * q;
      if (v8) {
        st_global_v8(dst, hv[0], hv[1], hv[2], hv[3], hv[4], hv[5], hv[6], hv[7]);
        st_global_v8(dst + 16, hv[8], hv[9], hv[10], hv[11], hv[12], hv[13], hv[14], hv[15]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4 *>(dst + 8 * k) = make_uint4(hv[4 * k], hv[4 * k + 1], hv[4 * k + 2], hv[4 * k + 3]);
      }
    }
    if (q < 7) tmem_wait_ld_regs(w[(q + 1) & 1]);
  }
}

// The zero output row half of an empty sequence (its lse is -inf).
template <typename T>
__device__ __noinline__ void zero_out(const FwdArgs &a, int seq, int split, int nsplit, int head, int g) {
  if (nsplit == 1) {
    uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<OutT<T> *>(a.out) + (int64_t)seq * a.o_batch_stride +
                                         (int64_t)head * a.o_head_stride + 256 * g);
    for (int i = 0; i < 32; ++i) o[i] = make_uint4(0, 0, 0, 0);
  } else {
    float4 *o = reinterpret_cast<float4 *>(a.oaccum) + ((int64_t)split * 128 + 64 * g) * a.h + head;
    for (int i = 0; i < 64; ++i) o[(int64_t)i * a.h] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <typename T>
__device__ void value_correction(const FwdArgs &a, uint8_t *smem, const Ctx &c, int part,
                                 uint32_t tmem, int head0, const CUtensorMap *omap) {
  using G = GeoOf<T>;
  Bars *b = c.bars;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sw = warp - 2;
  const int quad = warp & 3;
  const int g = sw >> 2;  // O columns [256 g, 256 g + 256)
  const int bar_id = 2 + g;
  const int r = 32 * quad + lane;
  const int head = head0 + r;
  const bool head_ok = head < a.h;
  const uint32_t tO = tmem + ((uint32_t)(32 * quad) << 16) + 256 * g;
  uint32_t sb = 0;
  int observed = -1;  // last o_done phase (superblock index) of my half waited on
  auto wait_done = [&](int k) -> bool {
    while (observed < k) {
      const int n = observed + 1;
      if (!wait_bar<false>(c, &b->o_done[g][n & 1], (n >> 1) & 1, W_O_DONE)) return false;
      observed = n;
    }
    return true;
  };
  SegWalk walk(a, part);
  Seg s;
  while (walk.next(a, s)) {
    if (s.hi <= s.lo) {  // empty sequence: its output row is zero
      if (head_ok) zero_out<T>(a, s.seq, s.split, s.nsplit, head, g);
      continue;
    }
    const int nsb = (s.hi - s.lo + kSB - 1) / kSB;
    for (int j = 0; j < nsb; ++j, ++sb) {
      // the header travels in the superblock's P slot, behind its two tiles
      const uint32_t slot = sb % G::kNPSB;
      bool ok = wait_bar<false>(c, &b->p_full[slot], (sb / G::kNPSB) & 1, W_HDR_FULL);
      const Header *hdr =
          reinterpret_cast<const Header *>(smem + G::kOffPRing + slot * G::kSBSlot + 2 * G::kPTile);
      const uint32_t flags = hdr->flags;
      const float alpha = hdr->alpha[r];
      const float lrow = hdr->l[r];
      if (bar_red_or(bar_id, 128, !ok || c.aborted())) return;
      // O_done(sb - 2) keeps the o_ready barriers from running two phases ahead;
      // a warp whose heads moved their reference max rescales once the previous
      // superblock's MMAs into this half are complete
      const bool resc = __any_sync(0xffffffffu, alpha != 1.f);
      if (ok && (int)sb >= 2) ok = wait_done((int)sb - 2);
      if (ok && resc) ok = wait_done((int)sb - 1);
      if (ok && resc) {
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
          uint32_t w0[32], w1[32];
          tmem_ld32(tO + 64 * i, w0);
          tmem_ld32(tO + 64 * i + 32, w1);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            w0[e] = __float_as_uint(__uint_as_float(w0[e]) * alpha);
            w1[e] = __float_as_uint(__uint_as_float(w1[e]) * alpha);
          }
          tmem_st32(tO + 64 * i, w0);
          tmem_st32(tO + 64 * i + 32, w1);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      mbar_arrive(&b->o_ready[g][sb & 1]);
      if (flags & 2u) {  // epilogue
        if (ok) ok = wait_done((int)sb);
        // one split and nothing after this segment: `out` leaves by TMA stores from
        // the V ring, once both halves' MMAs are done with it
        const bool staged = s.nsplit == 1 && walk.done();
        if (ok && staged) ok = wait_bar<false>(c, &b->o_done[1 - g][sb & 1], (sb >> 1) & 1, W_O_DONE);
        if (bar_red_or(bar_id, 128, !ok || c.aborted())) return;
        tc_fence_after();
        write_out<T>(a, s.seq, s.split, s.nsplit, head, head_ok, g, tO, lrow,
                     staged ? smem_u32(smem + G::kOffV + (warp - 2) * 16384) : 0u, omap);
        tc_fence_before();
        mbar_arrive(&b->o_free);
      }
    }
  }
}

// ------------------------------------------------------------------------------ fused combine

// The grid barrier's counters: the high half of each word is the call's tag, the
// low half a count.  The first CTA retags both words at its start when they hold
// another call's tag (a fresh workspace holds anything); every CTA waits for its
// call's tag before it counts itself in with one atomic add (a compare-and-swap
// loop here, with ~150 CTAs arriving together, took ~100 us).  The last CTA out
// sets both counts back to zero, so a replay of the same launch (same tag) starts
// from zero.
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void grid_bar_retag(unsigned long long *w, unsigned long long tag) {
  const unsigned long long old = *reinterpret_cast<volatile unsigned long long *>(w);
  if ((old & 0xffffffff00000000ull) != tag) atomicCAS(w, old, tag);
}

// Waits (bounded) until pred(word) holds; false on timeout (reported).
template <typename Pred>
__device__ __forceinline__ bool grid_bar_wait(const FwdArgs &a, const unsigned long long *w, Pred pred) {
  const uint64_t t0 = globaltimer_ns();
  while (!pred(ld_acquire_gpu(w))) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report_error(a.err, MLA_ERR_DEVICE_TIMEOUT, MLA_WAIT_GRID);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// The persistent variant of the TileLang kernels synchronises its split and
// combine phases grid-wide ("用 TileLang 编写高性能 DeepSeek MLA 内核…", section
// 变体内核).  Here: every CTA arrives once its parts are done (its partial
// outputs and LSEs fenced first), waits (bounded) for all CTAs of the grid, and
// then the grid's warps share the combine of every split sequence, one 32-row x
// 32-column block per warp at a time.  The whole grid is resident (one CTA per
// SM, at most one part per cluster that fits), so the barrier does not wait on
// CTAs that have not started.
template <typename T>
__device__ __noinline__ void combine_phase(const FwdArgs &a, uint8_t *smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long ctas = (unsigned long long)gridDim.x * gridDim.y;
  const unsigned long long tag = (unsigned long long)a.token << 32;
  auto tagged = [tag](unsigned long long v) { return (v & 0xffffffff00000000ull) == tag; };
  __shared__ int passed;
  __threadfence();  // this thread's partial outputs and LSEs, before the arrival
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = grid_bar_wait(a, a.grid_bar, tagged);
    if (ok) {
      atomicAdd(a.grid_bar, 1ull);
      ok = grid_bar_wait(a, a.grid_bar, [tag, ctas](unsigned long long v) { return v == tag + ctas; });
    }
    passed = ok ? 1 : 0;
  }
  __syncthreads();
  if (!passed) return;
  __threadfence();
  uint4 (*tile)[4] = reinterpret_cast<uint4 (*)[4]>(smem + warp * 2048);
  const int per_seq = ((a.h + 31) / 32) * 16;  // 32-row groups x 32-column blocks
  const int64_t blocks = (int64_t)a.b * per_seq;
  const int64_t warps = (int64_t)ctas * (kThreads / 32);
  const int64_t u0 = (int64_t)(blockIdx.y * gridDim.x + blockIdx.x) * (kThreads / 32) + warp;
  for (int64_t u = u0; u < blocks; u += warps) {
    const int seq = (int)(u / per_seq), rem = (int)(u % per_seq);
    const int s0 = a.num_splits[seq], n = a.num_splits[seq + 1] - s0;
    if (n <= 1) continue;
    combine_block<OutT<T>>(a, seq, s0, n, 32 * (rem >> 4), kCombineChunks * (rem & 15), tile, lane);
  }
  __syncthreads();
  if (threadIdx.x == 0 && grid_bar_wait(a, a.grid_bar + 1, tagged) &&
      atomicAdd(a.grid_bar + 1, 1ull) + 1 == tag + ctas) {
    atomicExch(a.grid_bar, tag);
    atomicExch(a.grid_bar + 1, tag);
  }
}

// ------------------------------------------------------------------------------ kernel

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
split_tc_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap q_map,
                const __grid_constant__ CUtensorMap kpe_map,
                const __grid_constant__ CUtensorMap qpe_map,
                const __grid_constant__ CUtensorMap kv4_map, const __grid_constant__ CUtensorMap o_map,
                const FwdArgs a) {
  using G = GeoOf<T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  Bars *b = reinterpret_cast<Bars *>(smem + G::kOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t role = cluster_ctarank();  // 0: score CTA, 1: value CTA
  const int part = blockIdx.x >> 1;
  const int head0 = blockIdx.y * 128;

  if (threadIdx.x == 0) {
    for (int i = 0; i < G::kNK; ++i) {
      for (int h = 0; h < G::kKParts; ++h) {
        mbar_init(&b->k_full[2 * i + h], 1);
        mbar_init(&b->k_empty[2 * i + h], 1);
      }
    }
    for (int i = 0; i < 2; ++i) {
      for (int k = 0; k < 2; ++k) {
        mbar_init(&b->o_ready[i][k], 128);
        mbar_init(&b->o_done[i][k], 1);
      }
    }
    mbar_init(&b->q_free, 1);
    mbar_init(&b->qs_full, 1);
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&b->s_full[i], 1);
      mbar_init(&b->s_free[i], 128);  // the four warps of the half that reads the page
    }
    for (int i = 0; i < G::kNStage; ++i) {
      mbar_init(&b->stage_ready[i], 256);
      mbar_init(&b->stage_free[i], 1);
    }
    for (int i = 0; i < G::kNPSB; ++i) {
      mbar_init(&b->slot_free[i], 2);    // the last MMA commit of each O half
      mbar_init(&b->p_full[i], 1);
    }
    for (int i = 0; i < G::kNV; ++i) {
      mbar_init(&b->v_full[i], 1);
      mbar_init(&b->v_empty[i], 1);
    }
    mbar_init(&b->o_free, 256);
    b->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&k_map);
    tma_prefetch_desc(&q_map);
    tma_prefetch_desc(&kpe_map);
    tma_prefetch_desc(&qpe_map);
    tma_prefetch_desc(&kv4_map);
    tma_prefetch_desc(&o_map);
  }
  if (warp == 1) {
    tmem_alloc(&b->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // peer barriers initialised before any remote arrive or copy
  // everything above overlaps the previous kernel in the stream (launched with
  // programmatic stream serialisation); the metadata and the buffers it wrote are
  // read only after it has completed
  grid_dependency_wait();
  launch_dependents();
  if (a.fused_combine && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    grid_bar_retag(a.grid_bar, (unsigned long long)a.token << 32);
    grid_bar_retag(a.grid_bar + 1, (unsigned long long)a.token << 32);
  }
  const uint32_t tmem = b->tmem_base;
  const Ctx c{b, a.err, kWaitLimitNs};

  // forced-timeout test (a.forced_timeout): the load and copy warps issue nothing,
  // so nothing is in flight, and the score MMA warp's first wait for K data gives
  // up after 1 ms; every other role sees the abort and unwinds
  const bool loads = !a.forced_timeout;
  if (role == 0) {
    // warp 0: K producer, 1: MMA, 2-9: softmax, 10: P/header copier, 11: idle.  Each
    // role has a whole warp (a diverged spin loop would starve the other lanes' path,
    // and warp-uniform issue loops let one elected lane issue at full rate).
    if (warp == 0) {
      if (loads) score_producer<T>(a, &k_map, &q_map, &kpe_map, &qpe_map, &kv4_map, smem, c, part, head0);
    } else if (warp == 1) {
      score_mma<T>(a, smem, loads ? c : Ctx{b, a.err, kForcedWaitNs}, part, tmem);
    } else if (warp < 10) {
      score_softmax<T>(a, smem, c, part, tmem, head0);
    } else if (warp == 10) {
      if (loads) score_copier<T>(a, smem, c, part);
    }
  } else {
    // warp 0: V producer, 1 / 11: MMAs into O half 0 / 1, 2-5 / 6-9: correction and
    // epilogue of O half 0 / 1, 10: superblock receiver
    if (warp == 0) {
      if (loads) value_producer<T>(a, &kv4_map, smem, c, part);
    } else if (warp == 1 || warp == 11) {
      value_mma<T>(a, smem, c, part, tmem, warp == 1 ? 0 : 1);
    } else if (warp < 10) {
      value_correction<T>(a, smem, c, part, tmem, head0, &o_map);
    } else {
      value_receiver<T>(a, c, part);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*reinterpret_cast<volatile int *>(&b->abort)) {
    // a wait gave up: let this CTA's TMA loads and the peer's copies into it land
    // (they complete within microseconds) before the CTAs exit
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) {
    }
  }
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // several splits in some sequence: the grid combines them (shared memory is free:
  // every load and copy into it has been consumed)
  if (a.fused_combine && a.num_splits[a.b] > a.b) combine_phase<T>(a, smem);
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
constexpr CUtensorMapDataType map_dtype() {
  return kIsF8<T> ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                  : (std::is_same<T, __nv_bfloat16>::value ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

// One 3-D tiled map over a [outer][mid][cols] tensor of T (strides in elements),
// boxes of box_cols x box_mid, 128-byte swizzle, zero fill past the extents.
template <typename T>
cudaError_t make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t mid, uint64_t outer,
                     int64_t mid_stride, int64_t outer_stride, uint32_t box_cols, uint32_t box_mid) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  constexpr uint64_t es = sizeof(T);
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)mid, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)mid_stride * es, (cuuint64_t)outer_stride * es};
  cuuint32_t box[3] = {box_cols, box_mid, 1};
  cuuint32_t el[3] = {1, 1, 1};
  CUresult r = enc(m, map_dtype<T>(), 3, const_cast<void *>(base), dims, strides, box, el,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The kernel's dynamic shared-memory limit is an attribute of the function in the
// current device's context, so it is set once per device (and per element type).
constexpr int kMaxDevices = 64;
template <typename T>
cudaError_t smem_attr() {
  static std::atomic<bool> done[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = cudaFuncSetAttribute(split_tc_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           GeoOf<T>::kSmemBytes);
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

// A 4-D tiled map over the cache's rows as [pages][column blocks][page rows]
// [block_cols columns] (block stride block_cols elements, so a box of several
// blocks lands as that many swizzled [64 rows x block] atoms back to back).
template <typename T>
cudaError_t make_block_map(CUtensorMap *m, const void *base, uint32_t block_cols, uint64_t blocks,
                           uint32_t box_blocks, CUtensorMapSwizzle swizzle, const FwdArgs &a) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  constexpr uint64_t es = sizeof(T);
  cuuint64_t dims[4] = {block_cols, (cuuint64_t)a.page_size, blocks, (cuuint64_t)a.num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)a.kv_row_stride * es, block_cols * es,
                           (cuuint64_t)a.kv_page_stride * es};
  cuuint32_t box[4] = {block_cols, 64, box_blocks, 1};
  cuuint32_t el[4] = {1, 1, 1, 1};
  CUresult r = enc(m, map_dtype<T>(), 4, const_cast<void *>(base), dims, strides, box, el,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_typed(const FwdArgs &a, cudaStream_t s) {
  constexpr uint64_t kLatent = MLA_HEAD_DIM_V, kRope = MLA_HEAD_DIM - MLA_HEAD_DIM_V;
  CUtensorMap kmap, qmap, pemap, qpemap, map4, omap;
  cudaError_t e;
  if constexpr (kIsF8<T>) {
    // e4m3, RoPE columns inside the rows (the host rejects separate tensors).
    // K: a page of nine [64 rows x 64 B] blocks, 64-byte swizzle, in two boxes
    // (blocks 0..3 and 4..8).  V: the
    // first four 128-byte blocks, two per box (one O half of one page).  Q as
    // [b][h][576 B], boxes of 128 heads x 128 B; the RoPE box starts at column 512
    // and reads zeros past column 575.
    e = make_block_map<T>(&kmap, a.kv, 64, 9, GeoOf<T>::kKAtomsA, CU_TENSOR_MAP_SWIZZLE_64B, a);
    if (e == cudaSuccess)
      e = make_block_map<T>(&pemap, a.kv, 64, 9, 9 - GeoOf<T>::kKAtomsA, CU_TENSOR_MAP_SWIZZLE_64B, a);
    if (e == cudaSuccess) e = make_block_map<T>(&map4, a.kv, 128, 4, 2, CU_TENSOR_MAP_SWIZZLE_128B, a);
    if (e == cudaSuccess)
      e = make_map<T>(&qmap, a.q, MLA_HEAD_DIM, a.h, a.b, a.q_head_stride, a.q_batch_stride, 128, 128);
    qpemap = qmap;
  } else {
    // K: a page in two parts, latent blocks 0..3 (the V map's box) and blocks 4..8
    // of the 576-column rows (five blocks), or, with K_pe separate, latent blocks
    // 4..7 plus a [64 rows x 64] K_pe box.  V: the latent blocks, four per box (one
    // O half of one page).  Q and
    // Q_pe as [b][h][cols], boxes of 128 heads x 64 columns (rows past h read as
    // zeros).
    e = make_block_map<T>(&kmap, a.kv, 64, a.k_fused ? 9 : 8, a.k_fused ? 9 - GeoOf<T>::kKAtomsA : 8,
                          CU_TENSOR_MAP_SWIZZLE_128B, a);
    if (e == cudaSuccess)
      e = make_block_map<T>(&map4, a.kv, 64, kLatent / 64, 4, CU_TENSOR_MAP_SWIZZLE_128B, a);
    if (e == cudaSuccess)
      e = make_map<T>(&pemap, a.k_pe, kRope, a.page_size, a.num_pages, a.k_pe_row_stride,
                      a.k_pe_page_stride, 64, 64);
    if (e == cudaSuccess)
      e = make_map<T>(&qmap, a.q, kLatent, a.h, a.b, a.q_head_stride, a.q_batch_stride, 64, 128);
    if (e == cudaSuccess)
      e = make_map<T>(&qpemap, a.q_pe, kRope, a.h, a.b, a.q_pe_head_stride, a.q_pe_batch_stride, 64,
                      128);
  }
  // out as [b][rows][512] 16-bit, boxes of 32 rows x 64 columns (the epilogue's TMA
  // stores; rows past h are not written)
  if (e == cudaSuccess)
    e = make_map<OutT<T>>(&omap, a.out, MLA_HEAD_DIM_V, a.h, a.b, a.o_head_stride, a.o_batch_stride, 64, 32);
  if (e != cudaSuccess) return e;
  if ((e = smem_attr<T>()) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a.num_parts, (a.h + 127) / 128, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = GeoOf<T>::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, split_tc_kernel<T>, kmap, qmap, pemap, qpemap, map4, omap, a);
}

}  // namespace

cudaError_t launch_split_tc(const FwdArgs &a, cudaStream_t s) {
  switch (a.dtype) {
    case MLA_DTYPE_BF16: return launch_typed<__nv_bfloat16>(a, s);
    case MLA_DTYPE_FP16: return launch_typed<__half>(a, s);
    case MLA_DTYPE_E4M3: return launch_typed<__nv_fp8_e4m3>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t split_tc_num_sm(int device, int *num_sm) {
  int prev = 0;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return e;
  if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
  int clusters = 0;
  e = smem_attr<__nv_bfloat16>();
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 256, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = GeoOf<__nv_bfloat16>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&clusters, split_tc_kernel<__nv_bfloat16>, &cfg);
  }
  if (prev != device) {
    const cudaError_t r = cudaSetDevice(prev);
    if (e == cudaSuccess) e = r;
  }
  if (e != cudaSuccess) return e;
  *num_sm = 2 * clusters;
  return cudaSuccess;
}

}  // namespace mla
