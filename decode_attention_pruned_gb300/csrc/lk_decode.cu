// Decode attention over the split LeanK cache (one launch covers one or
// more layers).
//
// What it computes (LeanK article, framerc.cn, section 3.1 "fused
// computation"; FastGen article, mhpn.cn, section 3.2 stage 2): for every
// sequence b and kv head h, the G query heads of h score the full-width rows
// (sinks + window ring, LOCAL ring or SPECIAL rows) on all 128 channels and the
// middle rows of K_prun on the head's kept channels (q gathered to the kept
// channel list), s = q.k / sqrt(128); one online softmax runs over both
// regions and o = sum p V.  INT8 / FP8 caches hold complete 128-row middle blocks
// as codes with per-channel K / per-token V scales (KIVI-style, after the
// pruning); those blocks are scored on the dequantised values.
//
// How:
//   * The work line.  Each (layer, b, h) "entry" is a run of rows: full-width
//     rows, then sealed INT8 / FP8 rows, then bf16 kept-channel rows.  A row costs
//     the bytes it streams, so the line is measured in bytes.  CTA i of P
//     takes the rows whose line offset falls in [iC/P, (i+1)C/P), with P
//     such that every CTA takes at least 64 KB; the CTAs touching an entry
//     are exactly first..last and each writes one partial.
//   * Per CTA: warp 8 (one lane) issues one TMA load per K tile and one per V
//     tile (swizzled boxes), or one bulk copy per three consecutive sealed
//     blocks, into a FIFO ring of variable-size stages with sixteen
//     mbarrier slots; warps 0-7 each take 16 rows of every 128-row tile (of
//     every block of a stage at once).
//   * Tensor cores (mma.sync m16n8k16, fp32 accumulate) with tokens on M:
//     S^T[16 tok x 8] = K[16 x w] Q^T[w x 8] and O^T[128 x 8] += V^T P^T, so
//     the G <= 8 query heads only pad N.  P goes from the S^T accumulator to
//     the B operand of P.V with one movmatrix transpose per 8x8 block; it is
//     split into hi + lo halves (two mmas) so P.V keeps ~16 bits of P.  INT8 / FP8
//     codes enter the f16 mmas exactly; the scales fold into q and p.
//   * Segment end: warps merge through shared memory; a CTA that owns the
//     whole entry writes o, otherwise it writes (o, m, l) to its partial slot
//     and the last of the entry's CTAs (acquire-release counter add) merges
//     them.
//   * Instantiations: one per middle format, cache layout (contiguous or
//     paged) and launch size (at most 32 entries or more), picked on the
//     host.
//   * Fused append (lk_step, bf16 middle): the launch also appends one token
//     per sequence, as an append kernel followed by this decode would.  The
//     window slot the token replaces is left out of the scores; the CTA whose
//     range holds that slot (else full-width row 0) loads the token, the row
//     it evicts and the kept-channel list as one more stage, folds the token
//     (all channels) and the evicted row (kept channels) into its softmax,
//     and writes both into the cache after it has read the slot.  The
//     lengths advance once no CTA reads them again: right after every CTA's
//     work split when the launch has at most 32 entries (the split's copy in
//     shared memory serves the rest of the launch), else when the last CTA
//     finishes.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include <type_traits>

#include "lk_append.cuh"
#include "lk_device.cuh"
#include "lk_internal.h"
#include "lk_kernels.h"

namespace lk {
namespace {

constexpr int kConsumerWarps = 8;                       // two per SM sub-partition
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileRows = kTmaBoxRows;                  // 128 tokens per stage
static_assert(kTileRows == 16 * kConsumerWarps, "one 16-row block per consumer warp");
constexpr int kMergeSlots = 4;                          // (o, m, l) slots of the segment merge
constexpr int kQStride = kHeadDim + 8;                  // padded q row (bf16): conflict-free ldmatrix
// Stages live in a byte ring: a stage holds a K tile (128 rows x width) and a
// V tile (128 rows x 128), so narrow-K tiles (40 KB at k = 32) keep five
// stages in flight where full-width ones (64 KB) keep three; stages of
// three sealed blocks (62-99 KB) keep two or three.
constexpr int kSlots = 16;                              // barrier pairs = stages in flight at most (power of 2)
constexpr int kRingBytes = 200 * 1024;
// A launch over at most this many (layer, kv head) pairs keeps their head
// descriptors in shared memory, copied before the dependency wait: after it
// the work split and the producer read them there instead of through L2.
constexpr int kMaxSmemHeads = 56;
// Sealed blocks per stage: three (62 KB at k = 32 .. 99 KB at k = 128);
// at least two stages fit the ring.
constexpr int kQPerStage = 3;
static_assert(2 * kQPerStage * 132 * (128 + 128) <= kRingBytes, "stages of sealed blocks fit the ring");
constexpr int kUnitsA = 2 * kHeadDim * 2;               // line cost of a full-width row: its bytes
static_assert(kUnitsA == 2 * kHeadDim + 256, "a full-width row costs what a k = 128 middle row costs");
constexpr uint64_t kMinCtaBytes = 64 * 1024;            // line bytes a CTA takes at least (one full-width tile)
constexpr uint64_t kTokenUnits = 48 * 1024;             // line charge of a fused token stage (~1 us of streaming)
constexpr int kFirst = 1, kLast = 2;
constexpr uint64_t kDrainLimitNs = 1000000000ull;      // bound of the producer's final wait for its copies

struct StageDesc {
  int32_t e;           // entry = b * Hkv + h; < 0 ends the stream
  int32_t region;      // 0: full width, 1: kept channels (bf16), 2: sealed INT8 / FP8 blocks, 3: fused token
  int32_t rlo;         // first valid row of the tile (sealed blocks; else 0)
  int32_t nrows;       // valid rows of the tile: rlo .. rlo + nrows - 1
  int32_t width;       // K channels of the tile
  int32_t flags;       // kFirst / kLast of this CTA's segment of the entry
  int32_t first_cta;   // CTAs first..last hold partials of the entry
  int32_t last_cta;
  uint32_t koff;       // ring offset of the K tile; the V tile follows it
  int32_t mrow;        // tile row left out (fused append: the window slot being replaced), or -1
  int32_t n, cnt;      // region 3: the entry's length and special count before the append;
                       // region 2: n = sealed blocks in the stage
};
// region-3 descriptors: mrow holds these flags, width the kept channels of
// the evicted window row (0: none)
constexpr int kTokAlways = 1;        // FULL / LOCAL head: the token always enters
constexpr int kTokSpecialHead = 2;   // SPECIAL head: the token enters if its id is special ...
constexpr int kTokRoom = 4;          // ... and the head has a free row

struct SmemLayout {
  static constexpr int kRingOff = 0;
  static constexpr int kMergeOOff = kRingOff + kRingBytes;
  static constexpr int kMergeMOff = kMergeOOff + kMergeSlots * kMaxGroup * kHeadDim * 4;
  static constexpr int kMergeLOff = kMergeMOff + kMergeSlots * kMaxGroup * 4;
  static constexpr int kQOff = kMergeLOff + kMergeSlots * kMaxGroup * 4;     // q of the segment: all channels
  static constexpr int kQKOff = kQOff + kMaxGroup * kQStride * 2;             //   and kept channels first
  static constexpr int kDescOff = kQKOff + kMaxGroup * kQStride * 2;
  static constexpr int kBarOff = kDescOff + kSlots * (int)sizeof(StageDesc);
  static constexpr int kCBarOff = kBarOff + 2 * kSlots * 8;                  // consumer barrier
  static constexpr int kScanOff = kCBarOff + 8;
  static constexpr int kMiscOff = kScanOff + (kThreads / 32) * 8;
  static constexpr int kHeadsOff = kMiscOff + 12 * 8;                        // head descriptors of the launch
  static constexpr int kLensOff = kHeadsOff + kMaxSmemHeads * (int)sizeof(HeadDesc);   // lengths of <= 32 entries
  static constexpr int kSBarOff = kLensOff + 32 * 12;                        // split-done barrier
  static constexpr int kBytes = kSBarOff + 8;
};
static_assert(SmemLayout::kSBarOff % 8 == 0, "mbarrier alignment");
constexpr int kSmemBytes = SmemLayout::kBytes + 1024;   // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory per block");

// Region 3 (fused append): the new token's K, V rows, then -- when it evicts
// a window row into the middle -- that row's K, V and the kept-channel list.
constexpr uint32_t kTokenBytes = 2 * kHeadDim * 2;
constexpr uint32_t kTokenEvictBytes = 2 * kTokenBytes + kHeadDim * 2;

__device__ __forceinline__ uint32_t stage_bytes(int region, int width) {
  return region == 3   ? (width != 0 ? kTokenEvictBytes : kTokenBytes)
         : region == 2 ? (uint32_t)qblock_bytes(width)
                       : (uint32_t)kTileRows * (2 * width + 256);
}
// ring footprint of a stage: 1024-byte granules (swizzled TMA boxes need
// 1024-byte aligned destinations)
__device__ __forceinline__ uint32_t ring_bytes(int region, int width) {
  return (stage_bytes(region, width) + 1023u) & ~1023u;
}

// Lengths and special counts are read through L2 (they are written by the
// preceding append kernel).  The loads are split from the arithmetic so the
// producer can issue the next entry's loads one entry ahead.
struct EntryLen {
  int n;      // tokens of the sequence in this layer
  int cnt;    // special rows (SPECIAL heads), else 0
  int act;    // fused launches: the sequence takes the appended token
};
static_assert(sizeof(EntryLen) == 12, "shared-memory length table");

// Rows of an entry in line order: n_a full width, n_q in sealed blocks,
// n_b bf16 kept-channel rows (quantised caches: the open tail block).  mrow: the
// full-width row a fused append replaces (left out of the scores), or -1;
// len: what the geometry was computed from.
struct Entry {
  int n_a, n_q, n_b, kb, mrow;
  EntryLen len;
  int anc;    // fused launches: the full-width row the token stage follows, or -1
};

// Entry e of a launch = (layer offset lr, sequence b, kv head h), layers
// outermost.
struct EntryId {
  int lr, l, b, h;
};
// x / d and x mod d by a launch-fixed divisor (see FastDiv), 32-bit x
__device__ __forceinline__ uint32_t fdiv(uint32_t x, const FastDiv& f) {
  return f.m == 0 ? x : (uint32_t)__umul64hi((uint64_t)x, f.m);
}
__device__ __forceinline__ uint32_t fmod(uint32_t x, const FastDiv& f) { return x - fdiv(x, f) * f.d; }

__device__ __forceinline__ EntryId entry_id(const DecodeArgs& a, int e) {
  const CacheView& cv = a.cv;
  const int per_layer = cv.B * cv.Hkv;
  EntryId r;
  r.lr = (int)fdiv((uint32_t)e, a.div_bh);
  const int rem = e - r.lr * per_layer;
  r.b = (int)fdiv((uint32_t)rem, a.div_h);
  r.h = rem - r.b * cv.Hkv;
  r.l = a.layer + r.lr;
  return r;
}

// hb: the head descriptors of the launch's layers, [nlayers][Hkv] (in
// shared memory, or the cache's table from the launch's first layer on).
__device__ __forceinline__ EntryLen entry_len(const DecodeArgs& a, const HeadDesc* hb, int e) {
  const CacheView& cv = a.cv;
  const EntryId id = entry_id(a, e);
  const HeadDesc& hd = hb[id.lr * cv.Hkv + id.h];
  EntryLen r;
  r.n = __ldcg(&cv.len[id.l * cv.B + id.b]);
  r.cnt = hd.policy == kSpecial ? __ldcg(&cv.cnt[id.l * cv.B + id.b]) : 0;
  r.act = a.k_new != nullptr && __ldcg(&cv.active[id.b]) != 0 && r.n < cv.capacity;
  return r;
}

// Whether the token a fused launch appends for sequence b is special (its
// id in [0, vocab) and flagged).
__device__ __forceinline__ bool token_special(const DecodeArgs& a, int b) {
  if (a.ids == nullptr) return false;
  const int id = a.ids[b];
  return id >= 0 && id < a.cv.vocab && a.cv.is_special[id] != 0;
}

__device__ __forceinline__ Entry entry_from(const DecodeArgs& a, const HeadDesc* hb, int e, EntryLen len) {
  const CacheView& cv = a.cv;
  const EntryId id = entry_id(a, e);
  const HeadDesc& hd = hb[id.lr * cv.Hkv + id.h];
  const int N = len.n;
  Entry r{0, 0, 0, 0, -1, len, -1};
  if (hd.policy == kFull) {
    r.n_a = min(N, cv.S + cv.W);
    // a fused append into a full window replaces the slot of token N - W
    if (len.act && N >= cv.S + cv.W) r.mrow = cv.S + (int)fmod((uint32_t)(N - cv.S), a.div_w);
    if (hd.n_kept > 0) {
      const int m = max(0, N - cv.S - cv.W);
      if (kv_quantized(cv.kv_format)) {
        const int nblk = min(m / kQBlockRows, cv.max_pages > 0 ? cv.max_pages : hd.qblocks);
        r.n_q = nblk * kQBlockRows;
        r.n_b = m - m / kQBlockRows * kQBlockRows;
      } else {
        r.n_b = m;
      }
      r.kb = hd.n_kept;
    }
  } else if (hd.policy == kLocal) {
    r.n_a = min(N, cv.W_loc);
    if (len.act && N >= cv.W_loc) r.mrow = (int)fmod((uint32_t)N, a.div_wloc);
  } else {
    r.n_a = min(len.cnt, hd.cap_a);
  }
  r.n_a = min(r.n_a, hd.cap_a);
  r.n_b = min(r.n_b, hd.cap_b);
  r.anc = len.act && r.n_a > 0 ? (r.mrow >= 0 ? r.mrow : 0) : -1;
  return r;
}

__device__ __forceinline__ Entry entry_geometry(const DecodeArgs& a, const HeadDesc* hb, int e) {
  return entry_from(a, hb, e, entry_len(a, hb, e));
}

// line costs per row = bytes streamed per row
__device__ __forceinline__ uint64_t row_cost_b(int kb) { return (uint64_t)(2 * kb + 256); }
__device__ __forceinline__ uint64_t row_cost_q(int kb) { return (uint64_t)(qblock_bytes(kb) / kQBlockRows); }

// The token stage of a fused launch is charged kTokenUnits of line right
// after its anchor row, so the CTA that folds and writes the token streams
// correspondingly fewer rows.
__device__ __forceinline__ uint64_t token_units(const Entry& g) { return g.anc >= 0 ? kTokenUnits : 0; }

__device__ __forceinline__ uint64_t entry_cost(const Entry& g) {
  return (uint64_t)kUnitsA * g.n_a + token_units(g) + row_cost_q(g.kb) * g.n_q + row_cost_b(g.kb) * g.n_b;
}

// a / b for 64-bit a with a 32-bit path when it fits
__device__ __forceinline__ uint64_t udiv(uint64_t a, uint64_t b) {
  if ((a >> 32) == 0 && (b >> 32) == 0) return (uint32_t)a / (uint32_t)b;
  return a / b;
}

// x / c for a row cost c of the line, given c's FastDiv f: one multiply
// while x (an offset inside one entry) fits 32 bits.  The producer divides
// before its first copy of every entry.
__device__ __forceinline__ uint64_t div_cost(uint64_t x, const FastDiv& f) {
  return (x >> 32) == 0 ? fdiv((uint32_t)x, f) : udiv(x, f.d);
}

// Rows r in [0, n) of a region whose row r sits at line offset o0 + c*r and
// starts inside [start, end): r in [r0, r1).  f: the FastDiv of c.
__device__ __forceinline__ void rows_in_range(uint64_t o0, const FastDiv& f, int n, uint64_t start, uint64_t end,
                                              int& r0, int& r1) {
  const uint64_t c = f.d;
  if (n == 0) {
    r0 = r1 = 0;
    return;
  }
  r0 = start > o0 ? (int)min((uint64_t)n, div_cost(start - o0 + c - 1, f)) : 0;
  r1 = end > o0 ? (int)min((uint64_t)n, div_cost(end - o0 + c - 1, f)) : 0;
}

// The CTA whose range [floor(iC/P), floor((i+1)C/P)) holds offset x < C:
// floor(iC/P) <= x  <=>  iC < (x+1)P, so i = ceil((x+1)P/C) - 1.
__device__ __forceinline__ int range_owner(uint64_t x, uint64_t C, int P) {
  const uint64_t i = udiv((x + 1) * (uint64_t)P - 1, C);
  return (int)min(i, (uint64_t)P - 1);
}


__device__ __forceinline__ void record_status(const DecodeArgs& a, uint32_t bits) {
  atomicOr(&a.cv.hdr->status, bits);
}

// Barrier of the consumer warps, on an mbarrier (one arrival per warp) so it
// is bounded like every other wait: on time-out the warp records the status
// bit and goes on (its results are then garbage, and lk_check reports it).
__device__ __forceinline__ void consumer_sync(uint32_t cbar, uint32_t& phase, const DecodeArgs& a) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(cbar);
  if (!mbar_wait_bounded(cbar, phase, a.wait_limit_ns) && (threadIdx.x & 31) == 0) record_status(a, kStatusTimeout);
  phase ^= 1u;
}

// Codes of a sealed block as exact f16 pairs, from one 32-bit word of an
// ldmatrix fragment (bytes 0..3): (byte 0, byte 2) and (byte 1, byte 3).
// K codes: INT8 two's complement or e4m3.  V codes: INT8 offset binary,
// given as 1152 + code (the caller removes the bias), or e4m3.
template <int kFmt>
__device__ __forceinline__ void codes_to_f16x2(uint32_t w, uint32_t& even, uint32_t& odd) {
  if (kFmt == kKvFp8) e4m3x4_to_f16x2(w, even, odd);
  else i8x4_to_f16x2(w, even, odd);
}
template <int kFmt>
__device__ __forceinline__ void vcodes_to_f16x2(uint32_t w, uint32_t& even, uint32_t& odd) {
  if (kFmt == kKvFp8) e4m3x4_to_f16x2(w, even, odd);
  else u8x4_to_f16x2_biased(w, even, odd);
}

// LSE merge of NS shared-memory slots of HS head rows (o: [NS*HS][128],
// m, l: [NS*HS]) for head g, channels dd .. dd+3: acc = sum_w 2^(m_w - M) o_w,
// L = sum_w 2^(m_w - M) l_w, M = max_w m_w.
template <int NS, int HS>
__device__ __forceinline__ void merge_slots(const float* merge_o, const float* merge_m, const float* merge_l, int g,
                                            int dd, float4& acc, float& M, float& L) {
  M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NS; ++w) M = fmaxf(M, merge_m[w * HS + g]);
  acc = make_float4(0.f, 0.f, 0.f, 0.f);
  L = 0.f;
#pragma unroll
  for (int w = 0; w < NS; ++w) {
    const float mw = merge_m[w * HS + g];
    const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
    const float4 v = *reinterpret_cast<const float4*>(&merge_o[(w * HS + g) * kHeadDim + dd]);
    acc.x += f * v.x;
    acc.y += f * v.y;
    acc.z += f * v.z;
    acc.w += f * v.w;
    L += f * merge_l[w * HS + g];
  }
}

// One online-softmax step of a warp over NB groups of its 16 tile rows: x
// holds scaled scores (log2 units, -inf for masked rows) in the S^T
// accumulator layout (x[j][0], x[j][2]: head column 2tig; x[j][1], x[j][3]:
// column 2tig + 1), p receives 2^(x - m).  Lazy rescaling: the running max m
// of a column moves only when some score exceeds it by more than
// kRescaleGap (log2 units); otherwise p <= 2^kRescaleGap, exact in the fp32
// accumulators and in the hi/lo splits of P.  One warp vote replaces the
// column-max shuffles in the common case.  When m moves, l, o and the INT8
// bias sums c are rescaled with it.
template <int NB>
__device__ __forceinline__ void online_softmax(const float (&x)[NB][4], float (&p)[NB][4], float& m0, float& m1,
                                               float& l0, float& l1, float& c0, float& c1, float (&o)[8][4]) {
  float mx0 = fmaxf(x[0][0], x[0][2]), mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
  for (int j = 1; j < NB; ++j) {
    mx0 = fmaxf(mx0, fmaxf(x[j][0], x[j][2]));
    mx1 = fmaxf(mx1, fmaxf(x[j][1], x[j][3]));
  }
  constexpr float kRescaleGap = 8.f;
  if (__any_sync(0xffffffffu, mx0 > m0 + kRescaleGap || mx1 > m1 + kRescaleGap)) {
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    l0 *= al0;
    l1 *= al1;
    c0 *= al0;
    c1 *= al1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[i][0] *= al0;
      o[i][1] *= al1;
      o[i][2] *= al0;
      o[i][3] *= al1;
    }
  }
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    p[j][0] = exp2f(x[j][0] - m0);     // token gid
    p[j][1] = exp2f(x[j][1] - m1);
    p[j][2] = exp2f(x[j][2] - m0);     // token gid + 8
    p[j][3] = exp2f(x[j][3] - m1);
    l0 += p[j][0] + p[j][2];
    l1 += p[j][1] + p[j][3];
  }
}

// Shared-memory address of 16-byte chunk `c` (channels 8c..8c+7) of tile row
// `r`.  128-byte family (K128, V, K64): 64-channel halves of T rows x 128 B,
// 128-byte swizzle (chunk ^= row mod 8).  64-byte family (K32, K96):
// 32-channel stripes of T rows x 64 B, 64-byte swizzle (chunk ^= (row/2) mod 4).
__device__ __forceinline__ uint32_t tile_addr128(uint32_t base, int r, int c) {
  return base + (uint32_t)(c >> 3) * (kTileRows * 128) + (uint32_t)r * 128u +
         ((uint32_t)((c & 7) ^ (r & 7)) << 4);
}
__device__ __forceinline__ uint32_t tile_addr64(uint32_t base, int r, int c) {
  return base + (uint32_t)(c >> 2) * (kTileRows * 64) + (uint32_t)r * 64u +
         ((uint32_t)((c & 3) ^ ((r >> 1) & 3)) << 4);
}

// kFmt: the cache's middle format (KvFormat).  The quantised instantiations
// (INT8, FP8) handle sealed blocks; the bf16 one carries no code for them.
// kPaged: the middle rows live in pages (cv.max_pages > 0).  The layouts'
// producers differ per tile (page ids, tiles cut at page ends), so each is
// compiled on its own and a contiguous cache runs no paged code.
// kSmallE: the launch has at most 32 (layer, sequence, kv head) entries
// (the host picks it): one warp holds every entry's lengths, which the
// kernel then keeps in shared memory; larger launches carry none of that
// code.
template <int kFmt, bool kPaged, bool kSmallE>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeMaps maps, const DecodeArgs a) {
  constexpr bool kQ8 = kFmt != kKvBf16;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  float* merge_o = reinterpret_cast<float*>(sm + SmemLayout::kMergeOOff);
  float* merge_m = reinterpret_cast<float*>(sm + SmemLayout::kMergeMOff);
  float* merge_l = reinterpret_cast<float*>(sm + SmemLayout::kMergeLOff);
  StageDesc* desc = reinterpret_cast<StageDesc*>(sm + SmemLayout::kDescOff);
  const uint32_t bar_full = base + SmemLayout::kBarOff;
  const uint32_t bar_empty = bar_full + kSlots * 8;
  uint64_t* scan = reinterpret_cast<uint64_t*>(sm + SmemLayout::kScanOff);
  volatile int64_t* misc = reinterpret_cast<volatile int64_t*>(sm + SmemLayout::kMiscOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const CacheView& cv = a.cv;
  const int E = a.nlayers * cv.B * cv.Hkv;
  const int G = cv.G;
  // Launches of at most 32 entries keep the lengths each warp's split read
  // in shared memory and read them there from then on; a fused one then
  // advances the lengths as soon as every CTA has finished its split,
  // instead of at its end (see the early advance below).
  EntryLen* slens = reinterpret_cast<EntryLen*>(sm + SmemLayout::kLensOff);
  const uint32_t sbar = base + SmemLayout::kSBarOff;
  const bool early_len = !kQ8 && kSmallE && a.k_new != nullptr;

  static_assert(kSlots < 32, "one barrier pair per lane of warp 0, plus the consumer barrier");
  if (tid < kSlots) {
    mbar_init(bar_full + 8 * tid, 1);
    mbar_init(bar_empty + 8 * tid, kConsumerWarps);
    fence_barrier_init();
  } else if (tid == kSlots) {
    mbar_init(base + SmemLayout::kCBarOff, kConsumerWarps);
    fence_barrier_init();
  } else if (tid == kSlots + 1) {
    mbar_init(base + SmemLayout::kSBarOff, kThreads / 32);
    fence_barrier_init();
  }
  if (tid == 0) {
    misc[0] = E;       // first entry of this CTA
    misc[1] = 0;       // its line offset
    misc[2] = 0;       // last-CTA flag of a segment
    misc[3] = misc[4] = misc[5] = misc[6] = 0;   // geometry of the first entry
    misc[7] = -1;
    misc[8] = misc[9] = misc[10] = 0;
    misc[11] = -1;
  }
  // the flat maps; the block views (few boxes use them) load on first use
  if (warp == kConsumerWarps && lane < kMapAK) tma_prefetch_map(&maps.m[lane]);
  if (warp == kConsumerWarps && lane == 0) {
    // read every launch parameter the producer uses once, so their constant
    // cache lines arrive while the preceding kernel finishes
    uint64_t touch = (uint64_t)cv.hdr ^ (uint64_t)cv.len ^ (uint64_t)cv.cnt ^ (uint64_t)cv.page_table ^
                     (uint64_t)cv.heads ^ (uint64_t)cv.qpool ^ (uint64_t)cv.kept ^ (uint64_t)a.q ^ (uint64_t)a.o ^
                     (uint64_t)a.part ^ (uint64_t)a.part_ml ^ (uint64_t)a.counters ^ a.wait_limit_ns;
    touch ^= (uint64_t)(cv.B ^ cv.Hkv ^ cv.S ^ cv.W ^ cv.W_loc ^ cv.max_pages ^ cv.kv_format ^ a.layer ^ a.nlayers ^
                        cv.G ^ cv.Hq);
#pragma unroll
    for (int i = 0; i < kNumMaps; ++i) touch ^= (uint64_t)maps.block_rows[i];
    touch ^= a.div_bh.m ^ a.div_h.m ^ a.div_w.m ^ a.div_wloc.m ^ (uint64_t)a.scale_log2 ^ (uint64_t)a.k_new ^
             (uint64_t)a.v_new ^ (uint64_t)a.ids;
#pragma unroll
    for (int i = 0; i < 5; ++i) touch ^= a.div_cost_b[i].m ^ a.div_cost_q[i].m ^ a.div_cost_b[i].d ^ a.div_cost_q[i].d;
    asm volatile("" ::"l"(touch));
  }
  // The head table is static (written once at cache init): read it while
  // the preceding kernel finishes -- into shared memory when the launch has
  // few heads (the work split and the producer then read it there), else
  // touched, which also walks the page table for the cache header (a
  // prefetch may be dropped on a TLB miss; a load is not).  Lengths and
  // special counts are written by that kernel, so they are read only after
  // the dependency wait.
  const int nheads = a.nlayers * cv.Hkv;
  const bool heads_in_smem = nheads <= kMaxSmemHeads;
  HeadDesc* sheads = reinterpret_cast<HeadDesc*>(sm + SmemLayout::kHeadsOff);
  const HeadDesc* hb = heads_in_smem ? sheads : cv.heads + (size_t)a.layer * cv.Hkv;
  if (heads_in_smem) {
    static_assert(sizeof(HeadDesc) % 8 == 0, "head descriptors copy as 8-byte words");
    constexpr int kWords = (int)sizeof(HeadDesc) / 8;
    const uint64_t* src = reinterpret_cast<const uint64_t*>(cv.heads + (size_t)a.layer * cv.Hkv);
    uint64_t* dst = reinterpret_cast<uint64_t*>(sheads);
    for (int i = tid; i < nheads * kWords; i += kThreads) dst[i] = src[i];
  } else {
    int64_t touch = 0;
    for (int h = tid; h < nheads; h += kThreads) touch += cv.heads[a.layer * cv.Hkv + h].row_a;
    asm volatile("" ::"l"(touch));
  }
  {
    // warm L2 and the TLB for this thread's first length word (the line may
    // be rewritten by the preceding append: only L2 is touched, which stays
    // coherent)
    const int per0 = (E + kThreads - 1) / kThreads;
    const int e0 = min(E, tid * per0);
    if (e0 < E) {
      const EntryId id0 = entry_id(a, e0);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(&cv.len[id0.l * cv.B + id0.b]));
    }
  }
  // barrier inits and misc visible to every thread (before the dependency
  // wait, so it overlaps the preceding kernel)
  __syncthreads();
  const uint64_t policy = l2_policy_evict_first();
  grid_dependency_wait();
  grid_launch_dependents();

  // ---- the line: the total cost C, this CTA's range [start, end), and the
  // entry, line offset and geometry of its first row
  uint64_t C = 0, start = 0, end = 0;
  int P = 1;
  int first_e = E;
  uint64_t first_off = 0;
  Entry fg{0, 0, 0, 0, -1, {0, 0, 0}, -1};
  const int cta = blockIdx.x;
  // every CTA range holds at least kMinCtaBytes of rows (so at least one row
  // start): a small launch runs on fewer CTAs, with fewer partials to merge.
  // floor(iC/P) = i*(C/P) + floor(i*(C mod P)/P): one division of C by P,
  // then 32-bit arithmetic (i, C mod P < P <= 256)
  auto split_line = [&]() {
    P = (int)max((uint64_t)1, min((uint64_t)gridDim.x, C / kMinCtaBytes));
    const uint64_t cq = udiv(C, (uint64_t)P);
    const uint32_t cr = (uint32_t)(C - cq * (uint64_t)P);
    start = cta < P ? (uint64_t)cta * cq + ((uint32_t)cta * cr) / (uint32_t)P : C;
    end = cta < P ? (uint64_t)(cta + 1) * cq + ((uint32_t)(cta + 1) * cr) / (uint32_t)P : C;
  };
  if constexpr (kSmallE) {
    // few entries: every warp scans them all itself (lane = entry), so no
    // block barrier stands between the length loads and the first copy
    const Entry g = lane < E ? entry_geometry(a, hb, lane) : Entry{0, 0, 0, 0, -1, {0, 0, 0}, -1};
    // every warp writes the same values; each reads back its own writes
    if (lane < E) slens[lane] = g.len;
    __syncwarp();
    const uint64_t cost = entry_cost(g);
    uint64_t incl = cost;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    C = __shfl_sync(0xffffffffu, incl, 31);
    split_line();
    const unsigned hit = __ballot_sync(0xffffffffu, cost > 0 && incl - cost <= start && start < incl);
    const int src = hit ? __ffs(hit) - 1 : 0;
    if (hit) first_e = src;
    first_off = __shfl_sync(0xffffffffu, incl - cost, src);
    fg.n_a = __shfl_sync(0xffffffffu, g.n_a, src);
    fg.n_q = __shfl_sync(0xffffffffu, g.n_q, src);
    fg.n_b = __shfl_sync(0xffffffffu, g.n_b, src);
    fg.kb = __shfl_sync(0xffffffffu, g.kb, src);
    fg.mrow = __shfl_sync(0xffffffffu, g.mrow, src);
    fg.len.n = __shfl_sync(0xffffffffu, g.len.n, src);
    fg.len.cnt = __shfl_sync(0xffffffffu, g.len.cnt, src);
    fg.len.act = __shfl_sync(0xffffffffu, g.len.act, src);
    fg.anc = __shfl_sync(0xffffffffu, g.anc, src);
    // this warp's length loads are done (their values are in use)
    if (early_len && lane == 0) mbar_arrive(sbar);
  } else {
    // per-thread chunks of entries, block exclusive scan
    const int per = (E + kThreads - 1) / kThreads;
    const int e_lo = min(E, tid * per), e_hi = min(E, e_lo + per);
    // the first two entries of the chunk keep their geometry for the second
    // pass
    Entry g0{0, 0, 0, 0, -1, {0, 0, 0}, -1}, g1{0, 0, 0, 0, -1, {0, 0, 0}, -1};
    if (e_lo < e_hi) g0 = entry_geometry(a, hb, e_lo);
    if (e_lo + 1 < e_hi) g1 = entry_geometry(a, hb, e_lo + 1);
    uint64_t local = entry_cost(g0) + entry_cost(g1);
    for (int e = e_lo + 2; e < e_hi; ++e) local += entry_cost(entry_geometry(a, hb, e));
    uint64_t incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    uint64_t warp_base = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      if (w < warp) warp_base += scan[w];
      C += scan[w];
    }
    const uint64_t excl = warp_base + incl - local;
    split_line();
    if (local > 0 && excl <= start && start < excl + local) {
      // this chunk holds the CTA's first row: its entry, line offset and
      // geometry go to every warp through shared memory
      uint64_t acc = excl;
      int found = -1;
      Entry f{0, 0, 0, 0, -1, {0, 0, 0}, -1};
      for (int e = e_lo; found < 0 && e < e_hi; ++e) {
        const Entry g = e == e_lo ? g0 : e == e_lo + 1 ? g1 : entry_geometry(a, hb, e);
        const uint64_t c = entry_cost(g);
        if (acc + c > start) {
          found = e;
          f = g;
        } else {
          acc += c;
        }
      }
      misc[0] = found;
      misc[1] = (int64_t)acc;
      misc[3] = f.n_a;
      misc[4] = f.n_b;
      misc[5] = f.kb;
      misc[6] = f.n_q;
      misc[7] = f.mrow;
      misc[8] = f.len.n;
      misc[9] = f.len.cnt;
      misc[10] = f.len.act;
      misc[11] = f.anc;
    }
    __syncthreads();
    first_e = (int)misc[0];
    first_off = (uint64_t)misc[1];
    fg = Entry{(int)misc[3], (int)misc[6], (int)misc[4], (int)misc[5], (int)misc[7],
               {(int)misc[8], (int)misc[9], (int)misc[10]}, (int)misc[11]};
  }

  if (warp == kConsumerWarps) {
    // ================================================================ producer
    if (lane == 0) {
      // The ring is a FIFO of variable-size stages: the oldest in-flight
      // stage starts at `tail`, the next one goes at `head` (or at 0 when it
      // does not fit before the end).  `wrapped`: the in-flight bytes run
      // from tail to the end and on from 0 to head.  O(1) per stage.
      uint32_t issued = 0, freed = 0;     // stages issued / known released
      uint32_t head = 0, tail = 0;
      bool wrapped = false;
      bool ok = true;
      // Wait (bounded) until the oldest in-flight stage is released.
      auto free_oldest = [&]() -> bool {
        const uint32_t slot = freed & (kSlots - 1);
        if (!mbar_wait_bounded(bar_empty + 8 * slot, (freed / kSlots) & 1u, a.wait_limit_ns)) return false;
        ++freed;
        if (freed == issued) {
          head = tail = 0;
          wrapped = false;
        } else {
          const uint32_t t = desc[freed & (kSlots - 1)].koff;
          if (t < tail) wrapped = false;            // the oldest stage is now past the wrap
          tail = t;
        }
        return true;
      };
      // Ring offset for a stage of `bytes`, once a slot and the bytes are free.
      auto reserve = [&](uint32_t bytes, uint32_t& at) -> bool {
        while (true) {
          if (issued == freed) {
            at = 0;
            break;
          }
          if (issued - freed < (uint32_t)kSlots) {
            if (!wrapped) {
              if (head + bytes <= (uint32_t)kRingBytes) {
                at = head;
                break;
              }
              if (bytes <= tail) {
                at = 0;
                wrapped = true;
                break;
              }
            } else if (head + bytes <= tail) {
              at = head;
              break;
            }
          }
          if (!free_oldest()) return false;
        }
        head = at + bytes;
        return true;
      };
      const bool fused_launch = !kQ8 && a.k_new != nullptr;
      const int e0 = first_e;
      int e = e0;
      uint64_t off = first_off;
      // entry geometry: the first from the scan, later ones from lengths
      // loaded one entry ahead -- after the entry's first copy is issued, so
      // that no copy waits behind those loads
      Entry g = fg;
      EntryLen ahead{0, 0, 0};
      bool have_ahead = false;
      for (; ok && e < E && off < end; ++e) {
        if (e != e0) {
          g = entry_from(a, hb, e, have_ahead ? ahead : kSmallE ? slens[e] : entry_len(a, hb, e));
          have_ahead = false;
        }
        const uint64_t cost = entry_cost(g);
        const uint64_t cq = row_cost_q(g.kb), cb = row_cost_b(g.kb);
        const FastDiv& dq = a.div_cost_q[g.kb >> 5];
        const FastDiv& dbr = a.div_cost_b[g.kb >> 5];
        const FastDiv& da = a.div_cost_b[kHeadDim >> 5];     // a full-width row costs what a k = 128 row does
        const uint64_t xu = token_units(g);
        const uint64_t off_q = off + (uint64_t)kUnitsA * g.n_a + xu;
        const uint64_t off_b = off_q + cq * g.n_q;
        int a0, a1, q0, q1, b0, b1;
        if (xu == 0) {
          rows_in_range(off, da, g.n_a, start, end, a0, a1);
        } else {
          // full-width rows 0 .. anc, the token's charge, rows anc+1 .. n_a-1
          const int n1 = g.anc + 1;
          int p0, p1, s0, s1;
          rows_in_range(off, da, n1, start, end, p0, p1);
          rows_in_range(off + (uint64_t)kUnitsA * n1 + xu, da, g.n_a - n1, start, end, s0, s1);
          if (p1 > p0) {
            a0 = p0;
            a1 = s1 > s0 ? n1 + s1 : p1;
          } else if (s1 > s0) {
            a0 = n1 + s0;
            a1 = n1 + s1;
          } else {
            a0 = a1 = 0;
          }
        }
        rows_in_range(off_q, dq, g.n_q, start, end, q0, q1);
        rows_in_range(off_b, dbr, g.n_b, start, end, b0, b1);
        // paged bf16 region B: tiles end at page boundaries (a box that starts
        // inside a page is clipped at its end: the page is a block of the
        // view).  Sealed blocks: whole blocks loaded, rows outside the range
        // masked; a stage takes up to qper consecutive blocks (one bulk copy,
        // or one per page), so the producer's and the consumers' per-stage
        // work is paid once per 62-99 KB.
        constexpr bool paged = kPaged;
        constexpr bool bpaged = kPaged && kFmt == kKvBf16;
        const int nta = (a1 - a0 + kTileRows - 1) / kTileRows;
        const int qfirst = q0 / kQBlockRows;
        const int nqb = q1 <= q0 ? 0 : (q1 - 1) / kQBlockRows - qfirst + 1;   // sealed blocks in range
        const int qper = kQPerStage;
        const int ntq = (nqb + qper - 1) / qper;
        const int ntb = b1 <= b0   ? 0
                        : bpaged ? (b1 - 1) / kPageRows - b0 / kPageRows + 1
                                 : (b1 - b0 + kTileRows - 1) / kTileRows;
        const int nt = nta + ntq + ntb;
        if (nt > 0) {
          const EntryId id = entry_id(a, e);
          const int b = id.b;
          const HeadDesc& hd = hb[id.lr * cv.Hkv + id.h];
          const int32_t* pt =
              cv.page_table + (((int64_t)id.l * cv.B + b) * cv.Hkv + id.h) * cv.max_pages;
          const uint64_t last_row_off = g.n_b > 0   ? off_b + cb * (g.n_b - 1)
                                        : g.n_q > 0 ? off_q + cq * (g.n_q - 1)
                                                    : off + (uint64_t)kUnitsA * (g.n_a - 1) +
                                                          (g.n_a - 1 > g.anc ? xu : 0);
          // the entry's first / last owning CTA is read only from the segment's
          // last descriptor: work it out after the first load is in flight
          int fc = -1, lc = -1;
          if (nt == 1) {
            fc = range_owner(off, C, P);
            lc = range_owner(last_row_off, C, P);
          }
          // Fused append: the CTA holding the entry's anchor row -- the window
          // slot the new token replaces, else full-width row 0 -- loads the
          // token (and the row it evicts into the middle) as a region-3 stage
          // right after that row's tile, so the slot is overwritten only
          // after this CTA has read it; no other CTA reads it.
          const int anc = g.anc;
          const int xj = fused_launch && anc >= 0 && anc >= a0 && anc < a1 ? (anc - a0) / kTileRows : -1;
          int32_t pq0 = 0, pq1 = 0, pq2 = 0, pq3 = 0;     // page ids of the next middle-row tiles
          int32_t qpg_ahead[kQPerStage] = {};
          for (int j = 0; j < nt; ++j) {
            const int region = j < nta ? 0 : j < nta + ntq ? 2 : 1;
            const int width = region == 0 ? kHeadDim : g.kb;
            int r, rend, rlo = 0, nq = 0;
            int32_t page = 0;
            int32_t qpg[kQPerStage] = {};
            if (region == 0) {
              r = a0 + j * kTileRows;
              rend = min(a1, r + kTileRows);
            } else if (region == 2) {
              const int blk = qfirst + (j - nta) * qper;
              nq = min(qper, qfirst + nqb - blk);
              r = max(q0, blk * kQBlockRows);
              rend = min(q1, (blk + nq) * kQBlockRows);
              rlo = r - blk * kQBlockRows;
              if (paged) {
                // page ids load one stage ahead (and before the slot wait); a
                // missing page (status already recorded) reads page 0
#pragma unroll
                for (int i = 0; i < kQPerStage; ++i) {
                  if (j == nta && i < nq) qpg_ahead[i] = __ldcg(pt + blk + i);
                  qpg[i] = max(0, qpg_ahead[i]);
                }
                if (j + 1 < nta + ntq) {
                  const int nb = blk + qper, nq2 = min(qper, qfirst + nqb - nb);
#pragma unroll
                  for (int i = 0; i < kQPerStage; ++i)
                    if (i < nq2) qpg_ahead[i] = __ldcg(pt + nb + i);
                }
              } else {
                page = b * hd.qblocks + blk;
              }
            } else if (bpaged) {
              const int jb = j - nta - ntq;           // middle-row tile = page of the range
              const int pg = b0 / kPageRows + jb;
              r = max(b0, pg * kPageRows);
              rend = min(b1, (pg + 1) * kPageRows);
              // page ids load four tiles ahead (a one-tile lead leaves the
              // id's L2 round trip exposed whenever a ring slot is free at
              // once); a missing page (status already recorded) reads page 0
              if (jb == 0) {
                pq0 = __ldcg(pt + pg);
                pq1 = 1 < ntb ? __ldcg(pt + pg + 1) : 0;
                pq2 = 2 < ntb ? __ldcg(pt + pg + 2) : 0;
                pq3 = 3 < ntb ? __ldcg(pt + pg + 3) : 0;
              }
              page = max(0, pq0);
              pq0 = pq1;
              pq1 = pq2;
              pq2 = pq3;
              pq3 = jb + 4 < ntb ? __ldcg(pt + pg + 4) : 0;
            } else {
              r = b0 + (j - nta - ntq) * kTileRows;
              rend = min(b1, r + kTileRows);
            }
            const uint32_t bytes = region == 2 ? (uint32_t)(nq * qblock_bytes(width)) : stage_bytes(region, width);
            uint32_t at = 0;
            if (!reserve(region == 2 ? (bytes + 1023u) & ~1023u : ring_bytes(region, width), at)) {
              ok = false;
              break;
            }
            const uint32_t stage = issued & (kSlots - 1);
            StageDesc d;
            d.e = e;
            d.region = region;
            d.rlo = rlo;
            d.nrows = rend - r;
            d.width = width;
            d.flags = (j == 0 ? kFirst : 0) | (j + 1 == nt && j != xj ? kLast : 0);
            d.first_cta = fc;
            d.last_cta = lc;
            d.koff = at;
            d.mrow = region == 0 && g.mrow >= r && g.mrow < rend ? g.mrow - r : -1;
            d.n = nq;         // region 2: sealed blocks in the stage
            d.cnt = 0;
            desc[stage] = d;
            const uint32_t fb = bar_full + 8 * stage;
            mbar_arrive_expect_tx(fb, bytes);
            const uint32_t kdst = base + SmemLayout::kRingOff + at;
            const uint32_t vdst = kdst + (uint32_t)kTileRows * 2 * width;
            if (region == 0) {
              // a box past the end of the (head, sequence) block takes the
              // class's block view
              const int cls = hd.policy;
              if (r + kTileRows > hd.cap_a && maps.block_rows[kMapAK + cls] != 0) {
                tma_load_4d(kdst, &maps.m[kMapAK + cls], 0, r, hd.blk_a + b, 0, fb, policy);
                tma_load_4d(vdst, &maps.m[kMapAV + cls], 0, r, hd.blk_a + b, 0, fb, policy);
              } else {
                const int32_t row = (int32_t)(hd.row_a + (int64_t)b * hd.cap_a + r);
                tma_load_3d(kdst, &maps.m[kMapFlat + kPoolK128], 0, row, 0, fb, policy);
                tma_load_3d(vdst, &maps.m[kMapFlat + kPoolV], 0, row, 0, fb, policy);
              }
            } else if (region == 2) {
              const uint32_t qb = (uint32_t)qblock_bytes(width);
              if (!paged) {
                // a sequence's blocks are consecutive: one copy for the stage
                bulk_load(kdst, cv.qpool + hd.qoff + (int64_t)page * qb, bytes, fb, policy);
              } else {
#pragma unroll
                for (int i = 0; i < kQPerStage; ++i)
                  if (i < nq) bulk_load(kdst + i * qb, cv.qpool + hd.qoff + (int64_t)qpg[i] * qb, qb, fb, policy);
              }
            } else {
              // block: the sequence's region-B rows, or the page
              const int32_t blk = bpaged ? page : b;
              const int rr = bpaged ? r % kPageRows : r;
              const int pk = hd.pool_kb;
              const bool narrow = pk == kPoolK32 || pk == kPoolK64;     // one part per row
              const int32_t brows = maps.block_rows[kMapB + pk];
              if (brows != 0 && rr + kTileRows > brows) {
                const int32_t kz = hd.kblk_b + blk, vz = hd.vblk_b + blk;
                if (narrow)
                  tma_load_3d(kdst, &maps.m[kMapB + pk], 0, rr, kz, fb, policy);
                else
                  tma_load_4d(kdst, &maps.m[kMapB + pk], 0, rr, kz, 0, fb, policy);
                tma_load_4d(vdst, &maps.m[kMapB + kPoolV], 0, rr, vz, 0, fb, policy);
              } else {
                const int64_t rb = bpaged ? (int64_t)page * kPageRows + rr : (int64_t)b * hd.cap_b + r;
                const int32_t krow = (int32_t)(hd.krow_b + rb);
                const int32_t vrow = (int32_t)(hd.vrow_b + rb);
                if (narrow)
                  tma_load_2d(kdst, &maps.m[kMapFlat + pk], 0, krow, fb, policy);
                else
                  tma_load_3d(kdst, &maps.m[kMapFlat + pk], 0, krow, 0, fb, policy);
                tma_load_3d(vdst, &maps.m[kMapFlat + kPoolV], 0, vrow, 0, fb, policy);
              }
            }
            ++issued;
            if (j == 0 && e + 1 < E) {
              ahead = kSmallE ? slens[e + 1] : entry_len(a, hb, e + 1);
              have_ahead = true;
              if (paged) {
                // the next entry's page ids into L2
                const EntryId nid = entry_id(a, e + 1);
                asm volatile("prefetch.global.L2 [%0];" ::"l"(
                    cv.page_table + (((int64_t)nid.l * cv.B + nid.b) * cv.Hkv + nid.h) * cv.max_pages));
              }
            }
            if (fc < 0) {
              fc = range_owner(off, C, P);
              lc = range_owner(last_row_off, C, P);
            }
            if (j == xj) {
              const bool evict = hd.policy == kFull && g.kb > 0 && g.mrow >= 0;
              const uint32_t xbytes = stage_bytes(3, evict ? g.kb : 0);
              if (!reserve(ring_bytes(3, evict ? g.kb : 0), at)) {
                ok = false;
                break;
              }
              const uint32_t xs = issued & (kSlots - 1);
              StageDesc x;
              x.e = e;
              x.region = 3;
              x.rlo = x.nrows = 0;
              x.width = evict ? g.kb : 0;
              x.flags = j + 1 == nt ? kLast : 0;
              x.first_cta = fc;
              x.last_cta = lc;
              x.koff = at;
              x.mrow = hd.policy != kSpecial ? kTokAlways
                                             : kTokSpecialHead | (g.len.cnt < hd.cap_a ? kTokRoom : 0);
              x.n = g.len.n;
              x.cnt = g.len.cnt;
              desc[xs] = x;
              const uint32_t xb = bar_full + 8 * xs;
              mbar_arrive_expect_tx(xb, xbytes);
              const uint32_t dst = base + SmemLayout::kRingOff + at;
              const size_t src = (((size_t)id.lr * cv.B + b) * cv.Hkv + id.h) * kHeadDim;
              bulk_load(dst, a.k_new + src, kHeadDim * 2, xb, policy);
              bulk_load(dst + kHeadDim * 2, a.v_new + src, kHeadDim * 2, xb, policy);
              if (evict) {
                const int64_t srow = hd.row_a + (int64_t)b * hd.cap_a + g.mrow;
                bulk_load(dst + 2 * kHeadDim * 2, cv.pool[kPoolK128] + srow * kHeadDim, kHeadDim * 2, xb, policy);
                bulk_load(dst + 3 * kHeadDim * 2, cv.pool[kPoolV] + srow * kHeadDim, kHeadDim * 2, xb, policy);
                bulk_load(dst + 4 * kHeadDim * 2, cv.kept + ((size_t)id.l * cv.Hkv + id.h) * kHeadDim, kHeadDim * 2,
                          xb, policy);
              }
              ++issued;
            }
          }
        }
        off += cost;
      }
      // end of stream: a descriptor with e < 0 in the next slot
      if (ok && issued - freed == (uint32_t)kSlots) ok = free_oldest();
      if (ok) {
        const uint32_t stage = issued & (kSlots - 1);
        desc[stage].e = -1;
        mbar_arrive(bar_full + 8 * stage);
      } else {
        record_status(a, kStatusTimeout);
      }
      // Keep the CTA alive until every copy this thread issued has landed
      // (its full barrier completed), so no copy can write shared memory
      // after the consumers left on a timed-out wait.  Normally these waits
      // return at once or overlap the consumers' last tiles.
      for (uint32_t m = freed; m != issued; ++m)
        if (!mbar_wait_bounded(bar_full + 8 * (m & (kSlots - 1)), (m / kSlots) & 1u, kDrainLimitNs)) {
          record_status(a, kStatusTimeout);
          break;
        }
    }
    return;
  }

  // ================================================================ consumers
  const int ct = tid;                       // 0 .. 255
  const uint32_t cbar = base + SmemLayout::kCBarOff;
  uint32_t cphase = 0;
  const int gid = lane >> 2, tig = lane & 3;
  const int rk = (lane & 7) + ((lane >> 3) & 1) * 8;    // ldmatrix row of the K (A) operand
  const int ck = lane >> 4;                              // +0 / +1 chunk
  const int rv = (lane & 7) + (lane >> 4) * 8;          // ldmatrix.trans row of the V^T operand
  const int cvh = (lane >> 3) & 1;
  const float NEG_INF = -INFINITY;
  uint16_t* qa_s = reinterpret_cast<uint16_t*>(sm + SmemLayout::kQOff);
  uint16_t* qb_s = reinterpret_cast<uint16_t*>(sm + SmemLayout::kQKOff);
  // ldmatrix address of the q B-fragments: heads (lane & 7), 8-channel
  // column (lane >> 3) of a 32-channel group
  const uint32_t qa_lane = base + SmemLayout::kQOff + (uint32_t)((lane & 7) * kQStride + 8 * (lane >> 3)) * 2;
  const uint32_t qb_lane = base + SmemLayout::kQKOff + (uint32_t)((lane & 7) * kQStride + 8 * (lane >> 3)) * 2;

  // ---- fused append (bf16 caches, a.k_new set).  Entries with resident rows
  // take the token through a region-3 stage (below); entries without any
  // take it here, through global memory.  The last CTA of the grid advances
  // the lengths.  Scratch `ex` lives in the q staging area, free before the
  // first entry's q is staged.
  const bool fused = !kQ8 && a.k_new != nullptr;
  float* ex = reinterpret_cast<float*>(sm + SmemLayout::kQOff);
  constexpr int kExS = 0, kExE = kMaxGroup, kExVn = 2 * kMaxGroup, kExVe = kExVn + kHeadDim;
  static_assert(kExVe + kHeadDim <= kMaxGroup * kQStride / 2, "fused scratch fits the q area");
  // The tokens the append adds to entry e: the new token (all channels;
  // SPECIAL heads take it only if its id is special) and, when a FULL window
  // with kept channels is full, the token n - W leaving it for the middle
  // (kept channels, read from its window row before the edit replaces it).
  // Scores in log2 units (-inf: absent) and V rows as fp32 into ex.  All
  // consumer threads; callers sync before reading ex.
  auto fused_extras = [&](int e) {
    const EntryId id = entry_id(a, e);
    const HeadDesc& hd = hb[id.lr * cv.Hkv + id.h];
    const EntryLen len = kSmallE ? slens[e] : entry_len(a, hb, e);
    const bool add_new = len.act && (hd.policy != kSpecial || (token_special(a, id.b) && len.cnt < hd.cap_a));
    const bool add_ev = len.act && hd.policy == kFull && hd.n_kept > 0 && len.n >= cv.S + cv.W;
    const int64_t slot =
        hd.row_a + (int64_t)id.b * hd.cap_a + (add_ev ? cv.S + (int)fmod((uint32_t)(len.n - cv.S), a.div_w) : 0);
    const size_t src = (((size_t)id.lr * cv.B + id.b) * cv.Hkv + id.h) * kHeadDim;
    if (warp < G) {
      const uint16_t* qg = a.q + (((size_t)id.lr * cv.B + id.b) * cv.Hq + (size_t)id.h * G + warp) * kHeadDim;
      float sn = 0.f, se = 0.f;
      if (add_new) {
        const uint2 qw = reinterpret_cast<const uint2*>(qg)[lane];
        const uint2 kw = reinterpret_cast<const uint2*>(a.k_new + src)[lane];
        sn = bf16_lo(qw.x) * bf16_lo(kw.x) + bf16_hi(qw.x) * bf16_hi(kw.x) + bf16_lo(qw.y) * bf16_lo(kw.y) +
             bf16_hi(qw.y) * bf16_hi(kw.y);
      }
      if (add_ev) {
        const int16_t* kept = cv.kept + ((size_t)id.l * cv.Hkv + id.h) * kHeadDim;
        const uint16_t* k_old = cv.pool[kPoolK128] + slot * kHeadDim;
        for (int c = lane; c < hd.n_kept; c += 32) {
          const int ch = kept[c];
          se += bf16_to_f32(qg[ch]) * bf16_to_f32(k_old[ch]);
        }
      }
#pragma unroll
      for (int sh = 16; sh > 0; sh >>= 1) {
        sn += __shfl_xor_sync(0xffffffffu, sn, sh);
        se += __shfl_xor_sync(0xffffffffu, se, sh);
      }
      if (lane == 0) {
        ex[kExS + warp] = add_new ? sn * a.scale_log2 : NEG_INF;
        ex[kExE + warp] = add_ev ? se * a.scale_log2 : NEG_INF;
      }
    }
    if (ct < 64) {
      const int c4 = ct & 31;
      const bool on = ct < 32 ? add_new : add_ev;
      const uint2 w = !on ? make_uint2(0u, 0u)
                      : ct < 32 ? reinterpret_cast<const uint2*>(a.v_new + src)[c4]
                                : row8(cv.pool[kPoolV], slot)[c4];
      *reinterpret_cast<float4*>(&ex[(ct < 32 ? kExVn : kExVe) + 4 * c4]) =
          make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
    }
  };
  // The cache edit of entry e (one warp): the append of the token, after
  // fused_extras and a consumer barrier.
  auto fused_edit = [&](int e) {
    const EntryId id = entry_id(a, e);
    const EntryLen len = kSmallE ? slens[e] : entry_len(a, hb, e);
    if (!len.act) return;
    const size_t src = (((size_t)id.lr * cv.B + id.b) * cv.Hkv + id.h) * kHeadDim;
    append_head<false>(cv, id.l, id.b, id.h, len.n, len.cnt, token_special(a, id.b), a.k_new + src,
                       a.v_new + src, lane);
  };

  const int nlb = a.nlayers * cv.B;
  // next lengths of (layer, sequence) i, and whether its active sequence's
  // token id is outside [0, vocab) (then it counts as not special)
  auto next_len = [&](int i, int& lb, int& n1, int& c1, bool& bad) {
    const int b = i % cv.B;
    lb = (a.layer + i / cv.B) * cv.B + b;
    // independent loads first: one round trip (two with token ids)
    const int act = __ldcg(&cv.active[b]);
    const int n = __ldcg(&cv.len[lb]);
    const int c = __ldcg(&cv.cnt[lb]);
    const int id = a.ids != nullptr ? a.ids[b] : 0;
    const bool in_vocab = id >= 0 && id < cv.vocab;
    const bool sp = a.ids != nullptr && in_vocab && cv.is_special[id] != 0;
    n1 = act != 0 && n < cv.capacity ? n + 1 : -1;
    c1 = n1 > 0 && sp && c < cv.spec_cap ? c + 1 : -1;
    bad = a.ids != nullptr && act != 0 && !in_vocab;
  };

  // entries with no resident token, by CTA (e mod grid): o = 0, or with a
  // fused append the new token alone
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    if (entry_cost(entry_from(a, hb, e, kSmallE ? slens[e] : entry_len(a, hb, e))) != 0) continue;
    const EntryId id = entry_id(a, e);
    float* dst = a.o + (((size_t)id.lr * cv.B + id.b) * cv.Hq + (size_t)id.h * G) * kHeadDim;
    if (fused) {
      fused_extras(e);
      consumer_sync(cbar, cphase, a);
      for (int i = ct; i < G * kHeadDim; i += kConsumerWarps * 32) {
        const int g = i >> 7, c = i & (kHeadDim - 1);
        const float sn = ex[kExS + g], se = ex[kExE + g];
        const float M = fmaxf(sn, se);
        float out = 0.f;
        if (M != NEG_INF) {
          const float fn = sn == NEG_INF ? 0.f : exp2f(sn - M), fe = se == NEG_INF ? 0.f : exp2f(se - M);
          out = (fn * ex[kExVn + c] + fe * ex[kExVe + c]) / (fn + fe);
        }
        dst[i] = out;
      }
      if (warp == kConsumerWarps - 1) fused_edit(e);
      consumer_sync(cbar, cphase, a);
    } else {
      for (int i = ct; i < G * kHeadDim; i += kConsumerWarps * 32) dst[i] = 0.f;
    }
  }

  // Early length advance (fused launches of at most 32 entries): once every
  // warp of this CTA is past its split (the split-done barrier), nothing in
  // the CTA reads the lengths from memory again, so the CTA is counted; the
  // CTA that completes the count advances them, as the append kernel does
  // per sequence.  The last consumer warp does it while the first tiles are
  // in flight.  The barrier waits its fixed bound whatever the configured
  // limit: on time-out the status is set and the lengths stay.
  if (early_len && warp == kConsumerWarps - 1) {
    if (!mbar_wait_bounded(sbar, 0u, kDrainLimitNs)) {
      if (lane == 0) record_status(a, kStatusTimeout);
    } else {
      int last = 0;
      if (lane == 0) last = atomicAdd(&a.counters[E], 1) == (int)gridDim.x - 1 ? 1 : 0;
      if (__shfl_sync(0xffffffffu, last, 0)) {
        for (int i = lane; i < nlb; i += 32) {
          int lb, n1, c1;
          bool bad;
          next_len(i, lb, n1, c1, bad);
          if (n1 > 0) cv.len[lb] = n1;
          if (c1 > 0) cv.cnt[lb] = c1;
          if (bad) set_status(cv, kStatusBadId);
        }
        __syncwarp();
        if (lane == 0) a.counters[E] = 0;
      }
    }
  }

  float o[8][4];
  float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
  // INT8 tiles accumulate V codes as 1152 + code: o carries 1152 * sum(P')
  // per head column, removed at the segment end (c0, c1: this lane's share)
  float c0 = 0.f, c1 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  // q of entry e into shared memory: all channels (full-width rows) and the
  // kept channels in kept order (middle rows); the B operand of S^T = K Q^T
  // is read from there with ldmatrix.  Callers separate it from readers of
  // the previous q with a consumer barrier.
  auto stage_q = [&](int e) {
    const EntryId id = entry_id(a, e);
    const HeadDesc& hd = hb[id.lr * cv.Hkv + id.h];
    const int16_t* kept = cv.kept + ((size_t)id.l * cv.Hkv + id.h) * kHeadDim;
    const int kk = hd.policy == kFull ? hd.n_kept : 0;
    const uint16_t* qg = a.q + (((size_t)id.lr * cv.B + id.b) * cv.Hq + (size_t)id.h * G) * kHeadDim;
    for (int i = ct; i < kMaxGroup * kHeadDim; i += kConsumerWarps * 32) {
      const int g = i >> 7, c = i & (kHeadDim - 1);
      uint16_t va = 0, vb = 0;
      if (g < G) {
        va = qg[g * kHeadDim + c];
        if (c < kk) vb = qg[g * kHeadDim + kept[c]];
      }
      qa_s[g * kQStride + c] = va;
      qb_s[g * kQStride + c] = vb;
    }
  };
  auto prefetch_q = [&](int e) {
    const EntryId id = entry_id(a, e);
    if (ct < G * 2) {       // G rows of 256 B: two 128-byte lines each
      const uint16_t* qg = a.q + (((size_t)id.lr * cv.B + id.b) * cv.Hq + (size_t)id.h * G) * kHeadDim;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(qg + ct * 64));
    } else if (ct < G * 2 + 2) {
      const int16_t* kept = cv.kept + ((size_t)id.l * cv.Hkv + id.h) * kHeadDim;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(kept + (ct - G * 2) * 64));
    }
  };
  // the first entry's q loads while the first tile is in flight
  int q_entry = first_e;
  if (q_entry < E) stage_q(q_entry);

  // this warp's 16 rows of every tile
  const int r0 = 16 * warp;

  // A stage of NB sealed INT8 / FP8 blocks (valid rows d.rlo .. d.rlo +
  // d.nrows - 1 counted from the first block's row 0: blocks at a segment's
  // ends are shared with another CTA).  The warp takes its 16 rows of every
  // block at once: the blocks' score and P.V chains are independent until
  // one softmax step joins them, so the warp keeps NB mma chains in flight.
  //   S^T = K_codes (f16, exact) . Q'^T, Q' = q[kept] * (K scale of the
  //   channel in the block), split into f16 hi + lo;
  //   O^T += V_codes^T (f16, exact) . P'^T, P' = p * (V scale of the token),
  //   split into f16 hi + lo.
  auto qstage = [&](auto nbc, const StageDesc& d) {
    constexpr int NB = decltype(nbc)::value;
    const int kb = d.width;
    const uint32_t qbytes = (uint32_t)qblock_bytes(kb);
    const uint32_t sbase = base + SmemLayout::kRingOff + d.koff;
    const uint8_t* sptr = sm + SmemLayout::kRingOff + d.koff;
    const int t0 = r0 + gid;
    bool va[NB], vb[NB];
    bool any = false;     // warp-uniform: one of the warp's rows is valid
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int rlo = d.rlo - j * kQBlockRows, rhi = d.rlo + d.nrows - j * kQBlockRows;
      va[j] = t0 >= rlo && t0 < rhi;
      vb[j] = t0 + 8 >= rlo && t0 + 8 < rhi;
      any = any || max(r0, rlo) < min(r0 + 16, rhi);
    }
    if (!any) return;
    // two independent accumulators per block halve the mma dependency chain
    float sc[NB][4], sd[NB][4];
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[j][i] = sd[j][i] = 0.f;
    const int krow = r0 + rk;
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      if (2 * kp < (kb >> 4)) {
        uint32_t qv[4];
        ldsm_x4(qb_lane + 64u * kp, qv[0], qv[1], qv[2], qv[3]);
        const uint32_t krow_off = (uint32_t)(krow * kb + 16 * ((2 * kp + ck) ^ qswz(kb, krow)));
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          const float* ksc = reinterpret_cast<const float*>(sptr + j * qbytes + qblock_ksoff(kb));
          uint32_t bh[2][2], bl[2][2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = 16 * (2 * kp + u) + 2 * tig;
            const float2 s01 = *reinterpret_cast<const float2*>(&ksc[c]);
            const float2 s89 = *reinterpret_cast<const float2*>(&ksc[c + 8]);
            const float q0 = bf16_lo(qv[2 * u]) * s01.x, q1 = bf16_hi(qv[2 * u]) * s01.y;
            const float q8 = bf16_lo(qv[2 * u + 1]) * s89.x, q9 = bf16_hi(qv[2 * u + 1]) * s89.y;
            bh[u][0] = pack_f16x2(q0, q1);
            bh[u][1] = pack_f16x2(q8, q9);
            bl[u][0] = pack_f16x2(q0 - f16_lo(bh[u][0]), q1 - f16_hi(bh[u][0]));
            bl[u][1] = pack_f16x2(q8 - f16_lo(bh[u][1]), q9 - f16_hi(bh[u][1]));
          }
          uint32_t w0, w1, w2, w3;
          ldsm_x4(sbase + j * qbytes + krow_off, w0, w1, w2, w3);
          uint32_t f0, f1, f2, f3;
          codes_to_f16x2<kFmt>(w0, f0, f2);       // rows gid: k 2tig.. / 2tig+8..
          codes_to_f16x2<kFmt>(w1, f1, f3);       // rows gid + 8
          mma_f16_16816(sc[j], f0, f1, f2, f3, bh[0][0], bh[0][1]);
          mma_f16_16816(sd[j], f0, f1, f2, f3, bl[0][0], bl[0][1]);
          codes_to_f16x2<kFmt>(w2, f0, f2);
          codes_to_f16x2<kFmt>(w3, f1, f3);
          mma_f16_16816(sc[j], f0, f1, f2, f3, bh[1][0], bh[1][1]);
          mma_f16_16816(sd[j], f0, f1, f2, f3, bl[1][0], bl[1][1]);
        }
      }
    }
    float x[NB][4], p[NB][4];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      x[j][0] = va[j] ? (sc[j][0] + sd[j][0]) * a.scale_log2 : NEG_INF;
      x[j][1] = va[j] ? (sc[j][1] + sd[j][1]) * a.scale_log2 : NEG_INF;
      x[j][2] = vb[j] ? (sc[j][2] + sd[j][2]) * a.scale_log2 : NEG_INF;
      x[j][3] = vb[j] ? (sc[j][3] + sd[j][3]) * a.scale_log2 : NEG_INF;
    }
    online_softmax<NB>(x, p, m0, m1, l0, l1, c0, c1, o);
    uint32_t ph[NB][2], pr[NB][2];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const float* vsc = reinterpret_cast<const float*>(sptr + j * qbytes + qblock_vsoff(kb));
      const float sv0 = vsc[t0], sv1 = vsc[t0 + 8];
      const float q0 = p[j][0] * sv0, q1 = p[j][1] * sv0, q2 = p[j][2] * sv1, q3 = p[j][3] * sv1;
      if (kFmt == kKvInt8) {
        c0 += q0 + q2;
        c1 += q1 + q3;
      }
      const uint32_t h01 = pack_f16x2(q0, q1), h23 = pack_f16x2(q2, q3);
      const uint32_t r01 = pack_f16x2(q0 - f16_lo(h01), q1 - f16_hi(h01));
      const uint32_t r23 = pack_f16x2(q2 - f16_lo(h23), q3 - f16_hi(h23));
      ph[j][0] = movmatrix_trans(h01);
      ph[j][1] = movmatrix_trans(h23);
      pr[j][0] = movmatrix_trans(r01);
      pr[j][1] = movmatrix_trans(r23);
    }
#pragma unroll
    for (int i2 = 0; i2 < 4; ++i2) {
      const uint32_t vrow_off =
          (uint32_t)(qblock_voff(kb) + krow * kHeadDim + 16 * ((2 * i2 + ck) ^ (krow & 7)));
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        uint32_t w0, w1, w2, w3;
        ldsm_x4_trans(sbase + j * qbytes + vrow_off, w0, w1, w2, w3);
        uint32_t f0, f1, f2, f3;
        vcodes_to_f16x2<kFmt>(w0, f0, f1);  // tokens 2tig.. of rows 0-7: channels gid / gid + 8
        vcodes_to_f16x2<kFmt>(w1, f2, f3);  // tokens 2tig + 8..
        mma_f16_16816(o[2 * i2], f0, f1, f2, f3, ph[j][0], ph[j][1]);
        mma_f16_16816(o[2 * i2], f0, f1, f2, f3, pr[j][0], pr[j][1]);
        vcodes_to_f16x2<kFmt>(w2, f0, f1);
        vcodes_to_f16x2<kFmt>(w3, f2, f3);
        mma_f16_16816(o[2 * i2 + 1], f0, f1, f2, f3, ph[j][0], ph[j][1]);
        mma_f16_16816(o[2 * i2 + 1], f0, f1, f2, f3, pr[j][0], pr[j][1]);
      }
    }
  };

  int stage = 0;
  uint32_t phase = 0;
  while (true) {
    if (!mbar_wait_bounded(bar_full + 8 * stage, phase, a.wait_limit_ns)) {
      if (lane == 0) record_status(a, kStatusTimeout);
      break;
    }
    const StageDesc d = desc[stage];
    if (d.e < 0) break;
    if (d.flags & kFirst) {
      // q of the entry into shared memory (staged ahead for the CTA's first
      // entry); the next entry's q and kept list head for L2 meanwhile
      if (d.e != q_entry) stage_q(d.e);
      if (d.e + 1 < E) prefetch_q(d.e + 1);
      q_entry = -1;
      consumer_sync(cbar, cphase, a);
      m0 = m1 = NEG_INF;
      l0 = l1 = c0 = c1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }

    // A stage of sealed blocks holds d.n (1-3) consecutive blocks of the
    // entry; any other stage is one tile.
    if (kQ8 && d.region == 2) {
      if (d.n == 3)
        qstage(std::integral_constant<int, 3>(), d);
      else if (d.n == 2)
        qstage(std::integral_constant<int, 2>(), d);
      else
        qstage(std::integral_constant<int, 1>(), d);
    } else {
    // valid rows rlo .. rhi - 1 of the tile except mrow; the warp works if
    // one of its 16 rows is valid (a block of masked rows would leave the
    // running max at -inf)
    const int rlo = max(0, d.rlo), rhi = min(kTileRows, d.rlo + d.nrows);
    const uint32_t kbase = base + SmemLayout::kRingOff + d.koff;
    const int wlo = max(r0, rlo), whi = min(r0 + 16, rhi);
    if (whi - wlo - (d.mrow >= wlo && d.mrow < whi ? 1 : 0) > 0) {
      // two independent accumulators halve the mma dependency chain
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
      const bool fam128 = (d.width & 63) == 0;          // widths 64 / 128 use 128-byte rows
      const int nks = d.width >> 4;
      const uint32_t q_lane = d.region == 0 ? qa_lane : qb_lane;
      const int row = r0 + rk;
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        if (2 * kp < nks) {
          uint32_t qv[4];
          ldsm_x4(q_lane + 64u * kp, qv[0], qv[1], qv[2], qv[3]);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = 2 * (2 * kp + u) + ck;
            const uint32_t addr = fam128 ? tile_addr128(kbase, row, c) : tile_addr64(kbase, row, c);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(addr, a0, a1, a2, a3);
            if (u == 0)
              mma_bf16_16816(sc, a0, a1, a2, a3, qv[0], qv[1]);
            else
              mma_bf16_16816(sd, a0, a1, a2, a3, qv[2], qv[3]);
          }
        }
      }
      const int t0 = r0 + gid;
      const bool v0 = t0 >= rlo && t0 < rhi && t0 != d.mrow;
      const bool v1 = t0 + 8 >= rlo && t0 + 8 < rhi && t0 + 8 != d.mrow;
      const float x[1][4] = {{v0 ? (sc[0] + sd[0]) * a.scale_log2 : NEG_INF,
                              v0 ? (sc[1] + sd[1]) * a.scale_log2 : NEG_INF,
                              v1 ? (sc[2] + sd[2]) * a.scale_log2 : NEG_INF,
                              v1 ? (sc[3] + sd[3]) * a.scale_log2 : NEG_INF}};
      float p[1][4];
      online_softmax<1>(x, p, m0, m1, l0, l1, c0, c1, o);
      // P as a bf16 pair hi + lo (two mmas): P.V keeps ~16 mantissa bits
      const uint32_t vbase = kbase + (uint32_t)kTileRows * 2 * d.width;
      const uint32_t h01 = pack_bf16x2(p[0][0], p[0][1]), h23 = pack_bf16x2(p[0][2], p[0][3]);
      const uint32_t r01 = pack_bf16x2(p[0][0] - bf16_lo(h01), p[0][1] - bf16_hi(h01));
      const uint32_t r23 = pack_bf16x2(p[0][2] - bf16_lo(h23), p[0][3] - bf16_hi(h23));
      // S^T accumulator rows (tokens) -> B operand rows (k = tokens) of P^T
      const uint32_t ph0 = movmatrix_trans(h01), ph1 = movmatrix_trans(h23);
      const uint32_t pr0 = movmatrix_trans(r01), pr1 = movmatrix_trans(r23);
      const int vrow = r0 + rv;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(tile_addr128(vbase, vrow, 2 * i + cvh), a0, a1, a2, a3);
        mma_bf16_16816(o[i], a0, a1, a2, a3, ph0, ph1);
        mma_bf16_16816(o[i], a0, a1, a2, a3, pr0, pr1);
      }
    }
    }   // tile stage
    if (!kQ8 && d.region == 3) {
      // ---- fused append: the new token (and the window row it evicts into
      // the middle, scored on the kept channels) join warp 0's running
      // softmax of this segment; the last warp writes them into the cache
      // from the staged copies.  The descriptor carries what decides this
      // (mrow: kTok* flags; width: kept channels of an
      // evicted row, else 0), so warp 0 reads nothing but shared memory
      // unless the head is SPECIAL.
      const uint16_t* kn = reinterpret_cast<const uint16_t*>(sm + SmemLayout::kRingOff + d.koff);
      const uint16_t* vn = kn + kHeadDim;
      const uint16_t* ko = kn + 2 * kHeadDim;
      const uint16_t* vo = kn + 3 * kHeadDim;
      const int16_t* kl = reinterpret_cast<const int16_t*>(kn + 4 * kHeadDim);
      const EntryId id = entry_id(a, d.e);
      const bool special = (d.mrow & kTokSpecialHead) != 0 && token_special(a, id.b);
      const bool add_new = (d.mrow & kTokAlways) != 0 || (special && (d.mrow & kTokRoom) != 0);
      const int kk = d.width;
      const bool add_ev = kk != 0;
      if (warp == 0 && (add_new || add_ev)) {
        // the evicted row's kept channels as a 128-bit mask
        uint32_t km[4] = {0u, 0u, 0u, 0u};
        if (add_ev) {
          for (int c = lane; c < kk; c += 32) {
            const int ch = kl[c];
#pragma unroll
            for (int w = 0; w < 4; ++w) km[w] |= (ch >> 5) == w ? 1u << (ch & 31) : 0u;
          }
#pragma unroll
          for (int w = 0; w < 4; ++w) km[w] = __reduce_or_sync(0xffffffffu, km[w]);
        }
        // lane = 4 g + part: head g on channels 32 part .. 32 part + 31
        const int gq = lane >> 2, part = lane & 3;
        const uint32_t kmask = part == 0 ? km[0] : part == 1 ? km[1] : part == 2 ? km[2] : km[3];
        const uint16_t* qr = qa_s + gq * kQStride + 32 * part;
        float sn = 0.f, se = 0.f;
#pragma unroll 1
        for (int j = 0; j < 32; j += 8) {
          const uint4 qv = *reinterpret_cast<const uint4*>(qr + j);
          const uint4 nv = *reinterpret_cast<const uint4*>(kn + 32 * part + j);
          const uint4 ov = *reinterpret_cast<const uint4*>(ko + 32 * part + j);
          const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, nw[4] = {nv.x, nv.y, nv.z, nv.w};
          const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float q0 = bf16_lo(qw[t]), q1 = bf16_hi(qw[t]);
            sn += q0 * bf16_lo(nw[t]) + q1 * bf16_hi(nw[t]);
            const uint32_t bits = kmask >> (j + 2 * t);
            se += ((bits & 1u) ? q0 * bf16_lo(ow[t]) : 0.f) + ((bits & 2u) ? q1 * bf16_hi(ow[t]) : 0.f);
          }
        }
        sn += __shfl_xor_sync(0xffffffffu, sn, 1);
        se += __shfl_xor_sync(0xffffffffu, se, 1);
        sn += __shfl_xor_sync(0xffffffffu, sn, 2);
        se += __shfl_xor_sync(0xffffffffu, se, 2);
        // this lane's head columns 2 tig, 2 tig + 1 sit in lanes 8 tig, 8 tig + 4
        float xn0 = __shfl_sync(0xffffffffu, sn, 8 * tig), xn1 = __shfl_sync(0xffffffffu, sn, 8 * tig + 4);
        float xe0 = __shfl_sync(0xffffffffu, se, 8 * tig), xe1 = __shfl_sync(0xffffffffu, se, 8 * tig + 4);
        xn0 = add_new ? xn0 * a.scale_log2 : NEG_INF;
        xn1 = add_new ? xn1 * a.scale_log2 : NEG_INF;
        xe0 = add_ev ? xe0 * a.scale_log2 : NEG_INF;
        xe1 = add_ev ? xe1 * a.scale_log2 : NEG_INF;
        const float mn0 = fmaxf(m0, fmaxf(xn0, xe0)), mn1 = fmaxf(m1, fmaxf(xn1, xe1));
        const float al0 = mn0 > m0 ? (m0 == NEG_INF ? 0.f : exp2f(m0 - mn0)) : 1.f;
        const float al1 = mn1 > m1 ? (m1 == NEG_INF ? 0.f : exp2f(m1 - mn1)) : 1.f;
        m0 = mn0;
        m1 = mn1;
        const float pn0 = xn0 == NEG_INF ? 0.f : exp2f(xn0 - m0), pe0 = xe0 == NEG_INF ? 0.f : exp2f(xe0 - m0);
        const float pn1 = xn1 == NEG_INF ? 0.f : exp2f(xn1 - m1), pe1 = xe1 == NEG_INF ? 0.f : exp2f(xe1 - m1);
        // l is summed over the gid lanes at the segment end: count p once
        l0 = l0 * al0 + (gid == 0 ? pn0 + pe0 : 0.f);
        l1 = l1 * al1 + (gid == 0 ? pn1 + pe1 : 0.f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float vna = bf16_to_f32(vn[16 * i + gid]), vnb = bf16_to_f32(vn[16 * i + gid + 8]);
          const float voa = add_ev ? bf16_to_f32(vo[16 * i + gid]) : 0.f;
          const float vob = add_ev ? bf16_to_f32(vo[16 * i + gid + 8]) : 0.f;
          o[i][0] = o[i][0] * al0 + pn0 * vna + pe0 * voa;
          o[i][1] = o[i][1] * al1 + pn1 * vna + pe1 * voa;
          o[i][2] = o[i][2] * al0 + pn0 * vnb + pe0 * vob;
          o[i][3] = o[i][3] * al1 + pn1 * vnb + pe1 * vob;
        }
      }
      if (warp == kConsumerWarps - 1)
        append_head<false>(cv, id.l, id.b, id.h, d.n, d.cnt, special, kn, vn, lane, add_ev ? ko : nullptr,
                           add_ev ? vo : nullptr, add_ev ? kl : nullptr);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * stage);

    if (d.flags & kLast) {
      if (kFmt == kKvInt8) {
        // remove the 1152 bias of the INT8 V codes: o -= 1152 * sum(P')
        float s0 = c0, s1 = c1;
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
          s0 += __shfl_xor_sync(0xffffffffu, s0, sh);
          s1 += __shfl_xor_sync(0xffffffffu, s1, sh);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          o[i][0] = fmaf(-1152.f, s0, o[i][0]);
          o[i][1] = fmaf(-1152.f, s1, o[i][1]);
          o[i][2] = fmaf(-1152.f, s0, o[i][2]);
          o[i][3] = fmaf(-1152.f, s1, o[i][3]);
        }
      }
      // ---- merge the warps' (o, m, l) of this segment through shared
      // memory slots of hs head rows.  G <= 4: every warp publishes its own
      // slot (eight slots of four heads) and one barrier precedes the CTA
      // merge.  Otherwise warps 4..7 hand theirs to warps 0..3 first (four
      // slots of eight heads), which merge and publish.
      float lr0 = l0, lr1 = l1;
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        lr0 += __shfl_xor_sync(0xffffffffu, lr0, sh);
        lr1 += __shfl_xor_sync(0xffffffffu, lr1, sh);
      }
      const bool one_pass = G <= 4;
      const int hs = one_pass ? 4 : kMaxGroup;
      auto publish = [&](int slotw) {
        if (2 * tig < hs) {       // this lane's head columns 2tig, 2tig+1 exist in the slot
          float* ob = merge_o + slotw * hs * kHeadDim;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            ob[(2 * tig) * kHeadDim + 16 * i + gid] = o[i][0];
            ob[(2 * tig + 1) * kHeadDim + 16 * i + gid] = o[i][1];
            ob[(2 * tig) * kHeadDim + 16 * i + gid + 8] = o[i][2];
            ob[(2 * tig + 1) * kHeadDim + 16 * i + gid + 8] = o[i][3];
          }
          if (gid == 0) {
            merge_m[slotw * hs + 2 * tig] = m0;
            merge_m[slotw * hs + 2 * tig + 1] = m1;
            merge_l[slotw * hs + 2 * tig] = lr0;
            merge_l[slotw * hs + 2 * tig + 1] = lr1;
          }
        }
      };
      if (one_pass) {
        publish(warp);
      } else {
        const int slotw = warp & (kMergeSlots - 1);
        const float* ob = merge_o + slotw * kMaxGroup * kHeadDim;
        if (warp >= kMergeSlots) publish(slotw);
        consumer_sync(cbar, cphase, a);
        if (warp < kMergeSlots) {
          const float mo0 = merge_m[slotw * kMaxGroup + 2 * tig], mo1 = merge_m[slotw * kMaxGroup + 2 * tig + 1];
          const float lo0 = merge_l[slotw * kMaxGroup + 2 * tig], lo1 = merge_l[slotw * kMaxGroup + 2 * tig + 1];
          const float mn0 = fmaxf(m0, mo0), mn1 = fmaxf(m1, mo1);
          const float fa0 = m0 == NEG_INF ? 0.f : exp2f(m0 - mn0), fb0 = mo0 == NEG_INF ? 0.f : exp2f(mo0 - mn0);
          const float fa1 = m1 == NEG_INF ? 0.f : exp2f(m1 - mn1), fb1 = mo1 == NEG_INF ? 0.f : exp2f(mo1 - mn1);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[i][0] = o[i][0] * fa0 + ob[(2 * tig) * kHeadDim + 16 * i + gid] * fb0;
            o[i][1] = o[i][1] * fa1 + ob[(2 * tig + 1) * kHeadDim + 16 * i + gid] * fb1;
            o[i][2] = o[i][2] * fa0 + ob[(2 * tig) * kHeadDim + 16 * i + gid + 8] * fb0;
            o[i][3] = o[i][3] * fa1 + ob[(2 * tig + 1) * kHeadDim + 16 * i + gid + 8] * fb1;
          }
          lr0 = lr0 * fa0 + lo0 * fb0;
          lr1 = lr1 * fa1 + lo1 * fb1;
          m0 = mn0;
          m1 = mn1;
        }
        // warp w < 4 overwrites only slot w, which only it read: a warp-level
        // barrier separates its lanes' reads from the writes
        __syncwarp();
        if (warp < kMergeSlots) publish(slotw);
      }
      // the segment's state now lives in the merge slots (the next tile
      // starts a segment); free its registers for the combine below
      m0 = m1 = NEG_INF;
      l0 = l1 = c0 = c1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      const bool single = d.first_cta == d.last_cta;
      consumer_sync(cbar, cphase, a);
      const EntryId id = entry_id(a, d.e);
      float* dst = a.o + (((size_t)id.lr * cv.B + id.b) * cv.Hq + (size_t)id.h * G) * kHeadDim;
      const size_t slot = (size_t)blockIdx.x + d.e;
      // CTA-level merge, 4 channels per thread
      for (int q4 = ct; q4 < G * 32; q4 += kConsumerWarps * 32) {
        const int g = q4 >> 5, dd = (q4 & 31) * 4;
        float4 acc;
        float M, L;
        if (one_pass)
          merge_slots<kConsumerWarps, 4>(merge_o, merge_m, merge_l, g, dd, acc, M, L);
        else
          merge_slots<kMergeSlots, kMaxGroup>(merge_o, merge_m, merge_l, g, dd, acc, M, L);
        if (single) {
          const float inv = L > 0.f ? 1.f / L : 0.f;
          *reinterpret_cast<float4*>(&dst[g * kHeadDim + dd]) =
              make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else {
          *reinterpret_cast<float4*>(&a.part[(slot * G + g) * kHeadDim + dd]) = acc;
          if (dd == 0) a.part_ml[slot * G + g] = make_float2(M, L);
        }
      }
      if (!single) {
        // The barrier orders every thread's partial stores before thread 0's
        // acquire-release add on the counter, which releases them all
        // (release is cumulative); the entry's last CTA acquires the other
        // partials by the same add before its barrier hands them to its
        // threads.
        consumer_sync(cbar, cphase, a);
        if (ct == 0) {
          const int prev = atom_add_acq_rel_gpu(&a.counters[d.e], 1);
          misc[2] = prev == d.last_cta - d.first_cta ? 1 : 0;
        }
        consumer_sync(cbar, cphase, a);
        if (misc[2]) {
          // last CTA of the entry: LSE-merge the partials of CTAs first..last
          // (slots first+e .. last+e, consecutive).  Each thread owns 4
          // output channels of one query head and merges on its own: per
          // chunk of partials it issues every o and (m, l) load at once (one
          // round trip), then folds the chunk into a running (M, L, acc)
          // with weights 2^(m_c - M).
          const int np = d.last_cta - d.first_cta + 1;
          const size_t slot0 = (size_t)d.first_cta + d.e;
          const int q4 = ct;                                   // G * 32 <= 256 outputs
          if (q4 < G * 32) {
            const int g = q4 >> 5;
            const float4* src = reinterpret_cast<const float4*>(a.part) + slot0 * G * 32 + q4;
            const float2* mls = a.part_ml + slot0 * G + g;
            constexpr int kChunk = 16;
            float M = NEG_INF, L = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c0 = 0; c0 < np; c0 += kChunk) {
              float4 v[kChunk];
              float2 ml[kChunk];
#pragma unroll
              for (int u = 0; u < kChunk; ++u) {
                const int c = min(c0 + u, np - 1);        // past np: the last partial again
                v[u] = __ldcg(src + (size_t)c * G * 32);
                ml[u] = __ldcg(mls + (size_t)c * G);
              }
              float Mc = M;
#pragma unroll
              for (int u = 0; u < kChunk; ++u) Mc = fmaxf(Mc, ml[u].x);
              if (Mc != NEG_INF) {
                const float f = M == NEG_INF ? 0.f : exp2f(M - Mc);
                acc.x *= f;
                acc.y *= f;
                acc.z *= f;
                acc.w *= f;
                L *= f;
#pragma unroll
                for (int u = 0; u < kChunk; ++u) {
                  const float w = c0 + u < np && ml[u].x != NEG_INF ? exp2f(ml[u].x - Mc) : 0.f;
                  acc.x += w * v[u].x;
                  acc.y += w * v[u].y;
                  acc.z += w * v[u].z;
                  acc.w += w * v[u].w;
                  L += w * ml[u].y;
                }
                M = Mc;
              }
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            *reinterpret_cast<float4*>(&dst[q4 * 4]) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
          }
          if (ct == 0) a.counters[d.e] = 0;
        }
      }
      consumer_sync(cbar, cphase, a);
    }
    if (++stage == kSlots) {
      stage = 0;
      phase ^= 1u;
    }
  }

  if (fused && !early_len) {
    // Lengths move only when every CTA is done (each read them in its work
    // split): the last CTA to finish advances them, as the append kernel
    // does per sequence.  Every CTA loads the new values of its threads'
    // first (layer, sequence) before the count, which nothing can change
    // before the last CTA stores them.
    // (Every length this CTA reads was read before its consumers left the
    // loop: the producer's last loads precede its final arrive.  The count
    // orders nothing else -- the cache writes are for the next kernel.)
    int lb0 = 0, n0 = -1, cn0 = -1;
    bool bad0 = false;
    if (ct < nlb) next_len(ct, lb0, n0, cn0, bad0);
    if (ct == 0) misc[2] = atomicAdd(&a.counters[E], 1) == (int)gridDim.x - 1 ? 1 : 0;
    consumer_sync(cbar, cphase, a);
    if (misc[2]) {
      for (int i = ct; i < nlb; i += kConsumerWarps * 32) {
        int lb = lb0, n1 = n0, c1 = cn0;
        bool bad = bad0;
        if (i != ct) next_len(i, lb, n1, c1, bad);
        if (n1 > 0) cv.len[lb] = n1;
        if (c1 > 0) cv.cnt[lb] = c1;
        if (bad) set_status(cv, kStatusBadId);
      }
      if (ct == 0) a.counters[E] = 0;
    }
  }
}

}  // namespace

size_t decode_smem_bytes() { return kSmemBytes; }

// One instantiation: its shared-memory limit raised on first use on the
// device, then the launch.
template <int kFmt, bool kPaged, bool kSmallE>
static cudaError_t launch_one(const cudaLaunchConfig_t& cfg, const DecodeMaps& maps, const DecodeArgs& args) {
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t err = set_smem_limit_once(decode_kernel<kFmt, kPaged, kSmallE>, kSmemBytes, attr_done);
  if (err != cudaSuccess) return err;
  return cudaLaunchKernelEx(&cfg, decode_kernel<kFmt, kPaged, kSmallE>, maps, args);
}

// The instantiation of a format for the cache's layout and the launch's
// entry count.
template <int kFmt>
static cudaError_t launch_fmt(const cudaLaunchConfig_t& cfg, const DecodeMaps& maps, const DecodeArgs& args) {
  const bool paged = args.cv.max_pages > 0;
  const bool small = (int64_t)args.nlayers * args.cv.B * args.cv.Hkv <= 32;
  if (paged)
    return small ? launch_one<kFmt, true, true>(cfg, maps, args) : launch_one<kFmt, true, false>(cfg, maps, args);
  return small ? launch_one<kFmt, false, true>(cfg, maps, args) : launch_one<kFmt, false, false>(cfg, maps, args);
}

cudaError_t launch_decode(const DecodeMaps& maps, const DecodeArgs& args, int ctas, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (args.cv.kv_format == kKvInt8) return launch_fmt<kKvInt8>(cfg, maps, args);
  if (args.cv.kv_format == kKvFp8) return launch_fmt<kKvFp8>(cfg, maps, args);
  return launch_fmt<kKvBf16>(cfg, maps, args);
}

}  // namespace lk
