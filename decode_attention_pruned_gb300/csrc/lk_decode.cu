// Decode attention over the split LeanK cache (one launch covers one or
// more layers).
//
// What it computes (LeanK article, framerc.cn, section 3.1 "fused
// computation"; FastGen article, mhpn.cn, section 3.2 stage 2): for every
// sequence b and kv head h, the G query heads of h score the full-width rows
// (sinks + window ring, LOCAL ring or SPECIAL rows) on all 128 channels and the
// middle rows of K_prun on the head's kept channels (q gathered to the kept
// channel list), s = q.k / sqrt(128); one online softmax runs over both
// regions and o = sum p V.  INT8 caches hold complete 128-row middle blocks
// as codes with per-channel K / per-token V scales (KIVI-style, after the
// pruning); those blocks are scored on the dequantised values.
//
// How:
//   * The work line.  Each (layer, b, h) "entry" is a run of rows: full-width
//     rows, then sealed INT8 rows, then bf16 kept-channel rows.  A row costs
//     the bytes it streams, so the line is measured in bytes.  CTA i of P
//     takes the rows whose line offset falls in [iC/P, (i+1)C/P); the CTAs
//     touching an entry are exactly first..last and each writes one partial.
//   * Per CTA: warp 8 (one lane) issues one TMA load per K tile and one per V
//     tile (swizzled boxes), or one bulk copy per sealed INT8 block, into a
//     FIFO ring of variable-size stages with sixteen mbarrier slots; warps
//     0-7 each take 16 rows of every 128-row tile.
//   * Tensor cores (mma.sync m16n8k16, fp32 accumulate) with tokens on M:
//     S^T[16 tok x 8] = K[16 x w] Q^T[w x 8] and O^T[128 x 8] += V^T P^T, so
//     the G <= 8 query heads only pad N.  P goes from the S^T accumulator to
//     the B operand of P.V with one movmatrix transpose per 8x8 block; it is
//     split into hi + lo halves (two mmas) so P.V keeps ~16 bits of P.  INT8
//     codes enter the f16 mmas exactly; the scales fold into q and p.
//   * Segment end: warps merge through shared memory; a CTA that owns the
//     whole entry writes o, otherwise it writes (o, m, l) to its partial slot
//     and the last of the entry's CTAs (atomic counter) merges them.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

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
// stages in flight where full-width ones (64 KB) keep three; sealed INT8
// blocks (21-33 KB) keep up to nine.
constexpr int kSlots = 16;                              // barrier pairs = stages in flight at most (power of 2)
constexpr int kRingBytes = 204 * 1024;
constexpr int kUnitsA = 2 * kHeadDim * 2;               // line cost of a full-width row: its bytes
constexpr int kFirst = 1, kLast = 2;
constexpr uint64_t kDrainLimitNs = 1000000000ull;      // bound of the producer's final wait for its copies

struct StageDesc {
  int32_t e;           // entry = b * Hkv + h; < 0 ends the stream
  int32_t region;      // 0: full width, 1: kept channels (bf16), 2: sealed INT8 block
  int32_t rlo;         // first valid row of the tile (sealed blocks; else 0)
  int32_t nrows;       // valid rows of the tile: rlo .. rlo + nrows - 1
  int32_t width;       // K channels of the tile
  int32_t flags;       // kFirst / kLast of this CTA's segment of the entry
  int32_t first_cta;   // CTAs first..last hold partials of the entry
  int32_t last_cta;
  uint32_t koff;       // ring offset of the K tile; the V tile follows it
};

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
  static constexpr int kBytes = kMiscOff + 64;
};
constexpr int kSmemBytes = SmemLayout::kBytes + 1024;   // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory per block");

__device__ __forceinline__ uint32_t stage_bytes(int region, int width) {
  return region == 2 ? (uint32_t)qblock_bytes(width) : (uint32_t)kTileRows * (2 * width + 256);
}
// ring footprint of a stage: 1024-byte granules (swizzled TMA boxes need
// 1024-byte aligned destinations)
__device__ __forceinline__ uint32_t ring_bytes(int region, int width) {
  return (stage_bytes(region, width) + 1023u) & ~1023u;
}

// Rows of an entry in line order: n_a full width, n_q in sealed INT8 blocks,
// n_b bf16 kept-channel rows (INT8 caches: the open tail block).
struct Entry {
  int n_a, n_q, n_b, kb;
};

// Entry e of a launch = (layer offset lr, sequence b, kv head h), layers
// outermost.
struct EntryId {
  int lr, l, b, h;
};
__device__ __forceinline__ EntryId entry_id(const DecodeArgs& a, int e) {
  const CacheView& cv = a.cv;
  const int per_layer = cv.B * cv.Hkv;
  EntryId r;
  r.lr = e / per_layer;
  const int rem = e - r.lr * per_layer;
  r.b = rem / cv.Hkv;
  r.h = rem - r.b * cv.Hkv;
  r.l = a.layer + r.lr;
  return r;
}

// Lengths and special counts are read through L2 (they are written by the
// preceding append kernel).  The loads are split from the arithmetic so the
// producer can issue the next entry's loads one entry ahead.
struct EntryLen {
  int n;      // tokens of the sequence in this layer
  int cnt;    // special rows (SPECIAL heads), else 0
};
__device__ __forceinline__ EntryLen entry_len(const DecodeArgs& a, int e) {
  const CacheView& cv = a.cv;
  const EntryId id = entry_id(a, e);
  const HeadDesc& hd = cv.heads[id.l * cv.Hkv + id.h];
  EntryLen r;
  r.n = __ldcg(&cv.len[id.l * cv.B + id.b]);
  r.cnt = hd.policy == kSpecial ? __ldcg(&cv.cnt[id.l * cv.B + id.b]) : 0;
  return r;
}

__device__ __forceinline__ Entry entry_from(const DecodeArgs& a, int e, EntryLen len) {
  const CacheView& cv = a.cv;
  const EntryId id = entry_id(a, e);
  const HeadDesc& hd = cv.heads[id.l * cv.Hkv + id.h];
  const int N = len.n;
  Entry r{0, 0, 0, 0};
  if (hd.policy == kFull) {
    r.n_a = min(N, cv.S + cv.W);
    if (hd.n_kept > 0) {
      const int m = max(0, N - cv.S - cv.W);
      if (cv.kv_format == kKvInt8) {
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
  } else {
    r.n_a = min(len.cnt, hd.cap_a);
  }
  r.n_a = min(r.n_a, hd.cap_a);
  r.n_b = min(r.n_b, hd.cap_b);
  return r;
}

__device__ __forceinline__ Entry entry_geometry(const DecodeArgs& a, int e) { return entry_from(a, e, entry_len(a, e)); }

// line costs per row = bytes streamed per row
__device__ __forceinline__ uint64_t row_cost_b(int kb) { return (uint64_t)(2 * kb + 256); }
__device__ __forceinline__ uint64_t row_cost_q(int kb) { return (uint64_t)(qblock_bytes(kb) / kQBlockRows); }

__device__ __forceinline__ uint64_t entry_cost(const Entry& g) {
  return (uint64_t)kUnitsA * g.n_a + row_cost_q(g.kb) * g.n_q + row_cost_b(g.kb) * g.n_b;
}

// a / b for 64-bit a with a 32-bit path when it fits
__device__ __forceinline__ uint64_t udiv(uint64_t a, uint64_t b) {
  if ((a >> 32) == 0 && (b >> 32) == 0) return (uint32_t)a / (uint32_t)b;
  return a / b;
}

// Rows r in [0, n) of a region whose row r sits at line offset o0 + c*r and
// starts inside [start, end): r in [r0, r1).
__device__ __forceinline__ void rows_in_range(uint64_t o0, uint64_t c, int n, uint64_t start, uint64_t end,
                                              int& r0, int& r1) {
  r0 = start > o0 ? (int)min((uint64_t)n, udiv(start - o0 + c - 1, c)) : 0;
  r1 = end > o0 ? (int)min((uint64_t)n, udiv(end - o0 + c - 1, c)) : 0;
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

// kQ8: the cache's middle is INT8 (sealed blocks may occur); the bf16
// instantiation carries no INT8 code.
template <bool kQ8>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k128, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_k32, const __grid_constant__ CUtensorMap tm_k64,
                  const __grid_constant__ CUtensorMap tm_k96, const DecodeArgs a) {
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

  static_assert(kSlots < 32, "one barrier pair per lane of warp 0, plus the consumer barrier");
  if (tid < kSlots) {
    mbar_init(bar_full + 8 * tid, 1);
    mbar_init(bar_empty + 8 * tid, kConsumerWarps);
    fence_barrier_init();
  } else if (tid == kSlots) {
    mbar_init(base + SmemLayout::kCBarOff, kConsumerWarps);
    fence_barrier_init();
  }
  if (tid == 0) {
    misc[0] = E;       // first entry of this CTA
    misc[1] = 0;       // its line offset
    misc[2] = 0;       // last-CTA flag of a segment
    misc[3] = misc[4] = misc[5] = misc[6] = 0;   // geometry of the first entry
  }
  if (warp == kConsumerWarps && lane == 0) {
    tma_prefetch_map(&tm_k128);
    tma_prefetch_map(&tm_v);
    tma_prefetch_map(&tm_k32);
    tma_prefetch_map(&tm_k64);
    tma_prefetch_map(&tm_k96);
    // read every launch parameter the producer uses once, so their constant
    // cache lines arrive while the preceding kernel finishes
    uint64_t touch = (uint64_t)cv.hdr ^ (uint64_t)cv.len ^ (uint64_t)cv.cnt ^ (uint64_t)cv.page_table ^
                     (uint64_t)cv.heads ^ (uint64_t)cv.qpool ^ (uint64_t)cv.kept ^ (uint64_t)a.q ^ (uint64_t)a.o ^
                     (uint64_t)a.part ^ (uint64_t)a.part_ml ^ (uint64_t)a.counters ^ a.wait_limit_ns;
    touch ^= (uint64_t)(cv.B ^ cv.Hkv ^ cv.S ^ cv.W ^ cv.W_loc ^ cv.max_pages ^ cv.kv_format ^ a.layer ^ a.nlayers ^
                        cv.G ^ cv.Hq);
    asm volatile("" ::"l"(touch));
  }
  // the head table is static (written once at cache init): load it while
  // the preceding kernel finishes, which also walks the page table for the
  // cache header (a prefetch may be dropped on a TLB miss; a load is not).
  // Lengths and special counts are written by that kernel, so they are read
  // only after the dependency wait.
  {
    int64_t touch = 0;
    for (int h = tid; h < a.nlayers * cv.Hkv; h += kThreads) touch += cv.heads[a.layer * cv.Hkv + h].row_a;
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
  const uint64_t policy = l2_policy_evict_first();
  grid_dependency_wait();
  grid_launch_dependents();

  // ---- the line: per-thread chunks of entries, block exclusive scan
  const int per = (E + kThreads - 1) / kThreads;
  const int e_lo = min(E, tid * per), e_hi = min(E, e_lo + per);
  // the first two entries of the chunk keep their geometry for the second
  // pass (a whole single-layer launch fits that)
  Entry g0{0, 0, 0, 0}, g1{0, 0, 0, 0};
  if (e_lo < e_hi) g0 = entry_geometry(a, e_lo);
  if (e_lo + 1 < e_hi) g1 = entry_geometry(a, e_lo + 1);
  uint64_t local = entry_cost(g0) + entry_cost(g1);
  for (int e = e_lo + 2; e < e_hi; ++e) local += entry_cost(entry_geometry(a, e));
  uint64_t incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint64_t v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) scan[warp] = incl;
  __syncthreads();
  uint64_t warp_base = 0, C = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) warp_base += scan[w];
    C += scan[w];
  }
  const uint64_t excl = warp_base + incl - local;
  // every CTA range must hold at least one row start (a row costs <= 16)
  const int P = (int)max((uint64_t)1, min((uint64_t)gridDim.x, C / kUnitsA));
  const int cta = blockIdx.x;
  const uint64_t start = cta < P ? ((uint64_t)cta * C) / P : C;
  const uint64_t end = cta < P ? ((uint64_t)(cta + 1) * C) / P : C;
  if (local > 0 && excl <= start && start < excl + local) {
    // this chunk holds the CTA's first row: its entry, line offset and
    // geometry go to the producer through shared memory
    uint64_t acc = excl;
    int found = -1;
    Entry fg{0, 0, 0, 0};
    for (int e = e_lo; found < 0 && e < e_hi; ++e) {
      const Entry g = e == e_lo ? g0 : e == e_lo + 1 ? g1 : entry_geometry(a, e);
      const uint64_t c = entry_cost(g);
      if (acc + c > start) {
        found = e;
        fg = g;
      } else {
        acc += c;
      }
    }
    misc[0] = found;
    misc[1] = (int64_t)acc;
    misc[3] = fg.n_a;
    misc[4] = fg.n_b;
    misc[5] = fg.kb;
    misc[6] = fg.n_q;
  }
  __syncthreads();

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
      const int e0 = (int)misc[0];
      int e = e0;
      uint64_t off = (uint64_t)misc[1];
      // entry geometry: the first from the scan, later ones from lengths
      // loaded one entry ahead
      Entry g{(int)misc[3], (int)misc[6], (int)misc[4], (int)misc[5]};
      EntryLen ahead{0, 0};
      if (e + 1 < E) ahead = entry_len(a, e + 1);
      for (; ok && e < E && off < end; ++e) {
        if (e != e0) {
          g = entry_from(a, e, ahead);
          if (e + 1 < E) ahead = entry_len(a, e + 1);
        }
        const uint64_t cost = entry_cost(g);
        const uint64_t cq = row_cost_q(g.kb), cb = row_cost_b(g.kb);
        const uint64_t off_q = off + (uint64_t)kUnitsA * g.n_a;
        const uint64_t off_b = off_q + cq * g.n_q;
        int a0, a1, q0, q1, b0, b1;
        rows_in_range(off, kUnitsA, g.n_a, start, end, a0, a1);
        rows_in_range(off_q, cq, g.n_q, start, end, q0, q1);
        rows_in_range(off_b, cb, g.n_b, start, end, b0, b1);
        // paged bf16 region B: tiles end at page boundaries (the box may read
        // past a page end; those rows are beyond nrows and ignored).  Sealed
        // INT8 blocks: one tile per block, whole block loaded, rows masked.
        const bool paged = cv.max_pages > 0;
        const bool bpaged = paged && cv.kv_format == kKvBf16;
        const int nta = (a1 - a0 + kTileRows - 1) / kTileRows;
        const int ntq = q1 <= q0 ? 0 : (q1 - 1) / kQBlockRows - q0 / kQBlockRows + 1;
        const int ntb = b1 <= b0   ? 0
                        : bpaged ? (b1 - 1) / kPageRows - b0 / kPageRows + 1
                                 : (b1 - b0 + kTileRows - 1) / kTileRows;
        const int nt = nta + ntq + ntb;
        if (nt > 0) {
          const EntryId id = entry_id(a, e);
          const int b = id.b;
          const HeadDesc& hd = cv.heads[id.l * cv.Hkv + id.h];
          const int32_t* pt =
              cv.page_table + (((int64_t)id.l * cv.B + b) * cv.Hkv + id.h) * cv.max_pages;
          const uint64_t last_row_off = g.n_b > 0   ? off_b + cb * (g.n_b - 1)
                                        : g.n_q > 0 ? off_q + cq * (g.n_q - 1)
                                                    : off + (uint64_t)kUnitsA * (g.n_a - 1);
          // the entry's first / last owning CTA is read only from the segment's
          // last descriptor: work it out after the first load is in flight
          int fc = -1, lc = -1;
          if (nt == 1) {
            fc = range_owner(off, C, P);
            lc = range_owner(last_row_off, C, P);
          }
          int32_t page_ahead = 0;
          for (int j = 0; j < nt; ++j) {
            const int region = j < nta ? 0 : j < nta + ntq ? 2 : 1;
            const int width = region == 0 ? kHeadDim : g.kb;
            int r, rend, rlo = 0;
            int32_t page = 0;
            if (region == 0) {
              r = a0 + j * kTileRows;
              rend = min(a1, r + kTileRows);
            } else if (region == 2) {
              const int blk = q0 / kQBlockRows + (j - nta);
              r = max(q0, blk * kQBlockRows);
              rend = min(q1, (blk + 1) * kQBlockRows);
              rlo = r - blk * kQBlockRows;
              if (paged) {
                page = j == nta ? __ldcg(pt + blk) : page_ahead;
                if (j + 1 < nta + ntq) page_ahead = __ldcg(pt + blk + 1);
                page = max(0, page);
              } else {
                page = b * hd.qblocks + blk;
              }
            } else if (bpaged) {
              const int pg = b0 / kPageRows + (j - nta - ntq);
              r = max(b0, pg * kPageRows);
              rend = min(b1, (pg + 1) * kPageRows);
              // page ids load one tile ahead (and before the slot wait); a
              // missing page (status already recorded) reads page 0
              page = j == nta + ntq ? __ldcg(pt + pg) : page_ahead;
              if (j + 1 < nt) page_ahead = __ldcg(pt + pg + 1);
              page = max(0, page);
            } else {
              r = b0 + (j - nta - ntq) * kTileRows;
              rend = min(b1, r + kTileRows);
            }
            const uint32_t bytes = stage_bytes(region, width);
            uint32_t at = 0;
            if (!reserve(ring_bytes(region, width), at)) {
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
            d.flags = (j == 0 ? kFirst : 0) | (j + 1 == nt ? kLast : 0);
            d.first_cta = fc;
            d.last_cta = lc;
            d.koff = at;
            desc[stage] = d;
            const uint32_t fb = bar_full + 8 * stage;
            mbar_arrive_expect_tx(fb, bytes);
            const uint32_t kdst = base + SmemLayout::kRingOff + at;
            const uint32_t vdst = kdst + (uint32_t)kTileRows * 2 * width;
            if (region == 0) {
              const int32_t row = (int32_t)(hd.row_a + (int64_t)b * hd.cap_a + r);
              tma_load_3d(kdst, &tm_k128, 0, row, 0, fb, policy);
              tma_load_3d(vdst, &tm_v, 0, row, 0, fb, policy);
            } else if (region == 2) {
              bulk_load(kdst, cv.qpool + hd.qoff + (int64_t)page * bytes, bytes, fb, policy);
            } else {
              const int64_t rb = bpaged ? (int64_t)page * kPageRows + r % kPageRows : (int64_t)b * hd.cap_b + r;
              const int32_t krow = (int32_t)(hd.krow_b + rb);
              const int32_t vrow = (int32_t)(hd.vrow_b + rb);
              switch (hd.pool_kb) {
                case kPoolK32: tma_load_2d(kdst, &tm_k32, 0, krow, fb, policy); break;
                case kPoolK64: tma_load_2d(kdst, &tm_k64, 0, krow, fb, policy); break;
                case kPoolK96: tma_load_3d(kdst, &tm_k96, 0, krow, 0, fb, policy); break;
                default: tma_load_3d(kdst, &tm_k128, 0, krow, 0, fb, policy); break;
              }
              tma_load_3d(vdst, &tm_v, 0, vrow, 0, fb, policy);
            }
            ++issued;
            if (fc < 0) {
              fc = range_owner(off, C, P);
              lc = range_owner(last_row_off, C, P);
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

  // entries with no resident token: o = 0, written by CTA (e mod grid)
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    if (entry_cost(entry_geometry(a, e)) != 0) continue;
    const EntryId id = entry_id(a, e);
    float* dst = a.o + (((size_t)id.lr * cv.B + id.b) * cv.Hq + (size_t)id.h * G) * kHeadDim;
    for (int i = ct; i < G * kHeadDim; i += kConsumerWarps * 32) dst[i] = 0.f;
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
    const HeadDesc& hd = cv.heads[id.l * cv.Hkv + id.h];
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
  int q_entry = (int)misc[0];
  if (q_entry < E) stage_q(q_entry);

  // this warp's 16 rows of every tile
  const int r0 = 16 * warp;
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

    // valid rows rlo .. rhi - 1 of the tile (sealed blocks may be shared with
    // another CTA)
    const int rlo = d.rlo, rhi = d.rlo + d.nrows;
    const uint32_t kbase = base + SmemLayout::kRingOff + d.koff;
    if (r0 < rhi && r0 + 16 > rlo) {
      // two independent accumulators halve the mma dependency chain
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
      if (kQ8 && d.region == 2) {
        // ---- sealed INT8 block: S^T = K_codes (f16, exact) . Q'^T with
        // Q' = q[kept] * (K scale of the channel), split into f16 hi + lo
        const int kb = d.width;
        const float* ksc = reinterpret_cast<const float*>(sm + SmemLayout::kRingOff + d.koff + qblock_ksoff(kb));
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          if (2 * kp < (kb >> 4)) {
            uint32_t qv[4];
            ldsm_x4(qb_lane + 64u * kp, qv[0], qv[1], qv[2], qv[3]);
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
            const int row = r0 + rk;
            const int grp = 2 * kp + ck;
            uint32_t w0, w1, w2, w3;
            ldsm_x4(kbase + (uint32_t)(row * kb + 16 * (grp ^ qswz(kb, row))), w0, w1, w2, w3);
            uint32_t f0, f1, f2, f3;
            i8x4_to_f16x2(w0, f0, f2);       // rows gid: k 2tig.. / 2tig+8..
            i8x4_to_f16x2(w1, f1, f3);       // rows gid + 8
            mma_f16_16816(sc, f0, f1, f2, f3, bh[0][0], bh[0][1]);
            mma_f16_16816(sd, f0, f1, f2, f3, bl[0][0], bl[0][1]);
            i8x4_to_f16x2(w2, f0, f2);
            i8x4_to_f16x2(w3, f1, f3);
            mma_f16_16816(sc, f0, f1, f2, f3, bh[1][0], bh[1][1]);
            mma_f16_16816(sd, f0, f1, f2, f3, bl[1][0], bl[1][1]);
          }
        }
      } else {
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
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[i] += sd[i];
      const int t0 = r0 + gid;
      const bool v0 = t0 >= rlo && t0 < rhi, v1 = t0 + 8 >= rlo && t0 + 8 < rhi;
      const float x0 = v0 ? sc[0] * a.scale_log2 : NEG_INF;
      const float x1 = v0 ? sc[1] * a.scale_log2 : NEG_INF;
      const float x2 = v1 ? sc[2] * a.scale_log2 : NEG_INF;
      const float x3 = v1 ? sc[3] * a.scale_log2 : NEG_INF;
      // Lazy rescaling: the running max m of a column moves only when some
      // score of the tile exceeds it by more than kRescaleGap (log2 units);
      // otherwise p = 2^(s - m) <= 2^kRescaleGap, exact in the fp32
      // accumulators and in the hi/lo splits of P.  One warp vote replaces
      // the column-max shuffles in the common case.
      float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
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
      const float p0 = exp2f(x0 - m0), p1 = exp2f(x1 - m1);   // token gid
      const float p2 = exp2f(x2 - m0), p3 = exp2f(x3 - m1);   // token gid + 8
      l0 += p0 + p2;
      l1 += p1 + p3;
      if (kQ8 && d.region == 2) {
        // ---- O^T += V_codes^T (f16, exact) . P'^T, P' = p * (V scale of
        // the token), split into f16 hi + lo
        const uint32_t vbase = kbase + (uint32_t)qblock_voff(d.width);
        const float* vsc =
            reinterpret_cast<const float*>(sm + SmemLayout::kRingOff + d.koff + qblock_vsoff(d.width));
        const float sv0 = vsc[r0 + gid], sv1 = vsc[r0 + gid + 8];
        const float q0 = p0 * sv0, q1 = p1 * sv0, q2 = p2 * sv1, q3 = p3 * sv1;
        c0 += q0 + q2;
        c1 += q1 + q3;
        const uint32_t h01 = pack_f16x2(q0, q1), h23 = pack_f16x2(q2, q3);
        const uint32_t r01 = pack_f16x2(q0 - f16_lo(h01), q1 - f16_hi(h01));
        const uint32_t r23 = pack_f16x2(q2 - f16_lo(h23), q3 - f16_hi(h23));
        const uint32_t ph0 = movmatrix_trans(h01), ph1 = movmatrix_trans(h23);
        const uint32_t pr0 = movmatrix_trans(r01), pr1 = movmatrix_trans(r23);
        const int row = r0 + rk;
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          const int grp = 2 * i2 + ck;
          uint32_t w0, w1, w2, w3;
          ldsm_x4_trans(vbase + (uint32_t)(row * kHeadDim + 16 * (grp ^ (row & 7))), w0, w1, w2, w3);
          uint32_t f0, f1, f2, f3;
          u8x4_to_f16x2_biased(w0, f0, f1);  // tokens 2tig.. of rows 0-7: channels gid / gid + 8
          u8x4_to_f16x2_biased(w1, f2, f3);  // tokens 2tig + 8..
          mma_f16_16816(o[2 * i2], f0, f1, f2, f3, ph0, ph1);
          mma_f16_16816(o[2 * i2], f0, f1, f2, f3, pr0, pr1);
          u8x4_to_f16x2_biased(w2, f0, f1);
          u8x4_to_f16x2_biased(w3, f2, f3);
          mma_f16_16816(o[2 * i2 + 1], f0, f1, f2, f3, ph0, ph1);
          mma_f16_16816(o[2 * i2 + 1], f0, f1, f2, f3, pr0, pr1);
        }
      } else {
        // P as a bf16 pair hi + lo (two mmas): P.V keeps ~16 mantissa bits
        const uint32_t vbase = kbase + (uint32_t)kTileRows * 2 * d.width;
        const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
        const uint32_t r01 = pack_bf16x2(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
        const uint32_t r23 = pack_bf16x2(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
        // S^T accumulator rows (tokens) -> B operand rows (k = tokens) of P^T
        const uint32_t ph0 = movmatrix_trans(h01), ph1 = movmatrix_trans(h23);
        const uint32_t pr0 = movmatrix_trans(r01), pr1 = movmatrix_trans(r23);
        const int row = r0 + rv;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(tile_addr128(vbase, row, 2 * i + cvh), a0, a1, a2, a3);
          mma_bf16_16816(o[i], a0, a1, a2, a3, ph0, ph1);
          mma_bf16_16816(o[i], a0, a1, a2, a3, pr0, pr1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * stage);

    if (d.flags & kLast) {
      if (kQ8) {
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
      // ---- merge the warps' (o, m, l) of this segment: warps 4..7 hand
      // theirs to warps 0..3 through the merge slots, then 0..3 publish
      float lr0 = l0, lr1 = l1;
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        lr0 += __shfl_xor_sync(0xffffffffu, lr0, sh);
        lr1 += __shfl_xor_sync(0xffffffffu, lr1, sh);
      }
      const int slotw = warp & (kMergeSlots - 1);
      float* ob = merge_o + slotw * kMaxGroup * kHeadDim;
      if (warp >= kMergeSlots) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ob[(2 * tig) * kHeadDim + 16 * i + gid] = o[i][0];
          ob[(2 * tig + 1) * kHeadDim + 16 * i + gid] = o[i][1];
          ob[(2 * tig) * kHeadDim + 16 * i + gid + 8] = o[i][2];
          ob[(2 * tig + 1) * kHeadDim + 16 * i + gid + 8] = o[i][3];
        }
        if (gid == 0) {
          merge_m[slotw * kMaxGroup + 2 * tig] = m0;
          merge_m[slotw * kMaxGroup + 2 * tig + 1] = m1;
          merge_l[slotw * kMaxGroup + 2 * tig] = lr0;
          merge_l[slotw * kMaxGroup + 2 * tig + 1] = lr1;
        }
      }
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
      consumer_sync(cbar, cphase, a);
      if (warp < kMergeSlots) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ob[(2 * tig) * kHeadDim + 16 * i + gid] = o[i][0];
          ob[(2 * tig + 1) * kHeadDim + 16 * i + gid] = o[i][1];
          ob[(2 * tig) * kHeadDim + 16 * i + gid + 8] = o[i][2];
          ob[(2 * tig + 1) * kHeadDim + 16 * i + gid + 8] = o[i][3];
        }
        if (gid == 0) {
          merge_m[slotw * kMaxGroup + 2 * tig] = m0;
          merge_m[slotw * kMaxGroup + 2 * tig + 1] = m1;
          merge_l[slotw * kMaxGroup + 2 * tig] = lr0;
          merge_l[slotw * kMaxGroup + 2 * tig + 1] = lr1;
        }
      }
      // the segment's state now lives in the merge slots (the next tile
      // starts a segment); free its registers for the combine below
      m0 = m1 = NEG_INF;
      l0 = l1 = c0 = c1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      consumer_sync(cbar, cphase, a);
      const EntryId id = entry_id(a, d.e);
      float* dst = a.o + (((size_t)id.lr * cv.B + id.b) * cv.Hq + (size_t)id.h * G) * kHeadDim;
      const bool single = d.first_cta == d.last_cta;
      const size_t slot = (size_t)blockIdx.x + d.e;
      // CTA-level merge, 4 channels per thread
      for (int q4 = ct; q4 < G * 32; q4 += kConsumerWarps * 32) {
        const int g = q4 >> 5, dd = (q4 & 31) * 4;
        float M = NEG_INF;
#pragma unroll
        for (int w = 0; w < kMergeSlots; ++w) M = fmaxf(M, merge_m[w * kMaxGroup + g]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeSlots; ++w) {
          const float mw = merge_m[w * kMaxGroup + g];
          const float f = mw == NEG_INF ? 0.f : exp2f(mw - M);
          const float4 v = *reinterpret_cast<const float4*>(&merge_o[(w * kMaxGroup + g) * kHeadDim + dd]);
          acc.x += f * v.x;
          acc.y += f * v.y;
          acc.z += f * v.z;
          acc.w += f * v.w;
          L += f * merge_l[w * kMaxGroup + g];
        }
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
        __threadfence();
        consumer_sync(cbar, cphase, a);
        if (ct == 0) {
          const int prev = atomicAdd(&a.counters[d.e], 1);
          misc[2] = (prev == d.last_cta - d.first_cta) ? 1 : 0;
        }
        consumer_sync(cbar, cphase, a);
        if (misc[2]) {
          // last CTA of the entry: LSE-merge the partials of CTAs first..last
          // (slots first+e .. last+e, consecutive).  Each thread owns 4 output
          // channels: it issues the o loads of its first chunk of partials
          // while the (m, l) pairs are staged into shared memory, so a chunk
          // costs one round trip; a warp per query head turns the pairs into
          // weights w_c = 2^(m_c - M) / L.
          __threadfence();
          const int np = d.last_cta - d.first_cta + 1;
          const size_t slot0 = (size_t)d.first_cta + d.e;
          const float4* src = reinterpret_cast<const float4*>(a.part) + slot0 * G * 32;
          float2* mlb = reinterpret_cast<float2*>(merge_o);      // [np][G], np * G <= 2048
          constexpr int kChunk = 20;
          const int q4a = ct, q4b = ct + kConsumerWarps * 32;  // G * 32 <= 256 outputs
          float4 v[kChunk];
#pragma unroll
          for (int u = 0; u < kChunk; ++u) {
            const int c = min(u, np - 1);
            v[u] = q4a < G * 32 ? __ldcg(src + (size_t)c * G * 32 + q4a) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          for (int i = ct; i < np * G; i += kConsumerWarps * 32) mlb[i] = __ldcg(&a.part_ml[slot0 * G + i]);
          consumer_sync(cbar, cphase, a);
          for (int g = warp; g < G; g += kConsumerWarps) {
            float M = NEG_INF;
            for (int c = lane; c < np; c += 32) M = fmaxf(M, mlb[c * G + g].x);
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
            float L = 0.f;
            for (int c = lane; c < np; c += 32) {
              const float2 ml = mlb[c * G + g];
              L += ml.x == NEG_INF ? 0.f : exp2f(ml.x - M) * ml.y;
            }
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) L += __shfl_xor_sync(0xffffffffu, L, sh);
            const float inv = L > 0.f ? 1.f / L : 0.f;
            __syncwarp();
            for (int c = lane; c < np; c += 32) {
              const float mc = mlb[c * G + g].x;
              mlb[c * G + g].x = mc == NEG_INF ? 0.f : exp2f(mc - M) * inv;
            }
          }
          consumer_sync(cbar, cphase, a);
          for (int pass = 0; pass < 2; ++pass) {
            const int q4 = pass == 0 ? q4a : q4b;
            if (q4 >= G * 32) continue;
            const int g = q4 >> 5;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c0 = 0; c0 < np; c0 += kChunk) {
              if (pass == 1 || c0 > 0) {
#pragma unroll
                for (int u = 0; u < kChunk; ++u)
                  v[u] = __ldcg(src + (size_t)min(c0 + u, np - 1) * G * 32 + q4);
              }
#pragma unroll
              for (int u = 0; u < kChunk; ++u) {
                const float wgt = c0 + u < np ? mlb[(c0 + u) * G + g].x : 0.f;
                acc.x += wgt * v[u].x;
                acc.y += wgt * v[u].y;
                acc.z += wgt * v[u].z;
                acc.w += wgt * v[u].w;
              }
            }
            *reinterpret_cast<float4*>(&dst[q4 * 4]) = acc;
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
}

}  // namespace

size_t decode_smem_bytes() { return kSmemBytes; }

cudaError_t launch_decode(const CUtensorMap* maps, const DecodeArgs& args, int ctas, cudaStream_t stream) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t err = cudaFuncSetAttribute(decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_done = true;
  }
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
  if (args.cv.kv_format == kKvInt8)
    return cudaLaunchKernelEx(&cfg, decode_kernel<true>, maps[kPoolK128], maps[kPoolV], maps[kPoolK32],
                              maps[kPoolK64], maps[kPoolK96], args);
  return cudaLaunchKernelEx(&cfg, decode_kernel<false>, maps[kPoolK128], maps[kPoolV], maps[kPoolK32],
                            maps[kPoolK64], maps[kPoolK96], args);
}

}  // namespace lk
