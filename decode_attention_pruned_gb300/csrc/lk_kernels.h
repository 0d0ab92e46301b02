// Kernel argument blocks and launchers (internal).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "lk_internal.h"

namespace lk {

// TMA tensor maps of the decode kernel.  Flat maps: one per pool, over all
// its rows (a 128-row box that starts near the end of a (head, sequence)
// block reads rows of the next block).  Block views: one pool's rows seen as
// [blocks][rows per block][channels], a block being one (head, sequence) of
// region A of a policy class, or one sequence's region B of a head (paged:
// one page), so a box that runs past the block's end is clipped there (zero
// fill, no DRAM read).  Higher-rank boxes stream slightly slower, so only a
// box that would cross its block's end takes the block view.
constexpr int kMapFlat = 0;         // + pool: every row of the pool
constexpr int kMapAK = kNumPools;   // + policy class: region-A K rows (pool K128)
constexpr int kMapAV = kMapAK + 3;  // + policy class: region-A V rows (pool V)
constexpr int kMapB = kMapAV + 3;   // + pool: region-B rows of that pool (kPoolV: V rows)
constexpr int kNumMaps = kMapB + kNumPools;
struct DecodeMaps {
  CUtensorMap m[kNumMaps];
  // rows per block of each block view; below one box the view is not used
  int32_t block_rows[kNumMaps];
};

// x / d for a 32-bit x and a divisor fixed for a launch: m = ceil(2^64 / d)
// for d >= 2 (m = 0 stands for d = 1), q = high 64 bits of x * m.  Exact for
// every 32-bit x: x * m / 2^64 = x / d + x * eps / 2^64 with eps < 1, and
// x * eps / 2^64 < 1 / d because x * d < 2^64.
struct FastDiv {
  uint64_t m;
  uint32_t d;
  uint32_t pad;
};
inline FastDiv make_fastdiv(uint32_t d) {
  return FastDiv{d <= 1 ? 0ull : ~0ull / d + 1, d, 0u};
}

struct DecodeArgs {
  CacheView cv;
  int32_t layer;            // first layer
  int32_t nlayers;          // layers layer .. layer + nlayers - 1 in one launch
  const uint16_t* q;        // bf16 [nlayers][B][Hq][128]
  float* o;                 // fp32 [nlayers][B][Hq][128]
  float* part;              // fp32 [slots][G][128] split partials (unnormalised o)
  float2* part_ml;          // [slots][G] (running max in log2 units, sum of p)
  int32_t* counters;        // [nlayers*B*Hkv] CTAs done per entry, then CTAs done in all;
                            // self-resetting
  uint64_t wait_limit_ns;   // bound of every mbarrier wait
  float scale_log2;         // log2(e) / sqrt(128)
  // Fused append (bf16 caches): null for a plain decode.  Otherwise the
  // launch appends one token per active sequence and layer and attends to
  // it, as an append followed by a decode would.
  const uint16_t* k_new;    // bf16 [nlayers][B][Hkv][128]
  const uint16_t* v_new;
  const int32_t* ids;       // [B] or null
  // divisions of the work split and the producer, by divisors fixed for the
  // launch: sequences x kv heads, kv heads, window, LOCAL window; and the
  // line cost of a middle row per kept width (index k / 32): bf16 rows
  // 2k + 256 bytes, sealed INT8 / FP8 rows 132 (k + 128) / 128 bytes
  FastDiv div_bh, div_h, div_w, div_wloc;
  FastDiv div_cost_b[5], div_cost_q[5];
};

struct AppendArgs {
  CacheView cv;
  int32_t layer;            // first layer
  int32_t nlayers;          // layers layer .. layer + nlayers - 1 (grid.y)
  const uint16_t* k;        // bf16 [nlayers][B][Hkv][128]
  const uint16_t* v;
  const int32_t* ids;       // [B] or null (the same token for every layer)
};

struct PrefillArgs {
  CacheView cv;
  int32_t layer;
  int32_t b0, nb;           // sequences b0 .. b0 + nb - 1
  const uint16_t* k;        // bf16 [nb][n][Hkv][128]
  const uint16_t* v;
  const int32_t* ids;       // [nb][n] or null
  int32_t n;                // tokens per sequence in k / v / ids (the longest length)
};

// Raise kernel `fn`'s dynamic shared-memory limit to `bytes` on the current
// device the first time it launches there: the attribute is per device, so
// `done` keeps one bit per device ordinal (ordinals past 63 set it every
// time).  Concurrent first launches may both set it, which is harmless.
template <typename F>
inline cudaError_t set_smem_limit_once(F* fn, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const uint64_t bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return err;
}

size_t decode_smem_bytes();
cudaError_t launch_decode(const DecodeMaps& maps, const DecodeArgs& args, int ctas, cudaStream_t stream);
cudaError_t launch_append(const AppendArgs& args, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs& args, bool has_special, int num_sms, cudaStream_t stream);
cudaError_t launch_release(const CacheView& cv, int b, cudaStream_t stream);
cudaError_t launch_build_masks(const float* alpha, const uint8_t* eligible, int nh, double pct, int align,
                               int exact, uint8_t* masks, cudaStream_t stream);

}  // namespace lk
