// The static channel mask beta from learned importances alpha, on the device
// (LeanK article, framerc.cn, section 2.2 stage 2 "hardware-friendly mask"):
// a global percentile threshold over the eligible alphas, per-head kept
// counts brought to a multiple of the alignment (rounded down, or topped up
// to the exact aligned budget by largest remainder), and each head's top
// channels (equal alphas: lower channel index first).
//
// One CTA does it all; the data is small (L*H*128 floats).
//   1. Radix select (4 passes of 8 bits over order-preserving uint32 keys)
//      finds the two order statistics around position s/100 * (n-1).
//   2. threshold = x_i + frac * (x_j - x_i) in fp32 with no fused
//      multiply-add: it decides integer counts, so it is computed exactly as
//      the reference computes it.
//   3. A warp per head counts alpha >= threshold (ballot) and rounds down.
//   4. Exact budget: heads sorted by (remainder desc, index asc) with a
//      bitonic sort in shared memory, then +align handed out in that order.
//   5. A warp per head ranks its 128 channels and keeps the top ones.
#include <cuda_runtime.h>
#include <math.h>

#include "lk_internal.h"
#include "lk_kernels.h"

namespace lk {
namespace {

constexpr int kThreadsM = 1024;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

struct MaskArgs {
  const float* alpha;       // [L*H][128]
  const uint8_t* eligible;  // [L*H] or null
  uint8_t* masks;           // [L*H][128]
  int nh;                   // L * H
  double pct;
  int align;
  int exact;
};

__device__ __forceinline__ bool head_eligible(const MaskArgs& a, int h) {
  return a.eligible == nullptr || a.eligible[h] != 0;
}

// Key of the rank-th smallest eligible alpha (rank < n).
__device__ uint32_t radix_select(const MaskArgs& a, uint32_t rank, uint32_t* hist) {
  uint32_t prefix = 0, mask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < a.nh * kHeadDim; i += blockDim.x) {
      if (!head_eligible(a, i >> 7)) continue;
      const uint32_t k = order_key(a.alpha[i]);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    __shared__ uint32_t s_bin, s_below;
    if (threadIdx.x == 0) {
      uint32_t acc = 0, bin = 255;
      for (uint32_t b = 0; b < 256; ++b) {
        if (acc + hist[b] > rank) {
          bin = b;
          break;
        }
        acc += hist[b];
      }
      s_bin = bin;
      s_below = acc;
    }
    __syncthreads();
    rank -= s_below;
    prefix |= s_bin << shift;
    mask |= 0xFFu << shift;
    __syncthreads();
  }
  return prefix;
}

__global__ void __launch_bounds__(kThreadsM, 1) build_masks_kernel(const MaskArgs a) {
  extern __shared__ uint8_t smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);                    // [256]
  uint32_t* keys = hist + 256;                                           // [pow2 >= nh]
  uint8_t* above = reinterpret_cast<uint8_t*>(keys + 8192);              // [nh]
  uint8_t* keep = above + 8192;                                          // [nh]
  __shared__ int s_neligible;
  __shared__ float s_thr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;

  if (tid == 0) s_neligible = 0;
  __syncthreads();
  int local = 0;
  for (int h = tid; h < a.nh; h += blockDim.x) local += head_eligible(a, h) ? 1 : 0;
  atomicAdd(&s_neligible, local);
  __syncthreads();
  const int ne = s_neligible;
  const uint32_t n = (uint32_t)ne * kHeadDim;

  // ---- 1-2. percentile threshold
  if (n > 0) {
    const double pos = a.pct / 100.0 * (double)(n - 1);
    const uint32_t i = (uint32_t)floor(pos);
    const uint32_t j = min(i + 1, n - 1);
    const float xi = key_value(radix_select(a, i, hist));
    const float xj = key_value(radix_select(a, j, hist));
    if (tid == 0) {
      const float frac = (float)(pos - (double)i);
      s_thr = __fadd_rn(xi, __fmul_rn(frac, __fsub_rn(xj, xi)));
    }
  } else if (tid == 0) {
    s_thr = INFINITY;
  }
  __syncthreads();
  const float thr = s_thr;

  // ---- 3. per-head counts
  for (int h = warp; h < a.nh; h += nwarps) {
    const float* row = a.alpha + (size_t)h * kHeadDim;
    int cnt = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) cnt += __popc(__ballot_sync(0xffffffffu, row[q * 32 + lane] >= thr));
    if (lane == 0) {
      above[h] = (uint8_t)cnt;
      keep[h] = head_eligible(a, h) ? (uint8_t)(cnt / a.align * a.align) : (uint8_t)kHeadDim;
    }
  }
  __syncthreads();

  // ---- 4. exact budget: largest remainders first, ties by head index
  if (a.exact && ne > 0) {
    int pow2 = 1;
    while (pow2 < a.nh) pow2 <<= 1;
    for (int h = tid; h < pow2; h += blockDim.x) {
      if (h < a.nh) {
        const int rem = head_eligible(a, h) ? (int)above[h] - (int)keep[h] : -1;
        keys[h] = ((uint32_t)(127 - rem) << 13) | (uint32_t)h;
      } else {
        keys[h] = 0xFFFFFFFFu;
      }
    }
    __syncthreads();
    for (int size = 2; size <= pow2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int t = tid; t < pow2; t += blockDim.x) {
          const int p = t ^ stride;
          if (p > t) {
            const bool up = (t & size) == 0;
            const uint32_t x = keys[t], y = keys[p];
            if ((x > y) == up) {
              keys[t] = y;
              keys[p] = x;
            }
          }
        }
        __syncthreads();
      }
    }
    if (tid == 0) {
      long long total = 0;
      for (int h = 0; h < a.nh; ++h)
        if (head_eligible(a, h)) total += keep[h];
      const long long target =
          (long long)a.align * (long long)floor((1.0 - a.pct / 100.0) * ne * 128.0 / a.align + 0.5);
      long long deficit = target - total;
      while (deficit > 0) {
        bool given = false;
        for (int r = 0; r < a.nh && deficit > 0; ++r) {
          const int h = (int)(keys[r] & 0x1FFFu);
          if (head_eligible(a, h) && keep[h] + a.align <= kHeadDim) {
            keep[h] = (uint8_t)(keep[h] + a.align);
            deficit -= a.align;
            given = true;
          }
        }
        if (!given) break;
      }
    }
    __syncthreads();
  }

  // ---- 5. each head keeps its top `keep` channels
  for (int h = warp; h < a.nh; h += nwarps) {
    const float* row = a.alpha + (size_t)h * kHeadDim;
    float mine[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) mine[q] = row[q * 32 + lane];
    int rank[4] = {0, 0, 0, 0};
    for (int src = 0; src < kHeadDim; ++src) {
      const float v = __shfl_sync(0xffffffffu, mine[src >> 5], src & 31);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = q * 32 + lane;
        rank[q] += (v > mine[q] || (v == mine[q] && src < c)) ? 1 : 0;
      }
    }
    const int kh = keep[h];
#pragma unroll
    for (int q = 0; q < 4; ++q) a.masks[(size_t)h * kHeadDim + q * 32 + lane] = rank[q] < kh ? 1 : 0;
  }
}

constexpr int kMaskSmem = 256 * 4 + 8192 * 4 + 8192 * 2;

}  // namespace

cudaError_t launch_build_masks(const float* alpha, const uint8_t* eligible, int nh, double pct, int align,
                               int exact, uint8_t* masks, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t err = set_smem_limit_once(build_masks_kernel, kMaskSmem, attr_done);
  if (err != cudaSuccess) return err;
  MaskArgs a{alpha, eligible, masks, nh, pct, align, exact};
  build_masks_kernel<<<1, kThreadsM, kMaskSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace lk
