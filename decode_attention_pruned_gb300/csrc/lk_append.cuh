// Cache editing shared by the append kernel and the fused append + decode
// kernel: the per-head append of one token, with the paged and INT8 / FP8 paths
// (LeanK article, framerc.cn, sections 3.1-3.2; FastGen article, mhpn.cn,
// section 3.2 stage 2; KIVI-style sealing after the pruning, LeanK section
// 4.2 and the pruning white paper's section 5.2.1).  Every helper is
// file-local to the translation unit that includes this header.
#pragma once
#include <cuda_runtime.h>

#include "lk_internal.h"

namespace lk {
namespace {

__device__ __forceinline__ void set_status(const CacheView& cv, uint32_t bits) {
  atomicOr(&cv.hdr->status, bits);
}

__device__ __forceinline__ const uint2* row8(const uint16_t* base, int64_t row) {
  return reinterpret_cast<const uint2*>(base + row * kHeadDim);
}
__device__ __forceinline__ uint2* row8(uint16_t* base, int64_t row) {
  return reinterpret_cast<uint2*>(base + row * kHeadDim);
}

// Warp copies one middle token: K gathered to the kept channels, V whole.
__device__ __forceinline__ void write_middle(const CacheView& cv, const HeadDesc& hd, const int16_t* kept,
                                             int64_t brow_k, int64_t brow_v, const uint16_t* k_src,
                                             uint2 v_word, int lane) {
  uint16_t* kb = cv.pool[hd.pool_kb] + brow_k * hd.n_kept;
  for (int j = lane; j < hd.n_kept; j += 32) kb[j] = k_src[kept[j]];
  row8(cv.pool[kPoolV], brow_v)[lane] = v_word;
}

__device__ __forceinline__ int32_t* page_row(const CacheView& cv, int layer, int b, int h) {
  return cv.page_table + (((int64_t)layer * cv.B + b) * cv.Hkv + h) * cv.max_pages;
}

// Pops `k` pages of the head's class into dst[0..k) (page ids in the order the
// stack hands them out); on an empty stack restores the top, fills -1 and
// records kStatusCapacity.
__device__ void pop_pages(const CacheView& cv, const HeadDesc& hd, int k, int32_t* dst) {
  if (k <= 0) return;
  int* top = &cv.hdr->free_top[hd.pool_kb];
  const int t = atomicSub(top, k);
  if (t < k) {
    atomicAdd(top, k);
    set_status(cv, kStatusCapacity);
    for (int i = 0; i < k; ++i) dst[i] = -1;
    return;
  }
  for (int i = 0; i < k; ++i) dst[i] = __ldcg(&cv.free_list[hd.free_off + t - 1 - i]);
}

// K_prun / V rows of middle row `mid` of sequence b of a head; `page` is the
// page holding it (paged caches).  False if that page is missing (a pop found
// no free page).
__device__ __forceinline__ bool middle_rows(const CacheView& cv, const HeadDesc& hd, int b, int mid, int32_t page,
                                            int64_t& krow, int64_t& vrow) {
  if (kv_quantized(cv.kv_format)) {        // the open block: bf16 tail row mid mod 128
    krow = hd.krow_b + (int64_t)b * hd.cap_b + mid % kQBlockRows;
    vrow = hd.vrow_b + (int64_t)b * hd.cap_b + mid % kQBlockRows;
    return true;
  }
  if (cv.max_pages == 0) {
    krow = hd.krow_b + (int64_t)b * hd.cap_b + mid;
    vrow = hd.vrow_b + (int64_t)b * hd.cap_b + mid;
    return true;
  }
  if (page < 0) return false;
  const int64_t r = (int64_t)page * kPageRows + mid % kPageRows;
  krow = hd.krow_b + r;
  vrow = hd.vrow_b + r;
  return true;
}

// Region-B pages a (FULL, k > 0) head holds at n tokens: started pages
// (bf16) or sealed blocks (INT8 / FP8).
__device__ __forceinline__ int pages_at(const CacheView& cv, int n) {
  const int m = max(0, n - cv.S - cv.W);
  return kv_quantized(cv.kv_format) ? m / kQBlockRows : (m + kPageRows - 1) / kPageRows;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Symmetric INT8 code of x for scale s (s = max|x| / 127 in fp32): x / s in
// fp32 rounded half to even, clipped to [-127, 127]; s = 0 gives 0.
__device__ __forceinline__ int8_t quant8(float x, float s) {
  if (!(s > 0.f)) return 0;
  const int q = __float2int_rn(__fdiv_rn(x, s));
  return (int8_t)max(-127, min(127, q));
}

// e4m3 code of x for scale s (s = max|x| / 448 in fp32): x / s in fp32,
// rounded to the nearest e4m3 value (ties to the even code) and saturated at
// +-448 by the conversion instruction; a zero code keeps the sign of x;
// s = 0 gives 0.
__device__ __forceinline__ uint8_t quant_e4m3(float x, float s) {
  if (!(s > 0.f)) return 0;
  const float y = __fdiv_rn(x, s);
  uint16_t pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.f), "f"(y));
  uint8_t c = (uint8_t)(pair & 0xFFu);
  if ((c & 0x7Fu) == 0) c = signbit(y) ? 0x80 : 0x00;
  return c;
}

// Device address of sealed block j of (layer, b, h); null if its page is
// missing.
__device__ __forceinline__ uint8_t* qblock_addr(const CacheView& cv, const HeadDesc& hd, int layer, int b, int h,
                                                int j) {
  const int qb = qblock_bytes(hd.n_kept);
  if (cv.max_pages == 0) return cv.qpool + hd.qoff + ((int64_t)b * hd.qblocks + j) * qb;
  const int32_t page = __ldcg(&page_row(cv, layer, b, h)[j]);
  return page < 0 ? nullptr : cv.qpool + hd.qoff + (int64_t)page * qb;
}

// One warp seals a 128-row block in format fmt (INT8 or FP8): kv(r, c) /
// vv(r, c) give the bf16 bits of K row r at kept channel c (c < k) and of V
// row r at channel c.  K: one scale per channel (lane per channel); V: one
// scale per row (lane per four channels, warp max).  Codes go to their
// swizzled byte (qbyte).
template <class KF, class VF>
__device__ void seal_block(uint8_t* dst, int k, int fmt, KF kv, VF vv, int lane) {
  float* ks = reinterpret_cast<float*>(dst + qblock_ksoff(k));
  float* vs = reinterpret_cast<float*>(dst + qblock_vsoff(k));
  const bool fp8 = fmt == kKvFp8;
  const float qmax = fp8 ? 448.f : 127.f;
  for (int c = lane; c < k; c += 32) {
    float m = 0.f;
    for (int r = 0; r < kQBlockRows; ++r) m = fmaxf(m, fabsf(bf16_to_f32(kv(r, c))));
    const float sc = __fdiv_rn(m, qmax);
    ks[c] = sc;
    for (int r = 0; r < kQBlockRows; ++r) {
      const float x = bf16_to_f32(kv(r, c));
      dst[r * k + qbyte(k, r, c)] = fp8 ? quant_e4m3(x, sc) : (uint8_t)quant8(x, sc);
    }
  }
  uint8_t* vc = dst + qblock_voff(k);
  for (int r = 0; r < kQBlockRows; ++r) {
    float x[4];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[i] = bf16_to_f32(vv(r, 4 * lane + i));
      m = fmaxf(m, fabsf(x[i]));
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, sh));
    const float sc = __fdiv_rn(m, qmax);
    if (lane == 0) vs[r] = sc;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      vc[r * kHeadDim + qbyte(kHeadDim, r, 4 * lane + i)] =
          fp8 ? quant_e4m3(x[i], sc) : (uint8_t)(quant8(x[i], sc) + 128);   // INT8: offset binary
  }
}

// One warp appends token n of sequence b to kv head h of `layer`: k_src /
// v_src are its bf16 rows [128]; cnt / special are the layer's special-row
// count and whether the token's id is special.  FULL: sink row n, or ring
// row S + (n-S) mod W after moving the token n-W it replaces into the middle
// (K gathered to the kept channels; INT8 / FP8 caches write the bf16 tail and
// seal it into a block when it fills).  LOCAL: ring row n mod W_loc.
// SPECIAL: row cnt if the token is special.  The caller updates len / cnt
// afterwards.  kWithQ8 = false compiles the quantised paths out (callers that
// never see a quantised cache).  k_old / v_old / kept, when given, are copies
// of the evicted window row and of the head's kept-channel list (e.g. in
// shared memory) to read instead of the cache.
template <bool kWithQ8>
__device__ void append_head(const CacheView& cv, int layer, int b, int h, int n, int cnt, bool special,
                            const uint16_t* k_src, const uint16_t* v_src, int lane,
                            const uint16_t* k_old_src = nullptr, const uint16_t* v_old_src = nullptr,
                            const int16_t* kept_src = nullptr) {
  const HeadDesc& hd = cv.heads[layer * cv.Hkv + h];
  const uint2 kx = reinterpret_cast<const uint2*>(k_src)[lane];
  const uint2 vx = reinterpret_cast<const uint2*>(v_src)[lane];
  uint16_t* ka_pool = cv.pool[kPoolK128];
  uint16_t* va_pool = cv.pool[kPoolV];
  const int64_t abase = hd.row_a + (int64_t)b * hd.cap_a;
  int64_t row = -1;
  if (hd.policy == kFull) {
    int slot = n;
    if (n >= cv.S) {
      slot = cv.S + (n - cv.S) % cv.W;
      if (n - cv.S >= cv.W && hd.n_kept > 0) {
        const int mid = n - cv.W - cv.S;               // K_prun row of token n - W
        int32_t page = -1;
        if (cv.max_pages > 0 && !(kWithQ8 && kv_quantized(cv.kv_format))) {
          int32_t* pt = page_row(cv, layer, b, h) + mid / kPageRows;
          if (mid % kPageRows == 0) {         // first row of a new page
            if (lane == 0) {
              pop_pages(cv, hd, 1, &page);
              *pt = page;
            }
            page = __shfl_sync(0xffffffffu, page, 0);
          } else {
            page = __ldcg(pt);
          }
        }
        int64_t krow, vrow;
        if (middle_rows(cv, hd, b, mid, page, krow, vrow)) {
          const uint16_t* k_old = k_old_src != nullptr ? k_old_src : ka_pool + (abase + slot) * kHeadDim;
          const uint2 v_old = v_old_src != nullptr ? reinterpret_cast<const uint2*>(v_old_src)[lane]
                                                   : row8(va_pool, abase + slot)[lane];
          const int16_t* kept = kept_src != nullptr ? kept_src : cv.kept + ((size_t)layer * cv.Hkv + h) * kHeadDim;
          write_middle(cv, hd, kept, krow, vrow, k_old, v_old, lane);
        }
        __syncwarp();
        if (kWithQ8 && kv_quantized(cv.kv_format) && mid % kQBlockRows == kQBlockRows - 1) {
          // the tail block is complete: seal it into block mid / 128
          const int j = mid / kQBlockRows;
          uint8_t* dst;
          if (cv.max_pages > 0) {
            int32_t pg = -1;
            if (lane == 0) {
              pop_pages(cv, hd, 1, &pg);
              page_row(cv, layer, b, h)[j] = pg;
            }
            pg = __shfl_sync(0xffffffffu, pg, 0);
            dst = pg < 0 ? nullptr : cv.qpool + hd.qoff + (int64_t)pg * qblock_bytes(hd.n_kept);
          } else {
            dst = qblock_addr(cv, hd, layer, b, h, j);
          }
          if (dst != nullptr) {
            const int k = hd.n_kept;
            const uint16_t* kt = cv.pool[hd.pool_kb] + (hd.krow_b + (int64_t)b * hd.cap_b) * k;
            const uint16_t* vt = va_pool + (hd.vrow_b + (int64_t)b * hd.cap_b) * kHeadDim;
            seal_block(
                dst, k, cv.kv_format, [&](int r, int c) { return kt[(size_t)r * k + c]; },
                [&](int r, int c) { return vt[(size_t)r * kHeadDim + c]; }, lane);
            __syncwarp();
            // the open block restarts empty (zeros), as a prefill leaves it
            uint4* kz = reinterpret_cast<uint4*>(cv.pool[hd.pool_kb] + (hd.krow_b + (int64_t)b * hd.cap_b) * k);
            uint4* vz = reinterpret_cast<uint4*>(va_pool + (hd.vrow_b + (int64_t)b * hd.cap_b) * kHeadDim);
            const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
            for (int i = lane; i < kQBlockRows * k / 8; i += 32) kz[i] = zero;
            for (int i = lane; i < kQBlockRows * kHeadDim / 8; i += 32) vz[i] = zero;
          }
          __syncwarp();
        }
      }
    }
    row = abase + slot;
  } else if (hd.policy == kLocal) {
    row = abase + n % cv.W_loc;
  } else if (special) {
    if (cnt < hd.cap_a) {
      row = abase + cnt;
    } else if (lane == 0) {
      set_status(cv, kStatusCapacity);
    }
  }
  if (row >= 0) {
    row8(ka_pool, row)[lane] = kx;
    row8(va_pool, row)[lane] = vx;
  }
}

}  // namespace
}  // namespace lk
