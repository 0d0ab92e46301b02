// Cache editing: append one token per sequence, and prefill a layer from a
// dense history.  Pure data movement; every copy is bit-exact.
//
// Rules (LeanK article, framerc.cn, section 3.1 "cache partition" and 3.2;
// StreamingLLM sinks + sliding window as in the "intelligent pruning white
// paper", yyx235 blog, section 3.3.1; FastGen article, mhpn.cn, section 3.2
// stage 2), for the token at position n of sequence b:
//   FULL    n < S: sink row n.  Otherwise ring row S + (n-S) mod W; when the
//           window is full the token n-W held there leaves it first: its K
//           row is gathered to the kept channels into K_prun row n-W-S and
//           its V row copied beside it (both dropped when no channel is kept).
//   LOCAL   ring row n mod W_loc.
//   SPECIAL appended at row `count` only if its id is special.
// Prefill of n tokens writes each position where n successive appends leave
// it: sinks, the last W positions in their ring rows, the middle in K_prun.
#include <cuda_runtime.h>

#include "lk_device.cuh"
#include "lk_internal.h"
#include "lk_kernels.h"

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

__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
  grid_dependency_wait();
  grid_launch_dependents();
  const CacheView& cv = a.cv;
  const int b = blockIdx.x;
  const int layer = a.layer + (int)blockIdx.y;
  const int lb = layer * cv.B + b;
  const uint16_t* k_in = a.k + (size_t)blockIdx.y * cv.B * cv.Hkv * kHeadDim;
  const uint16_t* v_in = a.v + (size_t)blockIdx.y * cv.B * cv.Hkv * kHeadDim;
  __shared__ int s_n, s_cnt, s_special, s_ok;
  if (threadIdx.x == 0) {
    const int n = __ldcg(&cv.len[lb]);
    int special = 0;
    if (a.ids != nullptr) {
      const int id = a.ids[b];
      if (id >= 0 && id < cv.vocab) {
        special = cv.is_special[id] ? 1 : 0;
      } else {
        set_status(cv, kStatusBadId);
      }
    }
    s_n = n;
    s_cnt = __ldcg(&cv.cnt[lb]);
    s_special = special;
    s_ok = n < cv.capacity;
    if (!s_ok) set_status(cv, kStatusCapacity);
  }
  __syncthreads();
  if (!s_ok) return;
  const int n = s_n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  uint16_t* ka_pool = cv.pool[kPoolK128];
  uint16_t* va_pool = cv.pool[kPoolV];
  for (int h = warp; h < cv.Hkv; h += nw) {
    const HeadDesc& hd = cv.heads[layer * cv.Hkv + h];
    const size_t src = ((size_t)b * cv.Hkv + h) * kHeadDim;
    const uint2 kx = reinterpret_cast<const uint2*>(k_in + src)[lane];
    const uint2 vx = reinterpret_cast<const uint2*>(v_in + src)[lane];
    const int64_t abase = hd.row_a + (int64_t)b * hd.cap_a;
    int64_t row = -1;
    if (hd.policy == kFull) {
      int slot = n;
      if (n >= cv.S) {
        slot = cv.S + (n - cv.S) % cv.W;
        if (n - cv.S >= cv.W && hd.n_kept > 0) {
          const int mid = n - cv.W - cv.S;               // K_prun row of token n - W
          const uint16_t* k_old = ka_pool + (abase + slot) * kHeadDim;
          const uint2 v_old = row8(va_pool, abase + slot)[lane];
          write_middle(cv, hd, cv.kept + ((size_t)layer * cv.Hkv + h) * kHeadDim,
                       hd.krow_b + (int64_t)b * hd.cap_b + mid, hd.vrow_b + (int64_t)b * hd.cap_b + mid,
                       k_old, v_old, lane);
          __syncwarp();
        }
      }
      row = abase + slot;
    } else if (hd.policy == kLocal) {
      row = abase + n % cv.W_loc;
    } else if (s_special) {
      if (s_cnt < hd.cap_a) {
        row = abase + s_cnt;
      } else if (lane == 0) {
        set_status(cv, kStatusCapacity);
      }
    }
    if (row >= 0) {
      row8(ka_pool, row)[lane] = kx;
      row8(va_pool, row)[lane] = vx;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    cv.len[lb] = n + 1;
    if (s_special && s_cnt < cv.spec_cap) cv.cnt[lb] = s_cnt + 1;
  }
}

// The layer's per-sequence lengths are already in len[layer][b] (the host
// enqueues them first); inputs are padded to n_max tokens per sequence.
__global__ void __launch_bounds__(256) prefill_kernel(const PrefillArgs a) {
  grid_dependency_wait();
  const CacheView& cv = a.cv;
  const int nmax = a.n;
  const int lane = threadIdx.x & 31;
  const int64_t items = (int64_t)cv.B * nmax * cv.Hkv;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  uint16_t* ka_pool = cv.pool[kPoolK128];
  uint16_t* va_pool = cv.pool[kPoolV];
  for (int64_t it = (((int64_t)blockIdx.x * blockDim.x) + threadIdx.x) >> 5; it < items; it += nwarps) {
    const int h = (int)(it % cv.Hkv);
    const int64_t bt = it / cv.Hkv;              // b * n_max + t
    const int t = (int)(bt % nmax);
    const int b = (int)(bt / nmax);
    const int n = __ldcg(&cv.len[a.layer * cv.B + b]);
    if (t >= n) continue;
    const HeadDesc& hd = cv.heads[a.layer * cv.Hkv + h];
    const uint16_t* k_src = a.k + (size_t)it * kHeadDim;
    const uint16_t* v_src = a.v + (size_t)it * kHeadDim;
    const int64_t abase = hd.row_a + (int64_t)b * hd.cap_a;
    int64_t arow = -1, mid = -1;
    if (hd.policy == kFull) {
      if (t < cv.S) arow = t;
      else if (t >= n - cv.W) arow = cv.S + (t - cv.S) % cv.W;
      else if (hd.n_kept > 0) mid = t - cv.S;
    } else if (hd.policy == kLocal) {
      if (t >= n - cv.W_loc) arow = t % cv.W_loc;
    }
    if (arow >= 0) {
      row8(ka_pool, abase + arow)[lane] = reinterpret_cast<const uint2*>(k_src)[lane];
      row8(va_pool, abase + arow)[lane] = reinterpret_cast<const uint2*>(v_src)[lane];
    } else if (mid >= 0) {
      write_middle(cv, hd, cv.kept + ((size_t)a.layer * cv.Hkv + h) * kHeadDim,
                   hd.krow_b + (int64_t)b * hd.cap_b + mid, hd.vrow_b + (int64_t)b * hd.cap_b + mid,
                   k_src, reinterpret_cast<const uint2*>(v_src)[lane], lane);
    }
  }
}

// SPECIAL heads: one block per sequence ranks the special tokens in position
// order (ballot + warp scan per 1024-token chunk) and copies them to rows
// count, count+1, ...
__global__ void __launch_bounds__(1024) prefill_special_kernel(const PrefillArgs a) {
  grid_dependency_wait();
  const CacheView& cv = a.cv;
  const int b = blockIdx.x;
  const int nmax = a.n;
  const int n = __ldcg(&cv.len[a.layer * cv.B + b]);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ int s_warp[32];
  __shared__ int s_total;
  __shared__ int s_tok[1024];
  int base = 0;
  for (int c0 = 0; c0 < n; c0 += 1024) {
    const int t = c0 + tid;
    bool flag = false;
    if (t < n && a.ids != nullptr) {
      const int id = a.ids[(size_t)b * nmax + t];
      if (id >= 0 && id < cv.vocab) flag = cv.is_special[id] != 0;
      else set_status(cv, kStatusBadId);
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, flag);
    const int wrank = __popc(ballot & ((1u << lane) - 1u));
    if (lane == 0) s_warp[warp] = __popc(ballot);
    __syncthreads();
    if (warp == 0) {
      const int v = s_warp[lane];
      int incl = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += u;
      }
      s_warp[lane] = incl - v;
      if (lane == 31) s_total = incl;
    }
    __syncthreads();
    if (flag) s_tok[s_warp[warp] + wrank] = t;
    const int total = s_total;
    __syncthreads();
    for (int it = warp; it < total * cv.Hkv; it += 32) {
      const int j = it / cv.Hkv, h = it - j * cv.Hkv;
      const HeadDesc& hd = cv.heads[a.layer * cv.Hkv + h];
      if (hd.policy != kSpecial) continue;
      const int r = base + j;
      if (r >= hd.cap_a) {
        if (lane == 0) set_status(cv, kStatusCapacity);
        continue;
      }
      const size_t src = (((size_t)b * nmax + s_tok[j]) * cv.Hkv + h) * kHeadDim;
      const int64_t row = hd.row_a + (int64_t)b * hd.cap_a + r;
      row8(cv.pool[kPoolK128], row)[lane] = reinterpret_cast<const uint2*>(a.k + src)[lane];
      row8(cv.pool[kPoolV], row)[lane] = reinterpret_cast<const uint2*>(a.v + src)[lane];
    }
    base += total;
    __syncthreads();
  }
  if (tid == 0) cv.cnt[a.layer * cv.B + b] = min(base, cv.spec_cap);
}

}  // namespace

cudaError_t launch_append(const AppendArgs& args, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(args.cv.B, args.nlayers);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_kernel, args);
}

cudaError_t launch_prefill(const PrefillArgs& args, bool has_special, int num_sms, cudaStream_t stream) {
  const int64_t items = (int64_t)args.cv.B * args.n * args.cv.Hkv;
  int64_t blocks = (items + 7) / 8;
  if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
  if (blocks < 1) blocks = 1;
  prefill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(args);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || !has_special) return err;
  prefill_special_kernel<<<args.cv.B, 1024, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace lk
