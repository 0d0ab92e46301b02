// Cache editing: append one token per sequence, and prefill a layer from a
// dense history.  Pure data movement (every bf16 copy is bit-exact) plus the
// INT8 / FP8 sealing of complete middle blocks.
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
//
// Paged caches hold the middle of each (layer, sequence, head) in 128-row
// pages of its width class: an append whose eviction starts a new page pops
// one from the class's free stack (an atomic on the stack top), prefill pops
// all the pages a sequence needs at once, and release pushes them back.  The
// host checks that enough pages are free before it launches, so a pop that
// finds the stack empty only records kStatusCapacity.
//
// INT8 / FP8 caches (KIVI-style quantisation after the pruning; LeanK article
// sections 4.2 and 5.2, the white paper's section 5.2.1): middle rows go to a
// 128-row bf16 tail; the append that fills its last row seals it into a byte
// block of the Q pool (per-channel K and per-token V scales, absmax / 127 in
// fp32 and codes x / scale rounded half to even for INT8; absmax / 448 and
// codes x / scale rounded to the nearest e4m3 value for FP8) and clears the
// tail.  Prefill
// seals complete blocks straight from its inputs, so both give the same
// bytes; with paging the sealed blocks are the pages.
#include <cuda_runtime.h>

#include "lk_append.cuh"
#include "lk_device.cuh"
#include "lk_internal.h"
#include "lk_kernels.h"

namespace lk {
namespace {

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
    // a released slot takes no tokens until it is prefilled again
    s_ok = __ldcg(&cv.active[b]) != 0;
    if (s_ok && n >= cv.capacity) {
      s_ok = 0;
      set_status(cv, kStatusCapacity);
    }
  }
  __syncthreads();
  if (!s_ok) return;
  const int n = s_n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int h = warp; h < cv.Hkv; h += nw) {
    const size_t src = ((size_t)b * cv.Hkv + h) * kHeadDim;
    append_head<true>(cv, layer, b, h, n, s_cnt, s_special != 0, k_in + src, v_in + src, lane);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    cv.len[lb] = n + 1;
    if (s_special && s_cnt < cv.spec_cap) cv.cnt[lb] = s_cnt + 1;
  }
}

// The layer's per-sequence lengths are already in len[layer][b] (the host
// enqueues them first); inputs are padded to n_max tokens per sequence.
// Sequences b0 .. b0 + nb - 1 are filled; input sequence i is sequence b0 + i.
__global__ void __launch_bounds__(256) prefill_kernel(const PrefillArgs a) {
  grid_dependency_wait();
  const CacheView& cv = a.cv;
  const int nmax = a.n;
  const int lane = threadIdx.x & 31;
  const int64_t items = (int64_t)a.nb * nmax * cv.Hkv;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  uint16_t* ka_pool = cv.pool[kPoolK128];
  uint16_t* va_pool = cv.pool[kPoolV];
  for (int64_t it = (((int64_t)blockIdx.x * blockDim.x) + threadIdx.x) >> 5; it < items; it += nwarps) {
    const int h = (int)(it % cv.Hkv);
    const int64_t bt = it / cv.Hkv;              // i * n_max + t
    const int t = (int)(bt % nmax);
    const int b = a.b0 + (int)(bt / nmax);
    const int n = __ldcg(&cv.len[a.layer * cv.B + b]);
    if (t >= n) continue;
    const HeadDesc& hd = cv.heads[a.layer * cv.Hkv + h];
    const uint16_t* k_src = a.k + (size_t)it * kHeadDim;
    const uint16_t* v_src = a.v + (size_t)it * kHeadDim;
    const int64_t abase = hd.row_a + (int64_t)b * hd.cap_a;
    int arow = -1, mid = -1;
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
      // INT8 / FP8: rows of complete blocks are sealed from the inputs by
      // prefill_seal_kernel; only the open block's rows go to the bf16 tail
      if (kv_quantized(cv.kv_format) && mid < (n - cv.S - cv.W) / kQBlockRows * kQBlockRows) continue;
      const int32_t page = cv.max_pages > 0 && cv.kv_format == kKvBf16
                               ? __ldcg(&page_row(cv, a.layer, b, h)[mid / kPageRows])
                               : -1;
      int64_t krow, vrow;
      if (middle_rows(cv, hd, b, mid, page, krow, vrow))
        write_middle(cv, hd, cv.kept + ((size_t)a.layer * cv.Hkv + h) * kHeadDim, krow, vrow, k_src,
                     reinterpret_cast<const uint2*>(v_src)[lane], lane);
    }
  }
}

// Paged caches: before the copy, each (sequence, FULL head with k > 0) of the
// range pops the pages its middle rows need (the slots are empty).
__global__ void __launch_bounds__(256) prefill_pages_kernel(const PrefillArgs a) {
  grid_dependency_wait();
  const CacheView& cv = a.cv;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.nb * cv.Hkv) return;
  const int b = a.b0 + i / cv.Hkv, h = i % cv.Hkv;
  const HeadDesc& hd = cv.heads[a.layer * cv.Hkv + h];
  if (hd.policy != kFull || hd.n_kept == 0) return;
  const int n = __ldcg(&cv.len[a.layer * cv.B + b]);
  pop_pages(cv, hd, min(pages_at(cv, n), cv.max_pages), page_row(cv, a.layer, b, h));
}

// INT8 / FP8 caches: a warp per (sequence, head, complete block) quantises the
// block straight from the prefill inputs (K gathered to the kept channels),
// exactly as appends seal it from the bf16 tail.
__global__ void __launch_bounds__(256) prefill_seal_kernel(const PrefillArgs a, int max_blocks) {
  grid_dependency_wait();
  const CacheView& cv = a.cv;
  const int lane = threadIdx.x & 31;
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (w >= (int64_t)a.nb * cv.Hkv * max_blocks) return;
  const int j = (int)(w % max_blocks);
  const int h = (int)((w / max_blocks) % cv.Hkv);
  const int i = (int)(w / ((int64_t)max_blocks * cv.Hkv));
  const int b = a.b0 + i;
  const HeadDesc& hd = cv.heads[a.layer * cv.Hkv + h];
  if (hd.policy != kFull || hd.n_kept == 0) return;
  const int n = __ldcg(&cv.len[a.layer * cv.B + b]);
  if (j >= pages_at(cv, n)) return;
  uint8_t* dst = qblock_addr(cv, hd, a.layer, b, h, j);
  if (dst == nullptr) return;
  const int16_t* kept = cv.kept + ((size_t)a.layer * cv.Hkv + h) * kHeadDim;
  const int t0 = cv.S + j * kQBlockRows;
  const uint16_t* kin = a.k + (((size_t)i * a.n + t0) * cv.Hkv + h) * kHeadDim;
  const uint16_t* vin = a.v + (((size_t)i * a.n + t0) * cv.Hkv + h) * kHeadDim;
  const size_t rs = (size_t)cv.Hkv * kHeadDim;
  seal_block(
      dst, hd.n_kept, cv.kv_format, [&](int r, int c) { return kin[r * rs + kept[c]]; },
      [&](int r, int c) { return vin[r * rs + c]; }, lane);
}

// Empties slot b in every layer (block = layer): pushes its pages back on
// their class stacks, clears the page table, lengths and special counts, and
// marks the slot released.
__global__ void __launch_bounds__(128) release_kernel(const CacheView cv, int b) {
  const int layer = blockIdx.x;
  const int lb = layer * cv.B + b;
  const int n = __ldcg(&cv.len[lb]);
  if (cv.max_pages > 0) {
    for (int h = threadIdx.x; h < cv.Hkv; h += blockDim.x) {
      const HeadDesc& hd = cv.heads[layer * cv.Hkv + h];
      if (hd.policy != kFull || hd.n_kept == 0) continue;
      const int k = min(cv.max_pages, pages_at(cv, n));
      int32_t* pt = page_row(cv, layer, b, h);
      if (k > 0) {
        const int t = atomicAdd(&cv.hdr->free_top[hd.pool_kb], k);
        // reversed, so the next pops hand the pages out in table order
        for (int i = 0; i < k; ++i) cv.free_list[hd.free_off + t + i] = pt[k - 1 - i];
      }
      for (int i = 0; i < k; ++i) pt[i] = -1;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    cv.len[lb] = 0;
    cv.cnt[lb] = 0;
    if (layer == 0) cv.active[b] = 0;
  }
}

// SPECIAL heads: one block per sequence ranks the special tokens in position
// order (ballot + warp scan per 1024-token chunk) and copies them to rows
// count, count+1, ...
__global__ void __launch_bounds__(1024) prefill_special_kernel(const PrefillArgs a) {
  grid_dependency_wait();
  const CacheView& cv = a.cv;
  const int i = blockIdx.x;               // input sequence
  const int b = a.b0 + i;
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
      const int id = a.ids[(size_t)i * nmax + t];
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
      const size_t src = (((size_t)i * nmax + s_tok[j]) * cv.Hkv + h) * kHeadDim;
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
  if (args.cv.max_pages > 0) {
    const int threads = args.nb * args.cv.Hkv;
    prefill_pages_kernel<<<(threads + 255) / 256, 256, 0, stream>>>(args);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  const int64_t items = (int64_t)args.nb * args.n * args.cv.Hkv;
  int64_t blocks = (items + 7) / 8;
  if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
  if (blocks < 1) blocks = 1;
  prefill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(args);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (kv_quantized(args.cv.kv_format)) {
    const int max_blocks = max(0, args.n - args.cv.S - args.cv.W) / kQBlockRows;
    const int64_t warps = (int64_t)args.nb * args.cv.Hkv * max_blocks;
    if (warps > 0) {
      prefill_seal_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(args, max_blocks);
      err = cudaGetLastError();
      if (err != cudaSuccess) return err;
    }
  }
  if (!has_special) return cudaSuccess;
  prefill_special_kernel<<<args.nb, 1024, 0, stream>>>(args);
  return cudaGetLastError();
}

cudaError_t launch_release(const CacheView& cv, int b, cudaStream_t stream) {
  release_kernel<<<cv.L, 128, 0, stream>>>(cv, b);
  return cudaGetLastError();
}

}  // namespace lk
