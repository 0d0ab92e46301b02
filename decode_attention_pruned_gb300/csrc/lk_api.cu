// Host side of the C ABI declared in include/leank.h: validation, the plan
// (head grouping and kept-channel lists, LeanK article section 3.1), the
// cache layout inside the caller's buffer, TMA tensor maps and launches.
// No CPU compute path exists: every step of decode/append/prefill runs in the
// kernels of lk_decode.cu and lk_kv.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/leank.h"
#include "lk_internal.h"
#include "lk_kernels.h"

using namespace lk;

namespace {

thread_local std::string g_last_error;

lk_status fail(lk_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

lk_status cuda_fail(cudaError_t err, const char* what) {
  return fail(LK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr uint64_t kWaitLimitNs = 1000000000ull;      // 1 s bound on device waits
constexpr uint64_t kMaxWaitLimitNs = 10000000000ull;  // lk_set_wait_limit: at most 10 s
constexpr int64_t kMaxPoolRows = (1ll << 31) - 2 * kTmaBoxRows;

}  // namespace

struct lk_plan_s {
  lk_plan_desc d;
  std::vector<int32_t> policy;      // [L][Hkv]
  std::vector<int32_t> n_kept;      // [L][Hkv]
  std::vector<int16_t> kept;        // [L][Hkv][128] kept channels ascending, then the pruned ones
  std::vector<uint8_t> is_special;  // [vocab]
  std::vector<uint8_t> layer_special;
};

namespace {

struct Layout {
  size_t off_len, off_cnt, off_active, off_pt, off_free, off_heads, off_kept, off_spec, off_q;
  size_t q_bytes = 0;                    // INT8 / FP8: Q pool bytes
  int32_t kv_format = kKvBf16;
  size_t off_pool[kNumPools];
  int64_t pool_rows[kNumPools];
  size_t total;
  int32_t spec_cap;
  int32_t max_pages = 0;                 // 0: contiguous region B
  int32_t num_pages[kNumPools] = {};     // paged: pages of each width class
  int32_t free_off[kNumPools] = {};
  // decode TMA views: first row, rows per block and blocks of region A of
  // each policy class (pools K128 and V) and of region B of each pool
  int64_t a_base[3] = {}, a_blocks[3] = {};
  int32_t a_rows[3] = {};
  int64_t b_base[kNumPools] = {}, b_blocks[kNumPools] = {};
  int32_t b_rows = 0;
  std::vector<HeadDesc> heads;
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Region-B pages one (FULL, k > 0) head holds for a sequence of n tokens:
// every started page (bf16), or the sealed blocks only (INT8 / FP8; the open block
// is the head's bf16 tail).
inline int32_t pages_at(int n, int S, int W, int fmt) {
  const int m = std::max(0, n - S - W);
  return kv_quantized(fmt) ? m / kQBlockRows : (int32_t)ceil_div(m, kPageRows);
}

// middle_tokens < 0: region B contiguous per (layer, sequence, head), sized
// for `cap` tokens.  Otherwise paged: each FULL head with k > 0 gets pages for
// middle_tokens middle tokens summed over the batch, plus one partly filled
// page per sequence (and never more than batch x max_pages).
lk_status compute_layout(const lk_plan_s& p, int B, int cap, int64_t middle_tokens, int fmt, Layout* lay) {
  const lk_plan_desc& d = p.d;
  const int L = d.num_layers, H = d.num_kv_heads;
  const bool paged = middle_tokens >= 0;
  const bool q8 = kv_quantized(fmt);
  lay->kv_format = fmt;
  lay->max_pages = paged ? std::max<int32_t>(1, pages_at(cap, d.sink, d.local, fmt)) : 0;
  int64_t pages_per_head = 0;
  if (paged)
    pages_per_head = std::min<int64_t>(q8 ? middle_tokens / kQBlockRows : ceil_div(middle_tokens, kPageRows) + B,
                                       (int64_t)B * lay->max_pages);
  size_t off = align_up(sizeof(DevHeader), 1024);
  lay->off_len = off;
  off = align_up(off + (size_t)L * B * 4, 1024);
  lay->off_cnt = off;
  off = align_up(off + (size_t)L * B * 4, 1024);
  lay->off_active = off;
  off = align_up(off + (size_t)B * 4, 1024);
  lay->off_pt = off;
  off = align_up(off + (size_t)L * B * H * lay->max_pages * 4, 1024);

  lay->spec_cap = d.special_capacity > 0 ? std::min(d.special_capacity, cap) : cap;
  lay->heads.assign((size_t)L * H, HeadDesc{});
  int64_t rows[kNumPools] = {0, 0, 0, 0, 0};
  int64_t ra = 0;
  int64_t class_heads[kNumPools] = {0, 0, 0, 0, 0};
  // region A, one policy class after another: a class's rows are equal
  // blocks of cap_a rows, one per (head, sequence)
  for (int cls = kFull; cls <= kSpecial; ++cls) {
    const int32_t cap_a = cls == kFull    ? std::min(cap, d.sink + d.local)
                          : cls == kLocal ? std::min(cap, d.local_only_window)
                                          : lay->spec_cap;
    lay->a_base[cls] = ra;
    lay->a_rows[cls] = cap_a;
    int64_t blocks = 0;
    for (int i = 0; i < L * H; ++i) {
      if (p.policy[i] != cls) continue;
      HeadDesc& hd = lay->heads[i];
      hd.policy = cls;
      hd.n_kept = cls == kFull ? p.n_kept[i] : 0;
      hd.cap_a = cap_a;
      hd.row_a = ra;
      hd.blk_a = (int32_t)blocks;
      blocks += B;
      ra += (int64_t)B * cap_a;
      hd.pool_kb = kPoolK128;
      if (cls == kFull && hd.n_kept > 0) class_heads[pool_for_width(hd.n_kept)] += 1;
    }
    if (blocks > INT32_MAX) return fail(LK_ERR_CAPACITY, "%lld region-A blocks in one policy class", (long long)blocks);
    lay->a_blocks[cls] = blocks;
  }
  rows[kPoolK128] = ra;
  rows[kPoolV] = ra;
  int64_t page_k[kNumPools] = {0, 0, 0, 0, 0}, page_v[kNumPools] = {0, 0, 0, 0, 0};
  int64_t page_q[kNumPools] = {0, 0, 0, 0, 0};
  int64_t qbytes = 0;
  if (paged) {
    int64_t free_total = 0;
    for (int pl = 0; pl < kNumPools; ++pl) {
      const int64_t np = class_heads[pl] * pages_per_head;
      if (np > (int64_t)1 << 30)
        return fail(LK_ERR_CAPACITY, "width class %d needs %lld pages", pool_width(pl), (long long)np);
      lay->num_pages[pl] = (int32_t)np;
      lay->free_off[pl] = (int32_t)free_total;
      free_total += np;
      if (q8) {
        // sealed blocks are the pages; bf16 rows hold only the tails
        page_q[pl] = qbytes;
        qbytes += np * qblock_bytes(pool_width(pl));
      } else {
        page_k[pl] = rows[pl];
        rows[pl] += np * kPageRows;
        page_v[pl] = rows[kPoolV];
        rows[kPoolV] += np * kPageRows;
      }
    }
    if (free_total > ((int64_t)1 << 31) - 1) return fail(LK_ERR_CAPACITY, "%lld pages in all", (long long)free_total);
  }
  lay->off_free = off;
  {
    int64_t nfree = 0;
    for (int pl = 0; pl < kNumPools; ++pl) nfree += lay->num_pages[pl];
    off = align_up(off + (size_t)nfree * 4, 1024);
  }
  lay->off_heads = off;
  off = align_up(off + (size_t)L * H * sizeof(HeadDesc), 1024);
  lay->off_kept = off;
  off = align_up(off + (size_t)L * H * kHeadDim * 2, 1024);
  lay->off_spec = off;
  off = align_up(off + (size_t)std::max(d.vocab, 1), 1024);
  const int64_t mid_cap = std::max(0, cap - d.sink - d.local);
  for (int i = 0; i < L * H; ++i) {
    HeadDesc& hd = lay->heads[i];
    if (hd.policy == kFull && hd.n_kept > 0) {
      hd.pool_kb = pool_for_width(hd.n_kept);
      if (q8) {
        // bf16 tail of 128 rows per sequence; sealed blocks in the Q pool
        hd.cap_b = (int32_t)std::min<int64_t>(mid_cap, kQBlockRows);
        hd.krow_b = rows[hd.pool_kb];
        rows[hd.pool_kb] += (int64_t)B * hd.cap_b;
        hd.vrow_b = rows[kPoolV];
        rows[kPoolV] += (int64_t)B * hd.cap_b;
        if (paged) {
          hd.qoff = page_q[hd.pool_kb];
          hd.free_off = lay->free_off[hd.pool_kb];
          hd.qblocks = lay->max_pages;
        } else {
          hd.qblocks = (int32_t)(mid_cap / kQBlockRows);
          hd.qoff = qbytes;
          qbytes += (int64_t)B * hd.qblocks * qblock_bytes(hd.n_kept);
        }
      } else if (paged) {
        hd.cap_b = lay->max_pages * kPageRows;
        hd.krow_b = page_k[hd.pool_kb];
        hd.vrow_b = page_v[hd.pool_kb];
        hd.free_off = lay->free_off[hd.pool_kb];
      } else {
        hd.cap_b = std::max(0, cap - d.sink - d.local);
        hd.krow_b = rows[hd.pool_kb];
        rows[hd.pool_kb] += (int64_t)B * hd.cap_b;
        hd.vrow_b = rows[kPoolV];
        rows[kPoolV] += (int64_t)B * hd.cap_b;
      }
    }
  }
  // region-B views: blocks of one sequence's rows (INT8 / FP8: its bf16 tail), or
  // of one page, from the first region-B row of each pool
  {
    const int64_t rows_b = paged && !q8 ? kPageRows : q8 ? std::min<int64_t>(mid_cap, kQBlockRows) : mid_cap;
    lay->b_rows = (int32_t)std::max<int64_t>(1, rows_b);
    for (int pl = 0; pl < kNumPools; ++pl) {
      lay->b_base[pl] = pl == kPoolK128 || pl == kPoolV ? ra : 0;
      lay->b_blocks[pl] = std::max<int64_t>(1, (rows[pl] - lay->b_base[pl]) / lay->b_rows);
      if (lay->b_blocks[pl] > INT32_MAX)
        return fail(LK_ERR_CAPACITY, "pool %d needs %lld region-B blocks", pl, (long long)lay->b_blocks[pl]);
    }
    for (int i = 0; i < L * H; ++i) {
      HeadDesc& hd = lay->heads[i];
      if (hd.policy != kFull || hd.n_kept == 0 || rows_b == 0) continue;
      const int64_t kr = hd.krow_b - lay->b_base[hd.pool_kb], vr = hd.vrow_b - lay->b_base[kPoolV];
      if (kr % rows_b != 0 || vr % rows_b != 0)
        return fail(LK_ERR_STATE, "internal: region-B rows of head %d are not block aligned", i);
      hd.kblk_b = (int32_t)(kr / rows_b);
      hd.vblk_b = (int32_t)(vr / rows_b);
    }
  }
  for (int pl = 0; pl < kNumPools; ++pl) {
    const int64_t r = std::max<int64_t>(rows[pl], kTmaBoxRows);
    if (r > kMaxPoolRows)
      return fail(LK_ERR_CAPACITY, "pool %d needs %lld rows; at most %lld fit TMA coordinates", pl,
                  (long long)r, (long long)kMaxPoolRows);
    lay->pool_rows[pl] = r;
    lay->off_pool[pl] = off;
    off = align_up(off + (size_t)r * pool_width(pl) * 2, 1024);
  }
  lay->off_q = off;
  lay->q_bytes = (size_t)qbytes;
  off = align_up(off + (size_t)qbytes, 1024);
  lay->total = off;
  return LK_OK;
}

struct WsLayout {
  size_t off_counters, off_ml, off_part, off_q, off_k, off_v, off_ids, off_o, total;
};

// Workspace: split counters and partials for every (layer, sequence, kv head)
// entry (a launch may cover all layers), then the staging of lk_step_host.
WsLayout ws_layout(const lk_plan_desc& d, int B) {
  WsLayout w;
  const size_t E = (size_t)d.num_layers * B * d.num_kv_heads;
  const size_t G = (size_t)(d.num_q_heads / d.num_kv_heads);
  const size_t slots = (size_t)kMaxCtas + E;
  size_t off = 0;
  w.off_counters = off;                      // per entry, then one for the whole grid
  off = align_up(off + (E + 1) * 4, 256);
  w.off_ml = off;
  off = align_up(off + slots * G * 8, 256);
  w.off_part = off;
  off = align_up(off + slots * G * kHeadDim * 4, 256);
  w.off_q = off;
  off = align_up(off + (size_t)B * d.num_q_heads * kHeadDim * 2, 256);
  w.off_k = off;
  off = align_up(off + (size_t)B * d.num_kv_heads * kHeadDim * 2, 256);
  w.off_v = off;
  off = align_up(off + (size_t)B * d.num_kv_heads * kHeadDim * 2, 256);
  w.off_ids = off;
  off = align_up(off + (size_t)B * 4, 256);
  w.off_o = off;
  off = align_up(off + (size_t)B * d.num_q_heads * kHeadDim * 4, 256);
  w.total = off;
  return w;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

// ---------------------------------------------------------------------------
// Scratch of lk_decode_attn_static: the split counters and partials live in
// this fixed device array instead of a caller workspace, for callers that may
// not allocate device memory.  Every GPU that loads the library holds it
// until the process exits; all calls share it.
namespace {
constexpr size_t kStaticScratchBytes = 8u << 20;
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch in the current device's context.  Host
// code must not use the symbol itself: on the host it names a stand-in, not
// device memory.  The lookup allocates nothing and is repeated on every call,
// so a context that was torn down and created again (cudaDeviceReset) never
// leaves a stale address behind.  Nothing is cleared here: each call zeroes
// its counters on its own stream, and every partial is written before it is
// read.
lk_status static_scratch(void** out) {
  void* ptr = nullptr;
  cudaError_t err = cudaGetSymbolAddress(&ptr, g_decode_scratch);
  if (err != cudaSuccess) return cuda_fail(err, "lk_decode_attn_static: cudaGetSymbolAddress");
  *out = ptr;
  return LK_OK;
}
}  // namespace

struct lk_cache_s {
  lk_plan_s plan;
  Layout lay;
  CacheView cv;
  uint8_t* buf = nullptr;
  size_t bytes = 0;
  int B = 0, cap = 0;
  std::vector<int32_t> host_len;   // [L][B] tokens per layer and sequence (host mirror)
  std::vector<int32_t> len_upload; // [L][B] source of the prefill length copies
  std::vector<int32_t> active;     // [B] host mirror of the slot flags
  std::vector<int32_t> class_heads;  // [L][kNumPools] paged FULL heads of each width class
  int64_t host_free[kNumPools] = {}; // paged: free pages per class (host mirror)
  int32_t one = 1;                 // source of the slot-activation copy
  int32_t max_len(int layer) const {
    int32_t m = 0;
    for (int b = 0; b < B; ++b) m = std::max(m, host_len[(size_t)layer * B + b]);
    return m;
  }
  bool paged() const { return lay.max_pages > 0; }
  // pages per class that taking sequence b of `layer` from n0 to n1 tokens needs
  void pages_needed(int layer, int n0, int n1, int64_t* need) const {
    if (!paged()) return;
    const int d = pages_at(n1, cv.S, cv.W, lay.kv_format) - pages_at(n0, cv.S, cv.W, lay.kv_format);
    if (d == 0) return;
    for (int pl = 0; pl < kNumPools; ++pl) need[pl] += (int64_t)d * class_heads[(size_t)layer * kNumPools + pl];
  }
  lk_status take_pages(const int64_t* need, const char* who) {
    for (int pl = 0; pl < kNumPools; ++pl)
      if (need[pl] > host_free[pl])
        return fail(LK_ERR_CAPACITY, "%s: width class %d needs %lld pages; %lld are free", who, pool_width(pl),
                    (long long)need[pl], (long long)host_free[pl]);
    for (int pl = 0; pl < kNumPools; ++pl) host_free[pl] -= need[pl];
    return LK_OK;
  }
  DecodeMaps maps;
  int device = 0, num_sms = 0, decode_ctas = 0, step_mode = LK_STEP_AUTO;
  uint64_t wait_limit_ns = kWaitLimitNs;   // decode ring and segment waits
  std::vector<uint8_t> upload;     // host image of the tables (kept alive for the async copy)
};

namespace {
// CTAs of a decode launch.  A launch over few (sequence, head) entries
// streams a few long contiguous runs per CTA; there ~27/32 of the SMs reach
// a higher aggregate HBM rate than all of them (on 152 SMs: 128 CTAs take
// 86.5 us where 152 take 91.2 us on the 4-sequence 128K-token layer, and the
// 32K-token layer is flat).  Launches over many entries (the 32-layer
// steps) and quantised middles (bound by the tile math) use every SM.
int default_decode_ctas(const lk_cache_s* cache, int nlayers) {
  const int64_t entries = (int64_t)nlayers * cache->B * cache->cv.Hkv;
  if (cache->lay.kv_format == kKvBf16 && entries <= 64) return std::max(1, cache->num_sms * 27 / 32);
  return cache->num_sms;
}

// Resident K+V bytes of one (layer, head) entry at N tokens and `cnt`
// special rows: what a decode call streams for it.
uint64_t entry_bytes(const lk_cache_s* cache, const HeadDesc& hd, int N, int cnt) {
  const int S = cache->cv.S, W = cache->cv.W;
  uint64_t na = 0, nb = 0;
  if (hd.policy == kFull) {
    na = std::min(N, S + W);
    if (hd.n_kept > 0) nb = std::max(0, N - S - W);
  } else if (hd.policy == kLocal) {
    na = std::min(N, cache->cv.W_loc);
  } else {
    na = std::min(cnt, hd.cap_a);
  }
  if (kv_quantized(cache->lay.kv_format) && nb > 0) {
    const uint64_t sealed = nb / kQBlockRows, tail = nb % kQBlockRows;
    return na * (2 * kHeadDim * 2) + sealed * (uint64_t)qblock_bytes(hd.n_kept) +
           tail * (uint64_t)(hd.n_kept + kHeadDim) * 2;
  }
  return na * (2 * kHeadDim * 2) + nb * (uint64_t)(hd.n_kept + kHeadDim) * 2;
}

// Whether lk_step fuses the append into the decode launch.  Fusion removes a
// kernel boundary (~3.5 us) but puts the append's latency -- the token
// stage's copy, its fold into the softmax, the cache write -- on one CTA per
// entry.  A launch of at most 32 entries advances the lengths right after
// its work split, so fusing it costs nothing at the end and always pays
// (the 0.24 MB tiny layer: 12.2 -> 10.0 us per step).  A larger launch
// counts its CTAs at the end: fusion pays when each CTA streams long and
// meets few entries (the 16-sequence 32-layer FastGen step, 27 entries per
// CTA: 1.534 -> 1.524 ms) and loses when CTAs meet many entries (the
// 64-sequence 32-layer step, 108 per CTA: 2.926 -> 2.993 ms).  Lengths are
// the host's; SPECIAL rows count as 0.
bool fuse_step(const lk_cache_s* cache, int layer0, int nlayers) {
  if (cache->lay.kv_format != kKvBf16 || cache->step_mode == LK_STEP_SPLIT) return false;
  if (cache->step_mode == LK_STEP_FUSED) return true;
  const int B = cache->B, H = cache->cv.Hkv;
  const int64_t entries = (int64_t)nlayers * B * H;
  if (entries <= 32) return true;
  uint64_t bytes = 0;
  for (int l = layer0; l < layer0 + nlayers; ++l)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h)
        bytes += entry_bytes(cache, cache->lay.heads[(size_t)l * H + h], cache->host_len[(size_t)l * B + b], 0);
  const int ctas = cache->decode_ctas > 0 ? cache->decode_ctas : default_decode_ctas(cache, nlayers);
  // the kernel gives every CTA at least 64 KB of the work
  const uint64_t p = std::max<uint64_t>(1, std::min<uint64_t>((uint64_t)ctas, bytes / (64u << 10)));
  return bytes / p >= (256u << 10) && entries <= 32 * (int64_t)p;
}
}  // namespace

extern "C" {

const char* lk_last_error(void) { return g_last_error.c_str(); }

lk_status lk_build_plan(const lk_plan_desc* desc, const uint8_t* masks, const int32_t* policies,
                        const uint8_t* is_special, lk_plan* out) {
  if (!desc || !masks || !policies || !out) return fail(LK_ERR_ARG, "lk_build_plan: null argument");
  *out = nullptr;
  const lk_plan_desc& d = *desc;
  if (d.num_layers < 1 || d.num_layers > 4096) return fail(LK_ERR_ARG, "num_layers %d out of [1, 4096]", d.num_layers);
  if (d.num_kv_heads < 1 || d.num_kv_heads > 1024)
    return fail(LK_ERR_ARG, "num_kv_heads %d out of [1, 1024]", d.num_kv_heads);
  if (d.num_q_heads < d.num_kv_heads || d.num_q_heads % d.num_kv_heads != 0)
    return fail(LK_ERR_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", d.num_q_heads, d.num_kv_heads);
  if (d.num_q_heads / d.num_kv_heads > kMaxGroup)
    return fail(LK_ERR_UNSUPPORTED, "query heads per kv head %d > %d", d.num_q_heads / d.num_kv_heads, kMaxGroup);
  if (d.head_dim != kHeadDim) return fail(LK_ERR_UNSUPPORTED, "head_dim %d != 128", d.head_dim);
  if (d.sink < 0 || d.local < 0 || d.local_only_window < 0 || d.vocab < 0 || d.special_capacity < 0)
    return fail(LK_ERR_ARG, "negative sink/local/local_only_window/vocab/special_capacity");
  auto p = new lk_plan_s();
  p->d = d;
  const int LH = d.num_layers * d.num_kv_heads;
  p->policy.assign(policies, policies + LH);
  p->n_kept.assign(LH, 0);
  p->kept.assign((size_t)LH * kHeadDim, 0);
  p->layer_special.assign(d.num_layers, 0);
  bool any_full = false, any_local = false, any_special = false;
  for (int i = 0; i < LH; ++i) {
    const int pol = p->policy[i];
    if (pol != kFull && pol != kLocal && pol != kSpecial) {
      delete p;
      return fail(LK_ERR_ARG, "policy %d of head %d is not FULL/LOCAL/SPECIAL", pol, i);
    }
    any_full |= pol == kFull;
    any_local |= pol == kLocal;
    any_special |= pol == kSpecial;
    if (pol == kSpecial) p->layer_special[i / d.num_kv_heads] = 1;
    const uint8_t* m = masks + (size_t)i * kHeadDim;
    int cnt = 0;
    for (int c = 0; c < kHeadDim; ++c) {
      if (m[c] > 1) {
        delete p;
        return fail(LK_ERR_ARG, "mask of head %d channel %d is %d (must be 0 or 1)", i, c, m[c]);
      }
      cnt += m[c];
    }
    // kept channels ascending, then the pruned ones (the q permutation)
    int16_t* perm = &p->kept[(size_t)i * kHeadDim];
    int w = 0;
    for (int c = 0; c < kHeadDim; ++c)
      if (m[c]) perm[w++] = (int16_t)c;
    for (int c = 0; c < kHeadDim; ++c)
      if (!m[c]) perm[w++] = (int16_t)c;
    if (pol == kFull) {
      if (cnt % 32 != 0) {
        delete p;
        return fail(LK_ERR_ARG, "FULL head %d keeps %d channels; must be a multiple of 32", i, cnt);
      }
      p->n_kept[i] = cnt;
    }
  }
  if (any_full && d.local < 1) {
    delete p;
    return fail(LK_ERR_ARG, "FULL heads need local >= 1");
  }
  if (any_local && d.local_only_window < 1) {
    delete p;
    return fail(LK_ERR_ARG, "LOCAL heads need local_only_window >= 1");
  }
  if (any_special) {
    if (d.vocab < 1 || !is_special) {
      delete p;
      return fail(LK_ERR_ARG, "SPECIAL heads need vocab >= 1 and an is_special table");
    }
  }
  if (is_special && d.vocab > 0) {
    p->is_special.assign(is_special, is_special + d.vocab);
    for (auto& f : p->is_special) f = f ? 1 : 0;
  }
  *out = p;
  return LK_OK;
}

void lk_plan_destroy(lk_plan plan) { delete plan; }

lk_status lk_build_masks(const float* alpha, const uint8_t* eligible, int32_t num_layers, int32_t num_kv_heads,
                         double prune_pct, int32_t align, int32_t exact, uint8_t* masks, void* stream) {
  if (!alpha || !masks) return fail(LK_ERR_ARG, "lk_build_masks: null alpha or masks");
  if (!aligned(alpha, 4)) return fail(LK_ERR_ALIGN, "lk_build_masks: alpha must be 4-byte aligned");
  if (num_layers < 1 || num_kv_heads < 1 || (int64_t)num_layers * num_kv_heads > 8192)
    return fail(LK_ERR_ARG, "lk_build_masks: layers x kv heads must be in [1, 8192]");
  if (align != 32 && align != 64 && align != 128)
    return fail(LK_ERR_ARG, "lk_build_masks: align %d is not 32, 64 or 128", align);
  if (!(prune_pct >= 0.0 && prune_pct <= 100.0))
    return fail(LK_ERR_ARG, "lk_build_masks: prune_pct %g outside [0, 100]", prune_pct);
  if (exact != 0 && exact != 1) return fail(LK_ERR_ARG, "lk_build_masks: exact must be 0 or 1");
  cudaError_t err = launch_build_masks(alpha, eligible, num_layers * num_kv_heads, prune_pct, align, exact, masks,
                                       static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_build_masks launch");
  return LK_OK;
}

lk_status lk_plan_head(lk_plan plan, int32_t layer, int32_t kv_head, int32_t* policy, int32_t* n_kept,
                       int16_t* kept_channels) {
  if (!plan) return fail(LK_ERR_ARG, "lk_plan_head: null plan");
  if (layer < 0 || layer >= plan->d.num_layers || kv_head < 0 || kv_head >= plan->d.num_kv_heads)
    return fail(LK_ERR_ARG, "lk_plan_head: (layer %d, kv_head %d) out of range", layer, kv_head);
  const int i = layer * plan->d.num_kv_heads + kv_head;
  if (policy) *policy = plan->policy[i];
  if (n_kept) *n_kept = plan->n_kept[i];
  if (kept_channels) std::memcpy(kept_channels, &plan->kept[(size_t)i * kHeadDim], kHeadDim * 2);
  return LK_OK;
}

static lk_status cache_bytes_impl(lk_plan plan, int32_t batch, int32_t capacity_tokens, int64_t middle_tokens,
                                  int32_t fmt, size_t* bytes) {
  if (!plan || !bytes) return fail(LK_ERR_ARG, "lk_cache_bytes: null argument");
  if (batch < 1 || (int64_t)batch * plan->d.num_kv_heads > (1 << 20))
    return fail(LK_ERR_ARG, "batch %d out of range", batch);
  if (capacity_tokens < 1 || capacity_tokens > (1 << 30))
    return fail(LK_ERR_ARG, "capacity_tokens %d out of [1, 2^30]", capacity_tokens);
  if (fmt != kKvBf16 && fmt != kKvInt8 && fmt != kKvFp8)
    return fail(LK_ERR_ARG, "kv_format %d is not LK_KV_BF16, LK_KV_INT8 or LK_KV_FP8", fmt);
  Layout lay;
  lk_status st = compute_layout(*plan, batch, capacity_tokens, middle_tokens, fmt, &lay);
  if (st != LK_OK) return st;
  *bytes = lay.total;
  return LK_OK;
}

lk_status lk_cache_bytes(lk_plan plan, int32_t batch, int32_t capacity_tokens, size_t* bytes) {
  return cache_bytes_impl(plan, batch, capacity_tokens, -1, kKvBf16, bytes);
}

lk_status lk_cache_bytes_paged(lk_plan plan, int32_t batch, int32_t capacity_tokens, int64_t middle_tokens,
                               size_t* bytes) {
  if (middle_tokens < 0) return fail(LK_ERR_ARG, "lk_cache_bytes_paged: middle_tokens %lld < 0", (long long)middle_tokens);
  return cache_bytes_impl(plan, batch, capacity_tokens, middle_tokens, kKvBf16, bytes);
}

lk_status lk_cache_bytes_ex(lk_plan plan, int32_t batch, int32_t capacity_tokens, const lk_cache_options* opt,
                            size_t* bytes) {
  if (!opt) return fail(LK_ERR_ARG, "lk_cache_bytes_ex: null options");
  return cache_bytes_impl(plan, batch, capacity_tokens, opt->middle_tokens < 0 ? -1 : opt->middle_tokens,
                          opt->kv_format, bytes);
}

lk_status lk_workspace_bytes(lk_plan plan, int32_t batch, size_t* bytes) {
  if (!plan || !bytes) return fail(LK_ERR_ARG, "lk_workspace_bytes: null argument");
  if (batch < 1 || (int64_t)batch * plan->d.num_kv_heads > (1 << 20))
    return fail(LK_ERR_ARG, "batch %d out of range", batch);
  *bytes = ws_layout(plan->d, batch).total;
  return LK_OK;
}

static lk_status cache_init_impl(lk_plan plan, void* dev_buf, size_t bytes, int32_t batch, int32_t capacity_tokens,
                                 int64_t middle_tokens, int32_t fmt, void* stream, lk_cache* out) {
  if (!plan || !dev_buf || !out) return fail(LK_ERR_ARG, "lk_cache_init: null argument");
  *out = nullptr;
  if (!aligned(dev_buf, 256)) return fail(LK_ERR_ALIGN, "cache buffer must be 256-byte aligned");
  size_t need = 0;
  lk_status st = cache_bytes_impl(plan, batch, capacity_tokens, middle_tokens, fmt, &need);
  if (st != LK_OK) return st;
  if (bytes < need) return fail(LK_ERR_CAPACITY, "cache buffer has %zu bytes; %zu needed", bytes, need);
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(LK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");

  auto c = new lk_cache_s();
  c->plan = *plan;
  compute_layout(c->plan, batch, capacity_tokens, middle_tokens, fmt, &c->lay);
  c->buf = static_cast<uint8_t*>(dev_buf);
  c->bytes = bytes;
  c->B = batch;
  c->cap = capacity_tokens;
  const lk_plan_desc& d = plan->d;
  const int L = d.num_layers, H = d.num_kv_heads;
  c->host_len.assign((size_t)L * batch, 0);
  c->len_upload.assign((size_t)L * batch, 0);
  c->active.assign(batch, 1);
  c->class_heads.assign((size_t)L * kNumPools, 0);
  const Layout& lay = c->lay;
  if (c->paged()) {
    for (int i = 0; i < L * H; ++i) {
      const HeadDesc& hd = lay.heads[i];
      if (hd.policy == kFull && hd.n_kept > 0) c->class_heads[(size_t)(i / H) * kNumPools + hd.pool_kb] += 1;
    }
    for (int pl = 0; pl < kNumPools; ++pl) c->host_free[pl] = lay.num_pages[pl];
  }
  cudaError_t err = cudaGetDevice(&c->device);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  if (err != cudaSuccess) {
    delete c;
    return cuda_fail(err, "lk_cache_init: device query");
  }
  CacheView& cv = c->cv;
  cv.hdr = reinterpret_cast<DevHeader*>(c->buf);
  cv.len = reinterpret_cast<int32_t*>(c->buf + lay.off_len);
  cv.cnt = reinterpret_cast<int32_t*>(c->buf + lay.off_cnt);
  cv.active = reinterpret_cast<int32_t*>(c->buf + lay.off_active);
  cv.page_table = c->paged() ? reinterpret_cast<int32_t*>(c->buf + lay.off_pt) : nullptr;
  cv.free_list = reinterpret_cast<int32_t*>(c->buf + lay.off_free);
  cv.heads = reinterpret_cast<const HeadDesc*>(c->buf + lay.off_heads);
  cv.kept = reinterpret_cast<const int16_t*>(c->buf + lay.off_kept);
  cv.is_special = c->buf + lay.off_spec;
  for (int pl = 0; pl < kNumPools; ++pl) {
    cv.pool[pl] = reinterpret_cast<uint16_t*>(c->buf + lay.off_pool[pl]);
    cv.pool_rows[pl] = lay.pool_rows[pl];
  }
  cv.L = L;
  cv.B = batch;
  cv.Hq = d.num_q_heads;
  cv.Hkv = H;
  cv.G = d.num_q_heads / d.num_kv_heads;
  cv.S = d.sink;
  cv.W = d.local;
  cv.W_loc = d.local_only_window;
  cv.vocab = d.vocab;
  cv.capacity = capacity_tokens;
  cv.spec_cap = lay.spec_cap;
  cv.max_pages = lay.max_pages;
  cv.kv_format = lay.kv_format;
  cv.qpool = c->buf + lay.off_q;

  // host image of everything before the pools: header (free stack tops),
  // lengths 0, slots active, page table -1, free stacks (pops hand out page
  // 0, 1, 2, ... of each class), head table, kept channels, special table
  const size_t tab_hi = lay.off_pool[0];
  c->upload.assign(tab_hi, 0);
  uint8_t* img = c->upload.data();
  DevHeader* hdr = reinterpret_cast<DevHeader*>(img);
  for (int pl = 0; pl < kNumPools; ++pl) hdr->free_top[pl] = lay.num_pages[pl];
  int32_t* act = reinterpret_cast<int32_t*>(img + lay.off_active);
  for (int b = 0; b < batch; ++b) act[b] = 1;
  int32_t* pt = reinterpret_cast<int32_t*>(img + lay.off_pt);
  std::fill(pt, pt + (size_t)L * batch * H * lay.max_pages, -1);
  int32_t* fl = reinterpret_cast<int32_t*>(img + lay.off_free);
  for (int pl = 0; pl < kNumPools; ++pl)
    for (int32_t i = 0; i < lay.num_pages[pl]; ++i) fl[lay.free_off[pl] + i] = lay.num_pages[pl] - 1 - i;
  std::memcpy(img + lay.off_heads, lay.heads.data(), lay.heads.size() * sizeof(HeadDesc));
  std::memcpy(img + lay.off_kept, c->plan.kept.data(), c->plan.kept.size() * 2);
  if (!c->plan.is_special.empty()) std::memcpy(img + lay.off_spec, c->plan.is_special.data(), c->plan.is_special.size());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  err = cudaMemsetAsync(c->buf + tab_hi, 0, lay.total - tab_hi, s);
  if (err == cudaSuccess) err = cudaMemcpyAsync(c->buf, img, tab_hi, cudaMemcpyHostToDevice, s);
  if (err != cudaSuccess) {
    delete c;
    return cuda_fail(err, "lk_cache_init: upload");
  }
  // One TMA operation per tile and operand (bandwidth grows with the size of
  // each operation): 128-byte-row pools load as 64-channel halves with
  // 128-byte swizzle, 64-byte-row pools as 32-channel stripes with 64-byte
  // swizzle; the halves / stripes of a row fold into one box.  Flat maps are
  // {channels, rows, parts}; block views {channels, rows per block, blocks,
  // parts}, so that a box stops at the end of its (head, sequence) block or
  // page.
  std::memset(&c->maps, 0, sizeof(c->maps));
  auto encode_view = [&](int map, int pl, int64_t first_row, int64_t rows, int64_t blocks) -> CUresult {
    const int width = pool_width(pl);
    const bool fam128 = (width % 64) == 0;
    const int inner = fam128 ? 64 : 32;              // channels per half / stripe
    const int parts = width / inner;
    const cuuint64_t row_bytes = (cuuint64_t)width * 2;
    const bool blocked = blocks > 0;
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4];
    cuuint32_t rank = 0;
    dims[rank] = (cuuint64_t)inner;
    box[rank++] = (cuuint32_t)inner;
    dims[rank] = (cuuint64_t)rows;
    strides[rank - 1] = row_bytes;
    box[rank++] = (cuuint32_t)kTmaBoxRows;
    if (blocked) {
      dims[rank] = (cuuint64_t)blocks;
      strides[rank - 1] = (cuuint64_t)rows * row_bytes;
      box[rank++] = 1;
    }
    if (parts > 1) {
      dims[rank] = (cuuint64_t)parts;
      strides[rank - 1] = (cuuint64_t)inner * 2;
      box[rank++] = (cuuint32_t)parts;
    }
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    return encode(&c->maps.m[map], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, cv.pool[pl] + first_row * width, dims,
                  strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  fam128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  for (int map = 0; map < kNumMaps; ++map) {
    CUresult r;
    if (map < kMapAK) {
      r = encode_view(map, map - kMapFlat, 0, lay.pool_rows[map - kMapFlat], 0);
    } else {
      // block views shorter than a box are never used: encode them over one
      // box of the pool so that every map is valid
      const bool a = map < kMapB;
      const int cls = (map - kMapAK) % 3;
      const int pl = a ? (map < kMapAV ? kPoolK128 : kPoolV) : map - kMapB;
      const int64_t first = a ? lay.a_base[cls] : lay.b_base[pl];
      const int64_t rows = a ? lay.a_rows[cls] : lay.b_rows;
      const int64_t blocks = a ? lay.a_blocks[cls] : lay.b_blocks[pl];
      const bool usable = rows >= kTmaBoxRows && blocks > 0;
      c->maps.block_rows[map] = usable ? (int32_t)rows : 0;
      r = usable ? encode_view(map, pl, first, rows, blocks) : encode_view(map, pl, 0, kTmaBoxRows, 1);
    }
    if (r != CUDA_SUCCESS) {
      delete c;
      return fail(LK_ERR_CUDA, "cuTensorMapEncodeTiled failed for map %d (CUresult %d)", map, (int)r);
    }
  }
  *out = c;
  return LK_OK;
}

lk_status lk_cache_init(lk_plan plan, void* dev_buf, size_t bytes, int32_t batch, int32_t capacity_tokens,
                        void* stream, lk_cache* out) {
  return cache_init_impl(plan, dev_buf, bytes, batch, capacity_tokens, -1, kKvBf16, stream, out);
}

lk_status lk_cache_init_paged(lk_plan plan, void* dev_buf, size_t bytes, int32_t batch, int32_t capacity_tokens,
                              int64_t middle_tokens, void* stream, lk_cache* out) {
  if (out) *out = nullptr;
  if (middle_tokens < 0) return fail(LK_ERR_ARG, "lk_cache_init_paged: middle_tokens %lld < 0", (long long)middle_tokens);
  return cache_init_impl(plan, dev_buf, bytes, batch, capacity_tokens, middle_tokens, kKvBf16, stream, out);
}

lk_status lk_cache_init_ex(lk_plan plan, void* dev_buf, size_t bytes, int32_t batch, int32_t capacity_tokens,
                           const lk_cache_options* opt, void* stream, lk_cache* out) {
  if (out) *out = nullptr;
  if (!opt) return fail(LK_ERR_ARG, "lk_cache_init_ex: null options");
  return cache_init_impl(plan, dev_buf, bytes, batch, capacity_tokens, opt->middle_tokens < 0 ? -1 : opt->middle_tokens,
                         opt->kv_format, stream, out);
}

void lk_cache_destroy(lk_cache cache) { delete cache; }

lk_status lk_workspace_init(lk_cache cache, void* workspace, size_t ws_bytes, void* stream) {
  if (!cache || !workspace) return fail(LK_ERR_ARG, "lk_workspace_init: null argument");
  if (!aligned(workspace, 256)) return fail(LK_ERR_ALIGN, "workspace must be 256-byte aligned");
  const WsLayout w = ws_layout(cache->plan.d, cache->B);
  if (ws_bytes < w.total) return fail(LK_ERR_CAPACITY, "workspace has %zu bytes; %zu needed", ws_bytes, w.total);
  cudaError_t err = cudaMemsetAsync(workspace, 0, w.total, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_workspace_init");
  return LK_OK;
}

// Shared by the uniform, ragged and single-sequence prefill of sequences
// b0 .. b0 + nb - 1: lengths go to the device length row first, then the copy
// kernels read each sequence's length there.
static lk_status prefill_impl(lk_cache cache, int32_t layer, int32_t b0, int32_t nb, const void* k, const void* v,
                              const int32_t* ids, const int32_t* lens, int32_t n_max, void* stream) {
  if (!cache) return fail(LK_ERR_ARG, "lk_prefill: null cache");
  if (layer < 0 || layer >= cache->cv.L) return fail(LK_ERR_ARG, "lk_prefill: layer %d out of range", layer);
  if (n_max < 0) return fail(LK_ERR_ARG, "lk_prefill: n = %d < 0", n_max);
  const int B = cache->B;
  for (int b = b0; b < b0 + nb; ++b)
    if (cache->host_len[(size_t)layer * B + b] != 0)
      return fail(LK_ERR_STATE, "lk_prefill: sequence %d of layer %d already holds tokens", b, layer);
  if (n_max > cache->cap) return fail(LK_ERR_CAPACITY, "lk_prefill: n = %d exceeds capacity %d", n_max, cache->cap);
  int32_t* up = &cache->len_upload[(size_t)layer * B + b0];
  int64_t need[kNumPools] = {0, 0, 0, 0, 0};
  for (int i = 0; i < nb; ++i) {
    const int32_t n = lens ? lens[i] : n_max;
    if (n < 0 || n > n_max)
      return fail(LK_ERR_ARG, "lk_prefill: length %d of sequence %d outside [0, %d]", n, b0 + i, n_max);
    up[i] = n;
    cache->pages_needed(layer, 0, n, need);
  }
  if (n_max == 0) return LK_OK;
  if (!k || !v) return fail(LK_ERR_ARG, "lk_prefill: null k or v");
  if (!aligned(k, 16) || !aligned(v, 16)) return fail(LK_ERR_ALIGN, "lk_prefill: k and v must be 16-byte aligned");
  if (ids && !aligned(ids, 4)) return fail(LK_ERR_ALIGN, "lk_prefill: ids must be 4-byte aligned");
  lk_status st = cache->take_pages(need, "lk_prefill");
  if (st != LK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err =
      cudaMemcpyAsync(cache->cv.len + (size_t)layer * B + b0, up, (size_t)nb * 4, cudaMemcpyHostToDevice, s);
  if (err != cudaSuccess) return cuda_fail(err, "lk_prefill: length upload");
  PrefillArgs a;
  a.cv = cache->cv;
  a.layer = layer;
  a.b0 = b0;
  a.nb = nb;
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.ids = ids;
  a.n = n_max;
  err = launch_prefill(a, cache->plan.layer_special[layer] != 0, cache->num_sms, s);
  if (err != cudaSuccess) {
    for (int pl = 0; pl < kNumPools; ++pl) cache->host_free[pl] += need[pl];
    return cuda_fail(err, "lk_prefill launch");
  }
  for (int i = 0; i < nb; ++i) cache->host_len[(size_t)layer * B + b0 + i] = up[i];
  return LK_OK;
}

lk_status lk_prefill(lk_cache cache, int32_t layer, const void* k, const void* v, const int32_t* ids, int32_t n,
                     void* stream) {
  if (!cache) return fail(LK_ERR_ARG, "lk_prefill: null cache");
  return prefill_impl(cache, layer, 0, cache->B, k, v, ids, nullptr, n, stream);
}

lk_status lk_prefill_ragged(lk_cache cache, int32_t layer, const void* k, const void* v, const int32_t* ids,
                            const int32_t* lens, int32_t n_max, void* stream) {
  if (!cache) return fail(LK_ERR_ARG, "lk_prefill_ragged: null cache");
  if (!lens) return fail(LK_ERR_ARG, "lk_prefill_ragged: null lens");
  return prefill_impl(cache, layer, 0, cache->B, k, v, ids, lens, n_max, stream);
}

lk_status lk_prefill_sequence(lk_cache cache, int32_t layer, int32_t b, const void* k, const void* v,
                              const int32_t* ids, int32_t n, void* stream) {
  if (!cache) return fail(LK_ERR_ARG, "lk_prefill_sequence: null cache");
  if (b < 0 || b >= cache->B) return fail(LK_ERR_ARG, "lk_prefill_sequence: sequence %d out of range", b);
  lk_status st = prefill_impl(cache, layer, b, 1, k, v, ids, nullptr, n, stream);
  if (st != LK_OK || cache->active[b]) return st;
  cudaError_t err = cudaMemcpyAsync(cache->cv.active + b, &cache->one, 4, cudaMemcpyHostToDevice,
                                    static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_prefill_sequence: slot activation");
  cache->active[b] = 1;
  return LK_OK;
}

lk_status lk_release_sequence(lk_cache cache, int32_t b, void* stream) {
  if (!cache) return fail(LK_ERR_ARG, "lk_release_sequence: null cache");
  if (b < 0 || b >= cache->B) return fail(LK_ERR_ARG, "lk_release_sequence: sequence %d out of range", b);
  cudaError_t err = launch_release(cache->cv, b, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_release_sequence launch");
  for (int l = 0; l < cache->cv.L; ++l) {
    int32_t& n = cache->host_len[(size_t)l * cache->B + b];
    int64_t back[kNumPools] = {0, 0, 0, 0, 0};
    cache->pages_needed(l, 0, n, back);
    for (int pl = 0; pl < kNumPools; ++pl) cache->host_free[pl] += back[pl];
    n = 0;
  }
  cache->active[b] = 0;
  return LK_OK;
}

lk_status lk_cache_pages(lk_cache cache, int32_t width, int64_t* total, int64_t* free_pages) {
  if (!cache) return fail(LK_ERR_ARG, "lk_cache_pages: null cache");
  if (width != 32 && width != 64 && width != 96 && width != 128)
    return fail(LK_ERR_ARG, "lk_cache_pages: width %d is not 32, 64, 96 or 128", width);
  const int pl = pool_for_width(width);
  if (total) *total = cache->lay.num_pages[pl];
  if (free_pages) *free_pages = cache->host_free[pl];
  return LK_OK;
}

}  // extern "C"

namespace {

// Host side of an append over layers [layer0, layer0 + nlayers): argument
// and capacity checks, and the pages the appends will pop (taken from the
// host count into need; the caller returns them if its launch fails).
lk_status append_prepare(lk_cache cache, int32_t layer0, int32_t nlayers, const void* k, const void* v,
                         const int32_t* ids, const char* what, int64_t need[kNumPools]) {
  if (!cache) return fail(LK_ERR_ARG, "%s: null cache", what);
  if (nlayers < 1 || layer0 < 0 || layer0 + nlayers > cache->cv.L)
    return fail(LK_ERR_ARG, "%s: layers [%d, %d) out of range", what, layer0, layer0 + nlayers);
  if (!k || !v) return fail(LK_ERR_ARG, "%s: null k or v", what);
  if (!aligned(k, 16) || !aligned(v, 16)) return fail(LK_ERR_ALIGN, "%s: k and v must be 16-byte aligned", what);
  if (ids && !aligned(ids, 4)) return fail(LK_ERR_ALIGN, "%s: ids must be 4-byte aligned", what);
  const int B = cache->B;
  for (int pl = 0; pl < kNumPools; ++pl) need[pl] = 0;
  for (int l = layer0; l < layer0 + nlayers; ++l)
    for (int b = 0; b < B; ++b) {
      if (!cache->active[b]) continue;
      const int n = cache->host_len[(size_t)l * B + b];
      if (n >= cache->cap)
        return fail(LK_ERR_CAPACITY, "%s: sequence %d of layer %d is full (%d tokens)", what, b, l, cache->cap);
      cache->pages_needed(l, n, n + 1, need);
    }
  return cache->take_pages(need, what);
}

void append_commit(lk_cache cache, int32_t layer0, int32_t nlayers) {
  const int B = cache->B;
  for (int l = layer0; l < layer0 + nlayers; ++l)
    for (int b = 0; b < B; ++b)
      if (cache->active[b]) cache->host_len[(size_t)l * B + b] += 1;
}

void return_pages(lk_cache cache, const int64_t need[kNumPools]) {
  for (int pl = 0; pl < kNumPools; ++pl) cache->host_free[pl] += need[pl];
}

// The decode kernel's launch-fixed divisors.
void set_divisors(const lk_cache_s* cache, DecodeArgs& a) {
  const CacheView& cv = cache->cv;
  a.div_bh = make_fastdiv((uint32_t)(cv.B * cv.Hkv));
  a.div_h = make_fastdiv((uint32_t)cv.Hkv);
  a.div_w = make_fastdiv((uint32_t)std::max(1, cv.W));
  a.div_wloc = make_fastdiv((uint32_t)std::max(1, cv.W_loc));
  for (int i = 0; i < 5; ++i) {
    const int k = 32 * i;
    a.div_cost_b[i] = make_fastdiv((uint32_t)(2 * k + 256));
    a.div_cost_q[i] = make_fastdiv((uint32_t)(qblock_bytes(k) / kQBlockRows));
  }
}

// Host side of a decode launch: checks, and the kernel arguments (no fused
// append) and CTA count.
lk_status decode_prepare(lk_cache cache, int32_t layer0, int32_t nlayers, const void* q, float* o, void* workspace,
                         size_t ws_bytes, const char* what, DecodeArgs& a, int& ctas) {
  if (!cache) return fail(LK_ERR_ARG, "%s: null cache", what);
  if (nlayers < 1 || layer0 < 0 || layer0 + nlayers > cache->cv.L)
    return fail(LK_ERR_ARG, "%s: layers [%d, %d) out of range", what, layer0, layer0 + nlayers);
  if (!q || !o || !workspace) return fail(LK_ERR_ARG, "%s: null q, o or workspace", what);
  if (!aligned(q, 16) || !aligned(o, 16)) return fail(LK_ERR_ALIGN, "%s: q and o must be 16-byte aligned", what);
  if (!aligned(workspace, 256)) return fail(LK_ERR_ALIGN, "%s: workspace must be 256-byte aligned", what);
  const WsLayout w = ws_layout(cache->plan.d, cache->B);
  if (ws_bytes < w.total) return fail(LK_ERR_CAPACITY, "%s: workspace has %zu bytes; %zu needed", what, ws_bytes, w.total);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a = DecodeArgs{};
  a.cv = cache->cv;
  a.layer = layer0;
  a.nlayers = nlayers;
  a.q = static_cast<const uint16_t*>(q);
  a.o = o;
  a.part = reinterpret_cast<float*>(ws + w.off_part);
  a.part_ml = reinterpret_cast<float2*>(ws + w.off_ml);
  a.counters = reinterpret_cast<int32_t*>(ws + w.off_counters);
  a.wait_limit_ns = cache->wait_limit_ns;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)kHeadDim));
  a.k_new = a.v_new = nullptr;
  a.ids = nullptr;
  set_divisors(cache, a);
  ctas = cache->decode_ctas > 0 ? cache->decode_ctas : default_decode_ctas(cache, nlayers);
  ctas = std::max(1, std::min(ctas, kMaxCtas));
  return LK_OK;
}

}  // namespace

extern "C" {

lk_status lk_append_layers(lk_cache cache, int32_t layer0, int32_t nlayers, const void* k, const void* v,
                           const int32_t* ids, void* stream) {
  int64_t need[kNumPools];
  lk_status st = append_prepare(cache, layer0, nlayers, k, v, ids, "lk_append", need);
  if (st != LK_OK) return st;
  AppendArgs a;
  a.cv = cache->cv;
  a.layer = layer0;
  a.nlayers = nlayers;
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.ids = ids;
  cudaError_t err = launch_append(a, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) {
    return_pages(cache, need);
    return cuda_fail(err, "lk_append launch");
  }
  append_commit(cache, layer0, nlayers);
  return LK_OK;
}

lk_status lk_append(lk_cache cache, int32_t layer, const void* k, const void* v, const int32_t* ids,
                    void* stream) {
  return lk_append_layers(cache, layer, 1, k, v, ids, stream);
}

lk_status lk_decode_attn_layers(lk_cache cache, int32_t layer0, int32_t nlayers, const void* q, float* o,
                                void* workspace, size_t ws_bytes, void* stream) {
  DecodeArgs a;
  int ctas = 0;
  lk_status st = decode_prepare(cache, layer0, nlayers, q, o, workspace, ws_bytes, "lk_decode_attn", a, ctas);
  if (st != LK_OK) return st;
  cudaError_t err = launch_decode(cache->maps, a, ctas, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_decode_attn launch");
  return LK_OK;
}

lk_status lk_decode_attn(lk_cache cache, int32_t layer, const void* q, float* o, void* workspace,
                         size_t ws_bytes, void* stream) {
  return lk_decode_attn_layers(cache, layer, 1, q, o, workspace, ws_bytes, stream);
}

lk_status lk_step_layers(lk_cache cache, int32_t layer0, int32_t nlayers, const void* q, const void* k,
                         const void* v, const int32_t* ids, float* o, void* workspace, size_t ws_bytes,
                         void* stream) {
  DecodeArgs a;
  int ctas = 0;
  lk_status st = decode_prepare(cache, layer0, nlayers, q, o, workspace, ws_bytes, "lk_step", a, ctas);
  if (st != LK_OK) return st;
  if (!fuse_step(cache, layer0, nlayers)) {
    // quantised middles always: an append may seal a block, which changes the
    // values the decode reads
    st = lk_append_layers(cache, layer0, nlayers, k, v, ids, stream);
    if (st != LK_OK) return st;
    return lk_decode_attn_layers(cache, layer0, nlayers, q, o, workspace, ws_bytes, stream);
  }
  int64_t need[kNumPools];
  st = append_prepare(cache, layer0, nlayers, k, v, ids, "lk_step", need);
  if (st != LK_OK) return st;
  a.k_new = static_cast<const uint16_t*>(k);
  a.v_new = static_cast<const uint16_t*>(v);
  a.ids = ids;
  cudaError_t err = launch_decode(cache->maps, a, ctas, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) {
    return_pages(cache, need);
    return cuda_fail(err, "lk_step launch");
  }
  append_commit(cache, layer0, nlayers);
  return LK_OK;
}

lk_status lk_step(lk_cache cache, int32_t layer, const void* q, const void* k, const void* v, const int32_t* ids,
                  float* o, void* workspace, size_t ws_bytes, void* stream) {
  return lk_step_layers(cache, layer, 1, q, k, v, ids, o, workspace, ws_bytes, stream);
}

// Device address of a page-locked host buffer mapped into the device's
// address space (cudaHostAlloc, or cudaHostRegister with mapping -- torch's
// pin_memory), else null.
static const void* mapped_host(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

// A host-driven step whose buffers the device can address: the kernels read
// q, k, v, ids from host memory and write o there over the host link (on
// Grace, NVLink-C2C), with no staging copies.  Always the append and decode
// launches: the fused kernel loads the new token with bulk copies, which
// this path keeps away from host memory.  The decode launch is checked
// before the append commits the token.
static lk_status step_in_place(lk_cache cache, int32_t layer, const void* q, const void* k, const void* v,
                               const int32_t* ids, float* o, void* workspace, size_t ws_bytes, void* stream) {
  DecodeArgs a;
  int ctas = 0;
  lk_status st = decode_prepare(cache, layer, 1, q, o, workspace, ws_bytes, "lk_step_host", a, ctas);
  if (st != LK_OK) return st;
  st = lk_append_layers(cache, layer, 1, k, v, ids, stream);
  if (st != LK_OK) return st;
  cudaError_t err = launch_decode(cache->maps, a, ctas, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_step_host decode launch");
  return LK_OK;
}

// Append + decode from the inputs staged in the workspace, then copy o back.
static lk_status step_from_staging(lk_cache cache, int32_t layer, bool has_ids, float* o_host, void* workspace,
                            size_t ws_bytes, void* stream) {
  const WsLayout w = ws_layout(cache->plan.d, cache->B);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* o_dev = reinterpret_cast<float*>(ws + w.off_o);
  lk_status st = lk_step(cache, layer, ws + w.off_q, ws + w.off_k, ws + w.off_v,
                         has_ids ? reinterpret_cast<const int32_t*>(ws + w.off_ids) : nullptr, o_dev, workspace,
                         ws_bytes, stream);
  if (st != LK_OK) return st;
  const size_t ob = (size_t)cache->B * cache->plan.d.num_q_heads * kHeadDim * 4;
  cudaError_t err = cudaMemcpyAsync(o_host, o_dev, ob, cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_step_host: device to host copy");
  return LK_OK;
}

lk_status lk_step_host(lk_cache cache, int32_t layer, const void* q_host, const void* k_host, const void* v_host,
                       const int32_t* ids_host, float* o_host, void* workspace, size_t ws_bytes, void* stream) {
  if (!cache || !q_host || !k_host || !v_host || !o_host || !workspace)
    return fail(LK_ERR_ARG, "lk_step_host: null argument");
  const WsLayout w = ws_layout(cache->plan.d, cache->B);
  if (ws_bytes < w.total)
    return fail(LK_ERR_CAPACITY, "lk_step_host: workspace has %zu bytes; %zu needed", ws_bytes, w.total);
  if (layer < 0 || layer >= cache->cv.L) return fail(LK_ERR_ARG, "lk_step_host: layer %d out of range", layer);
  if (cache->max_len(layer) >= cache->cap)
    return fail(LK_ERR_CAPACITY, "lk_step_host: a sequence of layer %d is full (%d tokens)", layer, cache->cap);
  {
    const void* qd = mapped_host(q_host);
    const void* kd = mapped_host(k_host);
    const void* vd = mapped_host(v_host);
    const void* idd = ids_host ? mapped_host(ids_host) : nullptr;
    float* od = static_cast<float*>(const_cast<void*>(mapped_host(o_host)));
    if (qd && kd && vd && od && (!ids_host || idd))
      return step_in_place(cache, layer, qd, kd, vd, static_cast<const int32_t*>(idd), od, workspace, ws_bytes,
                           stream);
  }
  const lk_plan_desc& d = cache->plan.d;
  const size_t B = cache->B;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t qb = B * d.num_q_heads * kHeadDim * 2, kvb = B * d.num_kv_heads * kHeadDim * 2;
  cudaError_t err = cudaMemcpyAsync(ws + w.off_q, q_host, qb, cudaMemcpyHostToDevice, s);
  if (err == cudaSuccess) err = cudaMemcpyAsync(ws + w.off_k, k_host, kvb, cudaMemcpyHostToDevice, s);
  if (err == cudaSuccess) err = cudaMemcpyAsync(ws + w.off_v, v_host, kvb, cudaMemcpyHostToDevice, s);
  if (err == cudaSuccess && ids_host)
    err = cudaMemcpyAsync(ws + w.off_ids, ids_host, B * 4, cudaMemcpyHostToDevice, s);
  if (err != cudaSuccess) return cuda_fail(err, "lk_step_host: host to device copy");
  return step_from_staging(cache, layer, ids_host != nullptr, o_host, workspace, ws_bytes, stream);
}

lk_status lk_step_host_packed(lk_cache cache, int32_t layer, const void* host_in, int32_t has_ids, float* o_host,
                              void* workspace, size_t ws_bytes, void* stream) {
  if (!cache || !host_in || !o_host || !workspace) return fail(LK_ERR_ARG, "lk_step_host_packed: null argument");
  const WsLayout w = ws_layout(cache->plan.d, cache->B);
  if (ws_bytes < w.total)
    return fail(LK_ERR_CAPACITY, "lk_step_host_packed: workspace has %zu bytes; %zu needed", ws_bytes, w.total);
  if (layer < 0 || layer >= cache->cv.L) return fail(LK_ERR_ARG, "lk_step_host_packed: layer %d out of range", layer);
  if (cache->max_len(layer) >= cache->cap)
    return fail(LK_ERR_CAPACITY, "lk_step_host_packed: a sequence of layer %d is full (%d tokens)", layer,
                cache->cap);
  const lk_plan_desc& d = cache->plan.d;
  const size_t B = cache->B;
  const size_t qb = B * d.num_q_heads * kHeadDim * 2, kvb = B * d.num_kv_heads * kHeadDim * 2;
  const size_t bytes = qb + 2 * kvb + (has_ids ? B * 4 : 0);
  {
    const uint8_t* in = static_cast<const uint8_t*>(mapped_host(host_in));
    float* od = static_cast<float*>(const_cast<void*>(mapped_host(o_host)));
    if (in && od)
      return step_in_place(cache, layer, in, in + qb, in + qb + kvb,
                           has_ids ? reinterpret_cast<const int32_t*>(in + qb + 2 * kvb) : nullptr, od, workspace,
                           ws_bytes, stream);
  }
  // the staging areas q | k | v | ids are adjacent in the workspace
  if (w.off_k != w.off_q + qb || w.off_v != w.off_k + kvb || w.off_ids != w.off_v + kvb)
    return fail(LK_ERR_UNSUPPORTED, "lk_step_host_packed: staging areas are not adjacent");
  cudaError_t err = cudaMemcpyAsync(static_cast<uint8_t*>(workspace) + w.off_q, host_in, bytes, cudaMemcpyHostToDevice,
                                    static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_step_host_packed: host to device copy");
  return step_from_staging(cache, layer, has_ids != 0, o_host, workspace, ws_bytes, stream);
}

lk_status lk_step_layers_host_packed(lk_cache cache, int32_t layer0, int32_t nlayers, const void* host_in,
                                     int32_t has_ids, float* o_host, void* workspace, size_t ws_bytes,
                                     void* stream) {
  if (!cache || !host_in || !o_host || !workspace)
    return fail(LK_ERR_ARG, "lk_step_layers_host_packed: null argument");
  if (nlayers < 1 || layer0 < 0 || layer0 + nlayers > cache->cv.L)
    return fail(LK_ERR_ARG, "lk_step_layers_host_packed: layers %d .. %d out of range", layer0, layer0 + nlayers - 1);
  const uint8_t* in = static_cast<const uint8_t*>(mapped_host(host_in));
  float* od = static_cast<float*>(const_cast<void*>(mapped_host(o_host)));
  if (!in || !od)
    return fail(LK_ERR_ARG, "lk_step_layers_host_packed: host buffers must be page-locked and mapped");
  const lk_plan_desc& d = cache->plan.d;
  const size_t rows = (size_t)nlayers * cache->B;
  const size_t qb = rows * d.num_q_heads * kHeadDim * 2, kvb = rows * d.num_kv_heads * kHeadDim * 2;
  const int32_t* ids = has_ids ? reinterpret_cast<const int32_t*>(in + qb + 2 * kvb) : nullptr;
  // every check of the decode launch (workspace size and alignment, q and o
  // alignment) before the append, which commits the token
  DecodeArgs a;
  int ctas = 0;
  lk_status st = decode_prepare(cache, layer0, nlayers, in, od, workspace, ws_bytes, "lk_step_layers_host_packed",
                                a, ctas);
  if (st != LK_OK) return st;
  st = lk_append_layers(cache, layer0, nlayers, in + qb, in + qb + kvb, ids, stream);
  if (st != LK_OK) return st;
  cudaError_t err = launch_decode(cache->maps, a, ctas, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_step_layers_host_packed decode launch");
  return LK_OK;
}

lk_status lk_cache_length(lk_cache cache, int32_t layer, int32_t* n) {
  if (!cache || !n) return fail(LK_ERR_ARG, "lk_cache_length: null argument");
  if (layer < 0 || layer >= cache->cv.L) return fail(LK_ERR_ARG, "lk_cache_length: layer %d out of range", layer);
  *n = cache->max_len(layer);
  return LK_OK;
}

lk_status lk_cache_lengths(lk_cache cache, int32_t layer, int32_t* lens) {
  if (!cache || !lens) return fail(LK_ERR_ARG, "lk_cache_lengths: null argument");
  if (layer < 0 || layer >= cache->cv.L) return fail(LK_ERR_ARG, "lk_cache_lengths: layer %d out of range", layer);
  std::memcpy(lens, &cache->host_len[(size_t)layer * cache->B], (size_t)cache->B * 4);
  return LK_OK;
}

lk_status lk_cache_region(lk_cache cache, int32_t layer, int32_t b, int32_t kv_head, lk_region_info* out) {
  if (!cache || !out) return fail(LK_ERR_ARG, "lk_cache_region: null argument");
  if (layer < 0 || layer >= cache->cv.L || b < 0 || b >= cache->B || kv_head < 0 || kv_head >= cache->cv.Hkv)
    return fail(LK_ERR_ARG, "lk_cache_region: (layer %d, b %d, kv_head %d) out of range", layer, b, kv_head);
  const HeadDesc& hd = cache->lay.heads[(size_t)layer * cache->cv.Hkv + kv_head];
  const Layout& lay = cache->lay;
  const int64_t ra = hd.row_a + (int64_t)b * hd.cap_a;
  out->policy = hd.policy;
  out->n_kept = hd.n_kept;
  out->rows_a = hd.cap_a;
  out->rows_b = hd.cap_b;
  out->k_a_offset = lay.off_pool[kPoolK128] + (uint64_t)ra * kHeadDim * 2;
  out->v_a_offset = lay.off_pool[kPoolV] + (uint64_t)ra * kHeadDim * 2;
  out->page_rows = 0;
  out->max_pages = 0;
  out->page_table_offset = 0;
  out->kv_format = lay.kv_format;
  out->sealed_blocks = 0;
  const bool q8 = kv_quantized(lay.kv_format);
  if (q8 && hd.cap_b > 0)
    out->sealed_blocks =
        pages_at(cache->host_len[(size_t)layer * cache->B + b], cache->cv.S, cache->cv.W, lay.kv_format);
  if (hd.cap_b > 0 && cache->paged() && !q8) {
    out->rows_b = (int32_t)std::min<int64_t>((int64_t)lay.num_pages[hd.pool_kb] * kPageRows, INT32_MAX);
    out->k_b_offset = lay.off_pool[hd.pool_kb] + (uint64_t)hd.krow_b * hd.n_kept * 2;
    out->v_b_offset = lay.off_pool[kPoolV] + (uint64_t)hd.vrow_b * kHeadDim * 2;
    out->page_rows = kPageRows;
    out->max_pages = lay.max_pages;
    out->page_table_offset =
        lay.off_pt + ((((uint64_t)layer * cache->B + b) * cache->cv.Hkv + kv_head) * lay.max_pages) * 4;
  } else if (hd.cap_b > 0) {
    out->k_b_offset = lay.off_pool[hd.pool_kb] + (uint64_t)(hd.krow_b + (int64_t)b * hd.cap_b) * hd.n_kept * 2;
    out->v_b_offset = lay.off_pool[kPoolV] + (uint64_t)(hd.vrow_b + (int64_t)b * hd.cap_b) * kHeadDim * 2;
  } else {
    out->k_b_offset = out->v_b_offset = 0;
  }
  return LK_OK;
}

lk_status lk_cache_block(lk_cache cache, int32_t layer, int32_t b, int32_t kv_head, int32_t block, int8_t* k_codes,
                         float* k_scales, int8_t* v_codes, float* v_scales, void* stream) {
  if (!cache) return fail(LK_ERR_ARG, "lk_cache_block: null cache");
  if (!kv_quantized(cache->lay.kv_format))
    return fail(LK_ERR_STATE, "lk_cache_block: the cache is not INT8 or FP8");
  if (layer < 0 || layer >= cache->cv.L || b < 0 || b >= cache->B || kv_head < 0 || kv_head >= cache->cv.Hkv)
    return fail(LK_ERR_ARG, "lk_cache_block: (layer %d, b %d, kv_head %d) out of range", layer, b, kv_head);
  const HeadDesc& hd = cache->lay.heads[(size_t)layer * cache->cv.Hkv + kv_head];
  const int sealed = hd.cap_b > 0 ? pages_at(cache->host_len[(size_t)layer * cache->B + b], cache->cv.S,
                                             cache->cv.W, cache->lay.kv_format)
                                  : 0;
  if (block < 0 || block >= sealed)
    return fail(LK_ERR_ARG, "lk_cache_block: block %d not in [0, %d) sealed blocks", block, sealed);
  const int k = hd.n_kept;
  const int qb = qblock_bytes(k);
  cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  int64_t at = 0;
  if (cache->paged()) {
    int32_t page = -1;
    const int32_t* pt = cache->cv.page_table +
                        (((int64_t)layer * cache->B + b) * cache->cv.Hkv + kv_head) * cache->lay.max_pages + block;
    if (err == cudaSuccess) err = cudaMemcpy(&page, pt, 4, cudaMemcpyDeviceToHost);
    if (err == cudaSuccess && page < 0) return fail(LK_ERR_STATE, "lk_cache_block: block %d has no page", block);
    at = hd.qoff + (int64_t)page * qb;
  } else {
    at = hd.qoff + ((int64_t)b * hd.qblocks + block) * qb;
  }
  std::vector<uint8_t> img(qb);
  if (err == cudaSuccess) err = cudaMemcpy(img.data(), cache->cv.qpool + at, qb, cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return cuda_fail(err, "lk_cache_block");
  for (int r = 0; r < kQBlockRows; ++r) {
    if (k_codes)
      for (int c = 0; c < k; ++c) k_codes[r * k + c] = (int8_t)img[(size_t)r * k + qbyte(k, r, c)];
    if (v_codes)
      for (int c = 0; c < kHeadDim; ++c) {
        const int byte = img[qblock_voff(k) + (size_t)r * kHeadDim + qbyte(kHeadDim, r, c)];
        // INT8 V codes are stored offset binary; FP8 codes as they are
        v_codes[r * kHeadDim + c] = (int8_t)(uint8_t)(cache->lay.kv_format == kKvInt8 ? byte - 128 : byte);
      }
  }
  if (k_scales) std::memcpy(k_scales, img.data() + qblock_ksoff(k), (size_t)k * 4);
  if (v_scales) std::memcpy(v_scales, img.data() + qblock_vsoff(k), (size_t)kQBlockRows * 4);
  return LK_OK;
}

lk_status lk_resident_bytes(lk_cache cache, int32_t layer, void* stream, uint64_t* bytes) {
  if (!cache || !bytes) return fail(LK_ERR_ARG, "lk_resident_bytes: null argument");
  if (layer < 0 || layer >= cache->cv.L) return fail(LK_ERR_ARG, "lk_resident_bytes: layer %d out of range", layer);
  const int B = cache->B, H = cache->cv.Hkv;
  std::vector<int32_t> len(B), cnt(B);
  cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err == cudaSuccess)
    err = cudaMemcpy(len.data(), cache->cv.len + (size_t)layer * B, B * 4, cudaMemcpyDeviceToHost);
  if (err == cudaSuccess)
    err = cudaMemcpy(cnt.data(), cache->cv.cnt + (size_t)layer * B, B * 4, cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return cuda_fail(err, "lk_resident_bytes");
  uint64_t total = 0;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) total += entry_bytes(cache, cache->lay.heads[(size_t)layer * H + h], len[b], cnt[b]);
  *bytes = total;
  return LK_OK;
}

lk_status lk_set_step_mode(lk_cache cache, int32_t mode) {
  if (!cache) return fail(LK_ERR_ARG, "lk_set_step_mode: null cache");
  if (mode != LK_STEP_AUTO && mode != LK_STEP_FUSED && mode != LK_STEP_SPLIT)
    return fail(LK_ERR_ARG, "lk_set_step_mode: mode %d is not LK_STEP_AUTO, LK_STEP_FUSED or LK_STEP_SPLIT", mode);
  cache->step_mode = mode;
  return LK_OK;
}

lk_status lk_step_is_fused(lk_cache cache, int32_t layer0, int32_t nlayers, int32_t* fused) {
  if (!cache || !fused) return fail(LK_ERR_ARG, "lk_step_is_fused: null argument");
  if (nlayers < 1 || layer0 < 0 || layer0 + nlayers > cache->cv.L)
    return fail(LK_ERR_ARG, "lk_step_is_fused: layers [%d, %d) out of range", layer0, layer0 + nlayers);
  *fused = fuse_step(cache, layer0, nlayers) ? 1 : 0;
  return LK_OK;
}

lk_status lk_set_wait_limit(lk_cache cache, uint64_t ns) {
  if (!cache) return fail(LK_ERR_ARG, "lk_set_wait_limit: null cache");
  if (ns > kMaxWaitLimitNs)
    return fail(LK_ERR_ARG, "lk_set_wait_limit: %llu ns exceeds %llu ns", (unsigned long long)ns,
                (unsigned long long)kMaxWaitLimitNs);
  cache->wait_limit_ns = ns;
  return LK_OK;
}

lk_status lk_set_decode_ctas(lk_cache cache, int32_t ctas) {
  if (!cache) return fail(LK_ERR_ARG, "lk_set_decode_ctas: null cache");
  if (ctas < 0 || ctas > kMaxCtas) return fail(LK_ERR_ARG, "lk_set_decode_ctas: %d out of [0, %d]", ctas, kMaxCtas);
  cache->decode_ctas = ctas;
  return LK_OK;
}

lk_status lk_check(lk_cache cache, void* stream) {
  if (!cache) return fail(LK_ERR_ARG, "lk_check: null cache");
  cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_check: stream");
  err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err, "lk_check: pending error");
  uint32_t status = 0;
  err = cudaMemcpy(&status, &cache->cv.hdr->status, 4, cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return cuda_fail(err, "lk_check: status read");
  if (status == 0) return LK_OK;
  // clear on the caller's stream and wait for it: a plain cudaMemset would
  // run on the legacy stream, which non-blocking streams do not wait for, so
  // a bit set by the caller's next launch could be cleared after the fact
  err = cudaMemsetAsync(&cache->cv.hdr->status, 0, 4, static_cast<cudaStream_t>(stream));
  if (err == cudaSuccess) err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "lk_check: status clear");
  if (status & kStatusTimeout) return fail(LK_ERR_TIMEOUT, "a device-side wait ran out (status 0x%x)", status);
  if (status & kStatusCapacity)
    return fail(LK_ERR_CAPACITY, "a layer or a SPECIAL head ran out of rows (status 0x%x)", status);
  return fail(LK_ERR_ARG, "a token id was outside [0, vocab) (status 0x%x)", status);
}

lk_status lk_decode_attn_static(lk_cache cache, int32_t layer, const void* q, float* o, void* stream) {
  if (!cache) return fail(LK_ERR_ARG, "lk_decode_attn_static: null cache");
  if (layer < 0 || layer >= cache->cv.L)
    return fail(LK_ERR_ARG, "lk_decode_attn_static: layer %d out of range", layer);
  if (!q || !o) return fail(LK_ERR_ARG, "lk_decode_attn_static: null q or o");
  if (!aligned(q, 16) || !aligned(o, 16))
    return fail(LK_ERR_ALIGN, "lk_decode_attn_static: q and o must be 16-byte aligned");
  // counters + partial (m, l) + partial o of one layer's entries
  lk_plan_desc one = cache->plan.d;
  one.num_layers = 1;
  const WsLayout w = ws_layout(one, cache->B);
  const size_t need = w.off_q;
  if (need > kStaticScratchBytes)
    return fail(LK_ERR_CAPACITY,
                "lk_decode_attn_static: this cache needs %zu bytes of split scratch; the built-in array has %zu "
                "(batch x kv heads too large; use lk_decode_attn with a workspace)",
                need, kStaticScratchBytes);
  void* scratch = nullptr;
  lk_status st = static_scratch(&scratch);
  if (st != LK_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the counters must start at zero whatever an earlier call left behind
  cudaError_t err = cudaMemsetAsync(ws + w.off_counters, 0, (size_t)cache->B * cache->cv.Hkv * 4, s);
  if (err != cudaSuccess) return cuda_fail(err, "lk_decode_attn_static: counter clear");
  DecodeArgs a;
  a.cv = cache->cv;
  a.layer = layer;
  a.nlayers = 1;
  a.q = static_cast<const uint16_t*>(q);
  a.o = o;
  a.part = reinterpret_cast<float*>(ws + w.off_part);
  a.part_ml = reinterpret_cast<float2*>(ws + w.off_ml);
  a.counters = reinterpret_cast<int32_t*>(ws + w.off_counters);
  a.wait_limit_ns = cache->wait_limit_ns;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)kHeadDim));
  a.k_new = a.v_new = nullptr;
  a.ids = nullptr;
  set_divisors(cache, a);
  int ctas = cache->decode_ctas > 0 ? cache->decode_ctas : default_decode_ctas(cache, 1);
  ctas = std::max(1, std::min(ctas, kMaxCtas));
  err = launch_decode(cache->maps, a, ctas, s);
  if (err != cudaSuccess) return cuda_fail(err, "lk_decode_attn_static launch");
  return LK_OK;
}

}  // extern "C"
