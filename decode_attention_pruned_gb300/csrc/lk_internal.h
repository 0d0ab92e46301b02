// Internal data structures shared by the host API and the device kernels.
//
// Device layout of a cache buffer (every block 1024-byte aligned):
//   DevHeader | len[L][B] | cnt[L][B] | active[B] | page table | free lists
//   | HeadDesc[L][Hkv] | kept[L][Hkv][128] i16 | is_special[vocab] u8
//   | pool K128 | pool V | pool K32 | pool K64 | pool K96
//
// Pools are 2-D row arrays (rows x width bf16); heads of equal kept width
// share a pool (the head grouping of LeanK section 3.1).  Region A (full
// width: sinks + window ring, LOCAL ring, SPECIAL rows) of every head sits at
// the same row index in pools K128 and V, grouped by policy class so that a
// class's rows are equal blocks of cap_a rows per (head, sequence).
// Region B (middle tokens of FULL heads with k > 0) has its K rows in the
// pool of width k and its V rows after all region-A rows of pool V: either
// contiguous per (layer, sequence, head), or in 128-row pages drawn from a
// page area per width class (page p of class c: K rows krow_b + 128p.. of
// pool c, V rows vrow_b + 128p.. of pool V), located through the page table
// [L][B][Hkv][max_pages].  Free pages of each class sit on a device stack, so
// appends allocate pages inside the kernel (graph replays included).
//
// INT8 / FP8 caches (KIVI-style quantisation after pruning): region B keeps
// only its last, incomplete 128-row block in bf16 (the "tail", 128 rows per
// (layer, sequence, head) in pools K_k and V); every complete block is sealed
// into a byte block of the Q pool (contiguous per head and sequence, or a
// page of its width class):
//   [K codes 128 x k][V codes 128 x 128][K scales k x f32][V scales 128 x f32]
// Codes are row-major; within each 16-channel group a row stores channels
// (0, 8, 1, 9, ..., 7, 15) and its 16-byte groups are XOR-swizzled by row
// (qswz), so ldmatrix reads mma fragments without bank conflicts.  INT8: K
// codes are two's complement, V codes offset binary (code + 128).  FP8: K and
// V codes are e4m3 bytes.
#pragma once
#include <stdint.h>

namespace lk {

constexpr int kHeadDim = 128;
constexpr int kMaxGroup = 8;        // query heads per kv head handled by one mma n8 tile
constexpr int kMaxCtas = 256;       // decode grid cap (partial workspace; combine staging np*G <= 2048)
constexpr int kTmaBoxRows = 128;    // token rows per TMA box = decode tile rows
constexpr int kPageRows = 128;      // middle rows per page (paged caches)
constexpr int kQBlockRows = 128;    // rows per sealed INT8 / FP8 block (= one page, one tile)

enum KvFormat : int32_t { kKvBf16 = 0, kKvInt8 = 1, kKvFp8 = 2 };
// complete middle blocks are sealed into one-byte codes + fp32 scales
__host__ __device__ constexpr bool kv_quantized(int fmt) { return fmt != kKvBf16; }

// Bytes of a sealed block (INT8 or FP8: one byte per code) of width k and the
// offsets of its parts.
__host__ __device__ constexpr int qblock_bytes(int k) { return 132 * (k + 128); }
__host__ __device__ constexpr int qblock_voff(int k) { return 128 * k; }
__host__ __device__ constexpr int qblock_ksoff(int k) { return 128 * k + 128 * 128; }
__host__ __device__ constexpr int qblock_vsoff(int k) { return 128 * k + 128 * 128 + 4 * k; }
// 16-byte group swizzle of row r in a block row of `width` bytes
__host__ __device__ constexpr int qswz(int width, int r) {
  return width == 128 ? (r & 7) : width == 64 ? ((r >> 1) & 3) : ((r >> 2) & 1);
}
// byte of channel c (< width) in row r of a sealed block part of that width
__host__ __device__ constexpr int qbyte(int width, int r, int c) {
  return 16 * ((c >> 4) ^ qswz(width, r)) + ((c & 15) < 8 ? 2 * (c & 7) : 2 * (c & 7) + 1);
}

enum Policy : int32_t { kFull = 0, kLocal = 1, kSpecial = 2 };
enum Pool : int32_t { kPoolK128 = 0, kPoolV = 1, kPoolK32 = 2, kPoolK64 = 3, kPoolK96 = 4, kNumPools = 5 };

// Sticky device status bits (cache header).
enum StatusBits : uint32_t {
  kStatusTimeout = 1u << 0,     // a bounded wait ran out
  kStatusCapacity = 1u << 1,    // a SPECIAL head overflowed its rows, a layer was full or no page was free
  kStatusBadId = 1u << 2,       // token id outside [0, vocab)
};

struct HeadDesc {                 // one (layer, kv head)
  int32_t policy;
  int32_t n_kept;                 // k for FULL heads, 0 otherwise
  int32_t cap_a;                  // region-A rows per sequence
  int32_t cap_b;                  // region-B rows per sequence (0 if none)
  int32_t pool_kb;                // pool of region-B K rows (= its page class)
  int32_t free_off;               // paged: first entry of the class's free stack
  int64_t row_a;                  // first region-A row (sequence 0) in K128 and V
  int64_t krow_b;                 // first region-B row (sequence 0) in pool_kb; paged: page area
  int64_t vrow_b;                 // first region-B row (sequence 0) in V; paged: page area
  int64_t qoff;                   // INT8 / FP8: byte offset in the Q pool of sequence 0's blocks
                                  //       (paged: of the class's page area)
  int32_t qblocks;                // INT8 / FP8, contiguous: sealed blocks per sequence
  // decode TMA views (a pool's rows seen as equal blocks, one per sequence or
  // page): the block of sequence 0's region A in its policy class's view,
  // and of sequence 0's region-B K and V rows (paged: of the class's page 0)
  int32_t blk_a;
  int32_t kblk_b;
  int32_t vblk_b;
};
static_assert(sizeof(HeadDesc) == 72, "HeadDesc layout");

struct DevHeader {
  uint32_t status;
  int32_t free_top[kNumPools];    // paged: free pages on each class's stack
  uint32_t pad[58];
};
static_assert(sizeof(DevHeader) == 256, "DevHeader layout");

// Pointers into one cache buffer, filled at cache init.
struct CacheView {
  DevHeader* hdr;
  int32_t* len;                   // [L][B] tokens per layer and sequence
  int32_t* cnt;                   // [L][B] special-token rows per layer and sequence
  int32_t* active;                // [B] 0: released slot, appends skip it
  int32_t* page_table;            // [L][B][Hkv][max_pages] or null (contiguous region B)
  int32_t* free_list;             // free page ids, class stacks at HeadDesc::free_off
  const HeadDesc* heads;          // [L][Hkv]
  const int16_t* kept;            // [L][Hkv][128] kept channels ascending
  const uint8_t* is_special;      // [vocab]
  uint16_t* pool[kNumPools];      // bf16 rows
  uint8_t* qpool;                 // INT8 / FP8: sealed blocks
  int64_t pool_rows[kNumPools];
  int32_t L, B, Hq, Hkv, G, S, W, W_loc, vocab, capacity;
  int32_t spec_cap;               // rows of a SPECIAL head per sequence
  int32_t max_pages;              // pages per (layer, sequence, head); 0: not paged
  int32_t kv_format;              // KvFormat of region B
};

inline int pool_width(int pool) {
  switch (pool) {
    case kPoolK32: return 32;
    case kPoolK64: return 64;
    case kPoolK96: return 96;
    default: return 128;
  }
}

inline int pool_for_width(int k) {
  switch (k) {
    case 32: return kPoolK32;
    case 64: return kPoolK64;
    case 96: return kPoolK96;
    default: return kPoolK128;
  }
}

}  // namespace lk
