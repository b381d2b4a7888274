// Internal kernel arguments and launchers of libpf (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace pf {

constexpr int kTile = 128;        // query rows and keys per tile (= key block of the sparse path)
constexpr int kMaxSplit = 8;      // parts of one split dense unit (tail split)
constexpr int kAttnThreads = 384; // 8 softmax warps (2 slots x 4), TMA warp, MMA warp, 2 V converters

// MODE_MASKB: an explicit mask read as the packing pass's bits.  A packed mask is launched
// twice, MODE_MASKB then MODE_MASK; each launch returns at once unless the pass's decision on
// the mask (binary or not) is its own, so each keeps its own register allocation.
enum AttnMode : int { MODE_CAUSAL = 0, MODE_MASK = 1, MODE_SPARSE = 2, MODE_MASKB = 3 };

struct AttnArgs {
  int B, Hq, Hkv, G, d, C, s, T;
  int n_qt;             // query tiles per (b, head)
  int slots;            // query heads per CTA sharing one K/V stream (1 or 2)
  int n_hp;             // head groups of `slots` heads per batch
  int n_hist_tiles;     // key tiles served by the history map (s / 128)
  int ab_type;          // 0 = f16, 1 = bf16 operands of S = Q K^T
  int convert_v;        // 1: V tiles are bf16 and are converted to fp16 in shared memory
  float scale_log2;     // scale * log2(e)
  // explicit additive mask (MODE_MASK)
  const void* mask;
  int mask_f16;         // 1 = fp16 mask, 0 = fp32
  int mask_vec;         // rows 16-byte aligned: vector loads allowed
  long long mask_ld;    // elements between mask rows
  // the same mask packed to bits when every value is 0 or <= -10000 (bit set = kept);
  // used only while *mask_nonbinary == 0 (the packing pass sets it otherwise)
  const uint32_t* mask_bits;  // [C][mask_words], rows padded to a multiple of 4 words
  int mask_words;
  const int* mask_nonbinary;
  // per 128-row query tile, a bit per 128-key tile that some row of the tile keeps (binary
  // masks only; null = visit every key tile)
  const uint32_t* mask_tiles;  // [n_qt][mask_tile_words]
  int mask_tile_words;
  // output
  void* out;
  float* lse;           // [B, Hq, C] log of each row's softmax denominator, or null
  int out_dtype;        // 0 f16, 1 bf16, 2 f32
  long long o_sb, o_st, o_sh;
  // block-sparse selection (MODE_SPARSE)
  const uint32_t* row_bits;   // [B, Hq, C, W]
  const int32_t* tile_list;   // [B, Hq, n_qt, nblk]
  const int32_t* tile_cnt;    // [B, Hq, n_qt]
  int words, nblk;
  float log2_nb;              // log2 of the pooled weight n_b (block size)
  // tail split (MODE_CAUSAL / MODE_MASK): units [0, n_whole) run whole, one CTA each; every
  // later unit runs as split_k CTAs over consecutive key-tile ranges, and the last of them to
  // finish merges the parts' partial results
  const int32_t* perm;  // sparse: CTA i runs unit perm[i] (longest first); null = natural order
  int n_whole;          // = number of units when nothing is split
  int split_k;          // parts per split unit (1 = no split)
  float* ws_part;       // per part and slot: O^T [d][128] then m [128] and l [128], fp32
  int* ws_cnt;          // finished parts per split unit, zero at launch
  // robustness
  unsigned* status;     // device status words (timeout flag, where)
  long long timeout;    // bounded-wait limit, SM cycles
  int withhold;         // test hook: never signal the first S tile
};

struct AttnMaps {
  CUtensorMap q, kh, kc, vh, vc, kbar, vbar;
  CUtensorMap out;  // [B, C, Hq, d] in the output type, box 128 bytes x 1 head x 128 rows
};

cudaError_t launch_attn(const AttnMaps& maps, const AttnArgs& a, int mode, cudaStream_t st);
// Packs an additive mask [C, T] (row stride ld) into bits [C][words] (kept iff the value is 0)
// and sets *nonbinary when a value is neither 0 nor <= -10000 or a row keeps no key; with
// tiles (zeroed, [ceil(C / 128)][tile_words]) it also ORs in the key tiles each query tile keeps.
// vec: rows start on 16-byte boundaries (base and ld * element size), so vector loads are allowed.
cudaError_t launch_mask_pack(const void* mask, int f16, int vec, int C, int T, long long ld, uint32_t* bits,
                             int words, int* nonbinary, uint32_t* tiles, int tile_words, cudaStream_t st);

// bf16 -> fp16, nvec 16-byte vectors (8 elements each); a value beyond fp16's range sets
// ST_VRANGE in status
cudaError_t launch_convert_f16(const void* src, void* dst, long long nvec, unsigned* status, cudaStream_t st);

// bit copy of the chunk's K and V into the cache layout (one launch for both)
cudaError_t launch_kv_relayout(const void* src_k, const void* src_v, void* dst_k, void* dst_v, int B, int C,
                               int H, int d, const long long ss[3], const long long ds[3], cudaStream_t st);

// mean-pool each key block: x [B, T, H, d] -> fp32 [B, H, nblk, d] (+ optional 16-bit copy)
struct PoolArgs {
  const void* x;
  int B, T, H, d, block, nblk;
  int cap;               // blocks per (b, h) in the outputs (>= nblk)
  int blk0;              // first block to pool (the ones before are already pooled)
  long long sb, st, sh;
  float* out_f32;        // [B, H, cap, d]
  void* out_lp;          // [B, H, cap, d] in the input type, may be null
  void* out_hi;          // [B, H, cap, d] 16-bit round of the mean, may be null
  void* out_lo;          // [B, H, cap, d] 16-bit round of (mean - hi), may be null
};
cudaError_t launch_pool(const PoolArgs& a, int bf16, cudaStream_t st);

// Longest-first order of the sparse attention's units (see order_units_kernel).
struct OrderArgs {
  const int32_t* tile_cnt;  // [B, Hq, n_qt]
  int B, Hq, n_qt, slots, n_hp, s, U;
  int32_t* perm;            // [U] out
};
cudaError_t launch_order_units(const OrderArgs& o, cudaStream_t st);

struct IndexArgs {
  int ab_type;           // 0 = f16, 1 = bf16 (q and the kbar hi/lo split)
  int B, Hq, Hkv, G, d, C, s, nblk, n_qt, words;
  int slots, n_hp;       // query heads per CTA (1 or 2) and head groups per batch
  float scale;
  float log_alpha;       // ln(alpha); -inf when alpha == 0
  // keep rules (all zero = the alpha rule alone)
  int sink_blocks;       // candidates b < sink_blocks are kept
  int local_blocks;      // candidates b >= ob - local_blocks are kept
  int tail_from;         // rows at positions p >= tail_from keep every candidate
  int row_group32;       // 1: the 32 rows of a warp share the union of their kept blocks
  uint32_t* row_bits;
  int32_t* tile_list;
  int32_t* tile_cnt;
  unsigned* status;
  long long timeout;
  int grid;              // CTAs to launch (one per SM); each runs units blockIdx.x + k * grid
};
struct IndexMaps {
  CUtensorMap q, hi, lo;
};
cudaError_t launch_index(const IndexMaps& maps, const IndexArgs& a, cudaStream_t st);
// Shared selection of a KV group: row bits ORed over the group's G query heads, written
// back to each, and each head's tile lists rebuilt from them.
cudaError_t launch_share_group(const IndexArgs& a, cudaStream_t st);

extern thread_local long long t_launches;

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device once: the
// attribute belongs to each device's copy of the kernel, so `done` holds the limit set so far
// per device (64 entries, zero-initialised).
inline cudaError_t ensure_dynamic_smem(const void* kernel, int bytes, std::atomic<int>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(bytes, std::memory_order_relaxed);
  return e;
}

}  // namespace pf
