// Packs an indexer's keep lists into per-row key bits and per-query-tile key-tile bitmaps.
//
// Method: "ANE Prefill Research", section "Folding a sparse indexer's selection into the
// mask": the indexer keeps compressed key blocks per query (keepIndices / keepCounts) and the
// keys after the last complete block stay visible.  The pages fold that selection into an
// additive mask of -30000; here it becomes the bit form of the same mask directly (no [C, T]
// float mask is written or read), which the attention kernel's bits mode consumes, skipping
// the 128-key tiles no row of a query tile sees.
#include "indexed.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace pf {
namespace {

// sets key bits [k0, k1) of a shared-memory row
__device__ __forceinline__ void set_key_range(uint32_t* rw, int k0, int k1) {
  while (k0 < k1) {
    const int b = k0 & 31;
    const int n = min(k1 - k0, 32 - b);
    const uint32_t m = (n == 32 ? 0xffffffffu : ((1u << n) - 1u)) << b;
    atomicOr(&rw[k0 >> 5], m);
    k0 += n;
  }
}

// Bits 0, 4, ..., 28 of x moved to bits 0 .. 7.
__device__ __forceinline__ uint32_t every_fourth(uint32_t x) {
  x &= 0x11111111u;
  x = (x | (x >> 3)) & 0x03030303u;
  x = (x | (x >> 6)) & 0x000F000Fu;
  return (x | (x >> 12)) & 0x000000FFu;
}

// A 128-key tile's bits in key order (bit i of word q = key 32q + i) in the packed-mask layout
// the attention kernel reads (bit L of word c = key 4L + c).
__device__ __forceinline__ uint4 to_packed_layout(const uint32_t (&o)[4]) {
  uint32_t w[4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
    w[c] = every_fourth(o[0] >> c) | (every_fourth(o[1] >> c) << 8) | (every_fourth(o[2] >> c) << 16) |
           (every_fourth(o[3] >> c) << 24);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One CTA per row (rows past the grid loop): the row's bits are built in key order in shared
// memory, then written 16 bytes (one 128-key tile) per thread in the packed-mask layout; a
// warp's 32 consecutive tiles become one tile-bitmap word through a ballot.
__global__ void __launch_bounds__(256) index_pack_kernel(const int32_t* __restrict__ keep_idx,
                                                         const int32_t* __restrict__ keep_cnt,
                                                         long long stride, int ratio, int C, int s,
                                                         uint32_t* __restrict__ bits, int words,
                                                         uint32_t* tiles, int tile_words,
                                                         unsigned* status) {
  extern __shared__ uint32_t rw[];
  const int n_kt = words / 4;
  for (int row = blockIdx.x; row < C; row += gridDim.x) {
    const int p = s + row;
    const int n_complete = (p + 1) / ratio;
    for (int w = threadIdx.x; w < words; w += blockDim.x) rw[w] = 0u;
    __syncthreads();
    int cnt = __ldg(keep_cnt + row);
    bool bad = cnt < 0 || cnt > stride;
    cnt = cnt < 0 ? 0 : (cnt > stride ? (int)stride : cnt);
    const int32_t* list = keep_idx + (long long)row * stride;
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
      const int c = __ldg(list + i);
      if (c < 0 || c >= n_complete) {
        bad = true;
        continue;
      }
      set_key_range(rw, c * ratio, c * ratio + ratio);
    }
    if (threadIdx.x == 0) set_key_range(rw, n_complete * ratio, p + 1);
    __syncthreads();
    bool any = false;
    uint4* out = reinterpret_cast<uint4*>(bits + (long long)row * words);
    for (int t0 = 0; t0 < n_kt; t0 += blockDim.x) {
      const int t = t0 + threadIdx.x;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (t < n_kt) {
        const uint32_t o[4] = {rw[4 * t], rw[4 * t + 1], rw[4 * t + 2], rw[4 * t + 3]};
        v = to_packed_layout(o);
        out[t] = v;
      }
      const bool seen = (v.x | v.y | v.z | v.w) != 0u;
      any |= seen;
      const uint32_t word = __ballot_sync(0xffffffffu, seen);
      if (tiles != nullptr && (threadIdx.x & 31) == 0 && word != 0u)
        atomicOr(&tiles[(long long)(row >> 7) * tile_words + (t >> 5)], word);
    }
    if (bad) record_error(status, ST_SELECTION, 0x500u);
    // also the barrier before the next row clears the shared row
    if (__syncthreads_or(any) == 0 && threadIdx.x == 0) record_error(status, ST_SELECTION, 0x501u);
  }
}

}  // namespace

cudaError_t launch_index_pack(const int32_t* keep_idx, const int32_t* keep_cnt, long long stride,
                              int ratio, int C, int s, uint32_t* bits, int words, uint32_t* tiles,
                              int tile_words, unsigned* status, cudaStream_t st) {
  const size_t smem = (size_t)words * 4;
  static std::atomic<int> configured[64];
  if (smem > 48 * 1024) {
    cudaError_t e =
        ensure_dynamic_smem(reinterpret_cast<const void*>(index_pack_kernel), (int)smem, configured);
    if (e != cudaSuccess) return e;
  }
  const int grid = C < 152 * 8 ? C : 152 * 8;
  index_pack_kernel<<<grid, 256, smem, st>>>(keep_idx, keep_cnt, stride, ratio, C, s, bits, words, tiles,
                                             tile_words, status);
  ++t_launches;
  return cudaGetLastError();
}

}  // namespace pf
