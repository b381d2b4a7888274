// Block pooling and block selection for the block-sparse path.
//
// "Porting FlashPrefill V2 to Apple silicon for faster prefill":
//   section "Compress keys before the heavy work"  -> pool_kernel (block means)
//   section "A cheap map of where the attention lives" and "The algorithm
//   starts here" -> index_kernel: one pooled score per query row per earlier
//   block, keep the blocks within ln(alpha) of the row's hottest block plus
//   the diagonal, and compact each query tile's union of kept blocks.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace pf {
namespace {

__device__ __forceinline__ void unpack8(const uint4 w, bool bf16, float (&f)[8]) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (bf16) {
      f[2 * e] = __uint_as_float(ww[e] << 16);
      f[2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
    } else {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&ww[e]));
      f[2 * e] = t.x;
      f[2 * e + 1] = t.y;
    }
  }
}

// One CTA per (key block, batch); thread t owns 8 consecutive elements of the
// [H, d] slab of every row of the block and sums them in fp32.
__global__ void pool_kernel(PoolArgs a, int bf16) {
  const int e0 = threadIdx.x * 8;
  const int h = e0 / a.d, e = e0 % a.d;
  const int blk = blockIdx.x, b = blockIdx.y;
  const int r0 = blk * a.block;
  const int n = min(a.T - r0, a.block);
  const uint16_t* base = static_cast<const uint16_t*>(a.x) + b * a.sb + (long long)r0 * a.st +
                         (long long)h * a.sh + e;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int i = 0;
  for (; i + 8 <= n; i += 8) {
    uint4 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) w[u] = __ldg(reinterpret_cast<const uint4*>(base + (long long)(i + u) * a.st));
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float f[8];
      unpack8(w[u], bf16 != 0, f);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] += f[k];
    }
  }
  for (; i < n; ++i) {
    float f[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(base + (long long)i * a.st)), bf16 != 0, f);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] += f[k];
  }
  const float inv = 1.f / (float)n;
  const long long o = (((long long)b * a.H + h) * a.nblk + blk) * a.d + e;
  float4* of = reinterpret_cast<float4*>(a.out_f32 + o);
  of[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  of[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  if (a.out_lp != nullptr) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = bf16 ? pack_bf16(acc[2 * k] * inv, acc[2 * k + 1] * inv)
                  : pack_f16(acc[2 * k] * inv, acc[2 * k + 1] * inv);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out_lp) + o) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void f32_to_lp_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst,
                                 long long n, int bf16) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; 2 * i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float2 v = reinterpret_cast<const float2*>(src)[i];
    reinterpret_cast<uint32_t*>(dst)[i] = bf16 ? pack_bf16(v.x, v.y) : pack_f16(v.x, v.y);
  }
}

constexpr int kChunk = 32;     // pooled blocks staged per step (one selection word)
constexpr int kMaxWords = 64;  // selection words per row (2048 blocks)

// One CTA per (query tile, batch, head); thread r owns query row q0 + r.
// Pass 1 finds the row's hottest candidate, pass 2 recomputes the scores and
// keeps b iff (s_b - s_max) * scale >= ln(alpha).
template <int D>
__global__ void __launch_bounds__(128) index_kernel(IndexArgs a) {
  __shared__ float kb[kChunk][D];
  __shared__ uint32_t uni[kMaxWords];
  const int per_qt = a.B * a.Hq;
  const int qt = a.n_qt - 1 - (int)blockIdx.x / per_qt;
  const int rem = (int)blockIdx.x % per_qt;
  const int b = rem / a.Hq, h = rem % a.Hq, g = h / a.G;
  const int r = threadIdx.x, lane = r & 31;
  const int q0 = qt * kTile, row = q0 + r;
  const bool valid = row < a.C;
  const int ob = (a.s + q0) / kTile;  // candidates: blocks 0 .. ob-1
  for (int w = r; w < kMaxWords; w += 128) uni[w] = 0u;

  float q[D];
  {
    const uint16_t* qp = static_cast<const uint16_t*>(a.q) + b * a.q_sb + (long long)(valid ? row : 0) * a.q_st +
                         (long long)h * a.q_sh;
#pragma unroll
    for (int v = 0; v < D / 8; ++v) {
      float f[8];
      unpack8(valid ? __ldg(reinterpret_cast<const uint4*>(qp) + v) : make_uint4(0, 0, 0, 0),
              a.ab_type == 1, f);
#pragma unroll
      for (int k = 0; k < 8; ++k) q[8 * v + k] = f[k];
    }
  }
  const float* kbar = a.kbar + ((long long)b * a.Hkv + g) * a.nblk * D;
  float smax = -INFINITY;
  uint32_t* bits = a.row_bits + ((long long)(b * a.Hq + h) * a.C + (valid ? row : 0)) * a.words;
  const int dword = ob >> 5;
  for (int pass = 0; pass < 2; ++pass) {
    for (int c0 = 0; c0 < ob; c0 += kChunk) {
      const int nc = min(kChunk, ob - c0);
      __syncthreads();
      for (int i = r; i < nc * D / 4; i += 128)
        reinterpret_cast<float4*>(&kb[0][0])[i] = reinterpret_cast<const float4*>(kbar + (long long)c0 * D)[i];
      __syncthreads();
      uint32_t word = 0u;
      for (int i = 0; i < nc; ++i) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int e = 0; e < D; e += 4) {
          const float4 k4 = *reinterpret_cast<const float4*>(&kb[i][e]);
          s0 = fmaf(q[e], k4.x, s0);
          s1 = fmaf(q[e + 1], k4.y, s1);
          s2 = fmaf(q[e + 2], k4.z, s2);
          s3 = fmaf(q[e + 3], k4.w, s3);
        }
        const float s = (s0 + s1) + (s2 + s3);
        if (pass == 0) {
          smax = fmaxf(smax, s);
        } else if ((s - smax) * a.scale >= a.log_alpha) {
          word |= 1u << i;
        }
      }
      if (pass == 1) {
        const int w = c0 >> 5;
        if (w == dword) word |= 1u << (ob & 31);
        if (valid) bits[w] = word;
        const uint32_t u = __reduce_or_sync(0xffffffffu, valid ? word : 0u);
        if (lane == 0 && u) atomicOr(&uni[w], u);
      }
    }
  }
  // words past the last candidate chunk: only the diagonal bit can be set
  const int w_first = (ob + kChunk - 1) / kChunk;
  for (int w = w_first; w < a.words; ++w) {
    const uint32_t word = (w == dword) ? (1u << (ob & 31)) : 0u;
    if (valid) bits[w] = word;
  }
  __syncthreads();
  if (r == 0) uni[dword] |= 1u << (ob & 31);
  __syncthreads();
  // compact the tile's union of kept blocks, ascending
  if (r < 32) {
    const long long t = (long long)(b * a.Hq + h) * a.n_qt + qt;
    int32_t* list = a.tile_list + t * a.nblk;
    int base = 0;
    for (int w0 = 0; w0 < a.words; w0 += 32) {
      const int w = w0 + lane;
      const uint32_t bw = (w < a.words) ? uni[w] : 0u;
      const int cnt = __popc(bw);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int pos = base + incl - cnt;
      uint32_t rb = bw;
      while (rb) {
        const int i = __ffs(rb) - 1;
        rb &= rb - 1u;
        list[pos++] = w * 32 + i;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) a.tile_cnt[t] = base;
  }
}

}  // namespace

cudaError_t launch_pool(const PoolArgs& a, int bf16, cudaStream_t st) {
  dim3 grid(a.nblk, a.B);
  pool_kernel<<<grid, a.H * a.d / 8, 0, st>>>(a, bf16);
  ++t_launches;
  return cudaGetLastError();
}

cudaError_t launch_f32_to_lp(const float* src, void* dst, long long n, int bf16, cudaStream_t st) {
  const long long pairs = n / 2;
  const int threads = 256;
  long long want = (pairs + threads - 1) / threads;
  const int grid = (int)(want < 152 * 8 ? (want > 0 ? want : 1) : 152 * 8);
  f32_to_lp_kernel<<<grid, threads, 0, st>>>(src, static_cast<uint16_t*>(dst), n, bf16);
  ++t_launches;
  return cudaGetLastError();
}

cudaError_t launch_index(const IndexArgs& a, cudaStream_t st) {
  const int grid = a.n_qt * a.B * a.Hq;
  if (a.d == 128)
    index_kernel<128><<<grid, 128, 0, st>>>(a);
  else
    index_kernel<64><<<grid, 128, 0, st>>>(a);
  ++t_launches;
  return cudaGetLastError();
}

}  // namespace pf
