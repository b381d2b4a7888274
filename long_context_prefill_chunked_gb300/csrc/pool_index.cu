// Block pooling for the block-sparse path ("Porting FlashPrefill V2 to Apple
// silicon for faster prefill", section "Compress keys before the heavy work":
// average the keys of each block into one pooled key; values likewise).
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

// One CTA per (key block, batch), blocks blk0 .. nblk - 1; thread t owns 8 consecutive
// elements of the [H, d] slab of every row of the block and sums them in fp32.
__global__ void pool_kernel(PoolArgs a, int bf16) {
  const int e0 = threadIdx.x * 8;
  const int h = e0 / a.d, e = e0 % a.d;
  const int blk = a.blk0 + (int)blockIdx.x, b = blockIdx.y;
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
  const long long o = (((long long)b * a.H + h) * a.cap + blk) * a.d + e;
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
  if (a.out_hi != nullptr) {
    // mean = hi + lo + O(2^-17 |mean|): the index scores q.hi + q.lo to that accuracy
    uint32_t wh[4], wl[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float m0 = acc[2 * k] * inv, m1 = acc[2 * k + 1] * inv;
      wh[k] = bf16 ? pack_bf16(m0, m1) : pack_f16(m0, m1);
      const float h0 = bf16 ? __uint_as_float(wh[k] << 16) : __half2float(__ushort_as_half((unsigned short)(wh[k] & 0xFFFFu)));
      const float h1 = bf16 ? __uint_as_float(wh[k] & 0xFFFF0000u) : __half2float(__ushort_as_half((unsigned short)(wh[k] >> 16)));
      wl[k] = bf16 ? pack_bf16(m0 - h0, m1 - h1) : pack_f16(m0 - h0, m1 - h1);
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out_hi) + o) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out_lo) + o) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
  }
}

// Longest-first order of the sparse attention's work units.  Unit u is the one the
// attention kernel runs as CTA u in its natural order (query tiles from the last);
// its cost in key tiles is its pooled tiles plus both heads' kept-list lengths (an
// upper bound on the union it executes).  One CTA counting-sorts the costs
// descending and writes perm[i] = the i-th heaviest unit, so that the hardware
// block scheduler hands the heavy units out first.
constexpr int kOrderBins = 8192;
__global__ void __launch_bounds__(1024) order_units_kernel(OrderArgs o) {
  __shared__ int bins[kOrderBins];
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x;
  auto cost = [&](int u) {
    const int per_qt = o.n_hp * o.B;
    const int qt = o.n_qt - 1 - u / per_qt;
    const int rem = u % per_qt;
    const int b = rem / o.n_hp;
    const int h0 = (rem % o.n_hp) * o.slots;
    const int ob = o.s / 128 + qt;
    int c = (ob + 127) / 128 + o.tile_cnt[(long long)(b * o.Hq + h0) * o.n_qt + qt];
    if (o.slots == 2) c += o.tile_cnt[(long long)(b * o.Hq + h0 + 1) * o.n_qt + qt];
    return min(max(c, 0), kOrderBins - 1);
  };
  for (int i = tid; i < kOrderBins; i += blockDim.x) bins[i] = 0;
  __syncthreads();
  for (int u = tid; u < o.U; u += blockDim.x) atomicAdd(&bins[cost(u)], 1);
  __syncthreads();
  // exclusive scan from the highest cost down: bins[c] = units costing more than c
  constexpr int per = kOrderBins / 1024;
  int loc[per], run = 0;
  const int hi = kOrderBins - 1 - tid * per;  // this thread's bins, descending
#pragma unroll
  for (int i = 0; i < per; ++i) {
    loc[i] = run;
    run += bins[hi - i];
  }
  int incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if ((tid & 31) >= off) incl += v;
  }
  if ((tid & 31) == 31) warp_sums[tid >> 5] = incl;
  __syncthreads();
  if (tid < 32) {
    int v = warp_sums[tid];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, off);
      if (tid >= off) v += t;
    }
    warp_sums[tid] = v;  // inclusive over warps
  }
  __syncthreads();
  const int before = (incl - run) + ((tid >> 5) > 0 ? warp_sums[(tid >> 5) - 1] : 0);
#pragma unroll
  for (int i = 0; i < per; ++i) bins[hi - i] = before + loc[i];
  __syncthreads();
  for (int u = tid; u < o.U; u += blockDim.x) o.perm[atomicAdd(&bins[cost(u)], 1)] = u;
}

}  // namespace

cudaError_t launch_order_units(const OrderArgs& o, cudaStream_t st) {
  order_units_kernel<<<1, 1024, 0, st>>>(o);
  ++t_launches;
  return cudaGetLastError();
}

cudaError_t launch_pool(const PoolArgs& a, int bf16, cudaStream_t st) {
  if (a.blk0 >= a.nblk) return cudaSuccess;  // every block already pooled
  dim3 grid(a.nblk - a.blk0, a.B);
  pool_kernel<<<grid, a.H * a.d / 8, 0, st>>>(a, bf16);
  ++t_launches;
  return cudaGetLastError();
}

}  // namespace pf
