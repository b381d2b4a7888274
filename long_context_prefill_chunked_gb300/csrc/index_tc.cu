// Block index on the tensor cores: pooled scores s_rb = q_r . kbar_b for every
// query row and every earlier key block, the row's hottest block, and the kept
// blocks (exp(s_rb - s_max) >= alpha, i.e. (s_rb - s_max) * scale >= ln alpha)
// plus the diagonal; then each query tile's union of kept blocks, ascending.
//
// Method: "Porting FlashPrefill V2 to Apple silicon for faster prefill",
// sections "A cheap map of where the attention lives" (one pooled score per
// query row per block, local block exact) and "The algorithm starts here"
// (keep blocks above alpha x the row's hottest block, plus the diagonal).
//
// The scores must decide a threshold the float64 definition decides, so they
// are computed to about 2^-17 relative error: kbar (fp32 block means) is split
// into kbar_hi = bf16(kbar) and kbar_lo = bf16(kbar - kbar_hi) and each score is
// accumulated in fp32 tensor memory as q . kbar_hi + q . kbar_lo (q is bf16 and
// exact).  Pass 1 streams every pooled tile (128 blocks; 64 at head dim 256) once
// to find the row maximum, pass 2 streams them again and thresholds.  A unit with
// at most two pooled tiles keeps pass 1's scores in its two tensor-memory buffers
// and pass 2 reads them again instead of recomputing them.
//
// One CTA = (batch, 128-row query tile, `slots` query heads of one KV group):
//   warps 0-3 / 4-7  row threads of slot 0 / 1 (thread t owns row t = TMEM lane t)
//   warp 8           TMA producer (Q once, then kbar hi/lo tiles, 2-stage ring)
//   warp 9           MMA issuer and TMEM owner (slot s, buffer u: columns 256s + 128u); the
//                    whole warp runs the issue loop, one elected lane issues
#include <math.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace pf {
namespace {

constexpr int XST = 2;                          // kbar tile ring stages
constexpr uint32_t X_Q = 0;                     // slot s: +32 KB * s
constexpr uint32_t X_K = 65536;                 // stage st: hi at +64 KB * st, lo at +32 KB
constexpr uint32_t X_BAR = X_K + XST * 65536;   // barriers, TMEM address, abort flag
constexpr uint32_t X_UNI = X_BAR + 256;         // per-slot union bitmaps, 64 words each
constexpr uint32_t X_BYTES = X_UNI + 2 * 256 + 16;
constexpr uint32_t X_ALLOC = X_BYTES + 1024;
constexpr int kIndexThreads = 320;
constexpr int kMaxWords = 64;

enum {
  I_Q = 0,
  I_QE = 1,            // the unit's MMAs are done reading its Q tile (the next one may load)
  I_KF = 2,            // hi/lo tile landed, per stage
  I_KE = I_KF + XST,   // stage free (both slots' MMAs on it done)
  I_SF = I_KE + XST,   // score buffer full, per (slot, buffer)
  I_SE = I_SF + 4,     // score buffer drained by the row threads, per (slot, buffer)
  I_DR = I_SE + 4,
  I_N = I_DR + 1
};
enum { R_PROD = 1, R_MMA = 2, R_ROW = 3 };

// Bits of word w (blocks 32w .. 32w + 31) for the blocks lo <= b < hi.
__device__ __forceinline__ uint32_t range_bits(int w, int lo, int hi) {
  const int a0 = max(lo - 32 * w, 0), a1 = min(hi - 32 * w, 32);
  if (a1 <= a0) return 0u;
  const uint32_t below_a1 = (a1 == 32) ? 0xFFFFFFFFu : ((1u << a1) - 1u);
  return below_a1 & ~((1u << a0) - 1u);
}

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, long long timeout,
                                         volatile int* abort_flag, unsigned* status,
                                         unsigned where) {
  bool ok = mbar_wait(bar, parity, timeout, abort_flag, status, where);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long timeout,
                                           unsigned* status) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > timeout) {
      record_error(status, ST_TIMEOUT, 0xFEu);
      return;
    }
  }
}

// WIDE: head dim 256 -- pooled tiles of 64 blocks (hi and lo tiles keep the 32 KB size), one
// query head per CTA (its 64 KB query tile fills both slots' room).
// One unit = (batch, 128-row query tile, `slots` query heads of one KV group).  The grid holds at
// most one CTA per SM and each CTA runs units blockIdx.x, blockIdx.x + gridDim.x, ... (heaviest
// first): tensor memory and barriers are set up once, the pooled-tile ring and the score buffers
// keep their phases from unit to unit, and the next unit's Q tile is loaded as soon as the
// previous unit's last MMA has read Q (I_QE), while its rows are still being thresholded.
struct IndexUnit {
  int b, h0, g, qt, q0, ob, np, nsteps, msteps;
  bool reuse;  // np <= 2: pass 1's scores stay in the two score buffers for pass 2
};

template <int PT>
__device__ __forceinline__ IndexUnit index_unit(const IndexArgs& a, int u) {
  IndexUnit x;
  const int per_qt = a.n_hp * a.B;
  x.qt = a.n_qt - 1 - u / per_qt;
  const int rem = u % per_qt;
  x.b = rem / a.n_hp;
  x.h0 = (rem % a.n_hp) * a.slots;
  x.g = x.h0 / a.G;
  x.q0 = x.qt * kTile;
  x.ob = (a.s + x.q0) / kTile;        // diagonal block; candidates 0 .. ob-1
  x.np = (x.ob + PT - 1) / PT;        // pooled tiles holding the candidates
  x.nsteps = 2 * x.np;                // row steps: pass 1 and pass 2
  // With at most two pooled tiles the slot's two score buffers hold every score of the row, so
  // pass 2 reads pass 1's scores again instead of recomputing them: np MMA steps, not 2 np.
  x.reuse = x.np <= 2;
  x.msteps = x.reuse ? x.np : x.nsteps;
  return x;
}

// One slot's scores for one pooled tile, issued by the whole warp (the elected lane issues):
// KQ = d / 16 k-steps of Q . kbar_hi, then KQ of Q . kbar_lo into the same accumulator.  The k-step
// count is a compile-time constant so that the issue runs as straight-line code.
template <int KQ, uint32_t PBOXT>
__device__ __forceinline__ void issue_hi_lo_w(uint32_t d_tmem, uint64_t aq, uint64_t bh, uint64_t bl,
                                              uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < KQ; ++kk) {
    const uint32_t offa = (16384u * (kk >> 2) + 32u * (kk & 3)) >> 4;
    const uint32_t offb = (PBOXT * (kk >> 2) + 32u * (kk & 3)) >> 4;
    mma_ss_w(d_tmem, aq + offa, bh + offb, idesc, kk > 0 ? 1u : 0u);
  }
#pragma unroll
  for (int kk = 0; kk < KQ; ++kk) {
    const uint32_t offa = (16384u * (kk >> 2) + 32u * (kk & 3)) >> 4;
    const uint32_t offb = (PBOXT * (kk >> 2) + 32u * (kk & 3)) >> 4;
    mma_ss_w(d_tmem, aq + offa, bl + offb, idesc, 1u);
  }
}

// WIDE: head dim 256 -- pooled tiles of 64 blocks (hi and lo tiles keep the 32 KB size), one
// query head per CTA (its 64 KB query tile fills both slots' room).
template <bool WIDE>
__global__ void __launch_bounds__(kIndexThreads, 1)
    index_tc_kernel(const __grid_constant__ IndexMaps maps, const IndexArgs a) {
  constexpr int PT = WIDE ? 64 : 128;     // pooled blocks per pooled tile (score columns)
  constexpr uint32_t PBOX = PT * 128u;    // bytes of one 64-column box of a pooled tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = sb + X_BAR;
#define XB(i) (bar0 + 8u * (uint32_t)(i))
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + X_BAR + 8 * I_N);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + X_BAR + 8 * I_N + 4);
  uint32_t* uni = reinterpret_cast<uint32_t*>(smem + X_UNI);  // [slot][64]
  const int n_units = a.n_qt * a.n_hp * a.B;

  if (threadIdx.x == 0) {
    mbar_init(XB(I_Q), 1);
    mbar_init(XB(I_QE), 1);
    for (int st = 0; st < XST; ++st) {
      mbar_init(XB(I_KF + st), 1);
      mbar_init(XB(I_KE + st), 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(XB(I_SF + i), 1);
      mbar_init(XB(I_SE + i), 4);
    }
    mbar_init(XB(I_DR), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 2 * kMaxWords; i += blockDim.x) uni[i] = 0u;
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const int nd = a.d / 64;
      const uint32_t box = 16384u;  // a query box: 128 rows x 64 columns
      int last[XST] = {-1, -1};
      int qloads = 0, last_q = -1;  // Q tiles loaded so far (units with candidates)
      long long tg = 0;             // ring steps so far, over all units
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const IndexUnit x = index_unit<PT>(a, u);
        if (x.nsteps == 0) continue;  // no candidate: nothing to score
        // the previous unit's MMAs must be done reading Q before it is overwritten
        if (qloads > 0 && !(ok = mbar_wait(XB(I_QE), (uint32_t)(qloads - 1) & 1u, a.timeout, abort_flag,
                                            a.status, (R_PROD << 8) | I_QE)))
          break;
        mbar_arrive_expect_tx(XB(I_Q), box * nd * (uint32_t)a.slots);
        for (int sl = 0; sl < a.slots; ++sl)
          for (int c = 0; c < nd; ++c)
            tma_load_4d(sb + X_Q + 32768u * sl + box * c, &maps.q, XB(I_Q), 64 * c, x.h0 + sl, x.q0, x.b);
        last_q = qloads++;
        for (int t = 0; t < x.msteps; ++t, ++tg) {
          const int st = (int)(tg % XST), use = (int)(tg / XST);
          const int pt = t % x.np;
          if (use > 0 && !(ok = mbar_wait(XB(I_KE + st), (uint32_t)(use - 1) & 1u, a.timeout, abort_flag,
                                          a.status, (R_PROD << 8) | (I_KE + st))))
            break;
          mbar_arrive_expect_tx(XB(I_KF + st), 2u * PBOX * nd);
          for (int c = 0; c < nd; ++c) {
            tma_load_4d(sb + X_K + 65536u * st + PBOX * c, &maps.hi, XB(I_KF + st), 64 * c, pt * PT, x.g, x.b);
            tma_load_4d(sb + X_K + 65536u * st + 32768u + PBOX * c, &maps.lo, XB(I_KF + st), 64 * c,
                        pt * PT, x.g, x.b);
          }
          last[st] = use;
        }
      }
      if (*abort_flag) {
        if (last_q >= 0) drain_wait(XB(I_Q), (uint32_t)last_q & 1u, a.timeout, a.status);
        for (int st = 0; st < XST; ++st)
          if (last[st] >= 0) drain_wait(XB(I_KF + st), last[st] & 1, a.timeout, a.status);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer (whole warp)
    {
      const uint32_t idesc = make_idesc_f16((uint32_t)a.ab_type, 128, PT, 0);  // -> fp32
      const int kq = a.d / 16;
      const uint64_t dq0 = make_sdesc_sw128(sb + X_Q, 16, 1024);
      const uint64_t dk0 = make_sdesc_sw128(sb + X_K, 16, 1024);
      bool ok = true;
      int qloads = 0;
      long long tg = 0;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const IndexUnit x = index_unit<PT>(a, u);
        if (x.nsteps == 0) continue;
        ok = wait_all(XB(I_Q), (uint32_t)qloads & 1u, a.timeout, abort_flag, a.status, (R_MMA << 8) | I_Q);
        ++qloads;
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; ok && t < x.msteps; ++t, ++tg) {
          const int st = (int)(tg % XST), ub = (int)(tg % 2);
          ok = wait_all(XB(I_KF + st), (uint32_t)(tg / XST) & 1u, a.timeout, abort_flag, a.status,
                        (R_MMA << 8) | (I_KF + st));
          if (!ok) break;
          for (int sl = 0; sl < a.slots; ++sl) {
            if (tg >= 2) {
              ok = wait_all(XB(I_SE + 2 * sl + ub), (uint32_t)(tg / 2 - 1) & 1u, a.timeout, abort_flag,
                            a.status, (R_MMA << 8) | (I_SE + 2 * sl + ub));
              if (!ok) break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + 256u * sl + 128u * ub;
            const uint64_t aq = dq0 + ((32768u * sl) >> 4);
            const uint64_t bh = dk0 + ((65536u * st) >> 4);
            const uint64_t bl = dk0 + ((65536u * st + 32768u) >> 4);
            if constexpr (WIDE) issue_hi_lo_w<16, PBOX>(d_tmem, aq, bh, bl, idesc);
            else if (kq == 8) issue_hi_lo_w<8, PBOX>(d_tmem, aq, bh, bl, idesc);
            else issue_hi_lo_w<4, PBOX>(d_tmem, aq, bh, bl, idesc);
            tc_commit_w(XB(I_SF + 2 * sl + ub));
          }
          if (!ok) break;
          tc_commit_w(XB(I_KE + st));
        }
        if (ok) tc_commit_w(XB(I_QE));  // this unit's MMAs are the last to read its Q
      }
      tc_commit_w(XB(I_DR));
      if (lane == 0) drain_wait(XB(I_DR), 0, a.timeout, a.status);
    }
    __syncwarp();
  } else if ((warp >> 2) < a.slots) {
    // ---------------------------------------------------------------- row threads
    const int sl = warp >> 2, quad = warp & 3;
    const int r = quad * 32 + lane;
    uint32_t* un = uni + kMaxWords * sl;
    const float thr_off = a.log_alpha / a.scale;  // -inf for alpha == 0: every candidate kept
    bool ok = true;
    long long tg = 0;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const IndexUnit x = index_unit<PT>(a, u);
      const int h = x.h0 + sl;
      const int row = x.q0 + r;
      const bool valid = row < a.C;
      uint32_t* bits = a.row_bits + ((long long)(x.b * a.Hq + h) * a.C + (valid ? row : 0)) * a.words;
      const int ob = x.ob, np = x.np;
      const int dword = ob >> 5;
      const uint32_t dbit = 1u << (ob & 31);
      float smax = -INFINITY;
      const bool tail_row = a.s + row >= a.tail_from;  // dense-tail rule: keep every candidate
      const long long tg0 = tg;  // this unit's first MMA step
      for (int t = 0; t < x.nsteps; ++t) {
        const int pass = t / np, pt = t % np;
        // the MMA step whose scores this row step reads: step t, or with reuse the pass-1 step
        // of the same pooled tile
        const long long m = x.reuse ? tg0 + pt : tg0 + t;
        const int ub = (int)(m % 2);
        const bool fresh = !x.reuse || pass == 0;  // scores not read yet: wait for the MMAs
        if (fresh) {
          ok = wait_all(XB(I_SF + 2 * sl + ub), (uint32_t)(m / 2) & 1u, a.timeout, abort_flag, a.status,
                        (R_ROW << 8) | (I_SF + 2 * sl + ub));
          if (!ok) break;
          tc_fence_after();
        }
        uint32_t xr[PT];
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + 256u * sl + 128u * ub;
        if constexpr (PT == 128) tmem_ld128_wait(taddr, xr);
        else tmem_ld64_wait(taddr, xr);
        tc_fence_before();
        __syncwarp();
        // the buffer is free once its last reader has loaded it (with reuse: in pass 2); one
        // release per MMA step either way
        if (lane == 0 && (!x.reuse || pass == 1)) mbar_arrive(XB(I_SE + 2 * sl + ub));
        const int lim = ob - pt * PT;  // columns c < lim are candidates
        if (pass == 0) {
          if (lim >= PT) {  // every column a candidate (all but a row's last pooled tile)
#pragma unroll
            for (int c = 0; c < PT; ++c) smax = fmaxf(smax, __uint_as_float(xr[c]));
          } else {
#pragma unroll
            for (int c = 0; c < PT; ++c)
              if (c < lim) smax = fmaxf(smax, __uint_as_float(xr[c]));
          }
        } else {
          // exp((s - smax) * scale) >= alpha  <=>  s >= smax + ln(alpha) / scale  (scale > 0): one
          // compare per column; the two roundings differ by about 1e-6 relative in the ratio, far
          // inside the 1e-4 band around alpha that the float64 definition leaves undecided
          const float thr = smax + thr_off;
#pragma unroll
          for (int q = 0; q < PT / 32; ++q) {
            uint32_t word = 0u;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (__uint_as_float(xr[32 * q + i]) >= thr) word |= 1u << i;
            word &= range_bits(pt * (PT / 32) + q, 0, ob);  // columns past the candidates
            const int w = pt * (PT / 32) + q;
            // keep rules on this word's candidates (blocks below ob): sinks, the local
            // window, the dense tail; then the 32-row query tile's union (a warp's rows are
            // one aligned 32-position tile)
            const uint32_t rule = tail_row ? 0xFFFFFFFFu
                                           : (range_bits(w, 0, a.sink_blocks) |
                                              range_bits(w, ob - a.local_blocks, ob));
            word |= rule & range_bits(w, 0, ob);
            if (a.row_group32) word = __reduce_or_sync(0xffffffffu, valid ? word : 0u);
            if (w == dword) word |= dbit;
            if (w < a.words) {
              if (valid) bits[w] = word;
              const uint32_t uw = __reduce_or_sync(0xffffffffu, valid ? word : 0u);
              if (lane == 0 && uw) atomicOr(&un[w], uw);
            }
          }
        }
      }
      tg = tg0 + x.msteps;
      if (ok) {
        // words past the pooled tiles: only the diagonal bit
        for (int w = (PT / 32) * np; w < a.words; ++w) {
          const uint32_t word = (w == dword) ? dbit : 0u;
          if (valid) bits[w] = word;
        }
        if (r == 0) atomicOr(&un[dword], dbit);
      }
      // the slot's four row warps finish their unions before warp 0 of the slot compacts, and
      // the compaction has read the union before it is cleared for the next unit; a bounded
      // wait that gave up in any of them ends the unit loop for all four alike
      if (!named_bar_and(1u + (uint32_t)sl, 128u, ok)) break;
      if (quad == 0) {
        const long long tl = (long long)(x.b * a.Hq + h) * a.n_qt + x.qt;
        int32_t* list = a.tile_list + tl * a.nblk;
        int base = 0;
        for (int w0 = 0; w0 < a.words; w0 += 32) {
          const int w = w0 + lane;
          const uint32_t bw = (w < a.words) ? un[w] : 0u;
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
        if (lane == 0) a.tile_cnt[tl] = base;
      }
      asm volatile("bar.sync %0, 128;" ::"r"(1 + sl) : "memory");
      for (int w = r; w < kMaxWords; w += 128) un[w] = 0u;
      asm volatile("bar.sync %0, 128;" ::"r"(1 + sl) : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
#undef XB
}

}  // namespace

// One CTA per (query tile, batch x KV head): each (row, word) element of the tile's rows is ORed
// over the KV head's G query heads and written back to each, with consecutive threads on
// consecutive words of the row-major bits (coalesced); the tile's union is then compacted into
// every head's tile list (ascending).
__global__ void __launch_bounds__(128) share_group_kernel(const IndexArgs a) {
  __shared__ uint32_t un[kMaxWords];
  const int qt = blockIdx.x;
  const int b = blockIdx.y / a.Hkv, g = blockIdx.y % a.Hkv;
  const int r = threadIdx.x, lane = r & 31;
  for (int w = r; w < kMaxWords; w += blockDim.x) un[w] = 0u;
  __syncthreads();
  const int rows = min(kTile, a.C - qt * kTile);
  const int n = rows * a.words;
  const long long head = (long long)a.C * a.words;  // one query head's bits
  const uint32_t* src = a.row_bits + (long long)(b * a.Hq + g * a.G) * head + (long long)qt * kTile * a.words;
  uint32_t* dst = a.row_bits + (long long)(b * a.Hq + g * a.G) * head + (long long)qt * kTile * a.words;
  for (int e = r; e < n; e += blockDim.x) {
    uint32_t acc = 0u;
    for (int j = 0; j < a.G; ++j) acc |= src[j * head + e];
    for (int j = 0; j < a.G; ++j) dst[j * head + e] = acc;
    if (acc != 0u) atomicOr(&un[e % a.words], acc);
  }
  __syncthreads();
  if (r < 32) {
    int base = 0;
    for (int w0 = 0; w0 < a.words; w0 += 32) {
      const int w = w0 + lane;
      const uint32_t bw = (w < a.words) ? un[w] : 0u;
      const int cnt = __popc(bw);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      for (int j = 0; j < a.G; ++j) {
        int32_t* list = a.tile_list + ((long long)(b * a.Hq + g * a.G + j) * a.n_qt + qt) * a.nblk;
        int pos = base + incl - cnt;
        uint32_t rb = bw;
        while (rb) {
          const int i = __ffs(rb) - 1;
          rb &= rb - 1u;
          list[pos++] = w * 32 + i;
        }
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0)
      for (int j = 0; j < a.G; ++j) a.tile_cnt[(long long)(b * a.Hq + g * a.G + j) * a.n_qt + qt] = base;
  }
}

cudaError_t launch_share_group(const IndexArgs& a, cudaStream_t st) {
  share_group_kernel<<<dim3(a.n_qt, a.B * a.Hkv), 128, 0, st>>>(a);
  ++t_launches;
  return cudaGetLastError();
}

template <bool WIDE>
cudaError_t launch_index_w(const IndexMaps& maps, const IndexArgs& a, cudaStream_t st) {
  static std::atomic<int> configured[64];
  cudaError_t e =
      ensure_dynamic_smem(reinterpret_cast<const void*>(index_tc_kernel<WIDE>), X_ALLOC, configured);
  if (e != cudaSuccess) return e;
  const int units = a.n_qt * a.n_hp * a.B;
  const int grid = units < a.grid ? units : a.grid;  // at most one CTA per SM; each loops over units
  index_tc_kernel<WIDE><<<grid, kIndexThreads, X_ALLOC, st>>>(maps, a);
  ++t_launches;
  return cudaGetLastError();
}

cudaError_t launch_index(const IndexMaps& maps, const IndexArgs& a, cudaStream_t st) {
  return a.d == 256 ? launch_index_w<true>(maps, a, st) : launch_index_w<false>(maps, a, st);
}

}  // namespace pf
