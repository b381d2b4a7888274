// Prefill attention forward for sm_103a: TMA-staged Q/K/V tiles, tcgen05 MMAs
// accumulating S = Q K^T and O += P V in tensor memory, exp2 online softmax.
//
// Method: "Flash attention on ANE: fast long-context prefill", section "Flash
// attention: the core insight" (tile Q and K/V, keep a running max and sum,
// accumulate weighted V, never materialise the score matrix); the chunk +
// history + additive-mask contract of "ANE Prefill Research", section "How the
// ANE prefill path works"; and for MODE_SPARSE the kept-block walk plus pooled
// correction of "Porting FlashPrefill V2 to Apple silicon for faster prefill",
// section "Compute the peaks, summarize the rest".
//
// One CTA = one work unit = (batch b, query tile of 128 rows, `slots` query
// heads of the same KV group), or one part of a unit's key range when the
// dense tail split is on (the last part to finish merges the parts' partial
// results).  The slots share every K/V tile (GQA): one TMA load feeds both
// heads' MMAs.  Units run heaviest first (sparse: through a longest-first
// permutation).
//   warps 0-3  softmax for slot 0 (thread t owns query row t = TMEM lane t)
//   warps 4-7  softmax for slot 1
//   warp  8    TMA producer (Q once, then K tiles through a 2-stage ring and V
//              tiles through a 3-stage ring)
//   warp  9    tcgen05 MMA issuer and TMEM owner
//   (warps 8 and 9 run their loops with all 32 lanes, so that descriptors, coordinates and
//   barrier addresses stay warp-uniform, and one elected lane issues each copy, MMA and
//   commit: measured 7-9% faster than the same loops run by lane 0 alone)
//   warps 10-11 V converters: for bf16 inputs they rewrite each landed V tile
//              in place as fp16, so that P * V runs as an fp16 MMA (P carries
//              11 significant bits instead of bf16's 8; bf16 -> fp16 is exact
//              for |v| <= 65504 and larger values are reported as an error)
// Tensor memory (512 columns): slot s uses columns [256s, 256s+128) for S (P
// is written back over its first half as fp16 pairs) and [256s+128,
// 256s+128+d) for the fp32 O accumulator.
// MMA order per key tile j: PV(slot0, j), S(slot0, j+1), PV(slot1, j),
// S(slot1, j+1); each softmax group works on its tile while the tensor core
// runs the other slot's pair.  K and V have separate rings: a K stage is freed
// as soon as both S MMAs that read it are done, so K tile j+1 is in flight
// while tile j's softmax runs.  The epilogue stages O / l in the freed Q and K
// stages and writes it with TMA tile stores (optionally also the row's
// log-sum-exp).
// Explicit masks: MODE_MASK reads the additive values; MODE_MASKB reads the bits of a binary
// mask packed by mask_pack_kernel and visits only the key tiles that some row of the query
// tile keeps (the key-tile bitmap walked like the sparse union).
// Values computed before the warp-role split reach the roles through shared
// memory or are recomputed: the producer warpgroup's setmaxnreg.dec may drop
// registers above its new limit.
#include <cuda_fp16.h>
#include <math.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace pf {
namespace {

constexpr int NSK = 2;                               // K ring stages
constexpr int NSV = 3;                               // V ring stages (V also waits for conversion)
constexpr int NTD = 4;                               // issue-iteration barriers (B_TD ring)
// Issue iteration k (k >= 1) issues PV(k-1) and QK(k); the iteration before the loop issues QK(0)
// as k = 0.  Its one commit, to B_TD + k % NTD, frees the K stage of tile k + 2 (QK(k) read it)
// and the V stage of tile k + 2 (PV(k-1) read it: stage (k + 2) mod 3 = (k - 1) mod 3), so the
// producer waits on that barrier before loading tile k + 2.
constexpr uint32_t SM_Q = 0;                         // slot s: +32 KB * s (two 64-column boxes)
constexpr uint32_t SM_K = 65536;                     // stage st: +32 KB * st
constexpr uint32_t SM_V = SM_K + NSK * 32768;
constexpr uint32_t SM_BAR = SM_V + NSV * 32768;      // mbarriers, TMEM address, abort flag
constexpr int kMaxBlocks = 2048;                     // sparse: key blocks per sequence (256K keys)
constexpr uint32_t SM_BM = SM_BAR + 256;             // sparse: union bitmap of kept key blocks
constexpr uint32_t SM_BYTES = SM_BM + kMaxBlocks / 8 + 16;
constexpr uint32_t SM_ALLOC = SM_BYTES + 1024;       // slack for 1024-byte alignment

enum {
  B_Q = 0,
  B_KF = 1,             // K tile landed, per K stage
  B_VF = B_KF + NSK,    // V tile landed, per V stage
  B_VC = B_VF + NSV,    // V tile converted to fp16 (bf16 inputs), per V stage
  B_TD = B_VC + NSV,    // issue iteration k's MMAs done (frees a K and a V stage), ring of NTD
  B_SF = B_TD + NTD,    // S ready, per slot
  B_PF = B_SF + 2,      // P written (and O rescaled), per slot
  B_OF = B_PF + 2,      // last PV done
  B_DR = B_OF + 1,      // drain: all issued MMAs done
  N_BARS = B_DR + 1
};

constexpr float kLog2e = 1.4426950408889634f;
// Lazy rescale: a row keeps its stale running max while the new tile's max
// exceeds it by at most 8 (log2 units), so P <= 256; the final O / l uses the
// same max for numerator and denominator, so the result is unchanged.
constexpr float kRescaleThreshold = 8.0f;

constexpr int kConvWarps = 2;  // warps 10..11

// where-codes recorded with a timeout: (role << 8) | barrier
enum { R_PROD = 1, R_MMA = 2, R_SOFT = 3, R_CONV = 4 };

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, long long timeout,
                                         volatile int* abort_flag, unsigned* status,
                                         unsigned where) {
  bool ok = mbar_wait(bar, parity, timeout, abort_flag, status, where);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait used only while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long timeout,
                                           unsigned* status) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > timeout) {
      record_error(status, ST_TIMEOUT, 0xFFu);
      return;
    }
  }
}

// S = Q K^T for one slot and one key tile, issued by the whole warp (one elected lane issues):
// KQ = d / 16 k-steps (Q boxes 16 KB apart, K boxes KBOXT apart).  A compile-time k-step count
// keeps the issue on straight-line code; a runtime bound costs a compare and branch per MMA.
template <int KQ, uint32_t KBOXT>
__device__ __forceinline__ void qk_steps(uint32_t d_tmem, uint64_t aq, uint64_t bk, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < KQ; ++kk) {
    const uint32_t offa = (16384u * (kk >> 2) + 32u * (kk & 3)) >> 4;
    const uint32_t offb = (KBOXT * (kk >> 2) + 32u * (kk & 3)) >> 4;
    mma_ss_w(d_tmem, aq + offa, bk + offb, idesc, kk > 0 ? 1u : 0u);
  }
}

// Walks the set bits of the kept-block bitmap in ascending order.
struct BlockWalk {
  const uint32_t* bm;
  int w;
  uint32_t rb;
  __device__ void init(const uint32_t* bitmap) { bm = bitmap; w = 0; rb = bitmap[0]; }
  __device__ int next() {
    while (rb == 0u) rb = bm[++w];
    const int t = __ffs(rb) - 1;
    rb &= rb - 1u;
    return w * 32 + t;
  }
  // passes over the first n set bits; the bitmap must hold more than n
  __device__ void skip(int n) {
    while (n >= __popc(rb)) {
      n -= __popc(rb);
      rb = bm[++w];
    }
    for (; n > 0; --n) rb &= rb - 1u;
  }
};

// Key tiles in order from a bitmap of 128-key blocks: each set bit gives `tpb` consecutive
// tiles of 128 / tpb keys (tpb = 1 or 2).
template <int TPB>
struct TileWalk {
  BlockWalk walk;
  int cur, half;
  // starts at the j0-th tile of the walk
  __device__ void init(const uint32_t* bitmap, int j0) {
    walk.init(bitmap);
    walk.skip(j0 / TPB);
    half = j0 % TPB;
    cur = half ? walk.next() : 0;
  }
  __device__ int next() {
    if (half == 0) cur = walk.next();
    const int kt = cur * TPB + half;
    half = (half + 1 == TPB) ? 0 : half + 1;
    return kt;
  }
};

// One row's scores of a key tile from tensor memory (KT = 128 or 64 columns).
template <int KT>
__device__ __forceinline__ void ld_row(uint32_t taddr, float (&x)[KT]) {
  uint32_t r[KT];
  if constexpr (KT == 128) tmem_ld128_wait(taddr, r);
  else tmem_ld64_wait(taddr, r);
#pragma unroll
  for (int i = 0; i < KT; ++i) x[i] = __uint_as_float(r[i]);
}

// 32 consecutive output values of one row, already divided by l, in the output type.
__device__ __forceinline__ void store_out32(const AttnArgs& a, long long off, const float (&v)[32]) {
  if (a.out_dtype == 2) {
    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + off);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = (a.out_dtype == 1) ? pack_bf16(v[8 * i + 2 * e], v[8 * i + 2 * e + 1])
                                  : pack_f16(v[8 * i + 2 * e], v[8 * i + 2 * e + 1]);
      dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// WIDE: head_dim 256.  Key tiles are 64 keys (a 128-key block is two tiles), pooled tiles 64
// pooled blocks, one query head per CTA; the Q tile (64 KB) and the K / V rings keep their sizes,
// and O (256 fp32 columns) sits at tensor-memory column 256.
template <int MODE, bool WIDE>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_kernel(const __grid_constant__ AttnMaps maps, const AttnArgs a) {
  constexpr int KT = WIDE ? 64 : 128;          // keys per key tile (S columns)
  constexpr int TPB = kTile / KT;              // key tiles per 128-key block
  constexpr int PT = WIDE ? 64 : 128;          // pooled blocks per pooled tile
  constexpr uint32_t O_COL = WIDE ? 256u : 128u;  // O's first column in the slot's tensor memory
  constexpr uint32_t KBOX = KT * 128u;         // bytes of one 64-column box of a K / V tile
  // a packed explicit mask is launched as bits, then as values: the launch that does not match
  // the packing pass's decision returns before it touches anything (the whole CTA alike)
  if (MODE == MODE_MASKB && __ldg(a.mask_nonbinary) != 0) return;
  if (MODE == MODE_MASK && a.mask_nonbinary != nullptr && __ldg(a.mask_nonbinary) == 0) return;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = sb + SM_BAR;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM_BAR + 8 * N_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_BAR + 8 * N_BARS + 4);
  int* n_ex_slot = reinterpret_cast<int*>(smem + SM_BAR + 8 * N_BARS + 8);
  int* last_part = reinterpret_cast<int*>(smem + SM_BAR + 8 * N_BARS + 12);
  const uint32_t* kept_bm = reinterpret_cast<const uint32_t*>(smem + SM_BM);

  // ---- work unit: heaviest query tiles first (longest causal key range).  CTAs past
  // n_whole are the parts of the last (lightest) units, split_k consecutive CTAs per unit.
  int unit = (MODE == MODE_SPARSE && a.perm != nullptr) ? __ldg(a.perm + blockIdx.x) : (int)blockIdx.x;
  int part = 0, split = -1;
  if (unit >= a.n_whole) {
    split = (unit - a.n_whole) / a.split_k;
    part = (unit - a.n_whole) % a.split_k;
    unit = a.n_whole + split;
  }
  const int per_qt = a.n_hp * a.B;
  const int qt = a.n_qt - 1 - unit / per_qt;
  const int rem = unit % per_qt;
  const int b = rem / a.n_hp;
  const int h0 = (rem % a.n_hp) * a.slots;
  const int g = h0 / a.G;
  const int q0 = qt * kTile;
  const int ob = (a.s + q0) / kTile;  // key block holding this tile's diagonal

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_Q), 1);
    for (int st = 0; st < NSK; ++st) {
      mbar_init(BAR(B_KF + st), 1);
    }
    for (int k = 0; k < NTD; ++k) mbar_init(BAR(B_TD + k), 1);
    for (int st = 0; st < NSV; ++st) {
      mbar_init(BAR(B_VF + st), 1);
      mbar_init(BAR(B_VC + st), kConvWarps);
    }
    for (int sl = 0; sl < 2; ++sl) {
      mbar_init(BAR(B_SF + sl), 1);
      mbar_init(BAR(B_PF + sl), 4);
    }
    mbar_init(BAR(B_OF), 1);
    mbar_init(BAR(B_DR), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (MODE == MODE_SPARSE && warp == 8) {
    // Union of the slots' kept-block lists, ascending, via a bitmap.  Only earlier
    // blocks (< ob) are taken from the lists and the diagonal block ob is always set,
    // so ob is the union's last block whatever the lists hold.  The count goes through
    // shared memory: every role reads it after its setmaxnreg (a value held in a
    // register across that point may be lost).
    uint32_t* bm = reinterpret_cast<uint32_t*>(smem + SM_BM);
    const long long t0 = (long long)(b * a.Hq + h0) * a.n_qt + qt;
    const int32_t* l0 = a.tile_list + t0 * a.nblk;
    const int32_t* l1 = l0 + (long long)a.n_qt * a.nblk;
    // the counts and the first 64 entries of both lists in one round trip (every list row
    // holds nblk entries, so the reads stay in bounds; entries past a count are ignored)
    const int raw0 = a.tile_cnt[t0];
    const int raw1 = (a.slots == 2) ? a.tile_cnt[t0 + a.n_qt] : 0;
    int e0[2], e1[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = lane + 32 * u;
      e0[u] = i < a.nblk ? l0[i] : -1;
      e1[u] = (a.slots == 2 && i < a.nblk) ? l1[i] : -1;
    }
    const int c0 = min(max(raw0, 0), a.nblk);
    const int c1 = min(max(raw1, 0), a.nblk);
    for (int w = lane; w < a.words; w += 32) bm[w] = 0u;
    __syncwarp();
    if (lane == 0) atomicOr(&bm[ob >> 5], 1u << (ob & 31));
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = lane + 32 * u;
      if (i < c0 && e0[u] >= 0 && e0[u] < ob) atomicOr(&bm[e0[u] >> 5], 1u << (e0[u] & 31));
      if (i < c1 && e1[u] >= 0 && e1[u] < ob) atomicOr(&bm[e1[u] >> 5], 1u << (e1[u] & 31));
    }
    for (int i = 64 + lane; i < c0; i += 32) {
      const int kb = l0[i];
      if (kb >= 0 && kb < ob) atomicOr(&bm[kb >> 5], 1u << (kb & 31));
    }
    for (int i = 64 + lane; i < c1; i += 32) {
      const int kb = l1[i];
      if (kb >= 0 && kb < ob) atomicOr(&bm[kb >> 5], 1u << (kb & 31));
    }
    __syncwarp();
    int cnt = 0;
    for (int w = lane; w < a.words; w += 32) cnt += __popc(bm[w]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    const int base = cnt;
    if (lane == 0) *n_ex_slot = base;
  }
  if (MODE == MODE_MASKB && warp == 8) {
    // A binary mask visits only the key tiles that some row of this query tile keeps (the
    // others add exactly nothing); -1 in the slot means every key tile.
    int cnt = -1;
    if (a.mask_tiles != nullptr) {
      uint32_t* bm = reinterpret_cast<uint32_t*>(smem + SM_BM);
      const uint32_t* src = a.mask_tiles + (long long)qt * a.mask_tile_words;
      cnt = 0;
      for (int w = lane; w < a.mask_tile_words; w += 32) {
        const uint32_t v = __ldg(src + w);
        bm[w] = v;
        cnt += __popc(v);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    }
    if (lane == 0) *n_ex_slot = cnt;
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int n_pool = 0, n_tiles;
  if (MODE == MODE_CAUSAL) {
    n_tiles = (ob + 1) * TPB;
  } else if (MODE == MODE_MASK) {
    n_tiles = (a.T + KT - 1) / KT;
  } else if (MODE == MODE_MASKB) {
    n_tiles = *n_ex_slot >= 0 ? *n_ex_slot * TPB : (a.T + KT - 1) / KT;
  } else {
    n_pool = (ob + PT - 1) / PT;
    n_tiles = n_pool + *n_ex_slot * TPB;
  }
  const int n_total = n_tiles;  // the unit's key tiles (a split part runs a range of them)
  // a split unit's part covers key tiles [j0, j0 + n_tiles); loops below count locally from 0
  int j0 = 0;
  const bool has_last_tile = split < 0 || part == a.split_k - 1;
  if (split >= 0) {
    j0 = part * n_tiles / a.split_k;
    n_tiles = (part + 1) * n_tiles / a.split_k - j0;
  }

  // 384 threads x 168 registers at launch; the softmax warpgroups take 216,
  // the producer/MMA/converter warpgroup keeps 72: 2*128*216 + 128*72 = 384*168.
  if (warp >= 8) {
    regs_dec<72>();
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    {  // the whole warp walks the tiles; the elected lane issues the copies
      const int nd = a.d / 64;
      const uint32_t tile_bytes = (uint32_t)nd * KBOX;  // one K or V tile: nd boxes of KT rows
      if (lane == 0) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.kh);
        tma_prefetch_desc(&maps.vh);
      }
      mbar_arrive_expect_tx_w(BAR(B_Q), (uint32_t)nd * 16384u * (uint32_t)a.slots);
      for (int sl = 0; sl < a.slots; ++sl)
        for (int c = 0; c < nd; ++c)
          tma_load_4d_w(sb + SM_Q + 32768u * sl + 16384u * c, &maps.q, BAR(B_Q), 64 * c, h0 + sl,
                        q0, b);
      int last_k[NSK], last_v[NSV];
      for (int st = 0; st < NSK; ++st) last_k[st] = -1;
      for (int st = 0; st < NSV; ++st) last_v[st] = -1;
      // key tiles come from the kept-block bitmap (sparse, binary masks) or in order
      const bool walked = MODE == MODE_SPARSE || (MODE == MODE_MASKB && *n_ex_slot >= 0);
      TileWalk<TPB> walk;
      if (walked) walk.init(kept_bm, MODE == MODE_MASKB ? j0 : 0);  // sparse units never split
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % NSK, use = j / NSK;
        const int sv = j % NSV, usev = j / NSV;
        const CUtensorMap *mk, *mv;
        int c1, c2;
        if (MODE == MODE_SPARSE && j < n_pool) {
          mk = &maps.kbar;  // pooled keys [B, Hkv, nblk, d]: rows = pooled blocks
          mv = &maps.vbar;
          c1 = j * PT;
          c2 = g;
        } else {
          const int kt = walked ? walk.next() : j0 + j;
          if (kt < a.n_hist_tiles) {
            mk = &maps.kh;
            mv = &maps.vh;
            c2 = kt * KT;
          } else {
            mk = &maps.kc;
            mv = &maps.vc;
            c2 = kt * KT - a.s;
          }
          c1 = g;
        }
        // tile j reuses the K stage of tile j - 2 and the V stage of tile j - 3: both freed by
        // issue iteration j - 2 (B_TD + (j - 2) % NTD, its ((j - 2) / NTD)-th phase; the next
        // phase of that barrier needs tile j + 2 loaded first, so it cannot be ahead)
        const int td = (j - 2) % NTD;
        if (j >= 2 && !wait_all(BAR(B_TD + td), (uint32_t)((j - 2) / NTD) & 1u, a.timeout, abort_flag, a.status,
                                (R_PROD << 8) | (B_TD + td)))
          break;
        mbar_arrive_expect_tx_w(BAR(B_KF + st), tile_bytes);
        for (int c = 0; c < nd; ++c)
          tma_load_4d_w(sb + SM_K + 32768u * st + KBOX * c, mk, BAR(B_KF + st), 64 * c, c1, c2, b);
        last_k[st] = use;
        mbar_arrive_expect_tx_w(BAR(B_VF + sv), tile_bytes);
        for (int c = 0; c < nd; ++c)
          tma_load_4d_w(sb + SM_V + 32768u * sv + KBOX * c, mv, BAR(B_VF + sv), 64 * c, c1, c2, b);
        last_v[sv] = usev;
      }
      if (lane == 0 && *abort_flag) {  // let this warp's copies land before the CTA exits
        drain_wait(BAR(B_Q), 0, a.timeout, a.status);
        for (int st = 0; st < NSK; ++st)
          if (last_k[st] >= 0) drain_wait(BAR(B_KF + st), last_k[st] & 1, a.timeout, a.status);
        for (int st = 0; st < NSV; ++st)
          if (last_v[st] >= 0) drain_wait(BAR(B_VF + st), last_v[st] & 1, a.timeout, a.status);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    {  // the whole warp runs the issue loop; mma_*_w / tc_commit_w issue from one elected lane
      const uint32_t idesc_qk = make_idesc_f16((uint32_t)a.ab_type, 128, KT, 0);
      const uint32_t idesc_pv = make_idesc_f16(0u, 128, (uint32_t)a.d, 1);  // fp16 P x fp16 V
      const int kq = a.d / 16;
      // descriptors are built once; a k-step only advances the start-address field.  Q boxes
      // (128 rows x 64 columns) are 16 KB apart, K / V boxes (KT rows) KBOX apart.
      const uint64_t dq0 = make_sdesc_sw128(sb + SM_Q, 16, 1024);
      const uint64_t dk0 = make_sdesc_sw128(sb + SM_K, 16, 1024);
      const uint64_t dv0 = make_sdesc_sw128(sb + SM_V, KBOX, 1024);
      auto issue_qk = [&](int sl, int st) {
        const uint32_t d_tmem = tmem + 256u * sl;
        const uint64_t aq = dq0 + ((32768u * sl) >> 4);
        const uint64_t bk = dk0 + ((32768u * st) >> 4);
        if constexpr (WIDE) qk_steps<16, KBOX>(d_tmem, aq, bk, idesc_qk);
        else if (kq == 8) qk_steps<8, KBOX>(d_tmem, aq, bk, idesc_qk);
        else qk_steps<4, KBOX>(d_tmem, aq, bk, idesc_qk);
      };
      auto issue_pv = [&](int sl, int st, bool acc) {
        const uint32_t d_tmem = tmem + 256u * sl + O_COL;
        const uint64_t bv = dv0 + ((32768u * st) >> 4);
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk)
          mma_ts_w(d_tmem, tmem + 256u * sl + 8u * kk, bv + ((2048u * kk) >> 4), idesc_pv,
                   (acc || kk > 0) ? 1u : 0u);
      };
      const int vbar_first = a.convert_v ? B_VC : B_VF;
      bool ok = wait_all(BAR(B_Q), 0, a.timeout, abort_flag, a.status, (R_MMA << 8) | B_Q);
      tc_fence_after();
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j % NSK;
        const uint32_t ph = (uint32_t)(j / NSK) & 1u;
        const int sv = j % NSV;
        const uint32_t phv = (uint32_t)(j / NSV) & 1u;
        if (j == 0) {
          ok = wait_all(BAR(B_KF + st), ph, a.timeout, abort_flag, a.status, (R_MMA << 8) | (B_KF + st));
          if (!ok) break;
          tc_fence_after();
          for (int sl = 0; sl < a.slots; ++sl) {
            issue_qk(sl, st);
            if (!a.withhold) tc_commit_w(BAR(B_SF + sl));
          }
          tc_commit_w(BAR(B_TD));  // issue iteration 0: QK(0)
        }
        ok = wait_all(BAR(vbar_first + sv), phv, a.timeout, abort_flag, a.status,
                      (R_MMA << 8) | (vbar_first + sv));
        if (!ok) break;
        tc_fence_after();
        const int st1 = (j + 1) % NSK;
        for (int sl = 0; sl < a.slots; ++sl) {
          ok = wait_all(BAR(B_PF + sl), (uint32_t)j & 1u, a.timeout, abort_flag, a.status,
                        (R_MMA << 8) | (B_PF + sl));
          if (!ok) break;
          tc_fence_after();
          issue_pv(sl, sv, j > 0);
          if (j + 1 < n_tiles) {
            if (sl == 0) {
              ok = wait_all(BAR(B_KF + st1), (uint32_t)((j + 1) / NSK) & 1u, a.timeout,
                            abort_flag, a.status, (R_MMA << 8) | (B_KF + st1));
              if (!ok) break;
              tc_fence_after();
            }
            issue_qk(sl, st1);
            tc_commit_w(BAR(B_SF + sl));
          }
        }
        if (!ok) break;
        tc_commit_w(BAR(B_TD + (j + 1) % NTD));  // issue iteration j + 1: PV(j), QK(j + 1)
      }
      if (ok) tc_commit_w(BAR(B_OF));
      tc_commit_w(BAR(B_DR));  // no MMA may still run when tensor memory is released
      if (lane == 0) drain_wait(BAR(B_DR), 0, a.timeout, a.status);
    }
    __syncwarp();
  } else if (warp >= 10 && a.convert_v) {
    // ------------------------------------------------------------ V converters
    const int ct = threadIdx.x - 320;  // 0 .. 32*kConvWarps-1
    const int nvec = KT * a.d / 8;       // 16-byte vectors per V tile
    float vmax = 0.f;                    // largest |v| seen (bf16 values are exact in fp32)
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % NSV;
      if (!wait_all(BAR(B_VF + st), (uint32_t)(j / NSV) & 1u, a.timeout, abort_flag, a.status,
                    (R_CONV << 8) | (B_VF + st)))
        break;
      uint4* v = reinterpret_cast<uint4*>(smem + SM_V + 32768u * st);
#pragma unroll 2
      for (int i = ct; i < nvec; i += 32 * kConvWarps) {
        uint4 w = v[i];
        uint32_t* ww = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(ww[e] << 16), hi = __uint_as_float(ww[e] & 0xFFFF0000u);
          vmax = max_nan(vmax, max_nan(fabsf(lo), fabsf(hi)));
          ww[e] = pack_f16(lo, hi);
        }
        v[i] = w;
      }
      fence_proxy_async();  // generic-proxy writes -> visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_VC + st));
    }
    // fp16 holds |v| <= 65504; anything larger (or inf / nan, which fails the test) is an error
    const bool bad = !(vmax <= 65504.f);
    if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(a.status, ST_VRANGE, R_CONV << 8);
  }
  } else {
    regs_inc<216>();
  if ((warp >> 2) < a.slots) {
    // ------------------------------------------------------------ softmax
    const int sl = warp >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t t_s = tmem + ((uint32_t)(quad * 32) << 16) + 256u * sl;
    const uint32_t t_o = t_s + O_COL;
    const int h = h0 + sl;
    const int row = q0 + r;
    const bool valid = row < a.C;
    const uint32_t* bits_row = nullptr;
    if (MODE == MODE_SPARSE && valid)
      bits_row = a.row_bits + ((long long)(b * a.Hq + h) * a.C + row) * a.words;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // MODE_MASKB: the tile's mask bits, one 16-byte word group per row and 128-key group (bit L of
    // word c = key 4L + c), loaded before the step's score wait (padding rows read none and mask
    // nothing).  In registers, key 4L + c of a KT-key tile is bit (c * KT / 4 + L) of the tile's
    // KT / 32 words: a 64-key tile takes its 16-bit half of each of its group's four words.
    // Loading a step ahead instead holds four more registers across the loop and spills: slower.
    const uint32_t* mbits = nullptr;
    if (MODE == MODE_MASKB && valid) mbits = a.mask_bits + (long long)row * a.mask_words;
    const bool mwalk = MODE == MODE_MASKB && *n_ex_slot >= 0;
    TileWalk<TPB> walk;
    if (MODE == MODE_SPARSE || mwalk) walk.init(kept_bm, mwalk ? j0 : 0);
    for (int j = 0; j < n_tiles; ++j) {
      uint32_t wq[KT / 32];
#pragma unroll
      for (int q = 0; q < KT / 32; ++q) wq[q] = 0xffffffffu;
      if (MODE == MODE_MASKB) {
        const int kt = mwalk ? walk.next() : j0 + j;
        if (mbits != nullptr) {
          if constexpr (KT == 128) {
            const uint4 bw = __ldg(reinterpret_cast<const uint4*>(mbits) + kt);
            wq[0] = bw.x;
            wq[1] = bw.y;
            wq[2] = bw.z;
            wq[3] = bw.w;
          } else {
            const uint4 bw = __ldg(reinterpret_cast<const uint4*>(mbits) + (kt >> 1));
            const uint32_t sel = (kt & 1) ? 0x7632u : 0x5410u;  // high or low halves
            wq[0] = __byte_perm(bw.x, bw.y, sel);
            wq[1] = __byte_perm(bw.z, bw.w, sel);
          }
        }
      }
      ok = wait_all(BAR(B_SF + sl), (uint32_t)j & 1u, a.timeout, abort_flag, a.status,
                    (R_SOFT << 8) | (B_SF + sl));
      if (!ok) break;
      tc_fence_after();
      float x[KT];
      ld_row<KT>(t_s, x);
      float xs = a.scale_log2, bias = 0.f;
      bool row_skip = false;  // sparse: this row did not keep the tile's block
      if (MODE == MODE_CAUSAL) {
        // the diagonal block's tiles (its last TPB): key q0 + off + c is visible iff off + c <= r
        const int gt = j0 + j;
        if (has_last_tile && gt >= n_total - TPB) {
          const int off = (gt - (n_total - TPB)) * KT;
#pragma unroll
          for (int c = 0; c < KT; ++c)
            if (c + off > r) x[c] = -INFINITY;
        }
      } else if (MODE == MODE_MASKB) {
        // bit set = kept (value 0); dropped keys (and keys past T, whose bits are 0) are -inf;
        // a word of 32 kept keys (most words of a causal-like mask) needs no selects
#pragma unroll
        for (int q = 0; q < KT / 32; ++q)
          if (wq[q] != 0xffffffffu) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              // bit i of word q is key 4L + c with c * KT / 4 + L = 32q + i
              constexpr int kL = KT / 4;
              const int c = (32 * q + i) / kL, L = (32 * q + i) % kL;
              if (!((wq[q] >> i) & 1u)) x[4 * L + c] = -INFINITY;
            }
          }
      } else if (MODE == MODE_MASK) {
        xs = 1.f;
        const int key0 = (j0 + j) * KT;
        if (valid && a.mask_vec && key0 + KT <= a.T) {
          if (a.mask_f16) {
            const uint4* mp = reinterpret_cast<const uint4*>(
                reinterpret_cast<const __half*>(a.mask) + (long long)row * a.mask_ld + key0);
#pragma unroll
            for (int q = 0; q < KT / 32; ++q) {  // 32 columns at a time keeps the loads in registers
              uint4 w4[4];
#pragma unroll
              for (int v = 0; v < 4; ++v) w4[v] = __ldg(mp + 4 * q + v);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const uint32_t ww[4] = {w4[v].x, w4[v].y, w4[v].z, w4[v].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[e]));
                  const int c = 32 * q + 8 * v + 2 * e;
                  x[c] = fmaf(x[c], a.scale_log2, f.x * kLog2e);
                  x[c + 1] = fmaf(x[c + 1], a.scale_log2, f.y * kLog2e);
                }
              }
              asm volatile("" ::: "memory");
            }
          } else {
            const float4* mp = reinterpret_cast<const float4*>(
                reinterpret_cast<const float*>(a.mask) + (long long)row * a.mask_ld + key0);
#pragma unroll
            for (int q = 0; q < KT / 32; ++q) {
              float4 w4[8];
#pragma unroll
              for (int v = 0; v < 8; ++v) w4[v] = __ldg(mp + 8 * q + v);
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                const int c = 32 * q + 4 * v;
                x[c + 0] = fmaf(x[c + 0], a.scale_log2, w4[v].x * kLog2e);
                x[c + 1] = fmaf(x[c + 1], a.scale_log2, w4[v].y * kLog2e);
                x[c + 2] = fmaf(x[c + 2], a.scale_log2, w4[v].z * kLog2e);
                x[c + 3] = fmaf(x[c + 3], a.scale_log2, w4[v].w * kLog2e);
              }
              asm volatile("" ::: "memory");
            }
          }
        } else {  // ragged last tile, unaligned rows or a padding row: element loads
#pragma unroll
          for (int q = 0; q < KT / 32; ++q) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int c = 32 * q + i;
              const int key = key0 + c;
              float mv = 0.f;
              if (valid && key < a.T) {
                const long long o = (long long)row * a.mask_ld + key;
                mv = a.mask_f16 ? __half2float(reinterpret_cast<const __half*>(a.mask)[o])
                                : reinterpret_cast<const float*>(a.mask)[o];
              }
              x[c] = (key < a.T) ? fmaf(x[c], a.scale_log2, mv * kLog2e) : -INFINITY;
            }
            asm volatile("" ::: "memory");
          }
        }
      } else {  // MODE_SPARSE
        if (j < n_pool) {
          // pooled keys: column c is block j*PT + c; a row takes it iff the
          // block is an earlier candidate (< ob) that the row did not keep
          bias = a.log2_nb;
#pragma unroll
          for (int q = 0; q < PT / 32; ++q) {
            const int wi = j * (PT / 32) + q;
            const uint32_t w = (bits_row != nullptr && wi < a.words) ? __ldg(bits_row + wi) : 0u;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int blk = wi * 32 + i;
              if (blk >= ob || ((w >> i) & 1u)) x[32 * q + i] = -INFINITY;
            }
          }
        } else {
          const int kt = walk.next();
          const int kb = kt / TPB;
          if (kb == ob) {  // the diagonal block: key q0 + off + c is visible iff off + c <= r
            const int off = (kt % TPB) * KT;
#pragma unroll
            for (int c = 0; c < KT; ++c)
              if (c + off > r) x[c] = -INFINITY;
          } else {
            // a row that did not keep the block gets P = 0 and leaves its max alone
            // (row max and offset -inf below) instead of masking 128 scores
            row_skip = bits_row != nullptr && !((__ldg(bits_row + (kb >> 5)) >> (kb & 31)) & 1u);
          }
        }
      }
      // ---- online softmax (log2 domain)
      float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
      for (int c = 4; c < KT; c += 4) {
        mx0 = fmaxf(mx0, x[c]);
        mx1 = fmaxf(mx1, x[c + 1]);
        mx2 = fmaxf(mx2, x[c + 2]);
        mx3 = fmaxf(mx3, x[c + 3]);
      }
      const float mraw = row_skip ? -INFINITY : fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      const float mt = (mraw == -INFINITY) ? -INFINITY : fmaf(mraw, xs, bias);
      const bool need = mt > m + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float mn = fmaxf(m, mt);
        const float f = (m == -INFINITY) ? 0.f : ex2(m - mn);
        l *= f;
        if (j > 0) {
          uint32_t o[32];
          for (int c0 = 0; c0 < a.d; c0 += 32) {
            tmem_ld32(t_o + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
            tmem_st32(t_o + c0, o);
          }
        }
        m = mn;
      }
      const float off = row_skip ? -INFINITY : bias - ((m == -INFINITY) ? 0.f : m);
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int q = 0; q < KT / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float y0, y1;
          fma2(y0, y1, x[32 * q + 2 * i], x[32 * q + 2 * i + 1], xs, xs, off, off);
          const float p0 = ex2(y0), p1 = ex2(y1);
          add2(ls0, ls1, p0, p1);
          pk[i] = pack_f16(p0, p1);
        }
        tmem_st16(t_s + 16u * q, pk);
      }
      l += ls0 + ls1;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_PF + sl));
    }
    // ---- epilogue: out = O / l
    if (ok)
      ok = wait_all(BAR(B_OF), 0, a.timeout, abort_flag, a.status, (R_SOFT << 8) | B_OF);
    const long long obase = (long long)b * a.o_sb + (long long)row * a.o_st + (long long)h * a.o_sh;
    // natural log of the softmax denominator: sum_j 2^(y_j) = 2^m * l in the log2 domain
    auto write_lse = [&](float mm, float ll) {
      if (a.lse != nullptr && valid)
        a.lse[((long long)b * a.Hq + h) * a.C + row] = (mm + __log2f(ll)) * 0.6931471805599453f;
    };
    if (split < 0) {
      // Rows are staged in shared memory (the Q and K stages are free once every MMA is
      // done: slot s uses [64 KB * s, 64 KB * (s + 1))) as 128-byte boxes, 16-byte chunks
      // swizzled the way the tile store reads them, then one thread per head stores the
      // head's tile; rows at or past C are dropped by the store.
      const int es = (a.out_dtype == 2) ? 4 : 2;
      const int box_cols = 128 / es;  // 32 fp32 or 64 16-bit values per 128-byte box row
      const int nbox = a.d / box_cols;
      uint8_t* stage = smem + SM_Q + 65536u * sl;
      if (ok) {
        tc_fence_after();
        write_lse(m, l);
        const float inv = 1.f / l;
        for (int bx = 0; bx < nbox; ++bx) {
          uint32_t wv[32];
          if (es == 4) {
            uint32_t o[32];
            tmem_ld32(t_o + 32u * bx, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) wv[i] = __float_as_uint(__uint_as_float(o[i]) * inv);
          } else {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint32_t o[32];
              tmem_ld32(t_o + 64u * bx + 32u * half, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float lo = __uint_as_float(o[2 * i]) * inv, hi = __uint_as_float(o[2 * i + 1]) * inv;
                wv[16 * half + i] = (a.out_dtype == 1) ? pack_bf16(lo, hi) : pack_f16(lo, hi);
              }
            }
          }
          uint4* rowp = reinterpret_cast<uint4*>(stage + 16384u * bx + 128u * r);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            rowp[c ^ (r & 7)] = make_uint4(wv[4 * c], wv[4 * c + 1], wv[4 * c + 2], wv[4 * c + 3]);
        }
      }
      fence_proxy_async();  // generic-proxy writes -> visible to the tile store
      named_bar_sync(2u + (uint32_t)sl, 128u);
      if (r == 0 && ok) {
        const uint32_t stage_s = sb + SM_Q + 65536u * sl;
        for (int bx = 0; bx < nbox; ++bx) tma_store_4d(&maps.out, stage_s + 16384u * bx, bx * box_cols, h, q0, b);
        bulk_commit();
        bulk_wait_all();
      }
    } else {
      // A part of a split unit: O (relative to this part's running max m), m and l go to
      // the workspace, column-major so that a warp's rows are contiguous; the last part to
      // finish combines them: out = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p.
      const long long pstride = (long long)kTile * (a.d + 2);
      float* wp = a.ws_part + ((long long)(split * a.split_k + part) * 2 + sl) * pstride;
      if (ok) {
        tc_fence_after();
        for (int c0 = 0; c0 < a.d; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(t_o + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)  // a part with no key tile holds O = 0 (TMEM never written)
            wp[(long long)(c0 + i) * kTile + r] = n_tiles > 0 ? __uint_as_float(o[i]) : 0.f;
        }
        wp[(long long)a.d * kTile + r] = m;
        wp[(long long)(a.d + 1) * kTile + r] = l;
      }
      __threadfence();
      named_bar_sync(1, 128u * (uint32_t)a.slots);
      if (threadIdx.x == 0)
        *last_part = (!*abort_flag && atomicAdd(a.ws_cnt + split, 1) == a.split_k - 1) ? 1 : 0;
      named_bar_sync(1, 128u * (uint32_t)a.slots);
      if (*last_part) {
        __threadfence();
        const float* p0 = a.ws_part + ((long long)split * a.split_k * 2 + sl) * pstride;
        float M = -INFINITY;
        for (int p = 0; p < a.split_k; ++p)
          M = fmaxf(M, __ldcg(p0 + p * 2 * pstride + (long long)a.d * kTile + r));
        float wgt[kMaxSplit], L = 0.f;
#pragma unroll
        for (int p = 0; p < kMaxSplit; ++p) {
          wgt[p] = 0.f;
          if (p < a.split_k) {
            const float mp = __ldcg(p0 + p * 2 * pstride + (long long)a.d * kTile + r);
            wgt[p] = (mp == -INFINITY) ? 0.f : ex2(mp - M);
            L += wgt[p] * __ldcg(p0 + p * 2 * pstride + (long long)(a.d + 1) * kTile + r);
          }
        }
        write_lse(M, L);
        const float inv = 1.f / L;
        for (int c0 = 0; c0 < a.d; c0 += 32) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
#pragma unroll
          for (int p = 0; p < kMaxSplit; ++p) {
            if (p < a.split_k) {
              const float* op = p0 + p * 2 * pstride + (long long)c0 * kTile + r;
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = fmaf(wgt[p], __ldcg(op + (long long)i * kTile), v[i]);
            }
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= inv;
          if (valid) store_out32(a, obase + c0, v);
        }
      }
    }
  }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
#undef BAR
}

// Packed mask bits: per row, four words per 128-key tile; bit L of word c is key 4L + c of the
// tile (set = kept, value 0).  It is the layout four warp ballots give when lane L holds keys
// 4L .. 4L + 3, one ballot per c, so the packing needs no shuffles.
//
// One CTA per mask row (rows past 65535 loop): lane L loads keys 4L + c of a tile (four scalar
// loads; for rows not on 16-byte boundaries) and each warp keeps kPackTiles tiles in flight
// before their ballots (the pass reads the mask once); the row's kept count decides whether a
// fully dropped row (a plain softmax over the raw scores with values, NaN with bits) forces the
// value path; the key tiles the row keeps are ORed into its query tile's tile bitmap (when
// tiles != null).
constexpr int kPackTiles = 2;
__global__ void __launch_bounds__(256) mask_pack_kernel(const void* __restrict__ mask, int f16, int C,
                                                        int T, long long ld, uint32_t* __restrict__ bits,
                                                        int words, int* nonbinary, uint32_t* tiles,
                                                        int tile_words) {
  __shared__ int kept_any;
  __shared__ uint32_t row_tiles[64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x / 32;
  const int groups = words / 4;  // 128-key tiles per row
  for (int row = blockIdx.y; row < C; row += gridDim.y) {
    if (threadIdx.x == 0) kept_any = 0;
    for (int t = threadIdx.x; t < 64; t += blockDim.x) row_tiles[t] = 0u;
    __syncthreads();
    bool nonbin = false, any = false;
    for (int m0 = warp * kPackTiles; m0 < groups; m0 += nwarps * kPackTiles) {
      float v[kPackTiles][4];
#pragma unroll
      for (int u = 0; u < kPackTiles; ++u) {  // every load first, then the ballots
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int key = (m0 + u) * kTile + 4 * lane + c;
          v[u][c] = 0.f;
          if (m0 + u < groups && key < T) {
            const long long o = (long long)row * ld + key;
            v[u][c] = f16 ? __half2float(reinterpret_cast<const __half*>(mask)[o])
                          : reinterpret_cast<const float*>(mask)[o];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kPackTiles; ++u) {
        const int m = m0 + u;
        if (m >= groups) break;  // uniform across the warp
        uint32_t wc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const bool inb = m * kTile + 4 * lane + c < T;
          nonbin |= inb && !(v[u][c] == 0.f || v[u][c] <= -10000.f);
          wc[c] = __ballot_sync(0xffffffffu, inb && v[u][c] == 0.f);
        }
        if (lane == 0)
          *reinterpret_cast<uint4*>(bits + (long long)row * words + 4 * m) = make_uint4(wc[0], wc[1], wc[2], wc[3]);
        const bool tile_kept = (wc[0] | wc[1] | wc[2] | wc[3]) != 0u;
        any |= tile_kept;
        if (lane == 0 && tiles != nullptr && tile_kept) atomicOr(&row_tiles[m >> 5], 1u << (m & 31));
      }
    }
    if (__any_sync(0xffffffffu, any) && lane == 0) kept_any = 1;
    if (__any_sync(0xffffffffu, nonbin) && lane == 0) atomicExch(nonbinary, 1);
    __syncthreads();
    if (threadIdx.x == 0 && !kept_any) atomicExch(nonbinary, 1);
    if (tiles != nullptr)
      for (int t = threadIdx.x; t < tile_words; t += blockDim.x)
        if (row_tiles[t] != 0u) atomicOr(&tiles[(long long)(row / kTile) * tile_words + t], row_tiles[t]);
    __syncthreads();
  }
}

// The same packing for masks whose rows start on 16-byte boundaries (the common case): each lane
// reads its four keys 4L .. 4L + 3 with one streaming vector load (16 bytes of fp32, 8 of fp16),
// so a warp covers one 128-key tile per load and keeps kPackGroups tiles in flight; the four
// ballots are the tile's four words.  The pass is bound by its instructions more than by the
// mask's bytes, so a tile wholly inside the row skips the per-key bounds tests.  Bits, flags and
// tile bitmap are those of mask_pack_kernel.
constexpr int kPackGroups = 4;
// The first n (< 4) mask values from element o on, one scalar load each; the rest 0.  Kept out of
// line: inlined, its per-key branches cost the packing kernel a stack frame.
__device__ __noinline__ float4 ragged_keys(const void* mask, int f16, long long o, int n) {
  float x[3] = {0.f, 0.f, 0.f};
  for (int c = 0; c < n && c < 3; ++c)
    x[c] = f16 ? __half2float(static_cast<const __half*>(mask)[o + c]) : static_cast<const float*>(mask)[o + c];
  return make_float4(x[0], x[1], x[2], 0.f);
}
__global__ void __launch_bounds__(256) mask_pack_vec_kernel(const void* __restrict__ mask, int f16, int C,
                                                            int T, long long ld, uint32_t* __restrict__ bits,
                                                            int words, int* nonbinary, uint32_t* tiles,
                                                            int tile_words) {
  __shared__ int kept_any;
  __shared__ uint32_t row_tiles[64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x / 32;
  const int groups = words / 4;  // 128-key tiles per row (words is a multiple of 4)
  for (int row = blockIdx.y; row < C; row += gridDim.y) {
    if (threadIdx.x == 0) kept_any = 0;
    for (int t = threadIdx.x; t < 64; t += blockDim.x) row_tiles[t] = 0u;
    __syncthreads();
    bool nonbin = false, any = false;
    const long long rbase = (long long)row * ld;
    for (int m0 = warp * kPackGroups; m0 < groups; m0 += nwarps * kPackGroups) {
      float v[kPackGroups][4];
      // uniform: every key of the round's kPackGroups tiles exists (all rounds but those at a row's end)
      if ((m0 + kPackGroups) * kTile <= T) {
#pragma unroll
        for (int u = 0; u < kPackGroups; ++u) {  // every load first, then the ballots
          const long long o = rbase + (m0 + u) * kTile + 4 * lane;
          if (f16) {
            const uint2 r = __ldcs(reinterpret_cast<const uint2*>(static_cast<const __half*>(mask) + o));
            v[u][0] = __half2float(__ushort_as_half((unsigned short)(r.x & 0xFFFFu)));
            v[u][1] = __half2float(__ushort_as_half((unsigned short)(r.x >> 16)));
            v[u][2] = __half2float(__ushort_as_half((unsigned short)(r.y & 0xFFFFu)));
            v[u][3] = __half2float(__ushort_as_half((unsigned short)(r.y >> 16)));
          } else {
            const float4 r = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(mask) + o));
            v[u][0] = r.x;
            v[u][1] = r.y;
            v[u][2] = r.z;
            v[u][3] = r.w;
          }
        }
        uint32_t kept_tiles = 0u;  // bit u: tile m0 + u keeps a key
#pragma unroll
        for (int u = 0; u < kPackGroups; ++u) {
          uint32_t wc[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            nonbin |= !(v[u][c] == 0.f || v[u][c] <= -10000.f);
            wc[c] = __ballot_sync(0xffffffffu, v[u][c] == 0.f);
          }
          if (lane == 0)
            *reinterpret_cast<uint4*>(bits + (long long)row * words + 4 * (m0 + u)) =
                make_uint4(wc[0], wc[1], wc[2], wc[3]);
          kept_tiles |= ((wc[0] | wc[1] | wc[2] | wc[3]) != 0u) ? (1u << u) : 0u;
        }
        any |= kept_tiles != 0u;
        // the round's four tiles share one bitmap word (m0 is a multiple of 4)
        if (lane == 0 && tiles != nullptr && kept_tiles != 0u)
          atomicOr(&row_tiles[m0 >> 5], kept_tiles << (m0 & 31));
        continue;
      }
#pragma unroll
      for (int u = 0; u < kPackGroups; ++u) {  // the row's last round: ragged or missing tiles
        const int key0 = (m0 + u) * kTile + 4 * lane;
#pragma unroll
        for (int c = 0; c < 4; ++c) v[u][c] = 0.f;
        if (m0 + u < groups && key0 < T) {
          if (key0 + 4 <= T) {
            if (f16) {
              const uint2 r = __ldcs(reinterpret_cast<const uint2*>(static_cast<const __half*>(mask) + rbase + key0));
              v[u][0] = __half2float(__ushort_as_half((unsigned short)(r.x & 0xFFFFu)));
              v[u][1] = __half2float(__ushort_as_half((unsigned short)(r.x >> 16)));
              v[u][2] = __half2float(__ushort_as_half((unsigned short)(r.y & 0xFFFFu)));
              v[u][3] = __half2float(__ushort_as_half((unsigned short)(r.y >> 16)));
            } else {
              const float4 r = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(mask) + rbase + key0));
              v[u][0] = r.x;
              v[u][1] = r.y;
              v[u][2] = r.z;
              v[u][3] = r.w;
            }
          } else {  // the row's ragged end: only keys below T exist
            const float4 r = ragged_keys(mask, f16, rbase + key0, T - key0);
            v[u][0] = r.x;
            v[u][1] = r.y;
            v[u][2] = r.z;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kPackGroups; ++u) {
        const int m = m0 + u;
        if (m >= groups) break;  // uniform across the warp
        uint32_t wc[4];
        if ((m + 1) * kTile <= T) {  // uniform: every key of the tile exists
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            nonbin |= !(v[u][c] == 0.f || v[u][c] <= -10000.f);
            wc[c] = __ballot_sync(0xffffffffu, v[u][c] == 0.f);
          }
        } else {  // the row's ragged last tile
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const bool inb = m * kTile + 4 * lane + c < T;
            nonbin |= inb && !(v[u][c] == 0.f || v[u][c] <= -10000.f);
            wc[c] = __ballot_sync(0xffffffffu, inb && v[u][c] == 0.f);
          }
        }
        if (lane == 0)
          *reinterpret_cast<uint4*>(bits + (long long)row * words + 4 * m) = make_uint4(wc[0], wc[1], wc[2], wc[3]);
        const bool tile_kept = (wc[0] | wc[1] | wc[2] | wc[3]) != 0u;
        any |= tile_kept;
        if (lane == 0 && tiles != nullptr && tile_kept) atomicOr(&row_tiles[m >> 5], 1u << (m & 31));
      }
    }
    if (__any_sync(0xffffffffu, any) && lane == 0) kept_any = 1;
    if (__any_sync(0xffffffffu, nonbin) && lane == 0) atomicExch(nonbinary, 1);
    __syncthreads();
    if (threadIdx.x == 0 && !kept_any) atomicExch(nonbinary, 1);
    if (tiles != nullptr)
      for (int t = threadIdx.x; t < tile_words; t += blockDim.x)
        if (row_tiles[t] != 0u) atomicOr(&tiles[(long long)(row / kTile) * tile_words + t], row_tiles[t]);
    __syncthreads();
  }
}

// The chunk's K and V rows [B, C, H, d] (strides s*) copied to the cache layout [B, H, C, d]
// (strides d*), both tensors in one pass: each CTA iteration takes one (batch, token) row, whose
// H * d elements are contiguous in the source, and writes each head's d elements as one
// contiguous run.  16-byte copies (d a multiple of 8; pointers and strides 16-byte aligned).
__global__ void __launch_bounds__(128) kv_relayout_kernel(const uint16_t* __restrict__ src_k,
                                                         const uint16_t* __restrict__ src_v,
                                                         uint16_t* __restrict__ dst_k, uint16_t* __restrict__ dst_v,
                                                         int B, int C, int H, int d, long long s0, long long s1,
                                                         long long s2, long long d0, long long d1, long long d2) {
  const int nv = d / 8;        // 16-byte vectors per head row
  const int per_row = H * nv;  // per (batch, token) row
  const long long rows = (long long)B * C;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const int b = (int)(r / C), t = (int)(r % C);
    for (int i = threadIdx.x; i < per_row; i += blockDim.x) {
      const int h = i / nv, v = i % nv;
      const long long so = b * s0 + t * s1 + h * s2, dof = b * d0 + h * d1 + t * d2;
      const uint4 wk = __ldg(reinterpret_cast<const uint4*>(src_k + so) + v);
      const uint4 wv = __ldg(reinterpret_cast<const uint4*>(src_v + so) + v);
      reinterpret_cast<uint4*>(dst_k + dof)[v] = wk;
      reinterpret_cast<uint4*>(dst_v + dof)[v] = wv;
    }
  }
}

// bf16 -> fp16 for a v that the attention kernels then read as fp16: the per-element
// conversion of the V-converter warps (bf16 bits to fp32 exactly, cvt.rn to fp16), done once
// per element instead of once per tile in every CTA that loads the tile.
__global__ void __launch_bounds__(256) convert_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                         long long nvec, unsigned* status) {
  float vmax = 0.f;  // largest |v| seen (bf16 values are exact in fp32)
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nvec;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 w = __ldcs(src + i);
    uint32_t o[4];
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(in[e] << 16), hi = __uint_as_float(in[e] & 0xFFFF0000u);
      vmax = max_nan(vmax, max_nan(fabsf(lo), fabsf(hi)));
      o[e] = pack_f16(lo, hi);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  const bool bad = !(vmax <= 65504.f);
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) record_error(status, ST_VRANGE, 6u << 8);
}

template <int MODE, bool WIDE>
cudaError_t launch_mode(const AttnMaps& maps, const AttnArgs& a, cudaStream_t st) {
  static std::atomic<int> configured[64];
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(attn_fwd_kernel<MODE, WIDE>), SM_ALLOC,
                                      configured);
  if (e != cudaSuccess) return e;
  const int units = a.n_qt * a.n_hp * a.B;
  const int grid = a.n_whole + (units - a.n_whole) * a.split_k;
  attn_fwd_kernel<MODE, WIDE><<<grid, kAttnThreads, SM_ALLOC, st>>>(maps, a);
  ++t_launches;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn(const AttnMaps& maps, const AttnArgs& a, int mode, cudaStream_t st) {
  if (a.d == 256) {
    switch (mode) {
      case MODE_CAUSAL: return launch_mode<MODE_CAUSAL, true>(maps, a, st);
      case MODE_MASK: return launch_mode<MODE_MASK, true>(maps, a, st);
      case MODE_MASKB: return launch_mode<MODE_MASKB, true>(maps, a, st);
      default: return launch_mode<MODE_SPARSE, true>(maps, a, st);
    }
  }
  switch (mode) {
    case MODE_CAUSAL: return launch_mode<MODE_CAUSAL, false>(maps, a, st);
    case MODE_MASK: return launch_mode<MODE_MASK, false>(maps, a, st);
    case MODE_MASKB: return launch_mode<MODE_MASKB, false>(maps, a, st);
    default: return launch_mode<MODE_SPARSE, false>(maps, a, st);
  }
}

cudaError_t launch_mask_pack(const void* mask, int f16, int vec, int C, int T, long long ld, uint32_t* bits,
                             int words, int* nonbinary, uint32_t* tiles, int tile_words, cudaStream_t st) {
  const dim3 grid(1, C < 65535 ? C : 65535);
  if (vec)
    mask_pack_vec_kernel<<<grid, 256, 0, st>>>(mask, f16, C, T, ld, bits, words, nonbinary, tiles, tile_words);
  else
    mask_pack_kernel<<<grid, 256, 0, st>>>(mask, f16, C, T, ld, bits, words, nonbinary, tiles, tile_words);
  ++t_launches;
  return cudaGetLastError();
}

cudaError_t launch_convert_f16(const void* src, void* dst, long long nvec, unsigned* status, cudaStream_t st) {
  const long long want = (nvec + 255) / 256;
  const int grid = (int)(want < 152 * 8 ? want : 152 * 8);
  convert_f16_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), nvec, status);
  ++t_launches;
  return cudaGetLastError();
}

cudaError_t launch_kv_relayout(const void* src_k, const void* src_v, void* dst_k, void* dst_v, int B, int C,
                               int H, int d, const long long ss[3], const long long ds[3], cudaStream_t st) {
  const long long rows = (long long)B * C;
  const int grid = (int)(rows < 152 * 16 ? rows : 152 * 16);  // up to 16 CTAs of 128 threads per SM
  kv_relayout_kernel<<<grid, 128, 0, st>>>(static_cast<const uint16_t*>(src_k), static_cast<const uint16_t*>(src_v),
                                           static_cast<uint16_t*>(dst_k), static_cast<uint16_t*>(dst_v), B, C, H,
                                           d, ss[0], ss[1], ss[2], ds[0], ds[1], ds[2]);
  ++t_launches;
  return cudaGetLastError();
}

}  // namespace pf
