// C ABI of libpf: argument validation, TMA descriptor encoding and launches.
// The operations and their contracts are documented in include/pf.h.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <string>

#include "indexed.cuh"
#include "kernels.cuh"
#include "pf.h"
#include "ptx.cuh"

namespace pf {
thread_local long long t_launches = 0;
}  // namespace pf

namespace {
thread_local std::string t_err;
}

namespace pf {
// Lets other translation units of the library report through pf_last_error().
void set_error_message(const char* msg) { t_err = msg; }
}  // namespace pf

// Device status words written by the kernels' bounded waits: [0] flags, [1] where.
static __device__ unsigned int g_status[2];

using namespace pf;

namespace {

long long g_timeout = 400000000LL;  // ~0.2 s at 2 GHz; legitimate waits take microseconds
int g_withhold = 0;

pf_status fail(pf_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}

pf_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PF_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device address of g_status on the current device (looked up once per device).
unsigned* status_words() {
  static unsigned* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned*>(p);
  }
  return addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int esize(pf_dtype t) { return t == PF_F32 ? 4 : 2; }

// Fill a (b, t, h) element-stride triple; zeros mean contiguous [B, T, H, d].
void strides_or_default(const int64_t in[3], int64_t T, int64_t H, int64_t d, long long out[3]) {
  if (in[0] == 0 && in[1] == 0 && in[2] == 0) {
    out[0] = T * H * d;
    out[1] = H * d;
    out[2] = d;
  } else {
    out[0] = in[0];
    out[1] = in[1];
    out[2] = in[2];
  }
}

bool strides_ok(const long long s[3], int es) {
  for (int i = 0; i < 3; ++i)
    if (s[i] < 0 || ((s[i] * es) & 15) != 0) return false;
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 4-D tiled map over a 16-bit tensor with element strides (s1, s2, s3) for
// dims 1..3 (dim 0 = d, contiguous); box = 64 elements x box1 x box2 x 1,
// 128-byte swizzle, zero fill out of bounds.
pf_status make_map(CUtensorMap* m, const void* base, pf_dtype dt, uint64_t d0, uint64_t d1,
                   uint64_t d2, uint64_t d3, long long s1, long long s2, long long s3,
                   uint32_t box1, uint32_t box2, const char* what) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(PF_ECUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {(cuuint64_t)s1 * 2, (cuuint64_t)s2 * 2, (cuuint64_t)s3 * 2};
  const cuuint32_t box[4] = {64, box1, box2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t =
      dt == PF_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(m, t, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PF_ECUDA, "tensor map for %s rejected (CUresult %d)", what, (int)r);
  return PF_OK;
}

// The output [B, C, Hq, d] (f32, bf16 or f16) for tile stores: dims (d, Hq, C, B), box
// 128 bytes of d x 1 head x 128 rows, 128-byte swizzle (the kernel stages rows swizzled).
pf_status map_out(CUtensorMap* m, void* base, pf_dtype dt, int B, int C, int Hq, int d,
                  const long long s[3]) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(PF_ECUDA, "cuTensorMapEncodeTiled is unavailable");
  const int es = dt == PF_F32 ? 4 : 2;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)Hq, (cuuint64_t)C, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)s[2] * es, (cuuint64_t)s[1] * es, (cuuint64_t)s[0] * es};
  const cuuint32_t box[4] = {(cuuint32_t)(128 / es), 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t = dt == PF_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                : dt == PF_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(m, t, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PF_ECUDA, "tensor map for out rejected (CUresult %d)", (int)r);
  return PF_OK;
}

// Token-major tensor [B, T, H, d] -> map dims (d, H, T, B), box 64 x 1 x rows (128; K / V
// tiles of head dim 256 are 64 keys).
pf_status map_tokens(CUtensorMap* m, const void* base, pf_dtype dt, int B, int T, int H, int d,
                     const long long s[3], const char* what, uint32_t rows = 128) {
  return make_map(m, base, dt, d, H, T, B, s[2], s[1], s[0], 1, rows, what);
}

// Keys per key tile of the attention kernel (and pooled blocks per pooled tile): 64 for head dim
// 256, whose 128-key tiles would not fit the shared-memory rings, else 128.
int key_tile(int d) { return d == 256 ? 64 : 128; }

pf_status check_common(const pf_shape* sh, int32_t start_pos) {
  if (sh == nullptr) return fail(PF_EINVAL, "shape is NULL");
  if (sh->B < 1 || sh->Hq < 1 || sh->Hkv < 1 || sh->C < 1)
    return fail(PF_EINVAL, "B, Hq, Hkv and C must be >= 1 (got %d, %d, %d, %d)", sh->B, sh->Hq,
                sh->Hkv, sh->C);
  if (sh->Hq % sh->Hkv != 0) return fail(PF_EINVAL, "Hq (%d) must be a multiple of Hkv (%d)", sh->Hq, sh->Hkv);
  if (sh->d != 64 && sh->d != 128 && sh->d != 256)
    return fail(PF_EUNSUPPORTED, "head dim %d (supported: 64, 128, 256)", sh->d);
  if (sh->in_dtype != PF_F16 && sh->in_dtype != PF_BF16)
    return fail(PF_EUNSUPPORTED, "q/k/v dtype must be f16 or bf16");
  if (sh->out_dtype != PF_F32 && sh->out_dtype != PF_BF16 && sh->out_dtype != PF_F16)
    return fail(PF_EINVAL, "bad out dtype");
  if (start_pos < 0) return fail(PF_EINVAL, "start_pos %d < 0", start_pos);
  if (start_pos % kTile != 0)
    return fail(PF_EUNSUPPORTED, "start_pos %d is not a multiple of %d", start_pos, kTile);
  if ((long long)start_pos + sh->C > (1LL << 30)) return fail(PF_EINVAL, "sequence too long");
  if (!(sh->scale >= 0.f) || isinf(sh->scale)) return fail(PF_EINVAL, "bad scale");
  if (sh->v_f16 != 0 && sh->v_f16 != 1) return fail(PF_EINVAL, "v_f16 must be 0 or 1 (got %d)", sh->v_f16);
  return PF_OK;
}

// Element type of v (v_hist, v_chunk, the sparse v and its pooled copy).
pf_dtype v_type(const pf_shape* sh) { return sh->v_f16 ? PF_F16 : sh->in_dtype; }

void fill_attn_common(const pf_shape* sh, int32_t start_pos, AttnArgs& a) {
  a.B = sh->B;
  a.Hq = sh->Hq;
  a.Hkv = sh->Hkv;
  a.G = sh->Hq / sh->Hkv;
  a.d = sh->d;
  a.C = sh->C;
  a.s = start_pos;
  a.T = start_pos + sh->C;
  a.n_qt = (sh->C + kTile - 1) / kTile;
  // two query heads of a KV group share each K / V tile; head dim 256 runs one head per CTA
  // (its 64 KB query tile fills both slots' room)
  a.slots = (a.G % 2 == 0 && sh->d != 256) ? 2 : 1;
  a.n_hp = sh->Hq / a.slots;
  a.ab_type = sh->in_dtype == PF_BF16 ? 1 : 0;
  a.convert_v = v_type(sh) == PF_BF16 ? 1 : 0;  // P * V is fp16: a bf16 v is converted per tile
  const float scale = sh->scale > 0.f ? sh->scale : 1.0f / sqrtf((float)sh->d);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out_dtype = sh->out_dtype == PF_F32 ? 2 : (sh->out_dtype == PF_BF16 ? 1 : 0);
  a.timeout = g_timeout;
  a.withhold = g_withhold;
  a.status = status_words();
  a.n_whole = a.n_qt * a.n_hp * a.B;  // no tail split unless a dense call plans one
  a.split_k = 1;
}

// SMs of the current device (cached per device).
int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

constexpr int kMinPartTiles = 4;      // a part gets at least this many key tiles
constexpr long long kCountBytes = 4096;  // counter area at the head of the workspace

long long dense_workspace_bytes(int d, int sms) {
  return kCountBytes + (long long)sms * 2 * kTile * (d + 2) * 4;
}

// The masked workspace: the dense one, then a 256-byte flag area, the query tiles' key-tile
// bitmaps and the packed mask bits [C][mask_words] (4 words = 128 keys per tile).
long long mask_words_of(long long T) { return (T + kTile - 1) / kTile * 4; }

long long mask_tile_words_of(long long T) { return ((T + kTile - 1) / kTile + 31) / 32; }

long long mask_tiles_bytes(int C, long long T) {
  return (((long long)C + kTile - 1) / kTile * mask_tile_words_of(T) * 4 + 255) / 256 * 256;
}

long long dense_masked_workspace_bytes(int d, int sms, int C, long long T) {
  return dense_workspace_bytes(d, sms) + 256 + mask_tiles_bytes(C, T) + (long long)C * mask_words_of(T) * 4;
}

// Tail split.  With U units and P SMs, the last wave holds W = U mod P units (all U when
// U < P) on P SMs; each of those units (the lightest, since units run heaviest first) is
// cut into k = P / W parts of consecutive key tiles so that the last wave fills the GPU.
// Needs W * k * 2 * 128 * (d + 2) floats of partials, at most P parts.
void plan_split(AttnArgs& a, int mode, void* ws) {
  const int P = sm_count();
  const int U = a.n_qt * a.n_hp * a.B;
  if (P <= 0 || ws == nullptr) return;
  const int W = (U < P) ? U : U % P;
  if (W == 0 || W > (int)(kCountBytes / 4)) return;
  const int kt = key_tile(a.d);
  const int min_tiles = (mode == MODE_CAUSAL) ? (a.s / kTile + 1) * (kTile / kt) : (a.T + kt - 1) / kt;
  int k = P / W;
  if (k > kMaxSplit) k = kMaxSplit;
  if (k > min_tiles / kMinPartTiles) k = min_tiles / kMinPartTiles;
  if (k < 2) return;
  a.n_whole = U - W;
  a.split_k = k;
  a.ws_cnt = static_cast<int*>(ws);
  a.ws_part = reinterpret_cast<float*>(static_cast<char*>(ws) + kCountBytes);
}

}  // namespace

namespace {

// An indexer's keep lists (pf_attn_indexed).
struct IndexSel {
  const int32_t* keep_idx;
  const int32_t* keep_cnt;
  int32_t keep_stride;
  int32_t ratio;
};

// pf_attn_dense, and pf_attn_indexed when isel != null (then mask is null and the selection is
// packed to bits in the workspace, which is required).
pf_status dense_entry(const pf_shape* sh, const void* q, const void* k_hist, const void* v_hist,
                      const void* k_chunk, const void* v_chunk, const void* mask, const IndexSel* isel,
                      int32_t start_pos, void* out, float* lse, void* out_k, void* out_v,
                      void* workspace, int64_t workspace_bytes, void* stream) {
  pf_status rc = check_common(sh, start_pos);
  if (rc != PF_OK) return rc;
  if (q == nullptr || k_chunk == nullptr || v_chunk == nullptr || out == nullptr)
    return fail(PF_EINVAL, "q, k_chunk, v_chunk and out must not be NULL");
  if (start_pos > 0 && (k_hist == nullptr || v_hist == nullptr))
    return fail(PF_EINVAL, "k_hist and v_hist are required when start_pos > 0");
  if ((out_k == nullptr) != (out_v == nullptr)) return fail(PF_EINVAL, "give both out_k and out_v, or neither");
  if (mask != nullptr && sh->mask_dtype != PF_F32 && sh->mask_dtype != PF_F16)
    return fail(PF_EUNSUPPORTED, "mask dtype must be f32 or f16 (bf16 cannot hold -30000 exactly)");
  if (isel != nullptr) {
    if (isel->keep_cnt == nullptr || (isel->keep_idx == nullptr && isel->keep_stride > 0))
      return fail(PF_EINVAL, "keep_cnt (and keep_idx when keep_stride > 0) must not be NULL");
    if (isel->keep_stride < 0) return fail(PF_EINVAL, "keep_stride %d < 0", isel->keep_stride);
    if (isel->ratio < 1 || isel->ratio > 128)
      return fail(PF_EINVAL, "compression ratio %d outside [1, 128]", isel->ratio);
    if ((reinterpret_cast<uintptr_t>(isel->keep_idx) & 3u) != 0u ||
        (reinterpret_cast<uintptr_t>(isel->keep_cnt) & 3u) != 0u)
      return fail(PF_EINVAL, "keep_idx and keep_cnt must be 4-byte aligned");
    if ((long long)start_pos + sh->C > kIndexedMaxKeys)
      return fail(PF_EUNSUPPORTED, "start_pos + C = %lld keys (index-driven attention supports %lld)",
                  (long long)start_pos + sh->C, kIndexedMaxKeys);
    if (workspace == nullptr) return fail(PF_EINVAL, "index-driven attention needs a workspace");
  }
  if (workspace != nullptr) {
    const int P = sm_count();
    if (P <= 0) return fail(PF_ECUDA, "no CUDA device");
    if (workspace_bytes < dense_workspace_bytes(sh->d, P))
      return fail(PF_EINVAL, "workspace of %lld bytes is smaller than pf_dense_workspace_bytes (%lld)",
                  (long long)workspace_bytes, dense_workspace_bytes(sh->d, P));
    const long long need = dense_masked_workspace_bytes(sh->d, P, sh->C, (long long)start_pos + sh->C);
    if (isel != nullptr && workspace_bytes < need)
      return fail(PF_EINVAL, "workspace of %lld bytes is smaller than pf_indexed_workspace_bytes (%lld)",
                  (long long)workspace_bytes, need);
  }
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0u)
    return fail(PF_EINVAL, "lse must be 4-byte aligned");
  const void* ptrs[] = {q, k_hist, v_hist, k_chunk, v_chunk, out, out_k, out_v, workspace};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return fail(PF_EINVAL, "every base pointer must be 16-byte aligned");
  const int B = sh->B, C = sh->C, Hq = sh->Hq, Hkv = sh->Hkv, d = sh->d, s = start_pos;
  long long qs[3], khs[3], kcs[3], os[3], okv[3];
  strides_or_default(sh->q_stride, C, Hq, d, qs);
  strides_or_default(sh->kh_stride, s, Hkv, d, khs);
  strides_or_default(sh->kc_stride, C, Hkv, d, kcs);
  strides_or_default(sh->o_stride, C, Hq, d, os);
  if (sh->okv_stride[0] == 0 && sh->okv_stride[1] == 0 && sh->okv_stride[2] == 0) {
    okv[0] = (long long)Hkv * C * d;
    okv[1] = (long long)C * d;
    okv[2] = d;
  } else {
    for (int i = 0; i < 3; ++i) okv[i] = sh->okv_stride[i];
  }
  if (!strides_ok(qs, 2) || !strides_ok(khs, 2) || !strides_ok(kcs, 2) || !strides_ok(okv, 2))
    return fail(PF_EINVAL, "q/k/v strides must be non-negative multiples of 16 bytes");
  if (!strides_ok(os, esize(sh->out_dtype))) return fail(PF_EINVAL, "out strides must be multiples of 16 bytes");

  AttnArgs a{};
  fill_attn_common(sh, start_pos, a);
  a.n_hist_tiles = s / key_tile(d);
  a.out = out;
  a.lse = lse;
  a.o_sb = os[0];
  a.o_st = os[1];
  a.o_sh = os[2];
  int mode = MODE_CAUSAL;
  if (mask != nullptr) {
    mode = MODE_MASK;
    a.mask = mask;
    a.mask_f16 = sh->mask_dtype == PF_F16 ? 1 : 0;
    a.mask_ld = sh->mask_ld > 0 ? sh->mask_ld : (long long)s + C;
    if (a.mask_ld < (long long)s + C) return fail(PF_EINVAL, "mask_ld %lld < start_pos + C", a.mask_ld);
    const int mes = a.mask_f16 ? 2 : 4;
    a.mask_vec = (aligned16(mask) && ((a.mask_ld * mes) & 15) == 0) ? 1 : 0;
  }

  AttnMaps maps;
  const pf_dtype dt = sh->in_dtype;
  if ((rc = map_tokens(&maps.q, q, dt, B, C, Hq, d, qs, "q")) != PF_OK) return rc;
  const uint32_t kt_rows = (uint32_t)key_tile(d);
  if ((rc = map_tokens(&maps.kc, k_chunk, dt, B, C, Hkv, d, kcs, "k_chunk", kt_rows)) != PF_OK) return rc;
  if ((rc = map_tokens(&maps.vc, v_chunk, v_type(sh), B, C, Hkv, d, kcs, "v_chunk", kt_rows)) != PF_OK)
    return rc;
  if (s > 0) {
    if ((rc = map_tokens(&maps.kh, k_hist, dt, B, s, Hkv, d, khs, "k_hist", kt_rows)) != PF_OK) return rc;
    if ((rc = map_tokens(&maps.vh, v_hist, v_type(sh), B, s, Hkv, d, khs, "v_hist", kt_rows)) != PF_OK)
      return rc;
  } else {
    maps.kh = maps.kc;
    maps.vh = maps.vc;
  }
  maps.kbar = maps.kc;
  maps.vbar = maps.vc;
  if ((rc = map_out(&maps.out, out, sh->out_dtype, B, C, Hq, d, os)) != PF_OK) return rc;

  if (a.status == nullptr) return fail(PF_ECUDA, "no CUDA device (status words unavailable)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (isel != nullptr) mode = MODE_MASKB;
  plan_split(a, mode, workspace);
  if ((mode == MODE_MASK || mode == MODE_MASKB) && workspace != nullptr &&
      workspace_bytes >= dense_masked_workspace_bytes(d, sm_count(), C, (long long)s + C)) {
    // binary masks (0 / <= -10000) are read as bits; the packing pass sets the flag and the
    // kernels keep the value path when the mask is not binary.  Layout: the flag (256 bytes),
    // the query tiles' key-tile bitmaps, the bits; one memset clears the first two.
    char* base = static_cast<char*>(workspace) + dense_workspace_bytes(d, sm_count());
    const long long T = (long long)s + C;
    const int words = (int)mask_words_of(T);
    const int tile_words = (int)mask_tile_words_of(T);
    const long long tile_bytes = mask_tiles_bytes(C, T);
    int* flag = reinterpret_cast<int*>(base);
    uint32_t* bits = reinterpret_cast<uint32_t*>(base + 256 + tile_bytes);
    // key-tile skipping needs the tile bitmap of a query tile in the kernel's 64-word bitmap
    uint32_t* tiles = tile_words <= 64 ? reinterpret_cast<uint32_t*>(base + 256) : nullptr;
    if ((e = cudaMemsetAsync(flag, 0, (size_t)(256 + (tiles != nullptr ? tile_bytes : 0)), st)) != cudaSuccess)
      return cuda_fail(e, "mask flag and tile bitmap");
    if (isel != nullptr) {
      // the keep lists become bits directly; the flag stays 0 (bits valid by construction)
      if ((e = launch_index_pack(isel->keep_idx, isel->keep_cnt, isel->keep_stride, isel->ratio, C, s,
                                 bits, words, tiles, tile_words, a.status, st)) != cudaSuccess)
        return cuda_fail(e, "keep-list packing launch");
    } else if ((e = launch_mask_pack(mask, a.mask_f16, a.mask_vec, C, (int)T, a.mask_ld, bits, words, flag, tiles,
                                     tile_words, st)) != cudaSuccess) {
      return cuda_fail(e, "mask packing launch");
    }
    a.mask_bits = bits;
    a.mask_words = words;
    a.mask_nonbinary = flag;
    a.mask_tiles = tiles;
    a.mask_tile_words = tile_words;
  }
  if (a.split_k > 1) {
    const int n_split = a.n_qt * a.n_hp * a.B - a.n_whole;
    if ((e = cudaMemsetAsync(a.ws_cnt, 0, sizeof(int) * n_split, st)) != cudaSuccess)
      return cuda_fail(e, "workspace counters");
  }
  if (mode == MODE_MASK && a.mask_nonbinary != nullptr &&
      (e = launch_attn(maps, a, MODE_MASKB, st)) != cudaSuccess)
    return cuda_fail(e, "attention launch (mask bits)");
  e = launch_attn(maps, a, mode, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  if (out_k != nullptr) {
    if ((e = launch_kv_relayout(k_chunk, v_chunk, out_k, out_v, B, C, Hkv, d, kcs, okv, st)) != cudaSuccess)
      return cuda_fail(e, "out_k / out_v copy");
  }
  return PF_OK;
}

}  // namespace

extern "C" {

const char* pf_last_error(void) { return t_err.c_str(); }

const char* pf_version(void) { return "libpf 0.1 sm_103a"; }

void pf_set_wait_timeout(int64_t cycles) { g_timeout = cycles > 1000 ? cycles : 1000; }

void pf_set_debug_withhold(int32_t on) { g_withhold = on ? 1 : 0; }

int64_t pf_launch_count(int32_t reset) {
  const long long n = t_launches;
  if (reset) t_launches = 0;
  return n;
}

pf_status pf_convert_f16(const void* src, void* dst, int64_t n, void* stream) {
  if (src == nullptr || dst == nullptr) return fail(PF_EINVAL, "src and dst must not be NULL");
  if (!aligned16(src) || !aligned16(dst)) return fail(PF_EINVAL, "src and dst must be 16-byte aligned");
  if (n < 0 || n % 8 != 0) return fail(PF_EINVAL, "n (%lld) must be a non-negative multiple of 8", (long long)n);
  if (n == 0) return PF_OK;
  unsigned* status = status_words();
  if (status == nullptr) return fail(PF_ECUDA, "no CUDA device (status words unavailable)");
  cudaError_t e = launch_convert_f16(src, dst, n / 8, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PF_OK : cuda_fail(e, "conversion launch");
}

pf_status pf_stream_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned w[2] = {0, 0};
  e = cudaMemcpyFromSymbol(w, g_status, sizeof(w));
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  if (w[0] == 0) return PF_OK;
  const unsigned zero[2] = {0, 0};
  cudaMemcpyToSymbol(g_status, zero, sizeof(zero));
  if ((w[0] & ST_TIMEOUT) == 0u && (w[0] & ST_SELECTION) != 0u)
    return fail(PF_EINVAL, "a keep list named a compressed block that is not complete at its row, a keep "
                           "count was outside [0, keep_stride], or a row saw no key (output invalid)");
  if ((w[0] & ST_TIMEOUT) == 0u && (w[0] & ST_VRANGE) != 0u)
    return fail(PF_ERANGE, "v holds a bf16 value outside the fp16 range of the P*V product "
                           "(|v| > 65504, inf or nan)");
  return fail(PF_ETIMEOUT, "a bounded device wait gave up (status 0x%x, role %u, barrier %u)", w[0],
              w[1] >> 8, w[1] & 0xFFu);
}

pf_status pf_dense_workspace_bytes_masked(const pf_shape* sh, int32_t start_pos, int64_t* bytes) {
  if (sh == nullptr || bytes == nullptr) return fail(PF_EINVAL, "NULL argument");
  if (sh->d != 64 && sh->d != 128 && sh->d != 256)
    return fail(PF_EUNSUPPORTED, "head dim %d (supported: 64, 128, 256)", sh->d);
  if (sh->C < 1 || start_pos < 0) return fail(PF_EINVAL, "C >= 1 and start_pos >= 0 required");
  const int P = sm_count();
  if (P <= 0) return fail(PF_ECUDA, "no CUDA device");
  *bytes = dense_masked_workspace_bytes(sh->d, P, sh->C, (long long)start_pos + sh->C);
  return PF_OK;
}

pf_status pf_dense_workspace_bytes(const pf_shape* sh, int64_t* bytes) {
  if (sh == nullptr || bytes == nullptr) return fail(PF_EINVAL, "NULL argument");
  if (sh->d != 64 && sh->d != 128 && sh->d != 256)
    return fail(PF_EUNSUPPORTED, "head dim %d (supported: 64, 128, 256)", sh->d);
  const int P = sm_count();
  if (P <= 0) return fail(PF_ECUDA, "no CUDA device");
  *bytes = dense_workspace_bytes(sh->d, P);
  return PF_OK;
}

pf_status pf_attn_dense(const pf_shape* sh, const void* q, const void* k_hist, const void* v_hist,
                        const void* k_chunk, const void* v_chunk, const void* mask,
                        int32_t start_pos, void* out, float* lse, void* out_k, void* out_v,
                        void* workspace, int64_t workspace_bytes, void* stream) {
  return dense_entry(sh, q, k_hist, v_hist, k_chunk, v_chunk, mask, nullptr, start_pos, out, lse, out_k,
                     out_v, workspace, workspace_bytes, stream);
}

pf_status pf_attn_indexed(const pf_shape* sh, const void* q, const void* k_hist, const void* v_hist,
                          const void* k_chunk, const void* v_chunk, const int32_t* keep_idx,
                          const int32_t* keep_cnt, int32_t keep_stride, int32_t ratio, int32_t start_pos,
                          void* out, float* lse, void* out_k, void* out_v, void* workspace,
                          int64_t workspace_bytes, void* stream) {
  const IndexSel isel{keep_idx, keep_cnt, keep_stride, ratio};
  return dense_entry(sh, q, k_hist, v_hist, k_chunk, v_chunk, nullptr, &isel, start_pos, out, lse, out_k,
                     out_v, workspace, workspace_bytes, stream);
}

pf_status pf_indexed_workspace_bytes(const pf_shape* sh, int32_t start_pos, int64_t* bytes) {
  return pf_dense_workspace_bytes_masked(sh, start_pos, bytes);
}

pf_status pf_sparse_query_sizes(const pf_shape* sh, int32_t start_pos, int32_t block,
                                pf_sparse_sizes* z) {
  if (sh == nullptr || z == nullptr) return fail(PF_EINVAL, "NULL argument");
  if (block != kTile) return fail(PF_EUNSUPPORTED, "block %d (supported: %d)", block, kTile);
  const long long T = (long long)start_pos + sh->C;
  z->nblk = (T + block - 1) / block;
  z->nqt = (sh->C + kTile - 1) / kTile;
  z->words = (z->nblk + 31) / 32;
  z->row_bits_elems = (long long)sh->B * sh->Hq * sh->C * z->words;
  z->tile_list_elems = (long long)sh->B * sh->Hq * z->nqt * z->nblk;
  z->tile_cnt_elems = (long long)sh->B * sh->Hq * z->nqt;
  const long long pe = (long long)sh->B * sh->Hkv * z->nblk * sh->d;  // pooled elements
  z->kbar_elems = 2 * pe;  // fp32 means, then the 16-bit hi and lo split of them
  const long long f32b = (pe * 4 + 255) / 256 * 256;
  const long long lpb = (pe * 2 + 255) / 256 * 256;
  z->pooled_bytes = f32b + 2 * lpb;
  return PF_OK;
}

namespace {

// The pooled layout of a call: blocks per (b, g) in kbar / vbar (cap) and the blocks an earlier
// call already pooled (p0).
pf_status pooled_layout(const pf_sel* sel, int32_t start_pos, int32_t block, const pf_sparse_sizes& z,
                        int* cap, int* p0) {
  *cap = sel->capacity > 0 ? sel->capacity : (int)z.nblk;
  if (sel->capacity < 0 || *cap < z.nblk)
    return fail(PF_EINVAL, "sel capacity %d is below the %lld key blocks of this call", sel->capacity, z.nblk);
  if (*cap > 2048) return fail(PF_EUNSUPPORTED, "sel capacity %d key blocks (at most 2048)", *cap);
  *p0 = sel->pooled_blocks;
  if (*p0 < 0 || *p0 > start_pos / block)
    return fail(PF_EINVAL, "pooled_blocks %d outside [0, start_pos / block = %d]", *p0, start_pos / block);
  return PF_OK;
}

pf_status check_sparse(const pf_shape* sh, int32_t start_pos, int32_t block, long long ks[3],
                       long long qs[3], pf_sparse_sizes* z) {
  pf_status rc = check_common(sh, start_pos);
  if (rc != PF_OK) return rc;
  if (block != kTile) return fail(PF_EUNSUPPORTED, "block %d (supported: %d)", block, kTile);
  if ((rc = pf_sparse_query_sizes(sh, start_pos, block, z)) != PF_OK) return rc;
  if (z->nblk > 2048) return fail(PF_EUNSUPPORTED, "%lld key blocks (at most 2048)", z->nblk);
  if (sh->Hkv * sh->d / 8 > 1024) return fail(PF_EUNSUPPORTED, "Hkv * d too large for pooling");
  strides_or_default(sh->q_stride, sh->C, sh->Hq, sh->d, qs);
  strides_or_default(sh->kh_stride, (long long)start_pos + sh->C, sh->Hkv, sh->d, ks);
  if (!strides_ok(qs, 2) || !strides_ok(ks, 2))
    return fail(PF_EINVAL, "q/k/v strides must be non-negative multiples of 16 bytes");
  return PF_OK;
}

}  // namespace

pf_status pf_block_index(const pf_shape* sh, const void* q, const void* k, int32_t start_pos,
                         int32_t block, float alpha, const pf_keep_rules* rules,
                         const pf_sel* sel, void* stream) {
  long long ks[3], qs[3];
  pf_sparse_sizes z;
  pf_status rc = check_sparse(sh, start_pos, block, ks, qs, &z);
  if (rc != PF_OK) return rc;
  if (!(alpha >= 0.f && alpha <= 1.f)) return fail(PF_EUNSUPPORTED, "alpha %g outside [0, 1]", alpha);
  pf_keep_rules kr{0, 0, 0, 1, 0};
  if (rules != nullptr) kr = *rules;
  if (kr.sink_tokens < 0 || kr.local_blocks < 0 || kr.dense_tail_rows < 0)
    return fail(PF_EINVAL, "keep-rule counts must be >= 0");
  if (kr.row_group != 1 && kr.row_group != 32)
    return fail(PF_EUNSUPPORTED, "row_group %d (supported: 1, 32)", kr.row_group);
  if (kr.share_kv_group != 0 && kr.share_kv_group != 1) return fail(PF_EINVAL, "share_kv_group must be 0 or 1");
  if (q == nullptr || k == nullptr || sel == nullptr || sel->row_bits == nullptr ||
      sel->tile_list == nullptr || sel->tile_cnt == nullptr || sel->kbar == nullptr)
    return fail(PF_EINVAL, "q, k and every pf_sel buffer must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(sel->kbar))
    return fail(PF_EINVAL, "q, k and kbar must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = start_pos + sh->C;
  const int B = sh->B, Hkv = sh->Hkv, d = sh->d, nblk = (int)z.nblk;
  int cap = 0, p0 = 0;
  if ((rc = pooled_layout(sel, start_pos, block, z, &cap, &p0)) != PF_OK) return rc;
  const long long pe = (long long)B * Hkv * cap * d;  // pooled elements at this capacity
  uint16_t* kb_hi = reinterpret_cast<uint16_t*>(sel->kbar + pe);
  uint16_t* kb_lo = kb_hi + pe;
  PoolArgs p{};
  p.x = k;
  p.B = B;
  p.T = T;
  p.H = Hkv;
  p.d = d;
  p.block = block;
  p.nblk = nblk;
  p.cap = cap;
  p.blk0 = p0;
  p.sb = ks[0];
  p.st = ks[1];
  p.sh = ks[2];
  p.out_f32 = sel->kbar;
  p.out_lp = nullptr;
  p.out_hi = kb_hi;
  p.out_lo = kb_lo;
  cudaError_t e = launch_pool(p, sh->in_dtype == PF_BF16 ? 1 : 0, st);
  if (e != cudaSuccess) return cuda_fail(e, "pool launch");
  IndexArgs ia{};
  ia.ab_type = sh->in_dtype == PF_BF16 ? 1 : 0;
  ia.B = B;
  ia.Hq = sh->Hq;
  ia.Hkv = Hkv;
  ia.G = sh->Hq / Hkv;
  ia.d = d;
  ia.C = sh->C;
  ia.s = start_pos;
  ia.nblk = nblk;
  ia.n_qt = (int)z.nqt;
  ia.words = (int)z.words;
  ia.slots = (ia.G % 2 == 0 && d != 256) ? 2 : 1;
  ia.n_hp = sh->Hq / ia.slots;
  ia.scale = sh->scale > 0.f ? sh->scale : 1.0f / sqrtf((float)d);
  ia.log_alpha = alpha > 0.f ? logf(alpha) : -INFINITY;
  ia.sink_blocks = (int)(((long long)kr.sink_tokens + kTile - 1) / kTile);
  ia.local_blocks = kr.local_blocks;
  ia.tail_from = (int)((long long)T - kr.dense_tail_rows);
  ia.row_group32 = kr.row_group == 32 ? 1 : 0;
  ia.row_bits = sel->row_bits;
  ia.tile_list = sel->tile_list;
  ia.tile_cnt = sel->tile_cnt;
  ia.status = status_words();
  ia.timeout = g_timeout;
  ia.grid = sm_count();
  if (ia.grid <= 0) return fail(PF_ECUDA, "no CUDA device");
  if (ia.status == nullptr) return fail(PF_ECUDA, "no CUDA device (status words unavailable)");
  IndexMaps maps;
  const long long pst[3] = {(long long)Hkv * cap * d, (long long)cap * d, (long long)d};
  if ((rc = map_tokens(&maps.q, q, sh->in_dtype, B, sh->C, sh->Hq, d, qs, "q")) != PF_OK) return rc;
  const uint32_t pt_rows = (uint32_t)key_tile(d);  // pooled blocks per pooled tile
  if ((rc = make_map(&maps.hi, kb_hi, sh->in_dtype, d, nblk, Hkv, B, pst[2], pst[1], pst[0], pt_rows, 1,
                     "kbar hi")) != PF_OK)
    return rc;
  if ((rc = make_map(&maps.lo, kb_lo, sh->in_dtype, d, nblk, Hkv, B, pst[2], pst[1], pst[0], pt_rows, 1,
                     "kbar lo")) != PF_OK)
    return rc;
  if ((e = launch_index(maps, ia, st)) != cudaSuccess) return cuda_fail(e, "index launch");
  if (kr.share_kv_group && ia.G > 1 && (e = launch_share_group(ia, st)) != cudaSuccess)
    return cuda_fail(e, "shared-selection launch");
  return PF_OK;
}

pf_status pf_attn_sparse(const pf_shape* sh, const void* q, const void* k, const void* v,
                         int32_t start_pos, int32_t block, const pf_sel* sel, void* pooled,
                         void* out, float* lse, void* stream) {
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0u)
    return fail(PF_EINVAL, "lse must be 4-byte aligned");
  long long ks[3], qs[3], os[3];
  pf_sparse_sizes z;
  pf_status rc = check_sparse(sh, start_pos, block, ks, qs, &z);
  if (rc != PF_OK) return rc;
  if (q == nullptr || k == nullptr || v == nullptr || sel == nullptr || pooled == nullptr ||
      out == nullptr || sel->row_bits == nullptr || sel->tile_list == nullptr ||
      sel->tile_cnt == nullptr || sel->kbar == nullptr)
    return fail(PF_EINVAL, "q, k, v, sel buffers, pooled and out must be non-NULL");
  const void* ptrs[] = {q, k, v, pooled, out, sel->kbar};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(PF_EINVAL, "every base pointer must be 16-byte aligned");
  strides_or_default(sh->o_stride, sh->C, sh->Hq, sh->d, os);
  if (!strides_ok(os, esize(sh->out_dtype))) return fail(PF_EINVAL, "out strides must be multiples of 16 bytes");
  const int B = sh->B, C = sh->C, Hq = sh->Hq, Hkv = sh->Hkv, d = sh->d, T = start_pos + C;
  const int nblk = (int)z.nblk;
  int cap = 0, p0 = 0;
  if ((rc = pooled_layout(sel, start_pos, block, z, &cap, &p0)) != PF_OK) return rc;
  const long long pe = (long long)B * Hkv * cap * d;  // pooled elements at this capacity
  const long long f32b = (pe * 4 + 255) / 256 * 256;
  const long long lpb = (pe * 2 + 255) / 256 * 256;
  float* vbar = static_cast<float*>(pooled);
  void* kbar_lp = sel->kbar + pe;  // the 16-bit round of the pooled keys written by pf_block_index
  void* vbar_lp = static_cast<char*>(pooled) + f32b + lpb;
  const int bf16 = v_type(sh) == PF_BF16 ? 1 : 0;  // v's type: pooled as read, copied in it
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  PoolArgs p{};
  p.x = v;
  p.B = B;
  p.T = T;
  p.H = Hkv;
  p.d = d;
  p.block = block;
  p.nblk = nblk;
  p.cap = cap;
  p.blk0 = p0;
  p.sb = ks[0];
  p.st = ks[1];
  p.sh = ks[2];
  p.out_f32 = vbar;
  p.out_lp = vbar_lp;
  p.out_hi = nullptr;
  p.out_lo = nullptr;
  cudaError_t e = launch_pool(p, bf16, st);
  if (e != cudaSuccess) return cuda_fail(e, "pool launch");

  AttnArgs a{};
  fill_attn_common(sh, start_pos, a);
  a.n_hist_tiles = 1 << 30;  // every exact key tile comes from the one K/V cache map
  a.out = out;
  a.lse = lse;
  a.o_sb = os[0];
  a.o_st = os[1];
  a.o_sh = os[2];
  a.row_bits = sel->row_bits;
  a.tile_list = sel->tile_list;
  a.tile_cnt = sel->tile_cnt;
  a.words = (int)z.words;
  a.nblk = nblk;
  a.log2_nb = log2f((float)block);

  AttnMaps maps;
  const pf_dtype dt = sh->in_dtype;
  const long long pst[3] = {(long long)Hkv * cap * d, (long long)cap * d, (long long)d};
  if ((rc = map_tokens(&maps.q, q, dt, B, C, Hq, d, qs, "q")) != PF_OK) return rc;
  const uint32_t kt_rows = (uint32_t)key_tile(d);
  if ((rc = map_tokens(&maps.kh, k, dt, B, T, Hkv, d, ks, "k", kt_rows)) != PF_OK) return rc;
  if ((rc = map_tokens(&maps.vh, v, v_type(sh), B, T, Hkv, d, ks, "v", kt_rows)) != PF_OK) return rc;
  // pooled [B, Hkv, nblk, d]: dims (d, nblk, Hkv, B), box 64 x 128 pooled rows
  if ((rc = make_map(&maps.kbar, kbar_lp, dt, d, nblk, Hkv, B, pst[2], pst[1], pst[0], kt_rows, 1,
                     "kbar")) != PF_OK)
    return rc;
  if ((rc = make_map(&maps.vbar, vbar_lp, v_type(sh), d, nblk, Hkv, B, pst[2], pst[1], pst[0], kt_rows, 1,
                     "vbar")) != PF_OK)
    return rc;
  maps.kc = maps.kh;
  maps.vc = maps.vh;
  if ((rc = map_out(&maps.out, out, sh->out_dtype, B, C, Hq, d, os)) != PF_OK) return rc;
  if (a.status == nullptr) return fail(PF_ECUDA, "no CUDA device (status words unavailable)");
  // longest-first unit order, kept in the workspace's spare 16-bit region when it fits
  const long long units = (long long)a.n_qt * a.n_hp * B;
  if (units * 4 <= lpb) {
    OrderArgs o{};
    o.tile_cnt = sel->tile_cnt;
    o.B = B;
    o.Hq = Hq;
    o.n_qt = a.n_qt;
    o.slots = a.slots;
    o.n_hp = a.n_hp;
    o.s = start_pos;
    o.U = (int)units;
    o.perm = reinterpret_cast<int32_t*>(static_cast<char*>(pooled) + f32b);
    if ((e = launch_order_units(o, st)) != cudaSuccess) return cuda_fail(e, "unit order launch");
    a.perm = o.perm;
  }
  if ((e = launch_attn(maps, a, MODE_SPARSE, st)) != cudaSuccess) return cuda_fail(e, "attention launch");
  return PF_OK;
}

}  // extern "C"
