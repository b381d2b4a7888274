// pf_attn_sparse_static: the block-sparse attention entry point for callers
// that cannot allocate device memory.
//
// pf_attn_sparse needs a caller-provided workspace (`pooled`).  Some callers
// have no way to provide one: a plug-in running inside a host framework that
// owns every device allocation and hands the plug-in only its inputs and
// outputs, or a latency-critical serving loop that must not call cudaMalloc
// (it can block on the device and takes far longer than the attention call).
// This entry point takes the same inputs and outputs but no workspace: the
// scratch lives in the fixed-size device array below, which is part of the
// library image and stays resident on every GPU that loads libpf until the
// process exits.  Nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
#include <stdio.h>

#include <mutex>

#include "pf.h"

namespace pf {
void set_error_message(const char* msg);  // defined in pf_abi.cu; feeds pf_last_error()
}

namespace {

// Scratch for the pooled means (fp32 vbar plus the 16-bit copies of kbar and
// vbar).  PF_STATIC_SCRATCH_BYTES (16 MiB) covers B * Hkv * nblk * d * 8 bytes
// up to 2^21 elements, e.g. 8 KV heads x head_dim 128 x 2048 key blocks (256K
// keys) at batch 1.
constexpr size_t kScratchBytes = PF_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_sparse_scratch[kScratchBytes];

// Device address of g_sparse_scratch, looked up once per device with that
// device current.  In host code the array's name is only a host-side stand-in;
// kernels must be given this address instead.
std::mutex g_mu;
void* g_addr[64] = {nullptr};

pf_status scratch_address(void** out, const char** why) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *why = "no current CUDA device";
    return PF_ECUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_sparse_scratch);
    if (e != cudaSuccess || p == nullptr) {
      *why = "cudaGetSymbolAddress failed for the static scratch buffer";
      return PF_ECUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return PF_OK;
}

}  // namespace

extern "C" {

pf_status pf_attn_sparse_static(const pf_shape* shape, const void* q, const void* k, const void* v,
                                int32_t start_pos, int32_t block, const pf_sel* sel, void* out,
                                float* lse, void* stream) {
  // A shape that pf_attn_sparse would reject as invalid is rejected the same way here, before
  // its scratch size is computed (a negative or overflowing size must not read as "too big").
  if (shape == nullptr) {
    pf::set_error_message("pf_attn_sparse_static: shape is NULL");
    return PF_EINVAL;
  }
  if (shape->B < 1 || shape->Hq < 1 || shape->Hkv < 1 || shape->d < 1 || shape->C < 1 || start_pos < 0) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "pf_attn_sparse_static: B, Hq, Hkv, d and C must be >= 1 and start_pos >= 0 (got %d, %d, %d, "
             "%d, %d, %d)", shape->B, shape->Hq, shape->Hkv, shape->d, shape->C, start_pos);
    pf::set_error_message(msg);
    return PF_EINVAL;
  }
  pf_sparse_sizes z;
  pf_status rc = pf_sparse_query_sizes(shape, start_pos, block, &z);
  if (rc != PF_OK) return rc;
  if (sel != nullptr && sel->pooled_blocks != 0) {
    pf::set_error_message("pf_attn_sparse_static: pooled_blocks must be 0 (the shared scratch cannot carry "
                          "one prompt's pooled blocks from call to call)");
    return PF_EUNSUPPORTED;
  }
  // the scratch covers sel->capacity blocks (nblk when 0)
  const long long cap = (sel != nullptr && sel->capacity > z.nblk) ? sel->capacity : z.nblk;
  const long long pe = (long long)shape->B * shape->Hkv * cap * shape->d;
  const long long need = (pe * 4 + 255) / 256 * 256 + 2 * ((pe * 2 + 255) / 256 * 256);
  // the same size in floating point: a product past int64 shows up here as too large
  const double approx = (double)shape->B * shape->Hkv * (double)cap * shape->d * 8.0;
  if (approx > (double)kScratchBytes * 2.0 || need < 0 || (size_t)need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "pf_attn_sparse_static: this problem needs %lld bytes of scratch but the static buffer "
             "holds %zu; use pf_attn_sparse with a caller-allocated workspace",
             need, kScratchBytes);
    pf::set_error_message(msg);
    return PF_EUNSUPPORTED;
  }
  void* scratch = nullptr;
  const char* why = nullptr;
  if ((rc = scratch_address(&scratch, &why)) != PF_OK) {
    char msg[256];
    snprintf(msg, sizeof(msg), "pf_attn_sparse_static: %s", why);
    pf::set_error_message(msg);
    return rc;
  }
  // Every byte of the workspace that the kernels read is written earlier in
  // the same call, so stale contents from a previous call do not matter.
  return pf_attn_sparse(shape, q, k, v, start_pos, block, sel, scratch, out, lse, stream);
}

}  // extern "C"
