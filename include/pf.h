/*
 * pf.h -- C ABI of libpf: long-context prefill attention on one GB300 (sm_103a).
 *
 * Three operations, each launched asynchronously on the caller's CUDA stream:
 *
 *   pf_attn_dense   a prompt chunk of queries attends to a token-major K/V
 *                   history plus its own keys under an additive mask, and the
 *                   chunk's K/V are re-emitted in cache layout.
 *                   ("ANE Prefill Research", section "How the ANE prefill path
 *                   works": chunk rows + token-major K/V history + additive
 *                   mask in; attention output + the chunk's cache-layout K/V
 *                   out; "Folding a sparse indexer's selection into the mask":
 *                   dropped keys carry -30000 so exp() gives exactly zero.)
 *   pf_block_index  mean-pools every key block, scores every query row
 *                   against the pooled keys and keeps the local diagonal plus
 *                   the blocks above alpha x the row's hottest block.
 *                   ("Porting FlashPrefill V2 to Apple silicon for faster
 *                   prefill", sections "Compress keys before the heavy work",
 *                   "A cheap map of where the attention lives", "The
 *                   algorithm starts here".)
 *   pf_attn_sparse  exact attention over the kept blocks plus a pooled
 *                   correction for the skipped ones (same page, section
 *                   "Compute the peaks, summarize the rest"): a skipped block b
 *                   adds n_b * exp(q . kbar_b * scale) to the softmax
 *                   denominator and that weight times vbar_b to the numerator.
 *
 * Conventions shared by every entry point
 *   - Positions are absolute: chunk row i is position start_pos + i; key j is
 *     position j (history rows first, then the chunk's rows).
 *   - Tensors are token-major with the head dimension d contiguous:
 *       q                 [B, C, Hq, d]
 *       k_hist, v_hist    [B, start_pos, Hkv, d]
 *       k_chunk, v_chunk  [B, C, Hkv, d]
 *       k, v (sparse)     [B, start_pos + C, Hkv, d]
 *     Strides are given in ELEMENTS for the (batch, token, head) axes; a
 *     stride triple of all zeros means "contiguous" for that tensor.
 *   - GQA: query head h reads KV head h / (Hq / Hkv).
 *   - Ownership: the caller allocates every buffer (device memory) and keeps it
 *     alive until the stream reaches the call.  The library allocates nothing
 *     per call and never synchronises the stream.
 *   - Errors: arguments are validated synchronously before anything is
 *     launched.  PF_EINVAL = bad pointer / shape / stride / alignment;
 *     PF_EUNSUPPORTED = a valid request outside what the kernels implement
 *     (they refuse rather than fall back); PF_ECUDA = a CUDA launch error.  A
 *     device-side bounded wait that gave up is reported as PF_ETIMEOUT by
 *     pf_stream_status().  pf_last_error() returns the calling thread's last
 *     message.  Nothing is written when a call returns an error.
 */
#ifndef PF_H_
#define PF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PF_OK = 0,
  PF_EINVAL = 1,
  PF_EUNSUPPORTED = 2,
  PF_ECUDA = 3,
  PF_ETIMEOUT = 4,
  PF_ERANGE = 5
} pf_status;

typedef enum { PF_F16 = 0, PF_BF16 = 1, PF_F32 = 2 } pf_dtype;

/* Problem description shared by the three entry points. */
typedef struct {
  int32_t B;            /* batch */
  int32_t Hq;           /* query heads */
  int32_t Hkv;          /* KV heads; Hq % Hkv == 0 */
  int32_t d;            /* head dim: 64, 128 or 256 */
  int32_t C;            /* query rows in this call (the chunk), >= 1 */
  pf_dtype in_dtype;    /* q/k/v element type: PF_F16 or PF_BF16 */
  pf_dtype out_dtype;   /* out element type: PF_F32, PF_BF16 or PF_F16 */
  pf_dtype mask_dtype;  /* PF_F32 or PF_F16 (a bf16 mask cannot hold -30000 exactly) */
  float scale;          /* logit scale; 0 means 1/sqrt(d) */
  int64_t q_stride[3];  /* q over (b, t, h) */
  int64_t kh_stride[3]; /* k_hist / v_hist over (b, t, h); sparse: k / v */
  int64_t kc_stride[3]; /* k_chunk / v_chunk over (b, t, h) */
  int64_t o_stride[3];  /* out over (b, t, h) */
  int64_t okv_stride[3];/* out_k / out_v over (b, h, t); zeros = [B, Hkv, C, d] */
  int64_t mask_ld;      /* elements between mask rows; 0 means start_pos + C */
  int32_t v_f16;        /* 1: v (v_hist, v_chunk; out_v receives a copy) is fp16 while q/k keep
                           in_dtype; 0: v is in_dtype.  P * V runs in fp16 either way: a bf16 v
                           is converted tile by tile inside the attention kernels, an fp16 v is
                           read as it is (see pf_convert_f16) */
} pf_shape;

/*
 * Dense chunked prefill.
 *   out[b, i, h, :] = sum_j w_j v_j / sum_j w_j,
 *   w_j = exp(l_j - max_j l_j),  l_j = (q[b,i,h] . k_j) * scale + M[i, j],
 * over all keys j < start_pos + C (k_j from k_hist for j < start_pos, else
 * from k_chunk).  mask: additive [C, start_pos + C] (row stride mask_ld),
 * shared by every batch and head; a key with -30000 contributes exactly zero
 * to any row that has a key above -1e4.  mask == NULL means causal
 * (M = 0 for j <= start_pos + i, else the key is excluded), the same result as
 * the explicit 0 / -30000 causal mask.  With an explicit mask visibility is
 * the mask alone.
 * out_k / out_v (optional, both or neither): bit copies of k_chunk / v_chunk
 * written at okv_stride, by default head-major [B, Hkv, C, d], so a caller can
 * point them at row start_pos of its own cache.
 * lse (optional, [B, Hq, C] fp32, contiguous, 4-byte aligned): the natural log
 * of each row's softmax denominator, log sum_j exp(l_j); results over disjoint
 * key sets (e.g. a short chunk split across a long history) merge as
 * lse = logaddexp(lse_a, lse_b), out = e^(lse_a - lse) out_a + e^(lse_b - lse) out_b.
 * workspace (optional, device memory owned by the caller, 16-byte aligned,
 * workspace_bytes >= pf_dense_workspace_bytes, PF_EINVAL otherwise): lets the
 * call split the key range of its last, partial wave of work units across the
 * idle SMs; the parts' partial results (O, running max, sum) are merged on the
 * device with the same softmax identity, so the output matches the unsplit
 * call up to fp32 rounding order.  NULL runs every unit whole.  Calls that can
 * overlap on the GPU need separate workspaces.
 * Requirements: start_pos % 128 == 0 (PF_EUNSUPPORTED otherwise); every base
 * pointer 16-byte aligned and every stride a multiple of 16 bytes (PF_EINVAL);
 * k_hist / v_hist may be NULL when start_pos == 0.
 */
pf_status pf_attn_dense(const pf_shape* shape, const void* q, const void* k_hist,
                        const void* v_hist, const void* k_chunk, const void* v_chunk,
                        const void* mask, int32_t start_pos, void* out, float* lse,
                        void* out_k, void* out_v, void* workspace, int64_t workspace_bytes,
                        void* stream);

/* Bytes of the optional pf_attn_dense workspace for shape->d on the current
 * device (about 20 MB for d = 128 on 152 SMs; independent of the sequence). */
pf_status pf_dense_workspace_bytes(const pf_shape* shape, int64_t* bytes);

/* Workspace bytes for a call with an explicit mask: the above plus room for the mask packed
 * to bits (C * ceil((start_pos + C) / 128) * 16 bytes) and, per 128-row query tile, a bitmap
 * of the 128-key tiles it keeps.  With a workspace of this size a mask whose values are all 0
 * or <= -10000 (and that keeps a key in every row) is read as bits, the same result as reading
 * the values, and a query tile skips every key tile that none of its rows keeps (when
 * start_pos + C <= 262144; longer calls visit every key tile); any other mask is read as
 * values. */
pf_status pf_dense_workspace_bytes_masked(const pf_shape* shape, int32_t start_pos, int64_t* bytes);

/* Index-driven attention over an indexer's compacted selection ("ANE Prefill Research",
 * section "Folding a sparse indexer's selection into the mask": keepIndices / keepCounts).
 * Row i (position p = start_pos + i) attends only to
 *   - the keys of its kept compressed blocks: block c covers keys ratio*c .. ratio*c + ratio - 1
 *     of [history ; chunk], and must be complete at the row, 0 <= c < floor((p + 1) / ratio);
 *   - the keys after the last complete block, ratio*floor((p + 1) / ratio) .. p.
 * The result equals pf_attn_dense with that selection folded into a 0 / -30000 mask, but no
 * [C, start_pos + C] mask is written or read: the lists are packed to bits on the device and
 * only the 128-key tiles that some row of a query tile sees are visited.
 * keep_idx [C][keep_stride] int32 (device, 4-byte aligned): row i's entries are its first
 * keep_cnt[i]; their order does not matter and a repeated entry counts once.
 * keep_cnt [C] int32 (device).  ratio in [1, 128] (PF_EINVAL otherwise).
 * start_pos + C <= 1048576 (PF_EUNSUPPORTED otherwise).
 * workspace is required: workspace_bytes >= pf_indexed_workspace_bytes (PF_EINVAL otherwise).
 * An entry outside the row's complete blocks, a count outside [0, keep_stride] or a row that
 * sees no key cannot be checked on the host: the entry is skipped, the output is invalid, and
 * the next pf_stream_status returns PF_EINVAL.
 * Every other argument as pf_attn_dense (shape->mask_dtype and mask_ld are not used). */
pf_status pf_attn_indexed(const pf_shape* shape, const void* q, const void* k_hist,
                          const void* v_hist, const void* k_chunk, const void* v_chunk,
                          const int32_t* keep_idx, const int32_t* keep_cnt, int32_t keep_stride,
                          int32_t ratio, int32_t start_pos, void* out, float* lse, void* out_k,
                          void* out_v, void* workspace, int64_t workspace_bytes, void* stream);

/* Workspace bytes for pf_attn_indexed (the same as pf_dense_workspace_bytes_masked). */
pf_status pf_indexed_workspace_bytes(const pf_shape* shape, int32_t start_pos, int64_t* bytes);

/* Block selection produced by pf_block_index and consumed by pf_attn_sparse.
 * nblk = ceil((start_pos + C) / block); nqt = ceil(C / 128); W = ceil(nblk / 32);
 * cap = capacity, or nblk when capacity is 0.
 *
 * Chunked prefill: the pooled keys and values of the history's blocks do not change from one
 * chunk to the next, so a prompt processed in chunks can keep ONE kbar buffer (and one
 * pf_attn_sparse workspace) for all its chunks, sized for its last chunk (capacity = that
 * chunk's nblk), and pass pooled_blocks = the blocks an earlier call of the same prompt has
 * already pooled into them: only blocks pooled_blocks .. nblk - 1 are pooled again. */
typedef struct {
  uint32_t* row_bits;  /* [B, Hq, C, W]: bit (b % 32) of word b / 32 set iff the row keeps block b */
  int32_t* tile_list;  /* [B, Hq, nqt, nblk]: ascending union of the kept blocks of the tile's rows */
  int32_t* tile_cnt;   /* [B, Hq, nqt]: valid entries of tile_list */
  float* kbar;         /* 2 * B*Hkv*cap*d floats: the fp32 pooled (mean) keys [B, Hkv, cap, d],
                          then the library's 16-bit split of them (hi = round(mean), lo =
                          round(mean - hi), each [B, Hkv, cap, d] in the q/k type); blocks
                          nblk .. cap - 1 are not touched */
  int32_t capacity;    /* key blocks per (batch, KV head) in kbar and in pf_attn_sparse's
                          workspace; 0 means nblk; otherwise >= nblk (PF_EINVAL) */
  int32_t pooled_blocks; /* leading blocks whose means kbar (pf_block_index) or the workspace
                          (pf_attn_sparse) already holds from an earlier call on the same keys
                          and values with the same capacity; 0 pools every block; at most
                          start_pos / block (only whole history blocks; PF_EINVAL otherwise) */
} pf_sel;

/* Element counts of the pf_sel buffers (kbar_elems counts floats) and the byte size of
 * the pf_attn_sparse workspace, for capacity = nblk.  For buffers shared by the chunks of
 * one prompt, query the last chunk: its kbar_elems and pooled_bytes cover every chunk. */
typedef struct {
  int64_t nblk, nqt, words;
  int64_t row_bits_elems, tile_list_elems, tile_cnt_elems, kbar_elems;
  int64_t pooled_bytes; /* workspace bytes for pf_attn_sparse */
} pf_sparse_sizes;

pf_status pf_sparse_query_sizes(const pf_shape* shape, int32_t start_pos, int32_t block,
                                pf_sparse_sizes* sizes);

/*
 * Block index.  For row i (p = start_pos + i) and head h: ob = p / block;
 * candidates are the blocks b < ob; s_ib = (q_i . kbar_b) * scale with kbar_b
 * the mean of block b's keys; candidate b is kept iff
 * s_ib - max_c s_ic >= ln(alpha) (alpha = 0 keeps every candidate); the
 * diagonal block ob is always kept.  q [B, C, Hq, d]; k [B, start_pos + C, Hkv, d]
 * (history and chunk contiguous in one cache, strides kh_stride).
 * rules (optional, NULL = the rule above alone): the keep rules of the Metal
 * port's selection map ("Porting FlashPrefill V2 to Apple silicon for faster
 * prefill", section "At 16k, only 28% of visible blocks run in full"), applied
 * in this order:
 *   sink_tokens      candidates holding keys j < sink_tokens are kept;
 *   local_blocks     the candidates ob - local_blocks .. ob - 1 are kept;
 *   dense_tail_rows  rows at p >= start_pos + C - dense_tail_rows keep every
 *                    candidate;
 *   row_group        1, or 32: the rows of each aligned 32-position query tile
 *                    share the union of their kept blocks;
 *   share_kv_group   0, or 1: the query heads of one KV head share the union
 *                    of their kept blocks (row by row).
 * Requirements: block == 128, 0 <= alpha <= 1, start_pos % 128 == 0; rule
 * counts >= 0 (PF_EINVAL); row_group in {1, 32} (PF_EUNSUPPORTED).
 */
typedef struct {
  int32_t sink_tokens, local_blocks, dense_tail_rows, row_group, share_kv_group;
} pf_keep_rules;

pf_status pf_block_index(const pf_shape* shape, const void* q, const void* k, int32_t start_pos,
                         int32_t block, float alpha, const pf_keep_rules* rules,
                         const pf_sel* sel, void* stream);

/*
 * Block-sparse attention with pooled correction.  Row i (p = start_pos + i),
 * head h, kept set K_i from sel (row_bits), skipped set R_i = {b < ob} \ K_i:
 *   out = (sum_{j <= p, j/block in K_i} e^(l_j - m) v_j + sum_{b in R_i} n_b e^(s_ib - m) vbar_b)
 *       / (sum_{j <= p, j/block in K_i} e^(l_j - m)     + sum_{b in R_i} n_b e^(s_ib - m)).
 * pooled: caller-allocated workspace of pf_sparse_sizes.pooled_bytes (for
 * sel->capacity blocks); on return it starts with vbar, the fp32 block means of
 * v, [B, Hkv, cap, d]; the rest is scratch, except that with sel->pooled_blocks
 * > 0 it must still hold what the earlier call of the same prompt left there.  sel must come from pf_block_index on the same q, k,
 * start_pos and block.  lse (optional, [B, Hq, C] fp32): the log of the
 * denominator above, exact and pooled terms, as for pf_attn_dense.
 */
pf_status pf_attn_sparse(const pf_shape* shape, const void* q, const void* k, const void* v,
                         int32_t start_pos, int32_t block, const pf_sel* sel, void* pooled,
                         void* out, float* lse, void* stream);

/*
 * pf_attn_sparse_static -- pf_attn_sparse for callers that cannot allocate
 * device memory.  The pages describe no counterpart of this entry point.
 *
 * Some callers have no way to give pf_attn_sparse its `pooled` workspace: a
 * plug-in inside a host framework that owns every device allocation and hands
 * the plug-in only its inputs and outputs, or a latency-critical serving loop
 * that must not call cudaMalloc (it can block on the device and costs far more
 * than the attention call).  This entry point takes the same arguments minus
 * `pooled` and computes the same output; its scratch is a static device buffer
 * of PF_STATIC_SCRATCH_BYTES inside libpf, resident on every GPU that loads the
 * library until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *   - Limit: a problem whose pf_sparse_query_sizes().pooled_bytes exceeds
 *     PF_STATIC_SCRATCH_BYTES (B * Hkv * nblk * d * 8 bytes, rounded) is
 *     rejected with PF_EUNSUPPORTED and a message in pf_last_error().
 *   - Set-up: the first call on each device looks up the buffer's device
 *     address (cudaGetSymbolAddress) with that device current; make that first
 *     call before any stream capture.  The address is looked up once per device
 *     for the life of the process and is not looked up again after a
 *     cudaDeviceReset: do not call this entry point after resetting a device.
 *   - Shapes: B, Hq, Hkv, d, C below 1 or a negative start_pos are refused
 *     with PF_EINVAL before the scratch size is considered.
 *   - Sharing: every call uses the same buffer, which keeps the previous call's
 *     contents; nothing in it needs to start at zero (each call writes what it
 *     reads).  Calls that overlap on the GPU (other streams, other host threads)
 *     race on the buffer: order them.
 *   - The pooled block means stay internal (no vbar output).  sel->pooled_blocks
 *     must be 0 (PF_EUNSUPPORTED otherwise): the shared buffer cannot carry one
 *     prompt's pooled blocks from call to call.
 */
#define PF_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

pf_status pf_attn_sparse_static(const pf_shape* shape, const void* q, const void* k,
                                const void* v, int32_t start_pos, int32_t block,
                                const pf_sel* sel, void* out, float* lse, void* stream);

/*
 * pf_convert_f16 -- bf16 -> fp16 element by element: dst[i] = fp16(src[i]), n elements, both
 * contiguous and 16-byte aligned, n a multiple of 8 (PF_EINVAL otherwise).  The attention
 * kernels compute P * V in fp16 and convert a bf16 v tile by tile in every CTA that reads the
 * tile; a caller that keeps v in fp16 (converting each chunk's v once with this call, and
 * passing v_f16 = 1) spares them that work.  The conversion is exact for |v| <= 65504 (bf16
 * values keep their 8 significant bits) and rounds to nearest below fp16's normal range; a
 * larger |v|, inf or nan is reported as PF_ERANGE by pf_stream_status, as the kernels' own
 * conversion reports it.  Asynchronous on `stream`; allocates nothing.
 */
pf_status pf_convert_f16(const void* src, void* dst, int64_t n, void* stream);

/* Synchronise `stream`, then report (and clear) a device-side error: PF_ETIMEOUT
 * if a bounded wait in a kernel gave up since the last check; PF_EINVAL if a
 * pf_attn_indexed selection was invalid; PF_ERANGE if a bf16 v held a value the
 * fp16 P*V product cannot represent (|v| > 65504, inf or nan; in an attention call or in
 * pf_convert_f16); the output of the call concerned is then invalid.  PF_ECUDA on a
 * CUDA error; else PF_OK. */
pf_status pf_stream_status(void* stream);

/* Bounded-wait limit in SM clock cycles (default 4e8, about 0.2 s). */
void pf_set_wait_timeout(int64_t cycles);

/* Test hook: nonzero makes the next attention launches withhold one MMA
 * completion signal so that the consumers' bounded waits run out. */
void pf_set_debug_withhold(int32_t on);

/* Kernel launches issued by this thread since the counter was last reset. */
int64_t pf_launch_count(int32_t reset);

const char* pf_last_error(void);
const char* pf_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PF_H_ */
