// Index-driven attention: an indexer's compacted selection (per query row, a list of kept
// compressed key blocks) packed into the bits the attention kernel's MODE_MASKB reads.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pf {

// device status bit beside ST_TIMEOUT (1) and ST_VRANGE (2): a keep list named a block that is
// not complete at its row, a count outside [0, stride], or a row saw no key
constexpr unsigned ST_SELECTION = 4u;

// Largest key count the packing pass holds in shared memory (one bit per key).
constexpr long long kIndexedMaxKeys = 1LL << 20;

// Row i (position p = s + i): bits of the keys of its kept blocks (block c covers keys
// ratio*c .. ratio*c + ratio - 1, and must be complete: c < (p + 1) / ratio) and of the keys
// ratio*((p + 1) / ratio) .. p, into bits [C][words]; with tiles (zeroed,
// [ceil(C / 128)][tile_words]) each query tile's rows OR in the 128-key tiles they see.
// A bad entry is skipped and sets ST_SELECTION in status.
cudaError_t launch_index_pack(const int32_t* keep_idx, const int32_t* keep_cnt, long long stride,
                              int ratio, int C, int s, uint32_t* bits, int words, uint32_t* tiles,
                              int tile_words, unsigned* status, cudaStream_t st);

}  // namespace pf
