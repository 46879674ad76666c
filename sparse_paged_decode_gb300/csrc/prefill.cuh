// prefill.cuh -- argument block, workspace size and launcher of the fused
// prefill score-to-selection call (msa_prefill_block_score).  Internal to the
// library; nothing here is part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace spd {

struct PrefillArgs {
    const void *q;               // [total_q, Hi, Di] index queries
    int64_t q_s0, q_s1, q_s2;
    const void *k;               // [P*128, 1, Di] index key cache
    int64_t k_s0, k_s2;
    const int32_t *bt;           // [R, NB] page ids
    int64_t bt_s0, bt_s1;
    const int32_t *slot_ids;     // [B] page-table row of each sequence
    int64_t sid_s0;
    const int32_t *cu_q;         // [B+1] query token offsets
    int64_t cuq_s0;
    const int32_t *seq_lens;     // [B] keys of each sequence
    int64_t sl_s0;
    const int32_t *prefix;       // [B] keys before each chunk
    int64_t pre_s0;
    const int32_t *cu_b;         // [B+1] query block (output row) offsets
    int64_t cub_s0;
    int32_t *out;                // [Hi, n_rows, topk]
    int64_t o_s0, o_s1, o_s2;
    int32_t q_dt, k_dt;
    int32_t total_q, Hi, Di, R, NB, B, n_rows, topk;
    int32_t bsq, init_blocks, local_blocks;
    int64_t P;
    float scale;
};

// Workspace: the token-level score sheet [Hi, total_q, NB] f32 and each
// token's key limit and page-table row.
size_t prefill_workspace_bytes(int64_t total_q, int64_t Hi, int64_t NB);

cudaError_t launch_prefill(const PrefillArgs &a, void *ws, cudaStream_t stream);

}  // namespace spd
