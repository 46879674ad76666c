// spd_dispatch.h -- choice of kernel for each stage and the workspace size of
// the attention calls.  Internal to the library.
#pragma once

#include <stddef.h>

#include "sdpa.cuh"
#include "spd_internal.cuh"

namespace spd {

cudaError_t dispatch_score(const ScoreArgs &a, cudaStream_t stream);
cudaError_t dispatch_select(const SelectArgs &a, cudaStream_t stream);
cudaError_t dispatch_attention(const AttnArgs &a, void *workspace, size_t workspace_bytes, cudaStream_t stream);
cudaError_t dispatch_sdpa(const SdpaArgs &a, cudaStream_t stream);

// Count of kernels enqueued by the library (spd_launch_count).
void count_launches(int n);
uint64_t launch_count();

// Kernel policy of a stage (1 score, 2 select, 3 attention, 4 dense attention;
// spd_set_kernel_policy)
// and the status word of a workspace (spd_workspace_status).
int set_kernel_policy(int stage, int policy);
int workspace_status(const void *workspace, cudaStream_t stream);

// Workspace bytes for the attention calls (capacities only).
size_t workspace_bytes(int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t NB);

}  // namespace spd
