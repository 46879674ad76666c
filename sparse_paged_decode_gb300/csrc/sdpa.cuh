// sdpa.cuh -- argument block and launcher of the dense GQA attention call
// (attention_sdpa).  Internal to the library; nothing here is part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace spd {

struct SdpaArgs {
    const void *q;          // [T, Hq, D]
    int64_t q_s0, q_s1, q_s2;
    const void *k;          // [S, Hkv, D]
    int64_t k_s0, k_s1, k_s2;
    const void *v;          // [S, Hkv, D]
    int64_t v_s0, v_s1, v_s2;
    void *out;              // [T, Hq, D]
    int64_t o_s0, o_s1, o_s2;
    int32_t in_dt, out_dt;  // spd_dtype of q/k/v and of out
    int32_t T, S, Hq, Hkv, D;
    int32_t causal;         // query t reads keys j <= t + S - T
    float sm_scale;
};

cudaError_t launch_sdpa(const SdpaArgs &a, cudaStream_t stream);

}  // namespace spd
