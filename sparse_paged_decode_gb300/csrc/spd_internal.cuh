// spd_internal.cuh -- argument blocks and launchers shared by the C ABI
// front end (spd_abi.cu) and the kernels.  Nothing here is part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "spd.h"

namespace spd {

constexpr int kBlock = 128;        // tokens per page (the only supported block size)
constexpr int kMaxNB = 1024;       // page-table capacity in blocks
constexpr int kMaxGroup = 16;      // q heads per kv head
constexpr int kMaxD = 256;         // attention head dim
constexpr int kMaxDi = 512;        // index head dim

// ------------------------------------------------------------ argument blocks

// Stage 1: block-max score sheet.
struct ScoreArgs {
    const void *q;          // [T, Hi, Di]
    int64_t q_s0, q_s1, q_s2;
    const void *k;          // [S, 1, Di]
    int64_t k_s0, k_s2;
    const int32_t *bt;      // [R, NB]
    int64_t bt_s0, bt_s1;
    const int32_t *sl;      // [T]
    int64_t sl_s0;
    const int32_t *ri;      // [T]
    int64_t ri_s0;
    float *out;             // [Hi, T, NB]
    int64_t o_s0, o_s1, o_s2;
    int32_t q_dt, k_dt;
    int32_t T, Hi, Di, R, NB;
    int64_t P;              // pool pages
    float idx_scale;
};

// Stage 2: top-k selection.
struct SelectArgs {
    const float *s;         // [Hi, T, NB]
    int64_t s_s0, s_s1, s_s2;
    int32_t *o;             // [Hi, T, K]
    int64_t o_s0, o_s1, o_s2;
    int32_t Hi, T, NB, K;
};

// Stage 3: paged decode attention (sparse when tk != nullptr).
struct AttnArgs {
    const void *q;          // [T, Hq, D]
    int64_t q_s0, q_s1, q_s2;
    const uint8_t *k;       // [S, Hkv, D] e4m3 or bf16 (kv_dt), innermost stride 1
    const uint8_t *v;
    int64_t k_s0, k_s1, v_s0, v_s1;
    const int32_t *bt;      // [R, NB]
    int64_t bt_s0, bt_s1;
    const int32_t *sl;      // [T]
    int64_t sl_s0;
    const int32_t *ri;      // [T]
    int64_t ri_s0;
    const int32_t *tk;      // [Hkv, T, K] or nullptr (dense)
    int64_t tk_s0, tk_s1, tk_s2;
    __nv_bfloat16 *out;     // [T, Hq, D]
    int64_t o_s0, o_s1, o_s2;
    int32_t q_dt, kv_dt;    // kv_dt: SPD_E4M3 or SPD_BF16 (both caches)
    int32_t T, Hq, Hkv, D, R, NB, K;
    int64_t P;
    float sm_scale, k_scale, v_scale;
};

// ------------------------------------------------------------------ launchers
// Each returns the cudaError_t of its launch(es).

cudaError_t launch_score_generic(const ScoreArgs &a, cudaStream_t stream);
cudaError_t launch_select_generic(const SelectArgs &a, cudaStream_t stream);
cudaError_t launch_select_rank(const SelectArgs &a, cudaStream_t stream);
cudaError_t launch_select_fast(const SelectArgs &a, cudaStream_t stream);  // sort for NB <= 256, else rank
cudaError_t launch_attention_generic(const AttnArgs &a, cudaStream_t stream);

// ------------------------------------------------------- per-device set-up
// Both are safe to call from several host threads and cache their answer per
// device ordinal (any ordinal the runtime reports).

// SMs of the current device (at least 1).
int device_sm_count();

// Opts `func` in to `bytes` of dynamic shared memory on the current device,
// once per (device, kernel); later calls with no more bytes do nothing.
cudaError_t opt_in_smem(const void *func, int bytes);

// ------------------------------------------------------------- device helpers

__device__ __forceinline__ float e4m3_to_float(uint8_t code) {
    __nv_fp8_e4m3 v;
    v.__x = code;
    return static_cast<float>(v);
}

__device__ __forceinline__ float load_float(const void *base, int dt, int64_t off) {
    if (dt == SPD_F32) return static_cast<const float *>(base)[off];
    if (dt == SPD_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[off]);
    if (dt == SPD_E4M3) return e4m3_to_float(static_cast<const uint8_t *>(base)[off]);
    return __half2float(static_cast<const __half *>(base)[off]);
}

// Element `off` of a K/V cache of dtype kv_dt (E4M3 or BF16) as fp32.
__device__ __forceinline__ float kv_value(const uint8_t *base, int kv_dt, int64_t off) {
    if (kv_dt == SPD_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[off]);
    return e4m3_to_float(base[off]);
}

// seq_len of query token t clipped to [0, NB*128]; 0 when its request row is
// outside the table.
__device__ __forceinline__ int64_t token_limit(const int32_t *ri, int64_t ri_s0,
                                               const int32_t *sl, int64_t sl_s0,
                                               int t, int R, int NB, int *row) {
    int r = ri[t * ri_s0];
    int64_t L = sl[t * sl_s0];
    *row = r;
    if (r < 0 || r >= R || L <= 0) return 0;
    int64_t cap = static_cast<int64_t>(NB) * kBlock;
    return L < cap ? L : cap;
}

}  // namespace spd
