// sdpa.cu -- dense GQA attention with a causal flag ("Kernel ABI" --
// attention.sdpa).
//
// Flash-style single pass over key tiles with an online softmax, fp32
// throughout on the CUDA cores.  A CTA takes 64 query rows -- (token, q head)
// pairs of one kv head, token-major, so the G heads of a token that share K
// and V sit together -- and streams that kv head's keys through shared
// memory 64 at a time:
//   * the rows' queries are staged once, pre-multiplied by sm_scale * log2(e)
//     so that the logits come out in base-2 units for exp2f;
//   * each K tile is stored transposed (dim-major, pitch 65) so lane i reads
//     keys i and i + 32 of a dim without bank conflicts, and each V tile
//     key-major so lane i reads dims i, i + 32, ...;
//   * each of the 8 warps owns 8 rows: every K value a lane loads feeds 8
//     rows' dot products and every V value 8 rows' accumulators, and the
//     queries and probabilities are read as broadcast float4s;
//   * at head dim 128 two CTAs (16 warps) fit an SM's shared memory and
//     registers; 4 warps per CTA (8 per SM) left the FMA pipe 29% busy
//     against 43% with 8, the kernel being bound by shared-memory latency.
// Keys past a row's causal limit are masked to -inf; tiles that no row of
// the CTA can read are not loaded, and under the causal flag the CTAs with
// the most keys are scheduled first.
#include <math.h>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sdpa.cuh"
#include "spd.h"

namespace spd {

namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 8;
constexpr int kRows = kWarps * kRowsPerWarp;  // query rows per CTA
constexpr int kKeys = 64;                     // keys per tile (two per lane)
constexpr int kKsPitch = kKeys + 1;           // odd pitch: conflict-free transposed stores
constexpr float kLog2e = 1.4426950408889634f;

template <int NPL>
constexpr size_t smem_floats() {
    // Qs [kRows][DP] + Ks [DP][kKsPitch] + Vs [kKeys][DP] + Ps [kRows][kKeys]
    return static_cast<size_t>(32 * NPL) * (kRows + kKsPitch + kKeys) + kRows * kKeys;
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(__half x) { return __half2float(x); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Keys query token t may read: all S, or j <= t + S - T under the causal flag.
__device__ __forceinline__ int readable_keys(const SdpaArgs &a, int64_t t) {
    if (!a.causal) return a.S;
    const int64_t n = t + (static_cast<int64_t>(a.S) - a.T) + 1;
    return n < 0 ? 0 : (n > a.S ? a.S : static_cast<int>(n));
}

__device__ __forceinline__ void store_out(const SdpaArgs &a, int64_t off, float x) {
    if (a.out_dt == SPD_BF16)
        static_cast<__nv_bfloat16 *>(a.out)[off] = __float2bfloat16_rn(x);
    else if (a.out_dt == SPD_F16)
        static_cast<__half *>(a.out)[off] = __float2half_rn(x);
    else
        static_cast<float *>(a.out)[off] = x;
}

// NPL = head dims per lane (D <= 32 * NPL); TIn = element type of q, k, v.
template <int NPL, typename TIn>
__global__ void __launch_bounds__(kWarps * 32) sdpa_kernel(const SdpaArgs a) {
    constexpr int DP = 32 * NPL;  // padded head dim (zeros past D)
    extern __shared__ float4 smem4[];
    float *Qs = reinterpret_cast<float *>(smem4);
    float *Ks = Qs + kRows * DP;
    float *Vs = Ks + DP * kKsPitch;
    float *Ps = Vs + kKeys * DP;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.y;
    const int G = a.Hq / a.Hkv;
    const int64_t n_rows = static_cast<int64_t>(a.T) * G;
    const int64_t tile = a.causal ? static_cast<int64_t>(gridDim.x - 1 - blockIdx.x) : blockIdx.x;
    const int64_t row0 = tile * kRows;
    const TIn *q = static_cast<const TIn *>(a.q);
    const TIn *k = static_cast<const TIn *>(a.k);
    const TIn *v = static_cast<const TIn *>(a.v);

    // stage the CTA's query rows, scaled into base-2 logit units
    const float qscale = a.sm_scale * kLog2e;
    for (int e = tid; e < kRows * DP; e += kWarps * 32) {
        const int r = e / DP, d = e % DP;
        const int64_t row = row0 + r;
        float x = 0.f;
        if (row < n_rows && d < a.D) {
            const int64_t t = row / G;
            const int64_t g = static_cast<int64_t>(h) * G + row % G;
            x = to_f(q[t * a.q_s0 + g * a.q_s1 + d * a.q_s2]) * qscale;
        }
        Qs[e] = x;
    }

    // readable keys of this warp's rows, of the warp and of the CTA (the
    // last row of a range has the largest token index)
    int lim[kRowsPerWarp];
    int warp_lim = 0;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int64_t row = row0 + warp * kRowsPerWarp + i;
        lim[i] = row < n_rows ? readable_keys(a, row / G) : 0;
        warp_lim = max(warp_lim, lim[i]);
    }
    const int64_t last_row = min(row0 + kRows, n_rows) - 1;
    const int cta_lim = last_row >= row0 ? readable_keys(a, last_row / G) : 0;

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][NPL];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < NPL; ++c) acc[i][c] = 0.f;
    }
    float *P = Ps + warp * kRowsPerWarp * kKeys;
    const float *Qw = Qs + warp * kRowsPerWarp * DP;

    for (int kt = 0; kt < cta_lim; kt += kKeys) {
        __syncthreads();  // the previous tile is consumed (first pass: Qs is staged)
        for (int e = tid; e < kKeys * DP; e += kWarps * 32) {
            const int j = e / DP, d = e % DP;
            const int key = kt + j;
            float kx = 0.f, vx = 0.f;
            if (key < a.S && d < a.D) {
                kx = to_f(k[key * a.k_s0 + static_cast<int64_t>(h) * a.k_s1 + d * a.k_s2]);
                vx = to_f(v[key * a.v_s0 + static_cast<int64_t>(h) * a.v_s1 + d * a.v_s2]);
            }
            Ks[d * kKsPitch + j] = kx;
            Vs[j * DP + d] = vx;
        }
        __syncthreads();
        if (kt >= warp_lim) continue;  // warp-uniform: no row of this warp reads the tile

        // logits of keys kt + lane and kt + lane + 32 for the warp's 8 rows
        float s0[kRowsPerWarp], s1[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) s0[i] = s1[i] = 0.f;
#pragma unroll 2
        for (int d = 0; d < DP; d += 4) {
            float k0[4], k1[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                k0[u] = Ks[(d + u) * kKsPitch + lane];
                k1[u] = Ks[(d + u) * kKsPitch + lane + 32];
            }
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                const float4 qv = *reinterpret_cast<const float4 *>(Qw + i * DP + d);
                s0[i] = fmaf(qv.x, k0[0], s0[i]);
                s0[i] = fmaf(qv.y, k0[1], s0[i]);
                s0[i] = fmaf(qv.z, k0[2], s0[i]);
                s0[i] = fmaf(qv.w, k0[3], s0[i]);
                s1[i] = fmaf(qv.x, k1[0], s1[i]);
                s1[i] = fmaf(qv.y, k1[1], s1[i]);
                s1[i] = fmaf(qv.z, k1[2], s1[i]);
                s1[i] = fmaf(qv.w, k1[3], s1[i]);
            }
        }

        // online softmax: new running maximum, rescale, probabilities to P
        const int j0 = kt + lane, j1 = kt + lane + 32;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const float z0 = j0 < lim[i] ? s0[i] : -INFINITY;
            const float z1 = j1 < lim[i] ? s1[i] : -INFINITY;
            const float mn = fmaxf(m[i], warp_max(fmaxf(z0, z1)));
            const float mref = mn == -INFINITY ? 0.f : mn;  // a row with nothing read yet stays at zero
            const float alpha = exp2f(m[i] - mref);
            const float p0 = exp2f(z0 - mref), p1 = exp2f(z1 - mref);
            m[i] = mn;
            l[i] = fmaf(l[i], alpha, p0 + p1);  // per-lane partial sum, reduced at the end
#pragma unroll
            for (int c = 0; c < NPL; ++c) acc[i][c] *= alpha;
            P[i * kKeys + lane] = p0;
            P[i * kKeys + lane + 32] = p1;
        }
        __syncwarp();

        // acc[i][c] += sum_j p[i][j] * V[j][lane + 32 c]
#pragma unroll 2
        for (int j = 0; j < kKeys; j += 4) {
            float4 p4[kRowsPerWarp];
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) p4[i] = *reinterpret_cast<const float4 *>(P + i * kKeys + j);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float vv[NPL];
#pragma unroll
                for (int c = 0; c < NPL; ++c) vv[c] = Vs[(j + u) * DP + lane + 32 * c];
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i) {
                    const float pu = u == 0 ? p4[i].x : u == 1 ? p4[i].y : u == 2 ? p4[i].z : p4[i].w;
#pragma unroll
                    for (int c = 0; c < NPL; ++c) acc[i][c] = fmaf(pu, vv[c], acc[i][c]);
                }
            }
        }
        __syncwarp();  // P is rewritten by the next tile
    }

    // normalise and store; a row that read no key writes zeros
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const float lt = warp_sum(l[i]);
        const int64_t row = row0 + warp * kRowsPerWarp + i;
        if (row >= n_rows) continue;
        const int64_t t = row / G;
        const int64_t g = static_cast<int64_t>(h) * G + row % G;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
        for (int c = 0; c < NPL; ++c) {
            const int d = lane + 32 * c;
            if (d < a.D) store_out(a, t * a.o_s0 + g * a.o_s1 + d * a.o_s2, acc[i][c] * inv);
        }
    }
}

template <int NPL, typename TIn>
cudaError_t launch_npl(const SdpaArgs &a, cudaStream_t stream) {
    const size_t smem = smem_floats<NPL>() * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(sdpa_kernel<NPL, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t n_rows = static_cast<int64_t>(a.T) * (a.Hq / a.Hkv);
    dim3 grid(static_cast<unsigned>((n_rows + kRows - 1) / kRows), static_cast<unsigned>(a.Hkv));
    sdpa_kernel<NPL, TIn><<<grid, kWarps * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_typed(const SdpaArgs &a, cudaStream_t stream) {
    if (a.D <= 32) return launch_npl<1, TIn>(a, stream);
    if (a.D <= 64) return launch_npl<2, TIn>(a, stream);
    if (a.D <= 128) return launch_npl<4, TIn>(a, stream);
    return launch_npl<8, TIn>(a, stream);
}

}  // namespace

cudaError_t launch_sdpa(const SdpaArgs &a, cudaStream_t stream) {
    if (a.in_dt == SPD_BF16) return launch_typed<__nv_bfloat16>(a, stream);
    if (a.in_dt == SPD_F16) return launch_typed<__half>(a, stream);
    return launch_typed<float>(a, stream);
}

}  // namespace spd
