// generic_kernels.cu -- the general-layout CUDA kernels of all three stages.
//
// These accept any strides and every shape of the capability domain.  They
// are the path for shapes the specialised kernels do not cover (for example
// head dim 64, fp32 queries) and the first correct implementation the
// specialised ones are checked against.  Plain CUDA-core fp32 arithmetic.
#include <math.h>

#include "spd_internal.cuh"

namespace spd {

namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------------ stage 1
// "Kernel ABI" -- attention.msa_block_score.  One warp per (h, t, block b);
// lane i takes tokens i, i+32, i+64, i+96 of the block.
constexpr int kScoreWarps = 4;

__global__ void __launch_bounds__(kScoreWarps * 32)
score_generic_kernel(ScoreArgs a) {
    extern __shared__ float qs[];  // [Di]
    const int t = blockIdx.x, h = blockIdx.z;
    for (int d = threadIdx.x; d < a.Di; d += blockDim.x)
        qs[d] = load_float(a.q, a.q_dt, t * a.q_s0 + h * a.q_s1 + d * a.q_s2);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y * kScoreWarps + warp;
    if (b >= a.NB) return;

    int r;
    const int64_t L = token_limit(a.ri, a.ri_s0, a.sl, a.sl_s0, t, a.R, a.NB, &r);
    float best = -INFINITY;
    if (static_cast<int64_t>(b) * kBlock < L) {
        const int64_t page = a.bt[r * a.bt_s0 + b * a.bt_s1];
        if (page >= 0 && page < a.P) {
            for (int i = lane; i < kBlock; i += 32) {
                if (static_cast<int64_t>(b) * kBlock + i >= L) break;
                const int64_t slot = page * kBlock + i;
                float dot = 0.f;
                for (int d = 0; d < a.Di; ++d)
                    dot = fmaf(qs[d], load_float(a.k, a.k_dt, slot * a.k_s0 + d * a.k_s2), dot);
                best = fmaxf(best, dot);
            }
        }
    }
    best = warp_max(best);
    if (lane == 0)
        a.out[h * a.o_s0 + t * a.o_s1 + b * a.o_s2] = (best == -INFINITY) ? -INFINITY : best * a.idx_scale;
}

// ------------------------------------------------------------------ stage 2
// Top-k by rank: a candidate's rank is the number of candidates ordered
// before it (higher score, or equal score and lower id); rank < K lands in
// output position rank.  One warp per row.
constexpr int kSelectWarps = 4;

__device__ __forceinline__ bool is_candidate(float v) { return !isnan(v) && v != -INFINITY; }

__global__ void __launch_bounds__(kSelectWarps * 32)
select_generic_kernel(SelectArgs a) {
    extern __shared__ float rows[];  // [kSelectWarps][NB]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kSelectWarps + warp;
    if (row >= a.Hi * a.T) return;
    const int h = row / a.T, t = row % a.T;
    float *s = rows + warp * a.NB;
    for (int b = lane; b < a.NB; b += 32) s[b] = a.s[h * a.s_s0 + t * a.s_s1 + b * a.s_s2];
    __syncwarp();

    int n_cand = 0;
    for (int i = lane; i < a.NB; i += 32) {
        const float vi = s[i];
        if (!is_candidate(vi)) continue;
        ++n_cand;
        int rank = 0;
        for (int j = 0; j < a.NB; ++j) {
            const float vj = s[j];
            rank += is_candidate(vj) && (vj > vi || (vj == vi && j < i));
        }
        if (rank < a.K) a.o[h * a.o_s0 + t * a.o_s1 + rank * a.o_s2] = i;
    }
    n_cand = warp_sum(n_cand);
    for (int k = n_cand + lane; k < a.K; k += 32) a.o[h * a.o_s0 + t * a.o_s1 + k * a.o_s2] = -1;
}

// The same ranks with the row held once per warp in shared memory (padded to
// a multiple of 4 with -inf, non-candidates stored as -inf) and compared in
// registers: each lane owns up to 8 candidates per pass and streams the row
// as broadcast float4 reads, so a comparison is a few ALU instructions.
constexpr int kSelectPer = 4;

__global__ void __launch_bounds__(kSelectWarps * 32)
select_rank_kernel(SelectArgs a, int nb4) {
    extern __shared__ float4 rows4[];  // [kSelectWarps][nb4]
    // launched with programmatic stream serialisation (see launch_select_rank)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kSelectWarps + warp;
    if (row >= a.Hi * a.T) return;
    const int h = row / a.T, t = row % a.T;
    float4 *s4 = rows4 + warp * nb4;
    float *s = reinterpret_cast<float *>(s4);
    int n_cand = 0;
    for (int b = lane; b < 4 * nb4; b += 32) {
        float v = -INFINITY;
        if (b < a.NB) {
            v = a.s[h * a.s_s0 + t * a.s_s1 + b * a.s_s2];
            if (!is_candidate(v)) v = -INFINITY;
        }
        n_cand += v != -INFINITY;
        s[b] = v;
    }
    __syncwarp();
    int32_t *o = a.o + h * a.o_s0 + t * a.o_s1;
    for (int base = 0; base < a.NB; base += 32 * kSelectPer) {
        float vi[kSelectPer];
        int ii[kSelectPer], rank[kSelectPer];
#pragma unroll
        for (int p = 0; p < kSelectPer; ++p) {
            ii[p] = base + p * 32 + lane;
            vi[p] = ii[p] < a.NB ? s[ii[p]] : -INFINITY;
            rank[p] = 0;
        }
        for (int j4 = 0; j4 < nb4; ++j4) {
            const float4 v = s4[j4];
            const float vj[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = 4 * j4 + e;
#pragma unroll
                for (int p = 0; p < kSelectPer; ++p)
                    rank[p] += (vj[e] > vi[p]) | ((vj[e] == vi[p]) & (j < ii[p]));
            }
        }
#pragma unroll
        for (int p = 0; p < kSelectPer; ++p)
            if (vi[p] != -INFINITY && rank[p] < a.K) o[rank[p] * a.o_s2] = ii[p];
    }
    n_cand = warp_sum(n_cand);
    for (int k = n_cand + lane; k < a.K; k += 32) o[k * a.o_s2] = -1;
}

// Top-k by sorting, for rows of at most 256 blocks.  Each score becomes a
// 64-bit key ordered by score (descending), then block id (ascending) -- the
// order the ranks above count in -- with non-candidates after every
// candidate; one warp sorts the row's 32E keys with a bitonic network, E
// keys per lane (lane l holds keys lE .. lE+E-1: partners E or more apart
// are exchanged by shuffles, nearer ones inside the lane).  The first K keys
// are the selection in output order.  About 28 (E = 4) to 36 (E = 8)
// exchange steps of a few instructions per key replace the NB^2 comparisons
// of the rank kernel.
constexpr uint64_t kNoKey = ~0ull;

__device__ __forceinline__ uint64_t order_key(float v, uint32_t b) {
    if (!is_candidate(v)) return kNoKey;
    if (v == 0.f) v = 0.f;  // -0 and +0 are equal scores
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // increasing in v
    return (static_cast<uint64_t>(~u) << 32) | b;      // decreasing in v, then increasing in b
}

template <int E>
__device__ __forceinline__ void warp_bitonic_sort(uint64_t (&x)[E], int lane) {
    constexpr int M = 32 * E;
#pragma unroll
    for (int k = 2; k <= M; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= E) {
                const int lj = j / E;
                const bool lower = (lane & lj) == 0;  // this lane holds the lower index of each pair
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const bool up = ((lane * E + e) & k) == 0;
                    const uint64_t y = __shfl_xor_sync(0xffffffffu, x[e], lj);
                    const bool lt = x[e] < y;
                    x[e] = (lower == up) ? (lt ? x[e] : y) : (lt ? y : x[e]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    if (e & j) continue;
                    const bool up = ((lane * E + e) & k) == 0;
                    const uint64_t p = x[e], q = x[e + j];
                    const bool swap = up ? (q < p) : (p < q);
                    x[e] = swap ? q : p;
                    x[e + j] = swap ? p : q;
                }
            }
        }
    }
}

template <int E>
__global__ void __launch_bounds__(kSelectWarps * 32)
select_sort_kernel(SelectArgs a) {
    // launched with programmatic stream serialisation (see launch_select_fast)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kSelectWarps + warp;
    if (row >= a.Hi * a.T) return;
    const int h = row / a.T, t = row % a.T;
    const float *s = a.s + h * a.s_s0 + t * a.s_s1;
    uint64_t key[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int b = lane * E + e;
        key[e] = (b < a.NB) ? order_key(s[b * a.s_s2], static_cast<uint32_t>(b)) : kNoKey;
    }
    warp_bitonic_sort<E>(key, lane);
    int32_t *o = a.o + h * a.o_s0 + t * a.o_s1;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = lane * E + e;
        if (i < a.K) o[i * a.o_s2] = (key[e] == kNoKey) ? -1 : static_cast<int32_t>(static_cast<uint32_t>(key[e]));
    }
    for (int i = 32 * E + lane; i < a.K; i += 32) o[i * a.o_s2] = -1;
}

// ------------------------------------------------------------------ stage 3
// "Kernel ABI" -- attention.decode.  One CTA per (query token t, kv head h)
// serves the G = Hq/Hkv q heads of that kv head.  Blocks are visited in
// ascending id; per block, thread i scores token i for every q head, then an
// online softmax (running max, rescaled sums) folds the block in, and thread
// d accumulates value column d.
constexpr int kAttnThreads = kBlock;
constexpr int kDPerThread = kMaxD / kAttnThreads;

__global__ void __launch_bounds__(kAttnThreads)
attention_generic_kernel(AttnArgs a) {
    __shared__ float qs[kMaxGroup][kMaxD];
    __shared__ float ps[kMaxGroup][kBlock];
    __shared__ float m_run[kMaxGroup], alpha_s[kMaxGroup], l_run[kMaxGroup];
    __shared__ unsigned char selected[kMaxNB];

    const int t = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int G = a.Hq / a.Hkv;

    for (int i = tid; i < G * a.D; i += blockDim.x) {
        const int g = i / a.D, d = i % a.D;
        qs[g][d] = load_float(a.q, a.q_dt, t * a.q_s0 + (h * G + g) * a.q_s1 + d * a.q_s2);
    }
    for (int b = tid; b < a.NB; b += blockDim.x) selected[b] = (a.tk == nullptr);
    if (tid < kMaxGroup) {
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.f;
    }
    __syncthreads();
    if (a.tk != nullptr) {
        for (int k = tid; k < a.K; k += blockDim.x) {
            const int b = a.tk[h * a.tk_s0 + t * a.tk_s1 + k * a.tk_s2];
            if (b >= 0 && b < a.NB) selected[b] = 1;
        }
    }
    __syncthreads();

    int r;
    const int64_t L = token_limit(a.ri, a.ri_s0, a.sl, a.sl_s0, t, a.R, a.NB, &r);
    const float zscale = a.sm_scale * a.k_scale;

    float acc[kDPerThread][kMaxGroup];
#pragma unroll
    for (int c = 0; c < kDPerThread; ++c)
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) acc[c][g] = 0.f;

    for (int b = 0; b < a.NB && static_cast<int64_t>(b) * kBlock < L; ++b) {
        if (!selected[b]) continue;
        const int64_t page = a.bt[r * a.bt_s0 + b * a.bt_s1];
        if (page < 0 || page >= a.P) continue;
        const int64_t base = page * kBlock;

        // logits of token tid for every q head
        const bool valid = static_cast<int64_t>(b) * kBlock + tid < L;
        if (valid) {
            const int64_t krow = (base + tid) * a.k_s0 + h * a.k_s1;
            float z[kMaxGroup];
#pragma unroll
            for (int g = 0; g < kMaxGroup; ++g) z[g] = 0.f;
            for (int d = 0; d < a.D; ++d) {
                const float kd = kv_value(a.k, a.kv_dt, krow + d);
#pragma unroll
                for (int g = 0; g < kMaxGroup; ++g)
                    if (g < G) z[g] = fmaf(qs[g][d], kd, z[g]);
            }
#pragma unroll
            for (int g = 0; g < kMaxGroup; ++g)
                if (g < G) ps[g][tid] = z[g] * zscale;
        } else {
            for (int g = 0; g < G; ++g) ps[g][tid] = -INFINITY;
        }
        __syncthreads();

        // block maximum and rescale factor per q head
        if (tid < G) {
            float bm = -INFINITY;
            for (int i = 0; i < kBlock; ++i) bm = fmaxf(bm, ps[tid][i]);
            const float m_new = fmaxf(m_run[tid], bm);
            alpha_s[tid] = (m_run[tid] == -INFINITY) ? 0.f : expf(m_run[tid] - m_new);
            m_run[tid] = m_new;
        }
        __syncthreads();

        for (int g = 0; g < G; ++g)
            ps[g][tid] = valid ? expf(ps[g][tid] - m_run[g]) : 0.f;
        __syncthreads();

        if (tid < G) {
            float s = 0.f;
            for (int i = 0; i < kBlock; ++i) s += ps[tid][i];
            l_run[tid] = l_run[tid] * alpha_s[tid] + s;
        }
        // only the block's valid prefix is read: the page tail past seq_len
        // may hold anything, and 0 * NaN would poison the sum
        const int n_valid = static_cast<int>(min(static_cast<int64_t>(kBlock), L - static_cast<int64_t>(b) * kBlock));
#pragma unroll
        for (int c = 0; c < kDPerThread; ++c) {
            const int d = tid + c * kAttnThreads;
            if (d >= a.D) continue;
            float part[kMaxGroup];
#pragma unroll
            for (int g = 0; g < kMaxGroup; ++g) part[g] = 0.f;
            for (int i = 0; i < n_valid; ++i) {
                const float vd = kv_value(a.v, a.kv_dt, (base + i) * a.v_s0 + h * a.v_s1 + d);
#pragma unroll
                for (int g = 0; g < kMaxGroup; ++g)
                    if (g < G) part[g] = fmaf(ps[g][i], vd, part[g]);
            }
#pragma unroll
            for (int g = 0; g < kMaxGroup; ++g)
                if (g < G) acc[c][g] = acc[c][g] * alpha_s[g] + part[g];
        }
        __syncthreads();
    }

#pragma unroll
    for (int c = 0; c < kDPerThread; ++c) {
        const int d = tid + c * kAttnThreads;
        if (d >= a.D) continue;
        for (int g = 0; g < G; ++g) {
            const float l = l_run[g];
            const float o = (l > 0.f) ? acc[c][g] * a.v_scale / l : 0.f;
            a.out[t * a.o_s0 + (h * G + g) * a.o_s1 + d * a.o_s2] = __float2bfloat16_rn(o);
        }
    }
}

}  // namespace

cudaError_t launch_score_generic(const ScoreArgs &a, cudaStream_t stream) {
    dim3 grid(a.T, (a.NB + kScoreWarps - 1) / kScoreWarps, a.Hi);
    score_generic_kernel<<<grid, kScoreWarps * 32, a.Di * sizeof(float), stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_select_fast(const SelectArgs &a, cudaStream_t stream) {
    if (a.NB > 256) return launch_select_rank(a, stream);
    const int rows = a.Hi * a.T;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows + kSelectWarps - 1) / kSelectWarps);
    cfg.blockDim = dim3(kSelectWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    // programmatic stream serialisation, as for the rank kernel
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.NB <= 32) return cudaLaunchKernelEx(&cfg, select_sort_kernel<1>, a);
    if (a.NB <= 64) return cudaLaunchKernelEx(&cfg, select_sort_kernel<2>, a);
    if (a.NB <= 128) return cudaLaunchKernelEx(&cfg, select_sort_kernel<4>, a);
    return cudaLaunchKernelEx(&cfg, select_sort_kernel<8>, a);
}

cudaError_t launch_select_rank(const SelectArgs &a, cudaStream_t stream) {
    const int rows = a.Hi * a.T;
    const int nb4 = (a.NB + 3) / 4;
    dim3 grid((rows + kSelectWarps - 1) / kSelectWarps);
    // programmatic stream serialisation: the kernel may be scheduled while
    // the score kernel drains and waits for it before reading the sheet
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kSelectWarps * 32);
    cfg.dynamicSmemBytes = kSelectWarps * nb4 * sizeof(float4);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, select_rank_kernel, a, nb4);
}

cudaError_t launch_select_generic(const SelectArgs &a, cudaStream_t stream) {
    const int rows = a.Hi * a.T;
    dim3 grid((rows + kSelectWarps - 1) / kSelectWarps);
    select_generic_kernel<<<grid, kSelectWarps * 32, kSelectWarps * a.NB * sizeof(float), stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attention_generic(const AttnArgs &a, cudaStream_t stream) {
    dim3 grid(a.T, a.Hkv);
    attention_generic_kernel<<<grid, kAttnThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace spd
