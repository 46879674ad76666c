// plan.cu -- the one-CTA device planner of the tensor-core decode attention
// (see plan.cuh for what it builds).
#include "plan.cuh"
#include "tc_ptx.cuh"

namespace spd {
namespace {

constexpr int kWarps = kPlanThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

// Exclusive prefix sum of one value per thread over the CTA.
__device__ int block_excl_sum(int v, int *total, int *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = scratch[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += n;
        }
        scratch[lane] = w;
    }
    __syncthreads();
    const int before = (warp > 0) ? scratch[warp - 1] : 0;
    *total = scratch[kWarps - 1];
    __syncthreads();
    return before + incl - v;
}

// Exclusive prefix maximum (identity -1) of one value per thread over the CTA.
__device__ int block_excl_max(int v, int *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl = max(incl, n);
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = scratch[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w = max(w, n);
        }
        scratch[lane] = w;
    }
    __syncthreads();
    int before = (warp > 0) ? scratch[warp - 1] : -1;
    const int up = __shfl_up_sync(kFull, incl, 1);
    if (lane > 0) before = max(before, up);
    __syncthreads();
    return before;
}

// dynamic shared memory: request row and key limit of each query row, and a
// per-warp mask word for each block of the page table
constexpr size_t kPlanSmem = sizeof(int) * 2 * kPlanMaxT + sizeof(uint32_t) * kWarps * kPlanMaxNB;

// Query rows -> three E4M3 terms each (one warp per row, 4 elements a lane).
__device__ void convert_queries(const PlanArgs &a) {
    const int lane = threadIdx.x & 31;
    const int warps = kWarps * (gridDim.x - 1);
    const int64_t n_rows = static_cast<int64_t>(a.T) * a.Hq;
    uint8_t *qt = reinterpret_cast<uint8_t *>(a.ws + a.lay.qterms);
    float *cf = reinterpret_cast<float *>(a.ws + a.lay.cfac);
    for (int64_t row = (blockIdx.x - 1) * kWarps + (threadIdx.x >> 5); row < n_rows; row += warps) {
        const int64_t t = row / a.Hq, hq = row % a.Hq;
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = load_float(a.q, a.q_dt, t * a.q_s0 + hq * a.q_s1 + (lane * 4 + e) * a.q_s2);
        float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        float scale = 1.f;
        if (amax > 0.f && amax < INFINITY) {
            int ex;
            frexpf(amax, &ex);
            scale = ldexpf(1.f, 8 - ex);  // amax * scale in [128, 256)
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] *= scale;
#pragma unroll
        for (int term = 0; term < kQueryTerms; ++term) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[e] = tc::round4(x[e]);
                x[e] -= v[e];
            }
            *reinterpret_cast<uint32_t *>(qt + (term * n_rows + row) * 128 + lane * 4) =
                tc::pack2x16(tc::f32x2_to_e4m3x2(v[1], v[0]), tc::f32x2_to_e4m3x2(v[3], v[2]));
        }
        if (lane == 0) cf[row] = a.zscale / scale;
    }
}

__device__ void plan_body(const PlanArgs &a);

__global__ void __launch_bounds__(kPlanThreads, 1) prepare_kernel(PlanArgs a) {
    if (blockIdx.x == 0)
        plan_body(a);
    else
        convert_queries(a);
}

__device__ void plan_body(const PlanArgs &a) {
    extern __shared__ int plan_smem[];
    int *s_r = plan_smem;
    int *s_L = plan_smem + kPlanMaxT;
    uint32_t *s_mask_all = reinterpret_cast<uint32_t *>(plan_smem + 2 * kPlanMaxT);
    __shared__ int scratch[32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(a.ws + a.lay.header);
    PlanGroup *groups = reinterpret_cast<PlanGroup *>(a.ws + a.lay.groups);
    PlanPair *pairs = reinterpret_cast<PlanPair *>(a.ws + a.lay.pairs);
    PlanEntry *lists = reinterpret_cast<PlanEntry *>(a.ws + a.lay.lists);
    PlanUnit *units = reinterpret_cast<PlanUnit *>(a.ws + a.lay.units);
    int32_t *counters = reinterpret_cast<int32_t *>(a.ws + a.lay.counters);

    // ---- per-row request and key limit
    const int T = a.T;
    const int items = (T + kPlanThreads - 1) / kPlanThreads;
    const int t_begin = tid * items, t_end = min(T, t_begin + items);
    for (int t = t_begin; t < t_end; ++t) {
        int r;
        s_L[t] = static_cast<int>(token_limit(a.ri, a.ri_s0, a.sl, a.sl_s0, t, a.R, a.NB, &r));
        s_r[t] = r;
    }
    __syncthreads();

    // ---- groups: runs of equal req_idx, cut every gmax rows from the run start
    int local_start = -1;
    for (int t = t_begin; t < t_end; ++t)
        if (t == 0 || s_r[t] != s_r[t - 1]) local_start = t;
    const int run_before = block_excl_max(local_start, scratch);
    int run_start = run_before, n_gs = 0;
    for (int t = t_begin; t < t_end; ++t) {
        if (t == 0 || s_r[t] != s_r[t - 1]) run_start = t;
        n_gs += ((t - run_start) % a.gmax) == 0;
    }
    int n_groups;
    int g = block_excl_sum(n_gs, &n_groups, scratch);
    run_start = run_before;
    for (int t = t_begin; t < t_end; ++t) {
        if (t == 0 || s_r[t] != s_r[t - 1]) run_start = t;
        if (((t - run_start) % a.gmax) == 0) {
            groups[g].t0 = t;
            groups[g].r = s_r[t];
            ++g;
        }
    }
    __syncthreads();
    // group sizes from consecutive starts (groups[] written above by this CTA)
    __threadfence_block();
    for (int gg = tid; gg < n_groups; gg += kPlanThreads) {
        const int t0 = groups[gg].t0;
        const int t1 = (gg + 1 < n_groups) ? groups[gg + 1].t0 : T;
        groups[gg].nt = t1 - t0;
    }
    __syncthreads();

    // ---- block list of every (group, kv head) pair
    const bool shared_sel = (a.tk == nullptr) || (a.tk_s0 == 0);
    const int heads_built = shared_sel ? 1 : a.Hkv;
    const int n_pairs = n_groups * a.Hkv;
    for (int item = warp; item < n_groups * heads_built; item += kWarps) {
        const int gg = item / heads_built, h = item % heads_built;
        const int t0 = groups[gg].t0, nt = groups[gg].nt, r = groups[gg].r;
        uint32_t *m = s_mask_all + warp * kPlanMaxNB;
        for (int b = lane; b < a.NB; b += 32) m[b] = 0;
        __syncwarp();
        if (a.tk == nullptr) {
            for (int b = lane; b < a.NB; b += 32) {
                uint32_t bits = 0;
                for (int j = 0; j < nt; ++j) bits |= static_cast<uint32_t>(b * kBlock < s_L[t0 + j]) << j;
                m[b] = bits;
            }
        } else {
            for (int j = 0; j < nt; ++j) {
                const int t = t0 + j, L = s_L[t];
                for (int k = lane; k < a.K; k += 32) {
                    const int b = a.tk[h * a.tk_s0 + t * a.tk_s1 + k * a.tk_s2];
                    if (b >= 0 && b < a.NB && b * kBlock < L) atomicOr(&m[b], 1u << j);
                }
            }
        }
        __syncwarp();
        const int list = (gg * a.Hkv + h) * a.NB;
        int count = 0;
        for (int b0 = 0; b0 < a.NB; b0 += 32) {
            const int b = b0 + lane;
            uint32_t bits = (b < a.NB) ? m[b] : 0u;
            int page = -1;
            if (bits) {
                page = a.bt[static_cast<int64_t>(r) * a.bt_s0 + static_cast<int64_t>(b) * a.bt_s1];
                if (page < 0 || page >= a.P) bits = 0;
            }
            const unsigned keep = __ballot_sync(kFull, bits != 0);
            if (bits) {
                PlanEntry e;
                e.page = page;
                e.block = static_cast<uint16_t>(b);
                e.mask = static_cast<uint16_t>(bits);
                lists[list + count + __popc(keep & ((1u << lane) - 1))] = e;
            }
            count += __popc(keep);
        }
        if (lane == 0) {
            if (shared_sel) {
                for (int hh = 0; hh < a.Hkv; ++hh) {
                    pairs[gg * a.Hkv + hh].list = list;
                    pairs[gg * a.Hkv + hh].n_blocks = count;
                }
            } else {
                pairs[gg * a.Hkv + h].list = list;
                pairs[gg * a.Hkv + h].n_blocks = count;
            }
        }
        __syncwarp();
    }
    __syncthreads();
    __threadfence_block();

    // ---- units.  Chunk c = total blocks / CTAs (at least 4; a little more
    // when that fits every unit in one wave): each pair's list is cut into
    // full chunks of c blocks and a remainder.  The unit
    // table holds the full chunks first (pair order), then the remainders
    // and unsplit pairs by decreasing size, so the dynamic scheduler claims
    // the longest work first.
    int blocks_local = 0;
    for (int p = tid; p < n_pairs; p += kPlanThreads) blocks_local += pairs[p].n_blocks;
    int total_blocks;
    block_excl_sum(blocks_local, &total_blocks, scratch);
    int chunk = max(4, (total_blocks + a.num_ctas - 1) / max(1, a.num_ctas));
    // One wave when it costs little: the warps try chunk, chunk+1, ... (up to
    // a quarter more) at once and the smallest whose unit count fits the grid
    // is taken -- every CTA then runs one unit, instead of a few CTAs running
    // a second one after everybody else.
    {
        __shared__ int s_best;
        if (tid == 0) s_best = 0x7fffffff;
        __syncthreads();
        const int c = chunk + warp;
        if (c <= kPlanMaxNB && 4 * c <= 5 * chunk + 4) {
            int cnt = 0;
            for (int p = lane; p < n_pairs; p += 32) cnt += max(1, (pairs[p].n_blocks + c - 1) / c);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
            if (lane == 0 && cnt <= a.num_ctas) atomicMin(&s_best, c);
        }
        __syncthreads();
        if (s_best != 0x7fffffff) chunk = s_best;
        __syncthreads();
    }
    int *hist = reinterpret_cast<int *>(s_mask_all);  // [chunk + 1] remainder-size bins (mask words are done)
    for (int attempt = 0; attempt < 24; ++attempt) {
        int nu = 0, rows = 0;
        for (int p = tid; p < n_pairs; p += kPlanThreads) {
            const int n = pairs[p].n_blocks;
            const int u = max(1, (n + chunk - 1) / chunk);
            nu += u;
            if (u > 1) rows += u * groups[p / a.Hkv].nt * a.G;
        }
        int tot_u, tot_rows;
        block_excl_sum(nu, &tot_u, scratch);
        block_excl_sum(rows, &tot_rows, scratch);
        if (tot_u <= a.lay.unit_cap && tot_rows <= a.lay.rows_cap) break;
        chunk *= 2;
    }
    chunk = min(chunk, kPlanMaxNB);
    for (int i = tid; i <= chunk; i += kPlanThreads) hist[i] = 0;
    __syncthreads();
    // full chunks, split rows and the size of each pair's last unit
    int n_full = 0, rows = 0;
    for (int p = tid; p < n_pairs; p += kPlanThreads) {
        const int n = pairs[p].n_blocks;
        const int u = max(1, (n + chunk - 1) / chunk);
        const int last = n - (u - 1) * chunk;  // 1..chunk, or 0 for an empty pair
        n_full += (last == chunk) ? u : u - 1;
        if (u > 1) rows += u * groups[p / a.Hkv].nt * a.G;
        if (last < chunk) atomicAdd(&hist[last], 1);
    }
    int tot_full, tot_rows;
    int f_off = block_excl_sum(n_full, &tot_full, scratch);
    int r_off = block_excl_sum(rows, &tot_rows, scratch);
    // bins in decreasing size: start of bin s = tot_full + units in bins > s
    // (thread i holds bin chunk-1-i; chunk <= 256 < kPlanThreads)
    {
        const int bin = chunk - 1 - tid;
        const int n = (bin >= 0) ? hist[bin] : 0;
        int n_rem;
        const int before = block_excl_sum(n, &n_rem, scratch);
        if (bin >= 0) hist[bin] = tot_full + before;
        if (tid == 0) hist[chunk] = tot_full + n_rem;  // total units
    }
    __syncthreads();
    const int tot_u = hist[chunk];
    for (int p = tid; p < n_pairs; p += kPlanThreads) {
        const int n = pairs[p].n_blocks;
        const int u = max(1, (n + chunk - 1) / chunk);
        const int last = n - (u - 1) * chunk;
        const PlanGroup gr = groups[p / a.Hkv];
        const int rows_per_unit = gr.nt * a.G;
        pairs[p].unit0 = f_off;
        pairs[p].n_units = u;
        for (int c = 0; c < u; ++c) {
            PlanUnit un;
            un.entry = pairs[p].list + c * chunk;
            un.count = (c + 1 < u) ? chunk : last;
            un.part_row = (u > 1) ? r_off + c * rows_per_unit : -1;
            un.pair = p;
            un.t0 = gr.t0;
            un.nt = static_cast<int16_t>(gr.nt);
            un.h = static_cast<int16_t>(p % a.Hkv);
            un.part_base = (u > 1) ? r_off : -1;
            un.n_split = u;
            const int slot = (un.count == chunk) ? f_off++ : atomicAdd(&hist[un.count], 1);
            units[slot] = un;
        }
        if (u > 1) r_off += u * rows_per_unit;
        counters[p] = 0;
    }
    if (tid == 0) {
        hdr->status = 0;
        hdr->n_groups = n_groups;
        hdr->n_pairs = n_pairs;
        hdr->n_units = tot_u;
        hdr->chunk = chunk;
        hdr->partial_rows = tot_rows;
        hdr->gmax = a.gmax;
        hdr->next_unit = 0;
    }
}

}  // namespace

cudaError_t launch_prepare(const PlanArgs &a, int conv_ctas, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(prepare_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kPlanSmem));
        if (e != cudaSuccess) return e;
        attr_set[dev & 63] = true;
    }
    prepare_kernel<<<1 + conv_ctas, kPlanThreads, kPlanSmem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace spd
