// plan.cu -- the device planner of the tensor-core decode attention and the
// query conversion that shares its unit launch (see plan.cuh for what the
// plan holds).
//
// The planner is latency-bound work on few SMs, so it is laid out for few
// dependent round trips and little code: the list kernel gives every list
// its own warp (topk_idx and the page table are each one round trip, all of
// a list's loads in flight together); the unit kernel runs on one CTA with
// its inputs staged in shared memory and one barrier per scan.
#include <algorithm>

#include "plan.cuh"
#include "tc_ptx.cuh"

namespace spd {
namespace {

constexpr int kWarps = kPlanThreads / 32;
constexpr unsigned kFull = 0xffffffffu;
// dynamic shared memory either planner kernel may take
constexpr int kPlanSmemMax = 160 * 1024;
constexpr int kVecs = 4;                  // topk_idx loads in flight per lane
constexpr int kChunks = kPlanMaxNB / 32;  // page-table loads in flight per lane
constexpr int kConvRows = 4;              // query rows per warp converted together

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Exclusive prefix sum over the CTA of one value per thread (thread order),
// with the total; one barrier.  `buf` (kWarps ints) is read after the
// barrier, so consecutive calls must alternate between two buffers.
__device__ int cta_scan(int v, int *total, int *buf) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) buf[warp] = incl;
    __syncthreads();
    const int w = (lane < kWarps) ? buf[lane] : 0;
    *total = warp_sum(w);
    return warp_sum(lane < warp ? w : 0) + incl - v;
}

// Query rows -> E4M3 terms (one warp per row, 4 elements a lane; kConvRows
// rows per warp with their loads issued together).  The row is scaled by a
// power of two so that its largest magnitude lies in [128, 256); each term is
// the remainder rounded to 4 significant bits.  bf16 queries need two terms
// (8 significant bits), other types get three.
template <int DT>
__device__ __forceinline__ float load_q(const void *q, int64_t off) {
    if (DT == SPD_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(q)[off]);
    if (DT == SPD_F16) return __half2float(static_cast<const __half *>(q)[off]);
    return static_cast<const float *>(q)[off];
}

template <int DT>
__device__ void convert_rows(const PlanArgs &a, int64_t first, int64_t warps) {
    constexpr int kT = (DT == SPD_BF16) ? 2 : kQueryTerms;
    const int lane = threadIdx.x & 31;
    const int64_t n_rows = static_cast<int64_t>(a.T) * a.Hq;
    uint8_t *qt = reinterpret_cast<uint8_t *>(a.ws + a.lay.qterms);
    float *cf = reinterpret_cast<float *>(a.ws + a.lay.cfac);
    for (int64_t base = first; base < n_rows; base += kConvRows * warps) {
        float x[kConvRows][4];
#pragma unroll
        for (int u = 0; u < kConvRows; ++u) {
            const int64_t row = base + u * warps;
            const int64_t t = row / a.Hq, hq = row - t * a.Hq;
            const int64_t off = t * a.q_s0 + hq * a.q_s1 + (lane * 4) * a.q_s2;
#pragma unroll
            for (int e = 0; e < 4; ++e) x[u][e] = (row < n_rows) ? load_q<DT>(a.q, off + e * a.q_s2) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kConvRows; ++u) {
            const int64_t row = base + u * warps;
            if (row >= n_rows) break;
            float amax = fmaxf(fmaxf(fabsf(x[u][0]), fabsf(x[u][1])), fmaxf(fabsf(x[u][2]), fabsf(x[u][3])));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
            float scale = 1.f;
            const uint32_t ebits = (__float_as_uint(amax) >> 23) & 0xFFu;  // biased exponent
            if (amax > 0.f && ebits != 0xFFu) {
                if (ebits >= 8u) {
                    scale = __uint_as_float((254u + 7u - ebits) << 23);  // 2^(7 - floor(log2 amax))
                } else {
                    int ex;
                    frexpf(amax, &ex);
                    scale = ldexpf(1.f, 8 - ex);
                }
            }
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = x[u][e] * scale;
#pragma unroll
            for (int term = 0; term < kT; ++term) {
                float r[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    r[e] = tc::round4(v[e]);
                    v[e] -= r[e];
                }
                *reinterpret_cast<uint32_t *>(qt + (term * n_rows + row) * 128 + lane * 4) =
                    tc::pack2x16(tc::f32x2_to_e4m3x2(r[1], r[0]), tc::f32x2_to_e4m3x2(r[3], r[2]));
            }
            if (lane == 0) cf[row] = a.zscale / scale;
        }
    }
}

__device__ void convert_queries(const PlanArgs &a, int first_cta) {
    const int64_t warps = static_cast<int64_t>(kWarps) * (gridDim.x - first_cta);
    const int64_t first = static_cast<int64_t>(blockIdx.x - first_cta) * kWarps + (threadIdx.x >> 5);
    if (a.q_dt == SPD_BF16)
        convert_rows<SPD_BF16>(a, first, warps);
    else if (a.q_dt == SPD_F16)
        convert_rows<SPD_F16>(a, first, warps);
    else
        convert_rows<SPD_F32>(a, first, warps);
}

// Shared memory of a list CTA: request and key limit per row, group starts,
// and one mask word per block for each warp.
__host__ __device__ inline size_t list_smem_bytes(int T, int NB) {
    return sizeof(int32_t) * (3 * static_cast<size_t>(T) + 8 + static_cast<size_t>(kWarps) * NB);
}

// Shared memory of the unit CTA: group starts and list lengths.
__host__ __device__ inline size_t unit_smem_bytes(int T, int hb) {
    return sizeof(int32_t) * (static_cast<size_t>(T) + 8 + static_cast<size_t>(T) * hb);
}

// Groups: runs of equal req_idx, cut every gmax rows from the run start.  A
// round covers kPlanThreads rows: the run start of a row is the last change
// at or before it (ballots within the warp, then the earlier warps' last
// changes, then the earlier rounds'), its group the count of group starts up
// to it.  Writes s_gt0[0..n_groups] (then T); returns n_groups.
__device__ int find_groups(const int32_t *s_r, int T, int gmax, int32_t *s_gt0, int (*buf)[kWarps]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lanes_le = (2u << lane) - 1u;
    int carry_run = 0, carry_g = 0;
    for (int base = 0; base < T; base += kPlanThreads) {
        const int t = base + tid;
        const bool valid = t < T;
        const bool change = valid && (t == 0 || s_r[t] != s_r[t - 1]);
        const unsigned bal = __ballot_sync(kFull, change);
        const unsigned below = bal & lanes_le;
        if (lane == 0) buf[0][warp] = bal ? base + 32 * warp + 31 - __clz(bal) : -1;
        __syncthreads();
        const int lc_warps = warp_max((lane < warp) ? buf[0][lane] : -1);
        const int lc_round = warp_max((lane < kWarps) ? buf[0][lane] : -1);
        const int run_start = below ? base + 32 * warp + 31 - __clz(below) : max(lc_warps, carry_run);
        const bool gs = valid && ((t - run_start) % gmax) == 0;
        const unsigned gbal = __ballot_sync(kFull, gs);
        if (lane == 0) buf[1][warp] = __popc(gbal);
        __syncthreads();
        const int w = (lane < kWarps) ? buf[1][lane] : 0;
        const int before = warp_sum((lane < warp) ? w : 0);
        if (gs) s_gt0[carry_g + before + __popc(gbal & lanes_le) - 1] = t;
        carry_run = max(carry_run, lc_round);
        carry_g += warp_sum(w);
    }
    if (tid == 0) s_gt0[carry_g] = T;
    __syncthreads();
    return carry_g;
}

// One list per warp: the union of the blocks its group's rows take (for
// sparse calls, those they selected; dense, every block below the key
// limit), ascending, with the row mask and page id of each.
__device__ void build_lists(const PlanArgs &a) {
    extern __shared__ int32_t plan_smem[];
    __shared__ int buf[2][kWarps];
    const int T = a.T, NB = a.NB, hb = a.heads_built;
    int32_t *s_r = plan_smem;
    int32_t *s_L = s_r + T;
    int32_t *s_gt0 = s_L + T;  // [T + 1]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t *m = reinterpret_cast<uint32_t *>(s_gt0 + T + 8) + warp * NB;

    for (int t = threadIdx.x; t < T; t += kPlanThreads) {
        int r;
        s_L[t] = static_cast<int>(token_limit(a.ri, a.ri_s0, a.sl, a.sl_s0, t, a.R, a.NB, &r));
        s_r[t] = r;
    }
    __syncthreads();
    const int n_groups = find_groups(s_r, T, a.gmax, s_gt0, buf);
    if (blockIdx.x == 0) {
        // the unit kernel reads the group starts
        int32_t *gstart = reinterpret_cast<int32_t *>(a.ws + a.lay.gstart);
        for (int g = threadIdx.x; g <= n_groups; g += kPlanThreads) gstart[g] = s_gt0[g];
        if (threadIdx.x == 0) reinterpret_cast<PlanHeader *>(a.ws + a.lay.header)->n_groups = n_groups;
    }

    PlanEntry *lists = reinterpret_cast<PlanEntry *>(a.ws + a.lay.lists);
    int32_t *lcount = reinterpret_cast<int32_t *>(a.ws + a.lay.lcount);
    const bool sparse = a.tk != nullptr;
    const bool vec = sparse && a.tk_s2 == 1 && (a.K % 4) == 0 && (a.tk_s1 % 4) == 0 && (a.tk_s0 % 4) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.tk) % 16) == 0;
    const int kv = vec ? 4 : 1, kq = max(1, a.K / kv);
    // lane -> (row, k vector) of its first load and the step between its loads
    const int j_first = lane / kq, k_first = lane % kq, j_step = 32 / kq, k_step = 32 % kq;
    const int n_items = n_groups * hb;
    for (int item = blockIdx.x * kWarps + warp; item < n_items; item += a.list_ctas * kWarps) {
        const int gg = item / hb, h = item % hb;
        const int t0 = s_gt0[gg], nt = s_gt0[gg + 1] - t0;
        for (int b = lane; b < NB; b += 32) {
            uint32_t bits = 0;
            if (!sparse)
                for (int j = 0; j < nt; ++j) bits |= static_cast<uint32_t>(b * kBlock < s_L[t0 + j]) << j;
            m[b] = bits;
        }
        __syncwarp();
        if (sparse) {
            const int nv = nt * (a.K / kv);
            int j = j_first, k = k_first;
            for (int v0 = lane; v0 < nv; v0 += kVecs * 32) {
                int4 x[kVecs];
                int jj[kVecs];
#pragma unroll
                for (int u = 0; u < kVecs; ++u) {
                    x[u] = make_int4(-1, -1, -1, -1);
                    jj[u] = j;
                    if (v0 + 32 * u < nv) {
                        const int32_t *src = a.tk + h * a.tk_s0 + (t0 + j) * a.tk_s1 + (k * kv) * a.tk_s2;
                        if (vec)
                            x[u] = __ldg(reinterpret_cast<const int4 *>(src));
                        else
                            x[u].x = __ldg(src);
                    }
                    k += k_step;
                    j += j_step;
                    if (k >= kq) {
                        k -= kq;
                        ++j;
                    }
                }
#pragma unroll
                for (int u = 0; u < kVecs; ++u) {
                    if (v0 + 32 * u >= nv) continue;
                    const int L = s_L[t0 + jj[u]];
                    const int bs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q < kv && bs[q] >= 0 && bs[q] < NB && bs[q] * kBlock < L) atomicOr(&m[bs[q]], 1u << jj[u]);
                }
            }
            __syncwarp();
        }
        // page ids of the taken blocks (all loads in flight), then compaction
        const int64_t row = static_cast<int64_t>(s_r[t0]) * a.bt_s0;
        uint32_t bits[kChunks];
        int page[kChunks];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            const int b = 32 * c + lane;
            bits[c] = (b < NB) ? m[b] : 0u;
            page[c] = bits[c] ? a.bt[row + static_cast<int64_t>(b) * a.bt_s1] : -1;
        }
        const int list = (gg * a.Hkv + h) * NB;
        int count = 0;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            if (32 * c >= NB) break;
            if (page[c] < 0 || page[c] >= a.P) bits[c] = 0;
            const unsigned keep = __ballot_sync(kFull, bits[c] != 0);
            if (bits[c]) {
                PlanEntry e;
                e.page = page[c];
                e.block = static_cast<uint16_t>(32 * c + lane);
                e.mask = static_cast<uint16_t>(bits[c]);
                lists[list + count + __popc(keep & ((1u << lane) - 1))] = e;
            }
            count += __popc(keep);
        }
        if (lane == 0) lcount[item] = count;
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kPlanThreads, 2) list_kernel(const __grid_constant__ PlanArgs a) {
    tc::pdl_wait();
    tc::pdl_trigger();
    build_lists(a);
}

// The unit table (one CTA).  Chunk c = total blocks / CTAs (at least 4; a little more
// when that fits every unit in one wave): each pair's list is cut into full
// chunks of c blocks and a remainder.  The table holds the full chunks first
// (pair order), then the remainders and unsplit pairs by decreasing size, so
// the dynamic scheduler claims the longest work first.  Each thread owns a
// contiguous range of pairs, so scans follow pair order.
__device__ void build_units(const PlanArgs &a);

// CTA 0 builds the unit table, the others convert the queries.
__global__ void __launch_bounds__(kPlanThreads, 2) unit_kernel(const __grid_constant__ PlanArgs a) {
    tc::pdl_wait();
    tc::pdl_trigger();
    if (blockIdx.x == 0)
        build_units(a);
    else
        convert_queries(a, 1);
}

__device__ void build_units(const PlanArgs &a) {
    extern __shared__ int32_t plan_smem[];
    __shared__ int buf[4][kWarps];
    __shared__ int hist[kPlanMaxNB + 1];
    __shared__ int s_best, s_fit0, s_ng;

    const int T = a.T, Hkv = a.Hkv, hb = a.heads_built;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t *s_gt0 = plan_smem;        // [T + 1]
    int32_t *s_cnt = plan_smem + T + 8;  // [T * hb]
    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(a.ws + a.lay.header);
    PlanUnit *units = reinterpret_cast<PlanUnit *>(a.ws + a.lay.units);
    int32_t *counters = reinterpret_cast<int32_t *>(a.ws + a.lay.counters);
    const int32_t *gstart = reinterpret_cast<const int32_t *>(a.ws + a.lay.gstart);
    const int32_t *lcount = reinterpret_cast<const int32_t *>(a.ws + a.lay.lcount);

    // inputs staged in shared memory (read up to their capacities, so no load
    // waits for the group count)
    if (tid == 0) {
        s_ng = hdr->n_groups;
        s_best = 0x7fffffff;
        s_fit0 = 0;
    }
    for (int i = tid; i <= T; i += kPlanThreads) s_gt0[i] = gstart[i];
    for (int i = tid; i < T * hb; i += kPlanThreads) s_cnt[i] = lcount[i];
    for (int i = tid; i <= kPlanMaxNB; i += kPlanThreads) hist[i] = 0;
    __syncthreads();
    const int n_groups = s_ng;
    const int n_pairs = n_groups * Hkv;
    const int ppt = (n_pairs + kPlanThreads - 1) / kPlanThreads;
    const int p_begin = min(n_pairs, tid * ppt), p_end = min(n_pairs, p_begin + ppt);
    auto count_of = [&](int p) { return s_cnt[hb == 1 ? p / Hkv : p]; };
    auto rows_of = [&](int p) { return (s_gt0[p / Hkv + 1] - s_gt0[p / Hkv]) * a.G; };
    int blocks_local = 0;
    for (int p = p_begin; p < p_end; ++p) blocks_local += count_of(p);
    int total_blocks;
    cta_scan(blocks_local, &total_blocks, buf[0]);
    const int chunk0 = min(kPlanMaxNB, max(4, (total_blocks + a.num_ctas - 1) / max(1, a.num_ctas)));
    // One wave when it costs little: chunk0 + i for i < 32 (two per warp, up
    // to a quarter more) are tried and the smallest whose unit count fits the
    // grid (and the unit and partial capacities) is taken -- every CTA then
    // runs one unit, instead of a few CTAs running a second one after
    // everybody else.
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        const int i = warp + kWarps * half;
        const int c = chunk0 + i;
        if (c <= kPlanMaxNB && (i == 0 || 4 * c <= 5 * chunk0 + 4)) {
            int nu = 0, rows = 0;
            for (int p = lane; p < n_pairs; p += 32) {
                const int u = max(1, (count_of(p) + c - 1) / c);
                nu += u;
                if (u > 1) rows += u * rows_of(p);
            }
            nu = warp_sum(nu);
            rows = warp_sum(rows);
            const bool caps = nu <= a.lay.unit_cap && rows <= a.lay.rows_cap;
            if (lane == 0 && caps && nu <= a.num_ctas) atomicMin(&s_best, c);
            if (lane == 0 && i == 0) s_fit0 = caps;
        }
    }
    __syncthreads();
    int chunk = (s_best != 0x7fffffff) ? s_best : chunk0;
    if (s_best == 0x7fffffff && !s_fit0) {
        // over a capacity: double the chunk until the table fits (rare)
        for (int attempt = 0; attempt < 24; ++attempt) {
            chunk *= 2;
            int nu = 0, rows = 0;
            for (int p = p_begin; p < p_end; ++p) {
                const int u = max(1, (count_of(p) + chunk - 1) / chunk);
                nu += u;
                if (u > 1) rows += u * rows_of(p);
            }
            int tot_u, tot_rows;
            cta_scan(nu, &tot_u, buf[2]);
            cta_scan(rows, &tot_rows, buf[3]);
            if (tot_u <= a.lay.unit_cap && tot_rows <= a.lay.rows_cap) break;
        }
    }
    chunk = min(chunk, kPlanMaxNB);
    // full chunks, split rows and the size of each pair's last unit
    int n_full = 0, rows = 0;
    for (int p = p_begin; p < p_end; ++p) {
        const int n = count_of(p);
        const int u = max(1, (n + chunk - 1) / chunk);
        const int last = n - (u - 1) * chunk;  // 1..chunk, or 0 for an empty pair
        n_full += (last == chunk) ? u : u - 1;
        if (u > 1) rows += u * rows_of(p);
        if (last < chunk) atomicAdd(&hist[last], 1);
    }
    int tot_full, tot_rows;
    int f_off = cta_scan(n_full, &tot_full, buf[0]);
    int r_off = cta_scan(rows, &tot_rows, buf[1]);
    // remainder bins in decreasing size start after the full chunks: warp 0,
    // each lane eight consecutive bins (chunk <= 256)
    if (warp == 0) {
        int cnt[8], loc = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int bin = chunk - 1 - (8 * lane + q);
            cnt[q] = (bin >= 0) ? hist[bin] : 0;
            loc += cnt[q];
        }
        int incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += n;
        }
        int start = tot_full + incl - loc;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int bin = chunk - 1 - (8 * lane + q);
            if (bin >= 0) hist[bin] = start;
            start += cnt[q];
        }
        if (lane == 31) hist[chunk] = tot_full + incl;  // total units
    }
    __syncthreads();
    const int tot_u = hist[chunk];
    for (int p = p_begin; p < p_end; ++p) {
        const int n = count_of(p);
        const int u = max(1, (n + chunk - 1) / chunk);
        const int last = n - (u - 1) * chunk;
        const int gg = p / Hkv, h = p % Hkv;
        const int t0 = s_gt0[gg], nt = s_gt0[gg + 1] - t0;
        const int rows_per_unit = nt * a.G;
        const int list = (gg * Hkv + (hb == 1 ? 0 : h)) * a.NB;
        for (int c = 0; c < u; ++c) {
            PlanUnit un;
            un.entry = list + c * chunk;
            un.count = (c + 1 < u) ? chunk : last;
            un.part_row = (u > 1) ? r_off + c * rows_per_unit : -1;
            un.pair = p;
            un.t0 = t0;
            un.nt = static_cast<int16_t>(nt);
            un.h = static_cast<int16_t>(h);
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
        hdr->n_pairs = n_pairs;
        hdr->n_units = tot_u;
        hdr->chunk = chunk;
        hdr->partial_rows = tot_rows;
        hdr->gmax = a.gmax;
        hdr->next_unit = 0;
    }
}

cudaError_t launch_pdl(const void *func, int grid, size_t smem, const PlanArgs &a, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<PlanArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, func, args);
}

}  // namespace

bool plan_configure(PlanArgs *a) {
    const bool shared_sel = (a->tk == nullptr) || (a->tk_s0 == 0);
    a->heads_built = shared_sel ? 1 : a->Hkv;
    if (list_smem_bytes(a->T, a->NB) > static_cast<size_t>(kPlanSmemMax)) return false;
    if (unit_smem_bytes(a->T, a->heads_built) > static_cast<size_t>(kPlanSmemMax)) return false;
    // a list per warp, for the most lists the rows can form
    const int64_t max_items = static_cast<int64_t>(a->T) * a->heads_built;
    a->list_ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(64, (max_items + kWarps - 1) / kWarps)));
    return true;
}

cudaError_t launch_prepare(const PlanArgs &a, int conv_ctas, cudaStream_t stream) {
    cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(list_kernel), kPlanSmemMax);
    if (e == cudaSuccess) e = opt_in_smem(reinterpret_cast<const void *>(unit_kernel), kPlanSmemMax);
    if (e != cudaSuccess) return e;
    e = launch_pdl(reinterpret_cast<const void *>(list_kernel), a.list_ctas, list_smem_bytes(a.T, a.NB), a, stream);
    if (e != cudaSuccess) return e;
    return launch_pdl(reinterpret_cast<const void *>(unit_kernel), 1 + conv_ctas,
                      unit_smem_bytes(a.T, a.heads_built), a, stream);
}

}  // namespace spd
