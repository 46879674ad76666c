// score_tc.cu -- the block-max score sheet ("Kernel ABI" --
// attention.msa_block_score / attention.msa_prefill_block_score) on the
// sm_103a tensor cores, for bf16 / f16 index tensors with Di a multiple of 64
// (at most 256).
//
// Orientation.  A CTA owns a tile of query lanes -- up to 128 (token, index
// head) pairs, head fastest -- and a chunk of block ids.  Per block and per
// run of consecutive lanes that read the same block-table row, one
// tcgen05.mma kind::f16 (fp32 accumulate, M = 128 query lanes, N = 128 keys
// of the block, K = Di) leaves that block's dot products in tensor memory
// with one query lane per TMEM lane.  The block maximum of a lane is then a
// reduction over its own 128 columns inside one thread: no shuffles, and the
// key mask (tokens at or beyond the lane's seq_len) is a column bound.
//
// An FP8-E4M3 index cache with bf16 index queries (Di = 128) takes the
// kind::f8f6f4 product instead: each lane's thread splits its query row,
// scaled by a power of two into E4M3 range, into two E4M3 terms (q = t0 + t1
// exactly for every element within 2^9 of the row's largest; below that t1
// is rounded in E4M3's subnormal range) written straight into the swizzled
// A tiles, the two terms accumulate into the same TMEM columns, and the
// epilogue undoes the scale.
//
// Keys are TMA-loaded straight from the paged index cache through the block
// table (128 tokens x 64 elements per box, 128-byte swizzle), double
// buffered; the two TMEM accumulators let the epilogue of one block overlap
// the product of the next.  Cells with no valid key are written -inf up front
// by the lane's own thread; a timed-out wait (a fault, never expected) leaves
// NaN in the cells it could not compute.
#include <math.h>

#include <algorithm>

#include "spd_internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace spd {

cudaError_t launch_score_tc(const ScoreArgs &a, cudaStream_t stream, bool *used);

namespace {

constexpr int kLanes = 128;       // query lanes per tile (M)
constexpr int kMaxStages = 4;     // key stages: 4 for Di = 64, else 2 (shared-memory budget)
constexpr int kMaxChunk = 8;      // block ids per CTA
constexpr int kThreadsSc = 192;   // warps 0-3 epilogue (TMEM quadrants), 4 TMA, 5 MMA
constexpr int kAtom = 128 * 128;  // one 64-element column chunk of 128 rows, bytes

struct ScoreTcArgs {
    const int32_t *bt;
    int64_t bt_s0, bt_s1;
    const int32_t *sl;
    int64_t sl_s0;
    const int32_t *ri;
    int64_t ri_s0;
    float *out;
    int64_t o_s0, o_s1, o_s2;
    int32_t T, Hi, Di, R, NB, tq, chunk;
    int64_t P;
    float idx_scale;
    uint32_t idesc;
    int32_t fp8;                    // E4M3 keys, bf16 queries split into two E4M3 terms
    const uint16_t *q;              // bf16 index queries (fp8 mode: read by the lanes' threads)
    int64_t q_s0, q_s1;
};

struct ScoreShared {
    uint64_t q_full, k_full[kMaxStages], k_empty[kMaxStages], acc_full[4], acc_empty[4];
    uint32_t tmem_base;
    int abort;
    int n_steps;
    int warp_starts[4];
    int lane_r[kLanes];
    int run_r[kLanes], run_lo[kLanes], run_hi[kLanes], run_lim[kLanes];
    int step_page[kMaxChunk * kLanes];
    uint16_t step_run[kMaxChunk * kLanes];
    uint8_t step_b[kMaxChunk * kLanes];
    uint32_t run_ok[kMaxChunk][kLanes / 32];  // bit j of word: run j has a valid page for that block
};

// Key stages and 128-column TMEM accumulators per CTA.  Up to Di = 128 a CTA
// takes at most ~110 KB of shared memory and 256 TMEM columns, so two CTAs
// share an SM: one's prologue (lane limits, page table, first loads)
// overlaps the other's products.  Wider keys keep the CTA alone on its SM,
// with four accumulators.
__host__ __device__ inline int key_stages(int nkc) { return nkc <= 1 ? 4 : 2; }
__device__ __forceinline__ int acc_count(int nkc) { return nkc >= 3 ? 4 : 2; }

// All 32 lanes wait; the warp goes on only if every lane saw the phase.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity));
}

// fp8 mode: the thread of query lane `lane` (row (t, h), valid when `row`)
// writes its query's two E4M3 terms into the swizzled A tiles (128-byte
// rows, K-major, 128-byte swizzle: term k at sQ + k * kAtom) and arrives on
// q_full.  The row is scaled by 2^e so that its largest magnitude lies in
// [128, 256) (E4M3 reaches 448), t0 = e4m3(y), t1 = e4m3(y - t0); returns
// 2^-e, the factor that takes the products back.  Lanes without a row write
// zeros.
__device__ __forceinline__ float split_query_row(const ScoreTcArgs &a, uint8_t *sQ, ScoreShared &sh, int lane,
                                                 bool row, int t, int h, bool needed) {
    float inv = 1.f;
    if (!needed) return inv;
    if (row) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.q + t * a.q_s0 + h * a.q_s1);
        float amax = 0.f;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
            const uint4 r = src[i];
            const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                amax = fmaxf(amax, fabsf(__uint_as_float(w4[j] << 16)));
                amax = fmaxf(amax, fabsf(__uint_as_float(w4[j] & 0xffff0000u)));
            }
        }
        // 2^s with s = 7 - floor(log2 amax), from the exponent bits
        const int eb = static_cast<int>((__float_as_uint(amax) >> 23) & 0xff);
        const int sb = min(253, max(1, 261 - eb));
        const float scale = __uint_as_float(static_cast<uint32_t>(sb) << 23);
        inv = __uint_as_float(static_cast<uint32_t>(254 - sb) << 23);
#pragma unroll 1
        for (int g = 0; g < 8; ++g) {  // 16 elements per group: two 16-byte loads
            const uint4 ra = src[2 * g], rb = src[2 * g + 1];
            const uint32_t w[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
            uint32_t p0[4], p1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // elements 16g + 4j .. +3
                const uint32_t wa = w[2 * j], wb = w[2 * j + 1];
                const float y0 = __uint_as_float(wa << 16) * scale, y1 = __uint_as_float(wa & 0xffff0000u) * scale;
                const float y2 = __uint_as_float(wb << 16) * scale, y3 = __uint_as_float(wb & 0xffff0000u) * scale;
                const uint16_t a01 = tc::f32x2_to_e4m3x2(y1, y0), a23 = tc::f32x2_to_e4m3x2(y3, y2);
                float z0, z1, z2, z3;
                tc::e4m3x2_to_f32x2(a01, z1, z0);
                tc::e4m3x2_to_f32x2(a23, z3, z2);
                const uint16_t b01 = tc::f32x2_to_e4m3x2(y1 - z1, y0 - z0);
                const uint16_t b23 = tc::f32x2_to_e4m3x2(y3 - z3, y2 - z2);
                p0[j] = static_cast<uint32_t>(a01) | (static_cast<uint32_t>(a23) << 16);
                p1[j] = static_cast<uint32_t>(b01) | (static_cast<uint32_t>(b23) << 16);
            }
            *reinterpret_cast<uint4 *>(sQ + tc::swz_offset(lane, 16 * g, 128)) = make_uint4(p0[0], p0[1], p0[2], p0[3]);
            *reinterpret_cast<uint4 *>(sQ + kAtom + tc::swz_offset(lane, 16 * g, 128)) =
                make_uint4(p1[0], p1[1], p1[2], p1[3]);
        }
    } else {
#pragma unroll 1
        for (int g = 0; g < 8; ++g) {
            *reinterpret_cast<uint4 *>(sQ + tc::swz_offset(lane, 16 * g, 128)) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(sQ + kAtom + tc::swz_offset(lane, 16 * g, 128)) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    tc::fence_proxy_async();
    tc::mbar_arrive(&sh.q_full);
    return inv;
}

__global__ void __launch_bounds__(kThreadsSc)
score_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const ScoreTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nkc = a.Di / 64;
    // bf16/f16: Q and each key stage are nkc 64-element atoms; fp8: two Q
    // term tiles and one 128-byte atom per key stage
    const int q_bytes = a.fp8 ? 2 * kAtom : nkc * kAtom;
    const int stage_bytes = a.fp8 ? kAtom : nkc * kAtom;
    uint8_t *sQ = smem;
    uint8_t *sK = smem + q_bytes;  // stage s at sK + s * stage_bytes
    const int n_stages = a.fp8 ? kMaxStages : key_stages(nkc);
    ScoreShared &sh = *reinterpret_cast<ScoreShared *>(sK + n_stages * stage_bytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * a.tq;
    const int b0 = blockIdx.y * a.chunk;
    const int nb = min(a.chunk, a.NB - b0);

    if (tid == 0) {
        tc::mbar_init(&sh.q_full, a.fp8 ? kLanes : 1);
        for (int i = 0; i < kMaxStages; ++i) {
            tc::mbar_init(&sh.k_full[i], 1);
            tc::mbar_init(&sh.k_empty[i], 1);
        }
        for (int i = 0; i < 4; ++i) {
            tc::mbar_init(&sh.acc_full[i], 1);
            tc::mbar_init(&sh.acc_empty[i], kLanes);
        }
        sh.abort = 0;
        sh.n_steps = 0;
        tc::fence_mbar_init();
    }
    const int n_acc = a.fp8 ? 2 : acc_count(nkc);
    if (warp == 5) tc::tmem_alloc(&sh.tmem_base, 128 * n_acc);
    // launched with programmatic stream serialisation: global memory only
    // after the previous kernel of the stream is done
    tc::pdl_wait();
    tc::pdl_trigger();

    // ---- lanes: (token t, head h) of each TMEM lane and its key limit
    const bool is_lane = tid < kLanes;
    const int tl = tid / a.Hi, h = tid % a.Hi, t = t0 + tl;
    const bool lane_row = is_lane && tl < a.tq && t < a.T;
    int my_r = -1;
    int my_lim = 0;
    if (lane_row) {
        int r;
        my_lim = static_cast<int>(token_limit(a.ri, a.ri_s0, a.sl, a.sl_s0, t, a.R, a.NB, &r));
        if (my_lim > 0) my_r = r;
    }
    if (is_lane) sh.lane_r[tid] = my_r;
    __syncthreads();

    // ---- runs: maximal spans of consecutive lanes with one block-table row
    const bool start = is_lane && my_r >= 0 && (tid == 0 || sh.lane_r[tid - 1] != my_r);
    const unsigned starts = __ballot_sync(0xffffffffu, start);
    if (lane == 0 && warp < 4) sh.warp_starts[warp] = __popc(starts);
    __syncthreads();
    int n_runs = 0, run_base = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        if (w < warp) run_base += sh.warp_starts[w];
        n_runs += sh.warp_starts[w];
    }
    const int my_run = my_r >= 0 ? run_base + __popc(starts & ((2u << lane) - 1u)) - 1 : -1;
    if (start) {
        sh.run_r[my_run] = my_r;
        sh.run_lo[my_run] = tid;
        sh.run_hi[my_run] = 0;
        sh.run_lim[my_run] = 0;
    }
    __syncthreads();
    if (my_run >= 0) {
        atomicMax(&sh.run_hi[my_run], tid + 1);
        atomicMax(&sh.run_lim[my_run], my_lim);
    }
    // ---- steps: (block, run) pairs with a valid page and some valid key
    // (the page table is read once, here)
    for (int i = tid; i < kMaxChunk * (kLanes / 32); i += kThreadsSc) (&sh.run_ok[0][0])[i] = 0u;
    __syncthreads();
    for (int idx = tid; idx < nb * n_runs; idx += kThreadsSc) {
        const int bl = idx / n_runs, j = idx % n_runs;
        const int b = b0 + bl;
        if (static_cast<int64_t>(b) * kBlock >= sh.run_lim[j]) continue;
        const int64_t page = a.bt[sh.run_r[j] * a.bt_s0 + b * a.bt_s1];
        if (page < 0 || page >= a.P) continue;
        atomicOr(&sh.run_ok[bl][j >> 5], 1u << (j & 31));
        const int s = atomicAdd(&sh.n_steps, 1);
        sh.step_page[s] = static_cast<int>(page);
        sh.step_run[s] = static_cast<uint16_t>(j);
        sh.step_b[s] = static_cast<uint8_t>(bl);
    }
    __syncthreads();
    // cells with no valid key: -inf now (the lane's own thread)
    if (lane_row) {
        for (int bl = 0; bl < nb; ++bl) {
            const int b = b0 + bl;
            bool empty = my_r < 0 || static_cast<int64_t>(b) * kBlock >= my_lim;
            if (!empty) empty = !((sh.run_ok[bl][my_run >> 5] >> (my_run & 31)) & 1u);
            if (empty) a.out[h * a.o_s0 + t * a.o_s1 + b * a.o_s2] = -INFINITY;
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const int n_steps = sh.n_steps;
    const uint32_t tmem = sh.tmem_base;

    if (warp == 4) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && n_steps > 0) {
            tc::prefetch_tmap(&tmap_k);
            if (!a.fp8) {
                tc::prefetch_tmap(&tmap_q);
                tc::mbar_arrive_expect_tx(&sh.q_full, static_cast<uint32_t>(nkc * a.tq * a.Hi * 128));
                for (int c = 0; c < nkc; ++c) tc::tma_load_3d(sQ + c * kAtom, &tmap_q, &sh.q_full, c * 64, 0, t0);
            }
            int s = 0;
            for (; s < n_steps; ++s) {
                const int st = s % n_stages;
                if (s >= n_stages && !tc::mbar_wait(&sh.k_empty[st], ((s / n_stages) - 1) & 1)) {
                    *reinterpret_cast<volatile int *>(&sh.abort) = 1;
                    break;
                }
                uint8_t *dst = sK + st * stage_bytes;
                tc::mbar_arrive_expect_tx(&sh.k_full[st], static_cast<uint32_t>(stage_bytes));
                if (a.fp8) {
                    tc::tma_load_2d(dst, &tmap_k, &sh.k_full[st], 0, sh.step_page[s] * kBlock);
                } else {
                    for (int c = 0; c < nkc; ++c)
                        tc::tma_load_2d(dst + c * kAtom, &tmap_k, &sh.k_full[st], c * 64, sh.step_page[s] * kBlock);
                }
            }
            // every issued copy lands before the CTA may exit
            if (!a.fp8) tc::mbar_wait(&sh.q_full, 0);
            for (int u = s > n_stages ? s - n_stages : 0; u < s; ++u)
                tc::mbar_wait(&sh.k_full[u % n_stages], (u / n_stages) & 1);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && n_steps > 0) {
            const uint32_t q_base = tc::smem_u32(sQ), k_base = tc::smem_u32(sK);
            bool ok = tc::mbar_wait(&sh.q_full, 0);
            int s = 0;
            for (; ok && s < n_steps; ++s) {
                const int st = s % n_stages, buf = s % n_acc;
                ok = tc::mbar_wait(&sh.k_full[st], (s / n_stages) & 1);
                if (ok && s >= n_acc) ok = tc::mbar_wait(&sh.acc_empty[buf], ((s / n_acc) - 1) & 1);
                if (!ok) break;
                tc::tc_fence_after();
                const uint32_t kb = k_base + st * stage_bytes;
                if (a.fp8) {
                    // two query terms x four 32-element k-steps into the same columns
                    for (int term = 0; term < 2; ++term)
                        for (int ks = 0; ks < 4; ++ks)
                            tc::mma_f8(tmem + buf * 128,
                                       tc::smem_desc(q_base + term * kAtom + ks * 32, 16, 1024, tc::kSw128),
                                       tc::smem_desc(kb + ks * 32, 16, 1024, tc::kSw128), a.idesc, term > 0 || ks > 0);
                } else {
                    for (int kc = 0; kc < a.Di / 16; ++kc) {
                        const uint32_t off = (kc >> 2) * kAtom + (kc & 3) * 32;
                        tc::mma_f16(tmem + buf * 128, tc::smem_desc(q_base + off, 16, 1024, tc::kSw128),
                                    tc::smem_desc(kb + off, 16, 1024, tc::kSw128), a.idesc, kc > 0);
                    }
                }
                tc::mma_commit(&sh.k_empty[st]);
                tc::mma_commit(&sh.acc_full[buf]);
            }
            if (!ok) *reinterpret_cast<volatile int *>(&sh.abort) = 1;
            // the issued products complete before TMEM is released
            if (s > 0) tc::mbar_wait(&sh.acc_full[(s - 1) % n_acc], ((s - 1) / n_acc) & 1);
        }
    } else {
        // --------------------------------------------------------- epilogue
        // Each warp reads its TMEM lane quadrant; a lane's block maximum is a
        // reduction over its own row of 128 key columns.
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float out_scale = a.idx_scale;
        if (a.fp8) out_scale *= split_query_row(a, sQ, sh, tid, lane_row, t, h, n_steps > 0);
        bool ok = true;
        for (int s = 0; s < n_steps; ++s) {
            const int buf = s % n_acc, j = sh.step_run[s];
            const int b = b0 + sh.step_b[s];
            const int lo = sh.run_lo[j], hi = sh.run_hi[j];
            const int lim = my_lim - b * kBlock;
            const bool mine = tid >= lo && tid < hi && lim > 0;
            if (ok) ok = warp_wait(&sh.acc_full[buf], (s / n_acc) & 1);
            if (!ok) {
                if (mine) a.out[h * a.o_s0 + t * a.o_s1 + b * a.o_s2] = NAN;
                continue;
            }
            tc::tc_fence_after();
            if (hi > warp * 32 && lo < warp * 32 + 32) {
                float best = -INFINITY;
                const uint32_t base = tmem + buf * 128 + lane_base;
                // 64 columns per tensor-memory round trip
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 64) {
                    float v[4][16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) tc::tmem_ld16(base + c0 + 16 * q, v[q]);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (lim >= 128) {
#pragma unroll
                            for (int k = 0; k < 16; ++k) best = fmaxf(best, v[q][k]);
                        } else {
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                if (c0 + 16 * q + k < lim) best = fmaxf(best, v[q][k]);
                        }
                    }
                }
                if (mine)
                    a.out[h * a.o_s0 + t * a.o_s1 + b * a.o_s2] = (best == -INFINITY) ? -INFINITY : best * out_scale;
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&sh.acc_empty[buf]);
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 5) tc::tmem_dealloc(tmem, 128 * n_acc);
}

bool make_tmap_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                  uint32_t box_rows) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 keys [rows, 128] (row stride in bytes, a multiple of 16) as a 2-D
// map whose box is 128 rows of 128 bytes, 128-byte swizzle.
bool make_tmap_2d_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t row_bytes) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {128, static_cast<cuuint32_t>(kBlock)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q_idx [T, Hi, Di] as a 3-D map: box = 64 elements x Hi heads x tq tokens,
// which lands as tq*Hi rows of 128 bytes (head fastest).
bool make_tmap_qidx(CUtensorMap *m, const ScoreArgs &a, int tq) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    const uint64_t s1 = a.Hi > 1 ? static_cast<uint64_t>(a.q_s1) * 2 : static_cast<uint64_t>(a.Di) * 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.Di), static_cast<cuuint64_t>(a.Hi),
                          static_cast<cuuint64_t>(a.T)};
    cuuint64_t strides[2] = {s1, static_cast<cuuint64_t>(a.q_s0) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(a.Hi), static_cast<cuuint32_t>(tq)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(a.q), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Covers: q_idx and k_idx_cache both bf16 or both f16, Di in {64, 128, 192,
// 256}, Hi <= 128, innermost strides 1, 16-byte aligned bases and row
// strides, at most 2^31 cache slots.  Anything else: *used stays false.
cudaError_t launch_score_tc(const ScoreArgs &a, cudaStream_t stream, bool *used) {
    *used = false;
    // E4M3 keys with bf16 queries of 128 dims: the f8 product
    const bool fp8 = a.k_dt == SPD_E4M3 && a.q_dt == SPD_BF16 && a.Di == 128;
    const int k_elem = fp8 ? 1 : 2;  // bytes per key element
    if (!fp8 && (a.q_dt != a.k_dt || (a.q_dt != SPD_BF16 && a.q_dt != SPD_F16))) return cudaSuccess;
    if (a.Di % 64 != 0 || a.Di > 256 || a.Hi > kLanes || a.Hi < 1) return cudaSuccess;
    if (a.q_s2 != 1 || a.k_s2 != 1) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(a.q) % 16) || (reinterpret_cast<uintptr_t>(a.k) % 16)) return cudaSuccess;
    if (a.q_s0 <= 0 || (a.q_s0 * 2) % 16 || a.k_s0 <= 0 || (a.k_s0 * k_elem) % 16) return cudaSuccess;
    if (a.Hi > 1 && (a.q_s1 <= 0 || (a.q_s1 * 2) % 16)) return cudaSuccess;
    if (a.P * kBlock > (int64_t(1) << 31) - 1) return cudaSuccess;

    const int sms = device_sm_count();
    const int nkc = a.Di / 64;
    const int smem = fp8 ? static_cast<int>(1024 + kAtom * (2 + kMaxStages) + sizeof(ScoreShared))
                         : static_cast<int>(1024 + nkc * kAtom * (1 + key_stages(nkc)) + sizeof(ScoreShared));
    {
        int smem_max = 0;
        for (int c = 1; c <= 4; ++c) {
            const int bytes = static_cast<int>(1024 + c * kAtom * (1 + key_stages(c)) + sizeof(ScoreShared));
            smem_max = bytes > smem_max ? bytes : smem_max;
        }
        cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(score_tc_kernel), smem_max);
        if (e != cudaSuccess) return e;
    }

    // A CTA runs its (request, block) steps one after another, so its time
    // grows with the steps it owns.  Decode batches (a few query rows per
    // page-table row) put many short requests in one lane tile, and the low
    // block ids, which every request has, carry the most steps: there a CTA
    // takes half a tile of lanes and one block id.  Prefill batches (long
    // runs of one request) keep full tiles and several block ids a CTA, so
    // each K tile serves many lanes.
    const bool decode_like = a.R > 0 && a.T <= 32LL * a.R;
    const int tq = decode_like ? std::max(1, kLanes / a.Hi / 2) : kLanes / a.Hi;
    const int64_t n_tiles = (a.T + tq - 1) / tq;
    int64_t chunk = decode_like ? 1 : (n_tiles * a.NB + 2 * sms - 1) / (2 * sms);
    chunk = chunk < 1 ? 1 : chunk > kMaxChunk ? kMaxChunk : chunk;
    const int64_t n_chunks = (a.NB + chunk - 1) / chunk;
    if (n_tiles > INT32_MAX) return cudaSuccess;

    CUtensorMap tq_map, tk_map;
    if (fp8) {
        // keys: 128-byte rows of E4M3 codes, one box = one block of 128 rows;
        // the query map is unused (the lanes' threads write the query terms)
        if (!make_tmap_2d_u8(&tk_map, a.k, static_cast<uint64_t>(a.P * kBlock), static_cast<uint64_t>(a.k_s0)))
            return cudaSuccess;
        tq_map = tk_map;
    } else {
        if (!make_tmap_qidx(&tq_map, a, tq)) return cudaSuccess;
        if (!make_tmap_2d(&tk_map, a.k, static_cast<uint64_t>(a.Di), static_cast<uint64_t>(a.P * kBlock),
                          static_cast<uint64_t>(a.k_s0) * 2, kBlock))
            return cudaSuccess;
    }

    ScoreTcArgs t{};
    t.bt = a.bt; t.bt_s0 = a.bt_s0; t.bt_s1 = a.bt_s1;
    t.sl = a.sl; t.sl_s0 = a.sl_s0;
    t.ri = a.ri; t.ri_s0 = a.ri_s0;
    t.out = a.out; t.o_s0 = a.o_s0; t.o_s1 = a.o_s1; t.o_s2 = a.o_s2;
    t.T = a.T; t.Hi = a.Hi; t.Di = a.Di; t.R = a.R; t.NB = a.NB;
    t.tq = tq;
    t.chunk = static_cast<int32_t>(chunk);
    t.P = a.P;
    t.idx_scale = a.idx_scale;
    t.idesc = fp8 ? tc::idesc_m128(128, false, false) : tc::idesc_f16_m128(128, a.q_dt == SPD_BF16);
    t.fp8 = fp8 ? 1 : 0;
    t.q = static_cast<const uint16_t *>(a.q);
    t.q_s0 = a.q_s0;
    t.q_s1 = a.q_s1;
    dim3 grid(static_cast<unsigned>(n_tiles), static_cast<unsigned>(n_chunks));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreadsSc);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, score_tc_kernel, tq_map, tk_map, t);
    if (e == cudaSuccess) *used = true;
    return e;
}

}  // namespace spd
