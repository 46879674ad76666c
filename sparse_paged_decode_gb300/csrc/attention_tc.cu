// attention_tc.cu -- paged sparse / dense GQA decode attention on the sm_103a
// tensor cores (tcgen05) with TMA-staged FP8 pages.
//
// What it computes is "Kernel ABI" -- attention.decode (see include/spd.h);
// how, in short:
//
//  * Work.  A device planner (plan.cu) groups the query rows of one request
//    that sit together (draft tokens of a verification row), unions the blocks
//    they selected per kv head, and cuts each (group, kv head) block list into
//    units.  A persistent grid walks the units; a pair cut into several units
//    merges its partials in the last unit to finish (an atomic counter, no
//    waiting on other CTAs).
//
//  * Staging.  Warp 0 streams each selected page's K and V tile (128 tokens x
//    128 bytes of one kv head) with TMA into a ring of shared-memory stages,
//    128-byte swizzled, straight from the paged cache through the block table.
//
//  * Contractions.  Warp 1 issues tcgen05.mma kind::f8f6f4 with fp32
//    accumulation in tensor memory.  Keys lie on the 128 TMEM lanes and the
//    group's query rows (rows x q heads, padded to N = 16/32/64) on columns:
//        S^T[tok][n]  = K[tok][:] . Qs[n][:]          (A = K tile, K-major)
//        O^T[d][n]   += V^T[d][tok] . P[tok][n]        (A = V tile, MN-major)
//    The E4M3 K/V bytes feed the tensor core unconverted.  Queries and
//    probabilities are split into two E4M3 terms, x = hi + lo with
//    hi = e4m3(x) and lo = e4m3(x - hi), accumulated along the contraction
//    (about 8 significant bits, like bf16), so no operand is converted from
//    FP8 and no precision below bf16 is lost.  Each query row is scaled by a
//    power of two into E4M3 range first; the factor comes out with the
//    softmax scale.
//
//  * Softmax.  Warps 2-5 own the 128 token lanes of S and the 128 d lanes of
//    O.  The exponent offset per query row is a running maximum that is only
//    raised when a logit exceeds it by more than 2^6 (then O is rescaled in
//    tensor memory): most blocks need no cross-lane reduction.  The row sums
//    accumulate per thread and are reduced once per unit.  Probabilities are
//    written to shared memory as the B operand of the next PV product.
//
// Synchronisation uses mbarriers between the roles, every wait bounded
// (a timeout sets bit 0 of the workspace status word and the CTA winds down).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "plan.cuh"
#include "spd_internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace spd {

cudaError_t launch_attention_tc(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream, bool *used);

namespace {

constexpr int kThreads = 192;         // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int kSoftThreads = 128;
constexpr int kStages = 3;
constexpr int kTile = 128 * 128;      // bytes of one K or V tile
constexpr int kNMax = 64;             // query rows per group (padded)
constexpr int kMaxEntries = kPlanMaxNB;
constexpr float kRaise = 6.0f;        // log2 headroom before the offset is raised (p <= 64)
constexpr int kD = 128;
constexpr int kTerms = kQueryTerms;   // E4M3 terms per query element (12 significant bits)
constexpr int kStride = kD + kPartialStride;

struct TcArgs {
    const int32_t *ri;
    int64_t ri_s0;
    const int32_t *sl;
    int64_t sl_s0;
    __nv_bfloat16 *out;
    int64_t o_s0, o_s1, o_s2;
    int32_t T, Hq, Hkv, G, R, NB, gmax;
    float v_scale;
    char *ws;
    PlanLayout lay;
};

struct __align__(16) Shared {
    float m_run[kNMax];   // running exponent offset per query row (log2 units)
    float cfac[kNMax];    // logit factor per query row
    float alpha[kNMax];   // rescale factor of the last offset raise
    float den[kNMax];     // merge: normaliser per row
    float red[4][kNMax];  // cross-warp reduction scratch
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], s_empty[2], p_full[2], pv_done[2];
    uint64_t q_full, q_empty, merge_bar;
    uint64_t unit_full[4], unit_empty[4];  // ring of unit records, producer -> MMA, softmax
    PlanUnit ring[4];
    uint32_t tmem_base;
    int abort;
    int combine;
    int rescale;
    int vote[2][4];
    int unit_vote[4];
    int Lj[16];                  // key limit of each group row
    PlanEntry ent[kMaxEntries];  // the unit's block list
};

// dynamic shared memory: E4M3 K and V stages, query terms, f16 V and P tiles
// (double buffered), Shared
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kStages * kTile;
constexpr int kQBytes = kNMax * 128;
constexpr int kOffQ = kOffV + kStages * kTile;
constexpr int kV16Tile = 128 * kD * 2;   // [2 d-halves][128 tokens][64 d] f16
constexpr int kP16Tile = 128 * kNMax * 2;  // [128 tokens][N] f16
constexpr int kOffV16 = kOffQ + kTerms * kQBytes;
constexpr int kOffP = kOffV16 + 2 * kV16Tile;
constexpr int kOffShared = kOffP + 2 * kP16Tile;
constexpr int kSmemBytes = kOffShared + static_cast<int>(sizeof(Shared)) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ int pow2_width(int n) { return n <= 16 ? 16 : n <= 32 ? 32 : 64; }

// swizzle of an f16 [tokens][n] tile whose rows are 2n bytes
__device__ __forceinline__ tc::Swizzle p_swizzle(int n) {
    return n == 16 ? tc::kSw32 : n == 32 ? tc::kSw64 : tc::kSw128;
}

__device__ __forceinline__ void named_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSoftThreads) : "memory"); }

__device__ __forceinline__ bool aborted(Shared &sh) { return *reinterpret_cast<volatile int *>(&sh.abort) != 0; }

__device__ __forceinline__ bool wait_or_abort(Shared &sh, uint64_t *bar, uint32_t parity, int32_t *status) {
    if (tc::mbar_wait(bar, parity)) return true;
    *reinterpret_cast<volatile int *>(&sh.abort) = 1;
    atomicOr(status, 1);
    return false;
}

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

// What a softmax thread needs besides the kernel arguments.
struct Soft {
    Shared *sh;
    uint8_t *smem;
    int32_t *status;
    int32_t *counters;
    float *partials;
    uint32_t tS0, tS1, tO, lane_base;
    int tok, lane, sw, st_id;
};

// The last unit of a split pair to finish merges all of them: the units'
// partial rows are pulled into the idle f16 V / P buffers with bulk copies
// (one wait for all of them), then per row the weights 2^(m_k - max m) and
// every output element's weighted sum.
__device__ __noinline__ void merge_partials(const Soft &c, const TcArgs &a, const PlanUnit &un,
                                            uint32_t &merge_uses) {
    Shared &sh = *c.sh;
    constexpr int kRowBytes = kStride * 4;
    constexpr int kStageBytes = 2 * kV16Tile + 2 * kP16Tile;
    const int rows = un.nt * a.G, ns = un.n_split;
    uint8_t *stage = c.smem + kOffV16;
    int R = rows;
    while (R > 1 && ns * R * (kRowBytes + 4) > kStageBytes) R = (R + 1) / 2;
    const float *pbase = c.partials + static_cast<int64_t>(un.part_base) * kStride;
    const float vs = a.v_scale * 256.f;
    const int d = c.tok;
    for (int r0 = 0; r0 < rows; r0 += R) {
        const int nr = min(R, rows - r0);
        float *wts = reinterpret_cast<float *>(stage + ns * nr * kRowBytes);
        if (c.st_id == 0) {
            tc::fence_proxy_async_global();
            tc::mbar_arrive_expect_tx(&sh.merge_bar, ns * nr * kRowBytes);
            for (int k = 0; k < ns; ++k)
                tc::bulk_load(stage + k * nr * kRowBytes, pbase + static_cast<int64_t>(k * rows + r0) * kStride,
                              nr * kRowBytes, &sh.merge_bar);
        }
        wait_or_abort(sh, &sh.merge_bar, merge_uses & 1, c.status);
        ++merge_uses;
        const float *st = reinterpret_cast<const float *>(stage);
        // weights 2^(m_k - max_k m) and the normaliser, one row per thread
        for (int r = c.st_id; r < nr; r += kSoftThreads) {
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            int k = 0;
            for (; k + 4 <= ns; k += 4)
#pragma unroll
                for (int j = 0; j < 4; ++j) m4[j] = fmaxf(m4[j], st[((k + j) * nr + r) * kStride + kD]);
            for (; k < ns; ++k) m4[0] = fmaxf(m4[0], st[(k * nr + r) * kStride + kD]);
            const float mstar = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            float den = 0.f;
            for (k = 0; k < ns; ++k) {
                const float mk = st[(k * nr + r) * kStride + kD];
                const float w = (mk == -INFINITY) ? 0.f : tc::ex2(mk - mstar);
                wts[k * nr + r] = w;
                den += w * st[(k * nr + r) * kStride + kD + 1];
            }
            sh.den[r] = den;
        }
        named_sync();
        // each thread one d of every row; four independent partial sums
        for (int r = 0; r < nr; ++r) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            int k = 0;
            for (; k + 4 <= ns; k += 4)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    acc[j] = fmaf(wts[(k + j) * nr + r], st[((k + j) * nr + r) * kStride + d], acc[j]);
            for (; k < ns; ++k) acc[0] = fmaf(wts[k * nr + r], st[(k * nr + r) * kStride + d], acc[0]);
            const float den = sh.den[r];
            const float sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            const float val = (den > 0.f) ? sum * vs / den : 0.f;
            const int t = un.t0 + (r0 + r) / a.G, g = (r0 + r) % a.G;
            a.out[t * a.o_s0 + (un.h * a.G + g) * a.o_s1 + d * a.o_s2] = __float2bfloat16_rn(val);
        }
        named_sync();  // the stage is reused by the next chunk
    }
}

// One unit's blocks and its epilogue for N = 16*NCH query columns.  Returns
// false when the CTA must stop (an abort, decided uniformly).
template <int NCH>
__device__ __forceinline__ bool unit_body(const Soft &c, const TcArgs &a, const PlanUnit &un, uint32_t gb) {
    constexpr int N = NCH * 16;
    Shared &sh = *c.sh;
    const int rows = un.nt * a.G;
    const uint64_t gmask = (a.G >= 64) ? ~0ull : ((1ull << a.G) - 1);
    float lsum[N];
#pragma unroll
    for (int col = 0; col < N; ++col) lsum[col] = 0.f;

    for (int i = 0; i < un.count; ++i) {
        const uint32_t b = gb + i;
        const int sb = b & 1, stg = b % kStages;
        const PlanEntry e = sh.ent[i];
        // columns valid on this token lane: selected by the column's row and
        // below that row's key limit
        uint64_t colmask = 0;
        for (int j = 0; j < un.nt; ++j)
            if (((e.mask >> j) & 1) && c.tok < sh.Lj[j] - e.block * 128) colmask |= gmask << (j * a.G);
        wait_or_abort(sh, &sh.s_full[sb], (b >> 1) & 1, c.status);
        tc::tc_fence_after();
        float s[N];
        const uint32_t sbase = (sb ? c.tS1 : c.tS0) + c.lane_base;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            float v[16];
            tc::tmem_ld16(sbase + ch * 16, v);
#pragma unroll
            for (int k = 0; k < 16; ++k) s[ch * 16 + k] = v[k];
        }
        tc::tmem_wait_ld();
        tc::tc_fence_before();
        tc::mbar_arrive(&sh.s_empty[sb]);

        bool need = false;
#pragma unroll
        for (int c4 = 0; c4 < N; c4 += 4) {
            const float4 cf = *reinterpret_cast<const float4 *>(&sh.cfac[c4]);
            const float4 mr = *reinterpret_cast<const float4 *>(&sh.m_run[c4]);
            const float cfs[4] = {cf.x, cf.y, cf.z, cf.w}, mrs[4] = {mr.x, mr.y, mr.z, mr.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int col = c4 + k;
                s[col] = ((colmask >> col) & 1) ? s[col] * cfs[k] : -INFINITY;
                need |= s[col] > mrs[k] + kRaise;
            }
        }
        // votes alternate between two slots by block parity: a warp can be at
        // most one block ahead of the slowest reader
        const int mine = (__any_sync(0xffffffffu, need) ? 1 : 0) | (aborted(sh) ? 2 : 0);
        if (c.lane == 0) sh.vote[sb][c.sw] = mine;
        named_sync();
        const int vote = sh.vote[sb][0] | sh.vote[sb][1] | sh.vote[sb][2] | sh.vote[sb][3];
        if (vote & 2) return false;
        if (vote & 1) {
            // raise the offsets to the block maximum; rescale O and the sums
#pragma unroll
            for (int col = 0; col < N; ++col) {
                const float mx = warp_max(s[col]);
                if (c.lane == 0) sh.red[c.sw][col] = mx;
            }
            named_sync();
            if (c.sw == 0) {
                bool any = false;
                for (int col = c.lane; col < N; col += 32) {
                    const float bm = fmaxf(fmaxf(sh.red[0][col], sh.red[1][col]), fmaxf(sh.red[2][col], sh.red[3][col]));
                    const float old = sh.m_run[col];
                    float al = 1.f;
                    if (bm > old) {
                        al = (old == -INFINITY) ? 0.f : tc::ex2(old - bm);
                        any |= old != -INFINITY;
                        sh.m_run[col] = bm;
                    }
                    sh.alpha[col] = al;
                }
                any = __any_sync(0xffffffffu, any);
                if (c.lane == 0) sh.rescale = any;
            }
            named_sync();
#pragma unroll
            for (int col = 0; col < N; ++col) lsum[col] *= sh.alpha[col];
            if (sh.rescale && i > 0) {
                // O holds blocks 0..i-1 of this unit: wait for the last PV
                wait_or_abort(sh, &sh.pv_done[(b - 1) & 1], ((b - 1) >> 1) & 1, c.status);
                tc::tc_fence_after();
                for (int ch = 0; ch < NCH; ++ch) {
                    float v[16];
                    tc::tmem_ld16(c.tO + c.lane_base + ch * 16, v);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[k] *= sh.alpha[ch * 16 + k];
                    tc::tmem_st16(c.tO + c.lane_base + ch * 16, v);
                }
                tc::tmem_wait_st();
                tc::tc_fence_before();
            }
        }

        // V and P buffers sb were read by the PV of block b-2
        if (b >= 2) wait_or_abort(sh, &sh.pv_done[sb], ((b >> 1) - 1) & 1, c.status);
        // this token's V row: E4M3 (128-byte swizzled TMA tile) -> f16 * 2^-8
        // (two 64-d halves, 128-byte swizzle), the A operand of P V; the E4M3
        // stage is then free for the next TMA load
        wait_or_abort(sh, &sh.kv_full[stg], (b / kStages) & 1, c.status);
        {
            const uint8_t *vsrc = c.smem + kOffV + stg * kTile + c.tok * 128;
            uint8_t *vdst = c.smem + kOffV16 + sb * kV16Tile + c.tok * 128;
            const int sw8 = c.tok & 7;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint4 x = *reinterpret_cast<const uint4 *>(vsrc + ((cc ^ sw8) << 4));
                uint32_t f[8];
                tc::e4m3x4_to_f16x4_scaled(x.x, f[0], f[1]);
                tc::e4m3x4_to_f16x4_scaled(x.y, f[2], f[3]);
                tc::e4m3x4_to_f16x4_scaled(x.z, f[4], f[5]);
                tc::e4m3x4_to_f16x4_scaled(x.w, f[6], f[7]);
                uint8_t *half = vdst + (cc >> 2) * (128 * 128);
                *reinterpret_cast<uint4 *>(half + ((((2 * cc) & 7) ^ sw8) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<uint4 *>(half + ((((2 * cc + 1) & 7) ^ sw8) << 4)) = make_uint4(f[4], f[5], f[6], f[7]);
            }
        }
        tc::fence_proxy_async();
        tc::mbar_arrive(&sh.kv_empty[stg]);
        // probabilities p = 2^(s - offset) <= 64 in f16 (11-bit significand,
        // normal down to 2^-14), the B operand of P V
        uint8_t *pb = c.smem + kOffP + sb * kP16Tile;
#pragma unroll
        for (int c8 = 0; c8 < N; c8 += 8) {
            const float4 m0 = *reinterpret_cast<const float4 *>(&sh.m_run[c8]);
            const float4 m1 = *reinterpret_cast<const float4 *>(&sh.m_run[c8 + 4]);
            const float mr[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
            float p[8];
#pragma unroll
            for (int e2 = 0; e2 < 8; ++e2) {
                const int col = c8 + e2;
                p[e2] = (s[col] == -INFINITY) ? 0.f : tc::ex2(s[col] - mr[e2]);
                lsum[col] += p[e2];
            }
            uint4 w;
            w.x = tc::f32x2_to_f16x2(p[0], p[1]);
            w.y = tc::f32x2_to_f16x2(p[2], p[3]);
            w.z = tc::f32x2_to_f16x2(p[4], p[5]);
            w.w = tc::f32x2_to_f16x2(p[6], p[7]);
            *reinterpret_cast<uint4 *>(pb + tc::swz_offset(c.tok, c8 * 2, 2 * N)) = w;
        }
        tc::fence_proxy_async();
        tc::mbar_arrive(&sh.p_full[sb]);
    }

    // ---- epilogue: row sums over the 128 token lanes, then O (d lane = tok)
#pragma unroll
    for (int col = 0; col < N; ++col) {
        const float v = warp_sum(lsum[col]);
        if (c.lane == 0) sh.red[c.sw][col] = v;
    }
    float o[N];
#pragma unroll
    for (int col = 0; col < N; ++col) o[col] = 0.f;
    if (un.count > 0) {
        const uint32_t last = gb + un.count - 1;
        wait_or_abort(sh, &sh.pv_done[last & 1], (last >> 1) & 1, c.status);
        tc::tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            float v[16];
            tc::tmem_ld16(c.tO + c.lane_base + ch * 16, v);
#pragma unroll
            for (int k = 0; k < 16; ++k) o[ch * 16 + k] = v[k];
        }
        tc::tmem_wait_ld();
        tc::tc_fence_before();
    }
    named_sync();
    const int d = c.tok;
    if (un.part_row < 0) {
#pragma unroll
        for (int col = 0; col < N; ++col) {
            if (col < rows) {
                const float l = sh.red[0][col] + sh.red[1][col] + sh.red[2][col] + sh.red[3][col];
                const float val = (l > 0.f) ? o[col] * (a.v_scale * 256.f) / l : 0.f;
                const int t = un.t0 + col / a.G, g = col % a.G;
                a.out[t * a.o_s0 + (un.h * a.G + g) * a.o_s1 + d * a.o_s2] = __float2bfloat16_rn(val);
            }
        }
    } else {
        // partial of a split pair: unnormalised O, offset and sum per row
#pragma unroll
        for (int col = 0; col < N; ++col) {
            if (col < rows) {
                float *prow = c.partials + static_cast<int64_t>(un.part_row + col) * kStride;
                prow[d] = o[col];
                if (d == 0) {
                    prow[kD] = sh.m_run[col];
                    prow[kD + 1] = sh.red[0][col] + sh.red[1][col] + sh.red[2][col] + sh.red[3][col];
                }
            }
        }
        tc::fence_proxy_async_global();  // the merge reads partials with bulk copies
        named_sync();
    }
    return true;
}

// A split unit takes a ticket on its pair's counter once its partial is
// written; whether it was the pair's last unit is looked at only after the
// next unit (so the atomic's round trip is hidden), and the last one merges.
struct PendingMerge {
    PlanUnit un;
    int ticket;  // thread st_id 0 only
};

__device__ __forceinline__ void take_ticket(const Soft &c, const PlanUnit &un, PendingMerge &pm) {
    pm.un = un;
    if (c.st_id == 0) {
        __threadfence();  // the CTA's partial writes (ordered by the barrier) before the ticket
        pm.ticket = atomicAdd(&c.counters[un.pair], 1);
    }
}

__device__ __forceinline__ void resolve_ticket(const Soft &c, const TcArgs &a, PendingMerge &pm,
                                               uint32_t &merge_uses) {
    Shared &sh = *c.sh;
    if (pm.un.pair < 0) return;
    if (c.st_id == 0) {
        sh.combine = (pm.ticket == pm.un.n_split - 1);
        if (sh.combine) __threadfence();  // the other units' partials before the merge reads them
    }
    named_sync();
    if (sh.combine) merge_partials(c, a, pm.un, merge_uses);
    named_sync();
    pm.un.pair = -1;
}

__global__ void __launch_bounds__(kThreads, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_q, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Shared &sh = *reinterpret_cast<Shared *>(smem + kOffShared);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(a.ws + a.lay.header);
    const PlanEntry *lists = reinterpret_cast<const PlanEntry *>(a.ws + a.lay.lists);
    const PlanUnit *units = reinterpret_cast<const PlanUnit *>(a.ws + a.lay.units);
    const int n_units = hdr->n_units;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&sh.kv_full[i], 1);
            tc::mbar_init(&sh.kv_empty[i], kSoftThreads);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&sh.s_full[i], 1);
            tc::mbar_init(&sh.s_empty[i], kSoftThreads);
            tc::mbar_init(&sh.p_full[i], kSoftThreads);
            tc::mbar_init(&sh.pv_done[i], 1);
        }
        tc::mbar_init(&sh.q_full, 1);
        tc::mbar_init(&sh.q_empty, 1);
        tc::mbar_init(&sh.merge_bar, 1);
        for (int i = 0; i < 4; ++i) {
            tc::mbar_init(&sh.unit_full[i], 1);
            tc::mbar_init(&sh.unit_empty[i], 1 + kSoftThreads);
        }
        sh.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(&sh.tmem_base, 4 * kNMax);  // S[2], O  (256 columns)
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const uint32_t tmem_S0 = tmem, tmem_S1 = tmem + kNMax, tmem_O = tmem + 2 * kNMax;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        // Metadata is software-pipelined: the next unit record and the next
        // list entry are loaded one step ahead of their use.
        if (lane == 0) {
            tc::prefetch_tmap(&tmap_k);
            tc::prefetch_tmap(&tmap_v);
            tc::prefetch_tmap(&tmap_q);
            const uint64_t policy = tc::policy_evict_first();
            const uint32_t qbox = static_cast<uint32_t>(a.G * a.gmax * 128);
            // Units are claimed from the global work counter (largest first
            // as the plan orders them) and handed to the MMA and softmax roles
            // through a 4-slot ring; claims run two units ahead so a record has
            // arrived by the time it is published.
            auto claim = [&]() -> PlanUnit {
                PlanUnit x{};
                x.pair = -1;
                const int uu = atomicAdd(&hdr->next_unit, 1);
                if (uu < n_units) x = units[uu];
                return x;
            };
            auto publish = [&](uint32_t k, const PlanUnit &x) {
                const int slot = k & 3;
                if (k >= 4) wait_or_abort(sh, &sh.unit_empty[slot], ((k >> 2) - 1) & 1, &hdr->status);
                sh.ring[slot] = x;
                tc::mbar_arrive(&sh.unit_full[slot]);
            };
            uint32_t lb = 0, uc = 0;  // blocks and units loaded by this CTA
            PlanUnit un = claim();
            publish(0, un);
            PlanUnit un_next = claim();
            while (!aborted(sh)) {
                publish(uc + 1, un_next);
                const PlanUnit un_after = claim();  // in flight while this unit's loads are issued
                if (un.pair < 0) break;
                // the group's query terms, once the previous unit's last Q K^T is done
                if (uc > 0 && !wait_or_abort(sh, &sh.q_empty, (uc - 1) & 1, &hdr->status)) break;
                tc::mbar_arrive_expect_tx(&sh.q_full, kTerms * qbox);
                for (int term = 0; term < kTerms; ++term)
                    tc::tma_load_3d(smem + kOffQ + term * kQBytes, &tmap_q, &sh.q_full, 0, un.h * a.G,
                                    term * a.T + un.t0, policy);
                ++uc;
                PlanEntry e_next{};
                if (un.count > 0) e_next = lists[un.entry];
                bool ok = true;
                for (int i = 0; i < un.count; ++i, ++lb) {
                    const PlanEntry e = e_next;
                    if (i + 1 < un.count) e_next = lists[un.entry + i + 1];
                    const int st = lb % kStages;
                    if (lb >= kStages && !wait_or_abort(sh, &sh.kv_empty[st], ((lb / kStages) - 1) & 1, &hdr->status)) {
                        ok = false;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&sh.kv_full[st], 2 * kTile);
                    tc::tma_load_3d(smem + kOffK + st * kTile, &tmap_k, &sh.kv_full[st], 0, un.h, e.page * 128, policy);
                    tc::tma_load_3d(smem + kOffV + st * kTile, &tmap_v, &sh.kv_full[st], 0, un.h, e.page * 128, policy);
                }
                if (!ok) break;
                un = un_next;
                un_next = un_after;
            }
            // let every issued copy land before the CTA may exit
            const uint32_t first = lb > kStages ? lb - kStages : 0;
            for (uint32_t b = first; b < lb; ++b) tc::mbar_wait(&sh.kv_full[b % kStages], (b / kStages) & 1);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t gb = 0, uc = 0;
            const uint32_t sK = tc::smem_u32(smem + kOffK), sV = tc::smem_u32(smem + kOffV);
            const uint32_t sQ = tc::smem_u32(smem + kOffQ);
            const uint32_t sV16 = tc::smem_u32(smem + kOffV16);
            const uint32_t sP = tc::smem_u32(smem + kOffP);
            while (!aborted(sh)) {
                const int slot = uc & 3;
                if (!wait_or_abort(sh, &sh.unit_full[slot], (uc >> 2) & 1, &hdr->status)) break;
                const PlanUnit un = sh.ring[slot];
                if (un.pair < 0) break;
                const int n = pow2_width(un.nt * a.G);
                const uint32_t idesc_qk = tc::idesc_m128(n, false, false);  // E4M3 x E4M3, both K-major
                const uint32_t idesc_pv = tc::idesc_m128(n, true, true);    // F16 x F16, both MN-major
                const tc::Swizzle psw = p_swizzle(n);
                const uint32_t prow = 2 * n;  // bytes per token row of the P tile
                if (!wait_or_abort(sh, &sh.q_full, uc & 1, &hdr->status)) break;
                tc::tc_fence_after();
                auto issue_qk = [&](uint32_t b) {
                    const int st = b % kStages, sb = b & 1;
                    if (!wait_or_abort(sh, &sh.kv_full[st], (b / kStages) & 1, &hdr->status)) return false;
                    if (b >= 2 && !wait_or_abort(sh, &sh.s_empty[sb], ((b >> 1) - 1) & 1, &hdr->status)) return false;
                    tc::tc_fence_after();
                    const uint32_t d = sb ? tmem_S1 : tmem_S0;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t ad = tc::smem_desc(sK + st * kTile + ks * 32, 16, 1024, tc::kSw128);
#pragma unroll
                        for (int term = 0; term < kTerms; ++term)
                            tc::mma_f8(d, ad, tc::smem_desc(sQ + term * kQBytes + ks * 32, 16, 1024, tc::kSw128),
                                       idesc_qk, ks > 0 || term > 0);
                    }
                    tc::mma_commit(&sh.s_full[sb]);
                    return true;
                };
                bool ok = un.count == 0 || issue_qk(gb);
                if (un.count <= 1) tc::mma_commit(&sh.q_empty);  // the unit's last Q K^T is issued
                for (int i = 0; ok && i < un.count; ++i) {
                    const uint32_t b = gb + i;
                    if (i + 1 < un.count) {
                        if (!issue_qk(b + 1)) { ok = false; break; }
                        if (i + 2 == un.count) tc::mma_commit(&sh.q_empty);
                    }
                    const int sb = b & 1;
                    if (!wait_or_abort(sh, &sh.p_full[sb], (b >> 1) & 1, &hdr->status)) { ok = false; break; }
                    tc::tc_fence_after();
                    // O^T[d][n] += V^T[d][tok] P[tok][n]: f16 V (two 64-d atoms, 16 KiB
                    // apart) and P, 16 tokens per instruction
                    const uint32_t vb = sV16 + sb * kV16Tile, pb = sP + sb * kP16Tile;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t ad = tc::smem_desc(vb + ks * 16 * 128, 128 * 128, 1024, tc::kSw128);
                        const uint64_t bd = tc::smem_desc(pb + ks * 16 * prow, 4096, 8 * prow, psw);
                        tc::mma_f16(tmem_O, ad, bd, idesc_pv, i > 0 || ks > 0);
                    }
                    tc::mma_commit(&sh.pv_done[sb]);
                }
                gb += un.count;
                tc::mbar_arrive(&sh.unit_empty[slot]);
                ++uc;
                if (!ok) break;
            }
            if (gb > 0) tc::mbar_wait(&sh.pv_done[(gb - 1) & 1], ((gb - 1) >> 1) & 1);
        }
    } else {
        // ------------------------------------------------ softmax / epilogue
        // The four softmax warps meet at named barriers, so they leave their
        // loops only together: an abort (a timed-out wait anywhere in the
        // CTA) is folded into the per-block vote and acted on after it.
        // Between barriers a timed-out wait only records the abort.
        Soft c;
        c.sh = &sh;
        c.smem = smem;
        c.status = &hdr->status;
        c.counters = reinterpret_cast<int32_t *>(a.ws + a.lay.counters);
        c.partials = reinterpret_cast<float *>(a.ws + a.lay.partials);
        c.st_id = threadIdx.x - 64;
        c.lane = lane;
        c.sw = warp - 2;
        const int quad = warp & 3;                 // TMEM lane quadrant
        c.tok = quad * 32 + lane;                  // token lane of S, d lane of O
        c.lane_base = static_cast<uint32_t>(quad * 32) << 16;
        c.tS0 = tmem_S0;
        c.tS1 = tmem_S1;
        c.tO = tmem_O;
        uint32_t gb = 0, merge_uses = 0;
        bool stop = false;
        const float *cfac = reinterpret_cast<const float *>(a.ws + a.lay.cfac);

        // per-unit metadata is loaded one unit ahead into registers: up to two
        // list entries, one key limit and one logit factor per thread
        PlanEntry pe0{}, pe1{};
        int pL = 0;
        float pcf = 0.f;
        auto prefetch = [&](const PlanUnit &x) {
            pe0 = (c.st_id < x.count) ? lists[x.entry + c.st_id] : PlanEntry{};
            pe1 = (c.st_id + kSoftThreads < x.count) ? lists[x.entry + c.st_id + kSoftThreads] : PlanEntry{};
            int r;
            pL = (c.st_id < x.nt)
                     ? static_cast<int>(token_limit(a.ri, a.ri_s0, a.sl, a.sl_s0, x.t0 + c.st_id, a.R, a.NB, &r))
                     : 0;
            pcf = (c.st_id < x.nt * a.G)
                      ? cfac[static_cast<int64_t>(x.t0 + c.st_id / a.G) * a.Hq + x.h * a.G + c.st_id % a.G]
                      : 0.f;
        };
        uint32_t uc = 0;
        PendingMerge pending{};
        pending.un.pair = -1;
        PlanUnit un{};
        un.pair = -1;
        if (wait_or_abort(sh, &sh.unit_full[0], 0, c.status)) un = sh.ring[0];
        if (un.pair >= 0) prefetch(un);
        while (un.pair >= 0 && !stop) {
            // the next unit's record (published by the producer before it issues
            // this unit's loads) and its metadata, loaded during this unit
            PlanUnit un_next{};
            un_next.pair = -1;
            if (wait_or_abort(sh, &sh.unit_full[(uc + 1) & 3], ((uc + 1) >> 2) & 1, c.status))
                un_next = sh.ring[(uc + 1) & 3];
            if (c.st_id < un.count) sh.ent[c.st_id] = pe0;
            if (c.st_id + kSoftThreads < un.count) sh.ent[c.st_id + kSoftThreads] = pe1;
            if (c.st_id < 16) sh.Lj[c.st_id] = pL;
            if (c.st_id < kNMax) {
                sh.cfac[c.st_id] = pcf;
                sh.m_run[c.st_id] = -INFINITY;
            }
            named_sync();
            if (un_next.pair >= 0) prefetch(un_next);

            const int nch = pow2_width(un.nt * a.G) / 16;
            bool ok;
            if (nch == 1) ok = unit_body<1>(c, a, un, gb);
            else if (nch == 2) ok = unit_body<2>(c, a, un, gb);
            else ok = unit_body<4>(c, a, un, gb);
            if (!ok) break;
            gb += un.count;
            resolve_ticket(c, a, pending, merge_uses);
            if (un.part_row >= 0) take_ticket(c, un, pending);
            tc::mbar_arrive(&sh.unit_empty[uc & 3]);
            // unit-level abort decision, uniform over the four warps
            if (lane == 0) sh.unit_vote[c.sw] = aborted(sh) ? 1 : 0;
            named_sync();
            stop = (sh.unit_vote[0] | sh.unit_vote[1] | sh.unit_vote[2] | sh.unit_vote[3]) != 0;
            named_sync();
            un = un_next;
            ++uc;
        }
        if (!stop) resolve_ticket(c, a, pending, merge_uses);
    }

    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, 4 * kNMax);
}

// ------------------------------------------------------------------ host side

// Tensor map of a [slots, Hkv, D] E4M3 cache: box = 128 tokens x D bytes of
// one kv head, 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const uint8_t *base, int64_t slots, int64_t hkv, int64_t s0, int64_t s1) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(slots)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(s1), static_cast<cuuint64_t>(s0)};
    cuuint32_t box[3] = {kD, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the query terms qterms[term][t][hq][128 bytes]: box = the
// gmax rows x G heads of one group for one term, 128-byte swizzle.
bool make_tmap_q(CUtensorMap *m, const uint8_t *base, int64_t T, int64_t hq, int g, int gmax) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(hq),
                          static_cast<cuuint64_t>(kTerms * T)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(hq * kD)};
    cuuint32_t box[3] = {kD, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(gmax)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int sms = 0;
    bool attr_set = false;
};

DeviceInfo &device_info() {
    static DeviceInfo info[64];
    int dev = 0;
    cudaGetDevice(&dev);
    DeviceInfo &d = info[dev & 63];
    if (d.sms == 0) {
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (d.sms <= 0) d.sms = 1;
    }
    return d;
}

}  // namespace

// The fast path covers: head dim 128, E4M3 caches whose rows are 16-byte
// aligned, G*gmax <= 64, page tables of at most 256 blocks, at most 4096 rows.
cudaError_t launch_attention_tc(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream, bool *used) {
    *used = false;
    const int G = a.Hq / a.Hkv;
    if (a.D != kD || a.NB > kPlanMaxNB || a.T > kPlanMaxT || G > kNMax) return cudaSuccess;
    if ((a.k_s0 % 16) || (a.k_s1 % 16) || (a.v_s0 % 16) || (a.v_s1 % 16)) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(a.k) % 16) || (reinterpret_cast<uintptr_t>(a.v) % 16)) return cudaSuccess;
    if (a.P * 128 > (int64_t(1) << 31) - 1) return cudaSuccess;
    PlanLayout lay(a.T, a.Hq, a.Hkv, a.D, a.NB);
    if (ws == nullptr || ws_bytes < lay.total) return cudaSuccess;

    CUtensorMap tk, tv;
    if (!make_tmap(&tk, a.k, a.P * 128, a.Hkv, a.k_s0, a.k_s1)) return cudaSuccess;
    if (!make_tmap(&tv, a.v, a.P * 128, a.Hkv, a.v_s0, a.v_s1)) return cudaSuccess;

    DeviceInfo &dev = device_info();
    if (!dev.attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        dev.attr_set = true;
    }

    PlanArgs p{};
    p.ri = a.ri; p.ri_s0 = a.ri_s0;
    p.sl = a.sl; p.sl_s0 = a.sl_s0;
    p.bt = a.bt; p.bt_s0 = a.bt_s0; p.bt_s1 = a.bt_s1;
    p.tk = a.tk; p.tk_s0 = a.tk_s0; p.tk_s1 = a.tk_s1; p.tk_s2 = a.tk_s2;
    p.T = a.T; p.R = a.R; p.NB = a.NB; p.K = a.K; p.Hkv = a.Hkv; p.G = G;
    p.gmax = std::min(16, kNMax / G);
    p.P = a.P;
    p.num_ctas = dev.sms;
    p.units_per_cta = 4;
    p.ws = static_cast<char *>(ws);
    p.lay = lay;
    p.q = a.q; p.q_s0 = a.q_s0; p.q_s1 = a.q_s1; p.q_s2 = a.q_s2;
    p.q_dt = a.q_dt;
    p.Hq = a.Hq;
    p.zscale = a.sm_scale * a.k_scale * 1.4426950408889634f;

    CUtensorMap tq;
    if (!make_tmap_q(&tq, reinterpret_cast<const uint8_t *>(p.ws + lay.qterms), a.T, a.Hq, G, p.gmax))
        return cudaSuccess;

    const int64_t q_rows = static_cast<int64_t>(a.T) * a.Hq;
    const int conv_ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(dev.sms - 1, (q_rows + 31) / 32)));
    cudaError_t e = launch_prepare(p, conv_ctas, stream);
    if (e != cudaSuccess) return e;

    TcArgs t{};
    t.ri = a.ri; t.ri_s0 = a.ri_s0;
    t.sl = a.sl; t.sl_s0 = a.sl_s0;
    t.out = a.out; t.o_s0 = a.o_s0; t.o_s1 = a.o_s1; t.o_s2 = a.o_s2;
    t.T = a.T; t.Hq = a.Hq; t.Hkv = a.Hkv; t.G = G; t.R = a.R; t.NB = a.NB; t.gmax = p.gmax;
    t.v_scale = a.v_scale;
    t.ws = static_cast<char *>(ws);
    t.lay = lay;
    attention_tc_kernel<<<dev.sms, kThreads, kSmemBytes, stream>>>(tk, tv, tq, t);
    e = cudaGetLastError();
    if (e == cudaSuccess) *used = true;
    return e;
}

}  // namespace spd
