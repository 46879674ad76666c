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

namespace spd {

cudaError_t launch_attention_tc(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream, bool *used);

namespace {

constexpr int kThreads = 192;         // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int kSoftThreads = 128;
constexpr int kStages = 4;
constexpr int kTile = 128 * 128;      // bytes of one K or V tile
constexpr int kNMax = 64;             // query rows per group (padded)
constexpr float kRaise = 6.0f;        // log2 headroom before the offset is raised
constexpr float kPScale = 4.0f;       // probabilities are stored times 4 (<= 256)
constexpr int kD = 128;

struct TcArgs {
    const void *q;
    int64_t q_s0, q_s1, q_s2;
    const int32_t *ri;
    int64_t ri_s0;
    const int32_t *sl;
    int64_t sl_s0;
    __nv_bfloat16 *out;
    int64_t o_s0, o_s1, o_s2;
    int32_t q_dt;
    int32_t Hkv, G, R, NB;
    float zscale;  // sm_scale * k_scale * log2(e)
    float v_scale;
    char *ws;
    PlanLayout lay;
};

struct __align__(8) Shared {
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], s_empty[2], p_full[2], pv_done[2];
    uint64_t q_full;
    uint32_t tmem_base;
    int abort;
    int combine;
    int vote[2][4];
    int unit_vote[4];
    float m_run[kNMax];   // running exponent offset per query row (log2 units)
    float cfac[kNMax];    // logit factor per query row
    float red[4][kNMax];  // cross-warp reduction scratch
    int colj[kNMax];      // group row of each column
    int Lj[16];           // key limit of each group row
};

// dynamic shared memory: K[kStages], V[kStages], Qhi, Qlo, P[2][hi,lo], Shared
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kStages * kTile;
constexpr int kOffQhi = kOffV + kStages * kTile;
constexpr int kOffQlo = kOffQhi + kNMax * 128;
constexpr int kOffP = kOffQlo + kNMax * 128;
constexpr int kPTile = 128 * kNMax;
constexpr int kOffShared = kOffP + 4 * kPTile;
constexpr int kSmemBytes = kOffShared + static_cast<int>(sizeof(Shared)) + 1024;  // + alignment slack

__device__ __forceinline__ int pow2_width(int n) { return n <= 16 ? 16 : n <= 32 ? 32 : 64; }

__device__ __forceinline__ tc::Swizzle swz_of(int width) {
    return width == 16 ? tc::kSwNone : width == 32 ? tc::kSw32 : tc::kSw64;
}

__device__ __forceinline__ void named_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSoftThreads) : "memory"); }

__device__ __forceinline__ bool aborted(Shared &sh) { return *reinterpret_cast<volatile int *>(&sh.abort) != 0; }

__device__ __forceinline__ bool wait_or_abort(Shared &sh, uint64_t *bar, uint32_t parity, int32_t *status) {
    if (tc::mbar_wait(bar, parity)) return true;
    *reinterpret_cast<volatile int *>(&sh.abort) = 1;
    atomicOr(status, 1);
    return false;
}

__global__ void __launch_bounds__(kThreads, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Shared &sh = *reinterpret_cast<Shared *>(smem + kOffShared);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(a.ws + a.lay.header);
    const PlanGroup *groups = reinterpret_cast<const PlanGroup *>(a.ws + a.lay.groups);
    const PlanPair *pairs = reinterpret_cast<const PlanPair *>(a.ws + a.lay.pairs);
    const PlanEntry *lists = reinterpret_cast<const PlanEntry *>(a.ws + a.lay.lists);
    const PlanUnit *units = reinterpret_cast<const PlanUnit *>(a.ws + a.lay.units);
    int32_t *counters = reinterpret_cast<int32_t *>(a.ws + a.lay.counters);
    float *partials = reinterpret_cast<float *>(a.ws + a.lay.partials);
    const int n_units = hdr->n_units;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&sh.kv_full[i], 1);
            tc::mbar_init(&sh.kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&sh.s_full[i], 1);
            tc::mbar_init(&sh.s_empty[i], kSoftThreads);
            tc::mbar_init(&sh.p_full[i], kSoftThreads);
            tc::mbar_init(&sh.pv_done[i], 1);
        }
        tc::mbar_init(&sh.q_full, kSoftThreads);
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
        if (lane == 0) {
            tc::prefetch_tmap(&tmap_k);
            tc::prefetch_tmap(&tmap_v);
            const uint64_t policy = tc::policy_evict_first();
            uint32_t lb = 0;  // blocks loaded by this CTA
            for (int u = blockIdx.x; u < n_units && !aborted(sh); u += gridDim.x) {
                const PlanUnit un = units[u];
                const PlanPair pr = pairs[un.pair];
                const int h = un.pair % a.Hkv;
                for (int i = 0; i < un.count; ++i, ++lb) {
                    const int st = lb % kStages;
                    if (lb >= kStages && !wait_or_abort(sh, &sh.kv_empty[st], ((lb / kStages) - 1) & 1, &hdr->status))
                        break;
                    const PlanEntry e = lists[pr.list + un.first + i];
                    tc::mbar_arrive_expect_tx(&sh.kv_full[st], 2 * kTile);
                    tc::tma_load_3d(smem + kOffK + st * kTile, &tmap_k, &sh.kv_full[st], 0, h, e.page * 128, policy);
                    tc::tma_load_3d(smem + kOffV + st * kTile, &tmap_v, &sh.kv_full[st], 0, h, e.page * 128, policy);
                }
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
            const uint32_t sQh = tc::smem_u32(smem + kOffQhi), sQl = tc::smem_u32(smem + kOffQlo);
            const uint32_t sP = tc::smem_u32(smem + kOffP);
            for (int u = blockIdx.x; u < n_units && !aborted(sh); u += gridDim.x, ++uc) {
                const PlanUnit un = units[u];
                const PlanGroup gr = groups[un.pair / a.Hkv];
                const int n = pow2_width(gr.nt * a.G);
                const uint32_t idesc_qk = tc::idesc_e4m3(n, false, false);
                const uint32_t idesc_pv = tc::idesc_e4m3(n, true, true);
                const tc::Swizzle psw = swz_of(n);
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
                        tc::mma_f8(d, ad, tc::smem_desc(sQh + ks * 32, 16, 1024, tc::kSw128), idesc_qk, ks > 0);
                        tc::mma_f8(d, ad, tc::smem_desc(sQl + ks * 32, 16, 1024, tc::kSw128), idesc_qk, true);
                    }
                    tc::mma_commit(&sh.s_full[sb]);
                    return true;
                };
                if (un.count > 0 && !issue_qk(gb)) break;
                bool ok = true;
                for (int i = 0; i < un.count; ++i) {
                    const uint32_t b = gb + i;
                    if (i + 1 < un.count && !issue_qk(b + 1)) { ok = false; break; }
                    const int st = b % kStages, sb = b & 1;
                    if (!wait_or_abort(sh, &sh.p_full[sb], (b >> 1) & 1, &hdr->status)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t pbase = sP + sb * 2 * kPTile;
                    // P tile: [128 tokens][n bytes], MN-major; atoms of 8 tokens
                    const uint32_t atom = 8 * n;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t ad = tc::smem_desc(sV + st * kTile + ks * 32 * 128, kTile, 1024, tc::kSw128);
                        const uint32_t poff = ks * 32 * n;
                        const uint64_t bh = (psw == tc::kSwNone)
                                                ? tc::smem_desc(pbase + poff, 128, 4096, tc::kSwNone)
                                                : tc::smem_desc(pbase + poff, 4096, atom, psw);
                        const uint64_t bl = (psw == tc::kSwNone)
                                                ? tc::smem_desc(pbase + kPTile + poff, 128, 4096, tc::kSwNone)
                                                : tc::smem_desc(pbase + kPTile + poff, 4096, atom, psw);
                        tc::mma_f8(tmem_O, ad, bh, idesc_pv, i > 0 || ks > 0);
                        tc::mma_f8(tmem_O, ad, bl, idesc_pv, true);
                    }
                    tc::mma_commit(&sh.pv_done[sb]);
                    tc::mma_commit(&sh.kv_empty[st]);
                }
                gb += un.count;
                if (!ok) break;
            }
            if (gb > 0) tc::mbar_wait(&sh.kv_empty[(gb - 1) % kStages], ((gb - 1) / kStages) & 1);
        }
    } else {
        // ------------------------------------------------ softmax / epilogue
        // The four softmax warps meet at named barriers, so they leave their
        // loops only together: an abort (a timed-out wait anywhere in the
        // CTA) is folded into the per-block vote and acted on after it.
        // Between barriers a timed-out wait only records the abort.
        const int st_id = threadIdx.x - 64;        // 0..127
        const int quad = warp & 3;                 // TMEM lane quadrant
        const int tok = quad * 32 + lane;          // token lane of S, d lane of O
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const int sw = warp - 2;                   // softmax warp index 0..3
        uint32_t gb = 0, uc = 0;
        bool stop = false;
        float lsum[kNMax];

        for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x, ++uc) {
            const PlanUnit un = units[u];
            const PlanPair pr = pairs[un.pair];
            const PlanGroup gr = groups[un.pair / a.Hkv];
            const int h = un.pair % a.Hkv;
            const int rows = gr.nt * a.G;
            const int n = pow2_width(rows);
            const int nchunks = n / 16;

            // ---- queries of the group: power-of-two row scale, E4M3 hi + lo
            uint8_t *qhi = smem + kOffQhi, *qlo = smem + kOffQlo;
            for (int row = sw; row < kNMax; row += 4) {
                uint32_t hi4 = 0, lo4 = 0;
                if (row < rows) {
                    const int j = row / a.G, g = row % a.G;
                    const int t = gr.t0 + j;
                    float x[4];
                    float amax = 0.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        x[e] = load_float(a.q, a.q_dt, t * a.q_s0 + (h * a.G + g) * a.q_s1 + (lane * 4 + e) * a.q_s2);
                        amax = fmaxf(amax, fabsf(x[e]));
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                    float scale = 1.f;
                    if (amax > 0.f && amax < INFINITY) {
                        int ex;
                        frexpf(amax, &ex);
                        scale = ldexpf(1.f, 8 - ex);  // amax * scale in [128, 256)
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) x[e] *= scale;
                    const uint16_t h01 = tc::f32x2_to_e4m3x2(x[1], x[0]);
                    const uint16_t h23 = tc::f32x2_to_e4m3x2(x[3], x[2]);
                    float b0, b1, b2, b3;
                    tc::e4m3x2_to_f32x2(h01, b1, b0);
                    tc::e4m3x2_to_f32x2(h23, b3, b2);
                    const uint16_t l01 = tc::f32x2_to_e4m3x2(x[1] - b1, x[0] - b0);
                    const uint16_t l23 = tc::f32x2_to_e4m3x2(x[3] - b3, x[2] - b2);
                    hi4 = static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16);
                    lo4 = static_cast<uint32_t>(l01) | (static_cast<uint32_t>(l23) << 16);
                    if (lane == 0) {
                        sh.cfac[row] = a.zscale / scale;
                        sh.colj[row] = j;
                    }
                } else if (lane == 0) {
                    sh.cfac[row] = 0.f;
                    sh.colj[row] = 0;
                }
                const uint32_t off = tc::swz_offset(row, lane * 4, 128);
                *reinterpret_cast<uint32_t *>(qhi + off) = hi4;
                *reinterpret_cast<uint32_t *>(qlo + off) = lo4;
            }
            if (st_id < 16) {
                int r;
                sh.Lj[st_id] = (st_id < gr.nt)
                                   ? static_cast<int>(token_limit(a.ri, a.ri_s0, a.sl, a.sl_s0, gr.t0 + st_id, a.R,
                                                                  a.NB, &r))
                                   : 0;
            }
            if (st_id < kNMax) sh.m_run[st_id] = -INFINITY;
#pragma unroll
            for (int c = 0; c < kNMax; ++c) lsum[c] = 0.f;
            tc::fence_proxy_async();
            named_sync();
            tc::mbar_arrive(&sh.q_full);

            // ---- blocks of the unit
            for (int i = 0; i < un.count; ++i) {
                const uint32_t b = gb + i;
                const int sb = b & 1, stg = b % kStages;
                const PlanEntry e = lists[pr.list + un.first + i];
                // validity of this token lane for each group row
                uint32_t vbits = 0;
                int max_valid = 0;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (j < gr.nt && ((e.mask >> j) & 1)) {
                        const int lim = sh.Lj[j] - e.block * 128;
                        max_valid = max(max_valid, lim);
                        vbits |= static_cast<uint32_t>(tok < lim) << j;
                    }
                }
                wait_or_abort(sh, &sh.s_full[sb], (b >> 1) & 1, &hdr->status);
                tc::tc_fence_after();
                float s[kNMax];
                const uint32_t sbase = (sb ? tmem_S1 : tmem_S0) + lane_base;
#pragma unroll
                for (int c = 0; c < kNMax / 16; ++c) {
                    if (c < nchunks) {
                        float v[16];
                        tc::tmem_ld16(sbase + c * 16, v);
#pragma unroll
                        for (int k = 0; k < 16; ++k) s[c * 16 + k] = v[k];
                    }
                }
                tc::tmem_wait_ld();
                tc::tc_fence_before();
                tc::mbar_arrive(&sh.s_empty[sb]);

                bool need = false;
#pragma unroll
                for (int c = 0; c < kNMax; ++c) {
                    if (c < n) {
                        const bool valid = c < rows && ((vbits >> sh.colj[c]) & 1);
                        s[c] = valid ? s[c] * sh.cfac[c] : -INFINITY;
                        need |= s[c] > sh.m_run[c] + kRaise;
                    }
                }
                // votes alternate between two slots by block parity: a warp can
                // be at most one block ahead of the slowest reader
                const int mine = (__any_sync(0xffffffffu, need) ? 1 : 0) | (aborted(sh) ? 2 : 0);
                if (lane == 0) sh.vote[sb][sw] = mine;
                named_sync();
                const int vote = sh.vote[sb][0] | sh.vote[sb][1] | sh.vote[sb][2] | sh.vote[sb][3];
                if (vote & 2) {
                    stop = true;
                    break;
                }
                if (vote & 1) {
                    // raise the offsets to the block maximum; rescale O and the sums
#pragma unroll
                    for (int c = 0; c < kNMax; ++c) {
                        if (c < n) {
                            float mx = s[c];
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                            if (lane == 0) sh.red[sw][c] = mx;
                        }
                    }
                    named_sync();
                    float alpha[kNMax];
                    bool rescale = false;
#pragma unroll
                    for (int c = 0; c < kNMax; ++c) {
                        alpha[c] = 1.f;
                        if (c < n) {
                            const float bm =
                                fmaxf(fmaxf(sh.red[0][c], sh.red[1][c]), fmaxf(sh.red[2][c], sh.red[3][c]));
                            const float old = sh.m_run[c];
                            const float nw = fmaxf(old, bm);
                            if (nw > old) {
                                alpha[c] = (old == -INFINITY) ? 0.f : tc::ex2(old - nw);
                                rescale = true;
                            }
                            lsum[c] *= alpha[c];
                        }
                    }
                    named_sync();  // every thread has read the old offsets
                    if (sw == 0) {
                        for (int c = lane; c < n; c += 32) {
                            const float bm =
                                fmaxf(fmaxf(sh.red[0][c], sh.red[1][c]), fmaxf(sh.red[2][c], sh.red[3][c]));
                            sh.m_run[c] = fmaxf(sh.m_run[c], bm);
                        }
                    }
                    if (rescale && i > 0) {
                        // O holds blocks 0..i-1 of this unit: wait for the last PV
                        wait_or_abort(sh, &sh.pv_done[(b - 1) & 1], ((b - 1) >> 1) & 1, &hdr->status);
                        tc::tc_fence_after();
#pragma unroll
                        for (int c = 0; c < kNMax / 16; ++c) {
                            if (c < nchunks) {
                                float v[16];
                                tc::tmem_ld16(tmem_O + lane_base + c * 16, v);
                                tc::tmem_wait_ld();
#pragma unroll
                                for (int k = 0; k < 16; ++k) v[k] *= alpha[c * 16 + k];
                                tc::tmem_st16(tmem_O + lane_base + c * 16, v);
                            }
                        }
                        tc::tmem_wait_st();
                        tc::tc_fence_before();
                    }
                    named_sync();
                }

                // P buffer sb was read by the PV of block b-2
                if (b >= 2) wait_or_abort(sh, &sh.pv_done[sb], ((b >> 1) - 1) & 1, &hdr->status);
                // value rows past every row's key limit may hold anything
                // (0 * NaN is NaN in the product): zero them
                if (tok >= max_valid) {
                    wait_or_abort(sh, &sh.kv_full[stg], (b / kStages) & 1, &hdr->status);
                    uint4 *vrow = reinterpret_cast<uint4 *>(smem + kOffV + stg * kTile + tok * 128);
#pragma unroll
                    for (int k = 0; k < 8; ++k) vrow[k] = make_uint4(0, 0, 0, 0);
                }
                uint8_t *phi = smem + kOffP + sb * 2 * kPTile;
                uint8_t *plo = phi + kPTile;
#pragma unroll
                for (int c = 0; c < kNMax; c += 16) {
                    if (c < n) {
                        uint32_t wh[4], wl[4];
#pragma unroll
                        for (int k = 0; k < 16; k += 4) {
                            float p[4], hi[4];
#pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2) {
                                const int cc = c + k + e2;
                                p[e2] = (s[cc] == -INFINITY) ? 0.f : tc::ex2(s[cc] - sh.m_run[cc]) * kPScale;
                                lsum[cc] += p[e2];
                            }
                            const uint16_t h01 = tc::f32x2_to_e4m3x2(p[1], p[0]);
                            const uint16_t h23 = tc::f32x2_to_e4m3x2(p[3], p[2]);
                            tc::e4m3x2_to_f32x2(h01, hi[1], hi[0]);
                            tc::e4m3x2_to_f32x2(h23, hi[3], hi[2]);
                            const uint16_t l01 = tc::f32x2_to_e4m3x2(p[1] - hi[1], p[0] - hi[0]);
                            const uint16_t l23 = tc::f32x2_to_e4m3x2(p[3] - hi[3], p[2] - hi[2]);
                            wh[k / 4] = static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16);
                            wl[k / 4] = static_cast<uint32_t>(l01) | (static_cast<uint32_t>(l23) << 16);
                        }
                        const uint32_t off = tc::swz_offset(tok, c, n);
                        *reinterpret_cast<uint4 *>(phi + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                        *reinterpret_cast<uint4 *>(plo + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                    }
                }
                tc::fence_proxy_async();
                tc::mbar_arrive(&sh.p_full[sb]);
            }
            if (stop) break;
            const uint32_t last = gb + un.count - 1;
            gb += un.count;

            // ---- row sums over all 128 token lanes
#pragma unroll
            for (int c = 0; c < kNMax; ++c) {
                if (c < n) {
                    float v = lsum[c];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) sh.red[sw][c] = v;
                }
            }
            // ---- O of this unit (d lane = tok)
            float o[kNMax];
#pragma unroll
            for (int c = 0; c < kNMax; ++c) o[c] = 0.f;
            if (un.count > 0) {
                wait_or_abort(sh, &sh.pv_done[last & 1], (last >> 1) & 1, &hdr->status);
                tc::tc_fence_after();
#pragma unroll
                for (int c = 0; c < kNMax / 16; ++c) {
                    if (c < nchunks) {
                        float v[16];
                        tc::tmem_ld16(tmem_O + lane_base + c * 16, v);
#pragma unroll
                        for (int k = 0; k < 16; ++k) o[c * 16 + k] = v[k];
                    }
                }
                tc::tmem_wait_ld();
                tc::tc_fence_before();
            }
            named_sync();
            const int d = tok;
            if (un.part_row < 0) {
#pragma unroll
                for (int c = 0; c < kNMax; ++c) {
                    if (c < rows) {
                        const float l = sh.red[0][c] + sh.red[1][c] + sh.red[2][c] + sh.red[3][c];
                        const float val = (l > 0.f) ? o[c] * a.v_scale / l : 0.f;
                        const int t = gr.t0 + c / a.G, g = c % a.G;
                        a.out[t * a.o_s0 + (h * a.G + g) * a.o_s1 + d * a.o_s2] = __float2bfloat16_rn(val);
                    }
                }
            } else {
                // partial of a split pair: unnormalised O, offset and sum per row
#pragma unroll
                for (int c = 0; c < kNMax; ++c) {
                    if (c < rows) {
                        float *prow = partials + static_cast<int64_t>(un.part_row + c) * (kD + kPartialStride);
                        prow[d] = o[c];
                        if (d == 0) {
                            prow[kD] = sh.m_run[c];
                            prow[kD + 1] = sh.red[0][c] + sh.red[1][c] + sh.red[2][c] + sh.red[3][c];
                        }
                    }
                }
                __threadfence();
                named_sync();
                if (st_id == 0) {
                    const int done = atomicAdd(&counters[un.pair], 1);
                    sh.combine = (done == pr.n_units - 1);
                }
                named_sync();
                if (sh.combine) {
                    __threadfence();
                    // the last unit of the pair to finish merges all of them
                    for (int c = 0; c < rows; ++c) {
                        float mstar = -INFINITY;
                        for (int k = 0; k < pr.n_units; ++k) {
                            const PlanUnit uk = units[pr.unit0 + k];
                            const float *prow = partials + static_cast<int64_t>(uk.part_row + c) * (kD + kPartialStride);
                            mstar = fmaxf(mstar, __ldcg(prow + kD));
                        }
                        float num = 0.f, den = 0.f;
                        for (int k = 0; k < pr.n_units; ++k) {
                            const PlanUnit uk = units[pr.unit0 + k];
                            const float *prow = partials + static_cast<int64_t>(uk.part_row + c) * (kD + kPartialStride);
                            const float mk = __ldcg(prow + kD);
                            if (mk == -INFINITY) continue;
                            const float wgt = tc::ex2(mk - mstar);
                            num += wgt * __ldcg(prow + d);
                            den += wgt * __ldcg(prow + kD + 1);
                        }
                        const float val = (den > 0.f) ? num * a.v_scale / den : 0.f;
                        const int t = gr.t0 + c / a.G, g = c % a.G;
                        a.out[t * a.o_s0 + (h * a.G + g) * a.o_s1 + d * a.o_s2] = __float2bfloat16_rn(val);
                    }
                }
            }
            // unit-level abort decision, uniform over the four warps
            if (lane == 0) sh.unit_vote[sw] = aborted(sh) ? 1 : 0;
            named_sync();
            stop = (sh.unit_vote[0] | sh.unit_vote[1] | sh.unit_vote[2] | sh.unit_vote[3]) != 0;
            named_sync();
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, 4 * kNMax);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Tensor map of a [slots, Hkv, D] E4M3 cache: box = 128 tokens x D bytes of
// one kv head, 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const uint8_t *base, int64_t slots, int64_t hkv, int64_t s0, int64_t s1) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(slots)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(s1), static_cast<cuuint64_t>(s0)};
    cuuint32_t box[3] = {kD, 1, 128};
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
    p.units_per_cta = 8;
    p.ws = static_cast<char *>(ws);
    p.lay = lay;
    cudaError_t e = launch_plan(p, stream);
    if (e != cudaSuccess) return e;

    TcArgs t{};
    t.q = a.q; t.q_s0 = a.q_s0; t.q_s1 = a.q_s1; t.q_s2 = a.q_s2;
    t.ri = a.ri; t.ri_s0 = a.ri_s0;
    t.sl = a.sl; t.sl_s0 = a.sl_s0;
    t.out = a.out; t.o_s0 = a.o_s0; t.o_s1 = a.o_s1; t.o_s2 = a.o_s2;
    t.q_dt = a.q_dt;
    t.Hkv = a.Hkv; t.G = G; t.R = a.R; t.NB = a.NB;
    t.zscale = a.sm_scale * a.k_scale * 1.4426950408889634f;
    t.v_scale = a.v_scale;
    t.ws = static_cast<char *>(ws);
    t.lay = lay;
    attention_tc_kernel<<<dev.sms, kThreads, kSmemBytes, stream>>>(tk, tv, t);
    e = cudaGetLastError();
    if (e == cudaSuccess) *used = true;
    return e;
}

}  // namespace spd
