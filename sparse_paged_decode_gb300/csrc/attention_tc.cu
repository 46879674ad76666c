// attention_tc.cu -- paged sparse / dense GQA decode attention on the sm_103a
// tensor cores (tcgen05) with TMA-staged FP8 pages.
//
// What it computes is "Kernel ABI" -- attention.decode (see include/spd.h);
// how, in short:
//
//  * Work.  A device planner (plan.cu) groups the query rows of one request
//    that sit together (draft tokens of a verification row), unions the blocks
//    they selected per kv head, and cuts each (group, kv head) block list into
//    units.  A persistent grid claims units from a work counter; a pair cut
//    into several units merges its partials in the last unit to finish (an
//    atomic ticket, no waiting on other CTAs).
//
//  * Roles (16 warps).  Warp 0 streams each selected page's K and V tile
//    (128 tokens x 128 bytes of one kv head) with TMA into a ring of stages,
//    straight from the paged cache through the block table.  Warps 4-7 and
//    8-11 are two softmax groups that take alternate blocks of a unit, each
//    with its own accumulators, and combine them at the unit's end.  Warp 1
//    issues every Q K^T, warps 2 and 3 the P V of one group each (an MMA
//    costs its issuing thread over a hundred cycles however small the tile,
//    so the issue is spread over three threads).  Warps 12-15 widen V.
//
//  * Contractions.  Keys lie on the 128 TMEM lanes and the group's query rows
//    (rows x q heads, padded to N = 16/32/64) on columns:
//        S^T[tok][n]  = K[tok][:] . Qs[n][:]      kind::f8f6f4, E4M3 K as read
//        O^T[d][n]   += V^T[d][tok] . P[tok][n]    kind::f16, f16 V and P
//    Queries enter as E4M3 terms (q = t0 + t1 (+ t2), each row scaled by a
//    power of two so its largest magnitude lies in [128, 256), the factor
//    folded into the logit scale): for a bf16 query two terms (4 + 4
//    significant bits) are exact for every element within 2^9 of its row's
//    largest magnitude; a smaller element's second term falls in E4M3's
//    subnormal range and is rounded there, an absolute error of at most
//    2^-10 in the scaled units (2^-17 of the row's largest magnitude).  Other
//    query types take three terms.  Two terms of a narrow group are stacked along
//    N (one product per k-step, the softmax adds the halves); otherwise the
//    terms accumulate into the same columns.  V is
//    widened to f16 exactly (cvt.rn.f16x2.e4m3x2).  Probabilities are f16
//    (normal down to 2^-14, so tiny weights survive).
//
//  * Softmax.  A group owns the 128 token lanes of its S and the 128 d lanes
//    of its O.  A thread reads its lane's logits of a block from tensor
//    memory in one batch; its row sums stay in registers and are reduced
//    over the lanes once per unit.  The exponent offset per query row is a
//    running maximum raised only when a logit exceeds it by more than 2^14
//    (then O is rescaled in tensor memory): most blocks need no cross-lane
//    reduction.
//
// Synchronisation uses mbarriers between the roles, every wait bounded (a
// timeout sets bit 0 of the workspace status word and the CTA winds down).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "plan.cuh"
#include "spd_internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace spd {

cudaError_t launch_attention_tc(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream, bool *used);

namespace {

constexpr int kThreads = 512;         // 16 warps, roles above
constexpr int kWarpSoft = 4;          // first softmax warp
constexpr int kSoftThreads = 128;     // one softmax group
constexpr int kConvThreads = 128;     // warps 12-15
constexpr int kWarpConv = 12;         // first V-widening warp
constexpr int kStages = 3;
constexpr int kTile = 128 * 128;      // bytes of one K or V tile
constexpr int kNMax = 64;             // query rows per group (padded)
constexpr int kMaxEntries = kPlanMaxNB;
// log2 headroom before a column's offset is raised: p <= 2^14 stays inside
// f16's range with a factor of 4 to spare, and a raise (a group-wide maximum
// and an O rescale, about 2 us) is needed only when a block's logits run more
// than 2^14 above the offset
constexpr float kRaise = 14.0f;
constexpr int kD = 128;
constexpr int kTerms = kQueryTerms;   // E4M3 terms per query element (12 significant bits)
constexpr int kStride = kD + kPartialStride;

// tensor memory columns (512 allocated): two S buffers per softmax group
// (the group's k-th block uses buffer k % 2) at kColS + (2 w + k % 2) * kNMax,
// O of group w at kColO + w * kNMax
constexpr uint32_t kSCols = kNMax;
constexpr uint32_t kColS = 0, kColO = 4 * kSCols;
constexpr uint32_t kTmemCols = 512;
static_assert(kColO + 2 * kNMax <= kTmemCols, "tensor memory columns");

struct TcArgs {
    const int32_t *ri;
    int64_t ri_s0;
    const int32_t *sl;
    int64_t sl_s0;
    __nv_bfloat16 *out;
    int64_t o_s0, o_s1, o_s2;
    int32_t T, Hq, Hkv, G, R, NB, gmax;
    int32_t terms;      // E4M3 query terms: 2 for bf16 queries (exact), 3 otherwise
    int32_t per_token;  // query terms loaded token by token (G >= 8), else one box per group
    float v_scale;
    char *ws;
    PlanLayout lay;
};

// What the softmax needs of a block-list entry: the block and which rows
// selected it.
struct BlockRows {
    uint16_t block;
    uint16_t mask;
};

struct __align__(16) Shared {
    float m_run[2][kNMax];   // running exponent offset per group and query row (log2 units)
    float m_eff[2][kNMax];   // the offset, 0 while a column has none
    float thr[2][kNMax];     // logit above which a column needs a raise: 2^kRaise, -inf while it has no offset
    float cfac[2][kNMax];    // logit factor per query row (double-buffered by unit)
    float alpha[2][kNMax];   // rescale factor of a group's last offset raise
    float delta[2][kNMax];   // change of each offset in that raise
    // per group: per-warp block maxima during the blocks (a raise), per-warp
    // row sums at the unit's end (the two uses never overlap)
    union {
        float red[2][4][kNMax];
        float lsum[2][4][kNMax];
    };
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2][2], s_empty[2][2];  // [group][S buffer]
    uint64_t p_full[2], v_full[2], pv_done[2];
    uint64_t q_full, q_empty, drain[3];
    uint64_t meta_full[2], meta_empty[2];  // unit metadata buffers: V-widening warp 0 -> softmax
    uint64_t unit_full[4], unit_empty[4];  // ring of unit records, producer -> everyone
    PlanUnit ring[4];
    uint32_t tmem_base;
    int abort;
    int combine;
    int rescale[2];
    int vote[2][2][4];
    int unit_vote[8];
    int Lj[2][16];                  // key limit of each group row (double-buffered by unit)
    BlockRows ent[2][kMaxEntries];  // the unit's block list (double-buffered by unit)
    uint8_t nvalid[4][kMaxEntries];  // per V-widening warp: tokens of each block valid for some row
};

// dynamic shared memory: E4M3 K and V stages, query terms, f16 V and P tiles
// (one per softmax group), Shared
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kStages * kTile;
constexpr int kQBytes = kNMax * 128;
constexpr int kOffQ = kOffV + kStages * kTile;
constexpr int kV16Tile = 128 * kD * 2;     // [2 d-halves][128 tokens][64 d] f16
constexpr int kP16Tile = 128 * kNMax * 2;  // [128 tokens][N] f16
constexpr int kOffV16 = kOffQ + kTerms * kQBytes;
constexpr int kOffP = kOffV16 + 2 * kV16Tile;
constexpr int kOffShared = kOffP + 2 * kP16Tile;
constexpr int kSmemBytes = kOffShared + static_cast<int>(sizeof(Shared)) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// a unit record is released by the three MMA issuers, both softmax groups and
// the V-widening warps
constexpr uint32_t kUnitArrivals = 3 + 2 * kSoftThreads + kConvThreads;

// Registers: the launch gives 128 per thread (512 x 128 = 65536); warps 0-3
// (TMA, the MMA issuers, one idle warp) and the V-widening warps drop to 64,
// and the two softmax groups rise to 192: 256 x 64 + 256 x 192 = 65536.
constexpr uint32_t kRegsIssue = 64, kRegsConv = 64, kRegsSoft = 192;
static_assert(128 * kRegsIssue + 128 * kRegsConv + 256 * kRegsSoft <= kThreads * 128, "register split");

__device__ __forceinline__ int pow2_width(int n) { return n <= 16 ? 16 : n <= 32 ? 32 : 64; }

// Two query terms of a group of width n are stacked along N (one Q K^T per
// k-step, 2n logit columns that the softmax adds) when they fit one S buffer
// and the terms are loaded token by token; otherwise the terms accumulate
// into the same n columns.
__device__ __forceinline__ bool stacked_terms(int terms, int per_token, int n) {
    return terms == 2 && per_token && n <= 32;
}

// swizzle of an f16 [tokens][n] tile whose rows are 2n bytes
__device__ __forceinline__ tc::Swizzle p_swizzle(int n) {
    return n == 16 ? tc::kSw32 : n == 32 ? tc::kSw64 : tc::kSw128;
}

// named barriers: 1 + w = softmax group w, 3 = both groups
__device__ __forceinline__ void group_sync(int w) { asm volatile("bar.sync %0, 128;" ::"r"(1 + w) : "memory"); }
__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

__device__ __forceinline__ bool aborted(Shared &sh) { return *reinterpret_cast<volatile int *>(&sh.abort) != 0; }

__device__ __forceinline__ void set_abort(Shared &sh, int32_t *status) {
    *reinterpret_cast<volatile int *>(&sh.abort) = 1;
    atomicOr(status, 1);
}

__device__ __forceinline__ bool wait_or_abort(Shared &sh, uint64_t *bar, uint32_t parity, int32_t *status) {
    if (tc::mbar_wait(bar, parity)) return true;
    set_abort(sh, status);
    return false;
}

// Warp-uniform wait: every lane waits, the warp goes on only if all saw the
// phase (so a warp-collective tcgen05 access that follows is uniform).
__device__ __forceinline__ bool warp_wait(Shared &sh, uint64_t *bar, uint32_t parity, int32_t *status) {
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(bar, parity));
    if (!ok) set_abort(sh, status);
    return ok;
}

// What a softmax thread needs besides the kernel arguments.
struct Soft {
    Shared *sh;
    uint8_t *smem;
    int32_t *status;
    int32_t *counters;
    float *partials;
    uint32_t tmem, lane_base;
    int wg;     // softmax group
    int tok;    // token lane of S, d lane of O
    int lane;
    int sw;     // warp within the group
    int st_id;  // 0..255 over both groups
    int mb;     // metadata buffer of the current unit
};

// Reduction over the 32 lanes of a warp of 16 per-lane columns, transposed:
// lanes l and l+16 end with the reduction of column l & 15.
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce16(float (&v)[16], int lane) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float got = __shfl_xor_sync(0xffffffffu, v[i], 16);
        v[i] = kMax ? fmaxf(v[i], got) : v[i] + got;
    }
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float keep = upper ? v[i + o] : v[i];
            const float send = upper ? v[i] : v[i + o];
            const float got = __shfl_xor_sync(0xffffffffu, send, o);
            v[i] = kMax ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
}

// Copy of columns [16 ch, 16 ch + 16) of a per-thread column array (the
// switch keeps every index compile-time, so the array stays in registers and
// a loop over chunks can stay rolled).
__device__ __forceinline__ void chunk16(const float (&x)[kNMax], int ch, float (&v)[16]) {
    switch (ch) {
        case 0:
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = x[q];
            break;
        case 1:
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = x[16 + q];
            break;
        case 2:
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = x[32 + q];
            break;
        default:
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = x[48 + q];
            break;
    }
}

// This thread's logits of one block (its token lane, N = 16 * nch columns)
// read from S in one batch and masked (-inf where the column is not valid on
// the lane): u = s * cfac - m (log2 units), m the column's offset or 0 while
// it has none.  Returns whether some column needs a raise: a logit more than
// 2^kRaise above its offset, or a valid logit in a column without one.  The
// raise keeps both forms of each offset in shared memory (m or 0, and the
// threshold: 2^kRaise, or -inf without an offset), so a column costs one
// FMA, the mask and one compare.
__device__ __forceinline__ bool load_u(const Shared &sh, int wg, int mb, int nch, bool stacked, uint32_t tS,
                                       uint64_t colmask, float (&u)[kNMax]) {
    // stacked: the second term's logits follow in chunks nch..2nch-1
    const int nld = stacked ? 2 * nch : nch;
#pragma unroll
    for (int ch = 0; ch < kNMax / 16; ++ch)
        if (ch < nld) tc::tmem_ld16(tS + 16 * ch, *reinterpret_cast<float(*)[16]>(&u[16 * ch]));
    tc::tmem_wait_ld();
    if (stacked) {  // n = 16 or 32 (compile-time indices keep u in registers)
        if (nch == 1) {
#pragma unroll
            for (int col = 0; col < 16; ++col) u[col] += u[16 + col];
        } else {
#pragma unroll
            for (int col = 0; col < 32; ++col) u[col] += u[32 + col];
        }
    }
    bool need[4] = {false, false, false, false};
#pragma unroll
    for (int c4 = 0; c4 < kNMax; c4 += 4) {
        if (c4 < 16 * nch) {
            const float4 cf = *reinterpret_cast<const float4 *>(&sh.cfac[mb][c4]);
            const float4 me = *reinterpret_cast<const float4 *>(&sh.m_eff[wg][c4]);
            const float4 th = *reinterpret_cast<const float4 *>(&sh.thr[wg][c4]);
            const float cfs[4] = {cf.x, cf.y, cf.z, cf.w}, mes[4] = {me.x, me.y, me.z, me.w};
            const float ths[4] = {th.x, th.y, th.z, th.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int col = c4 + q;
                const float v = fmaf(u[col], cfs[q], -mes[q]);
                u[col] = ((colmask >> col) & 1) ? v : -INFINITY;
                need[q] |= u[col] > ths[q];
            }
        }
    }
    return need[0] | need[1] | need[2] | need[3];
}

// The blocks of one unit that fall to this softmax group (global block index
// b with b % 2 == group), N = 16 * nch query columns.  Returns false when the
// CTA must stop (an abort, decided uniformly within the group).
__device__ __forceinline__ bool unit_blocks(const Soft &c, const TcArgs &a, const PlanUnit &un, uint32_t gb) {
    Shared &sh = *c.sh;
    const int wg = c.wg, mb = c.mb;
    const int n = pow2_width(un.nt * a.G), nch = n / 16;
    const bool stacked = stacked_terms(a.terms, a.per_token, n);
    const uint64_t gmask = (a.G >= 64) ? ~0ull : ((1ull << a.G) - 1);
    const uint32_t tO = c.tmem + kColO + wg * kNMax + c.lane_base;
    float *m_run = sh.m_run[wg];
    uint8_t *pb = c.smem + kOffP + wg * kP16Tile;
    // row sums of this thread's token lane, reduced over the group at the end
    float lsum[kNMax];
#pragma unroll
    for (int col = 0; col < kNMax; ++col) lsum[col] = 0.f;
    bool ok = true;

    for (int i = ((gb & 1u) == static_cast<uint32_t>(wg)) ? 0 : 1; i < un.count; i += 2) {
        const uint32_t b = gb + i;  // b % 2 == wg
        const uint32_t k = b >> 1;  // this group's block ordinal
        const BlockRows e = sh.ent[mb][i];
        // columns valid on this token lane: selected by the column's row and
        // below that row's key limit
        uint64_t colmask = 0;
        for (int j = 0; j < un.nt; ++j)
            if (((e.mask >> j) & 1) && c.tok < sh.Lj[mb][j] - e.block * 128) colmask |= gmask << (j * a.G);
        // logits relative to the offsets; a column without an offset yet
        // (m = -inf) gives +inf where valid, which forces a raise.  The
        // group's first block of the unit has no offsets at all: it reads
        // s * cfac directly and always takes the raise path.
        float u[kNMax];
        bool need = false;
        const int sb = k & 1;  // S buffer of this block
        const uint32_t tS = c.tmem + kColS + (2 * wg + sb) * kSCols + c.lane_base;
        const bool have = warp_wait(sh, &sh.s_full[wg][sb], (k >> 1) & 1, c.status);
        if (have) {
            tc::tc_fence_after();
            need = load_u(sh, wg, mb, nch, stacked, tS, colmask, u);
        }
        // votes alternate between two slots by block parity: a warp can be at
        // most one block ahead of the slowest reader of its group
        const int mine = (__any_sync(0xffffffffu, need) ? 1 : 0) | (aborted(sh) ? 2 : 0);
        if (c.lane == 0) sh.vote[wg][k & 1][c.sw] = mine;
        group_sync(wg);
        const int vote = sh.vote[wg][k & 1][0] | sh.vote[wg][k & 1][1] | sh.vote[wg][k & 1][2] | sh.vote[wg][k & 1][3];
        if (vote & 2) {
            tc::tc_fence_before();
            tc::mbar_arrive(&sh.s_empty[wg][sb]);
            ok = false;
            break;
        }
        if (vote & 1) {
            // raise: an offset moves to its column's block maximum of
            // s * cfac where that exceeds it by more than 2^kRaise (or where
            // the column had none); O and the sums are scaled by
            // 2^(old - new), and u shifts by the change of its offset.  The
            // block maxima come from u (u + m is s * cfac with m the column's
            // offset, 0 while unset).
#pragma unroll 1
            for (int ch = 0; ch < nch; ++ch) {
                float v[16];
                chunk16(u, ch, v);
                const float mx = warp_transpose_reduce16<true>(v, c.lane);
                if (c.lane < 16) sh.red[wg][c.sw][16 * ch + c.lane] = mx;
            }
            group_sync(wg);
            if (c.sw == 0) {
                bool any = false;
                for (int col = c.lane; col < n; col += 32) {
                    const float bu = fmaxf(fmaxf(sh.red[wg][0][col], sh.red[wg][1][col]),
                                           fmaxf(sh.red[wg][2][col], sh.red[wg][3][col]));
                    const float old = m_run[col];
                    const float meff = (old == -INFINITY) ? 0.f : old;
                    float al = 1.f, delta = 0.f;
                    if (bu != -INFINITY && (old == -INFINITY || bu > kRaise)) {
                        const float bm = meff + bu;
                        al = (old == -INFINITY) ? 0.f : tc::ex2(old - bm);
                        any |= old != -INFINITY;
                        m_run[col] = bm;
                        delta = bu;
                    }
                    sh.alpha[wg][col] = al;
                    sh.delta[wg][col] = delta;
                    const bool set = m_run[col] != -INFINITY;
                    sh.m_eff[wg][col] = set ? m_run[col] : 0.f;
                    sh.thr[wg][col] = set ? kRaise : -INFINITY;
                }
                any = __any_sync(0xffffffffu, any);
                if (c.lane == 0) sh.rescale[wg] = any;
            }
            group_sync(wg);
#pragma unroll
            for (int col = 0; col < kNMax; ++col) {
                if (col < n) {
                    lsum[col] *= sh.alpha[wg][col];
                    u[col] -= sh.delta[wg][col];  // -inf stays -inf
                }
            }
            if (sh.rescale[wg] && i >= 2) {
                // O holds this group's earlier blocks of the unit: wait for
                // its last product, then scale it in place
                if (warp_wait(sh, &sh.pv_done[wg], (k - 1) & 1, c.status)) {
                    tc::tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < nch; ++ch) {
                        float v[16];
                        tc::tmem_ld16(tO + 16 * ch, v);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 16; ++q) v[q] *= sh.alpha[wg][16 * ch + q];
                        tc::tmem_st16(tO + 16 * ch, v);
                        tc::tmem_wait_st();
                    }
                }
            }
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&sh.s_empty[wg][sb]);

        // this group's P tile was read by the product of its previous block
        if (b >= 2) wait_or_abort(sh, &sh.pv_done[wg], (k - 1) & 1, c.status);
        // probabilities p = 2^u <= 2^14 in f16 (11-bit significand, normal
        // from 2^-14 to 65504), the B operand of P V; masked columns have
        // u = -inf, p = 0
#pragma unroll
        for (int c8 = 0; c8 < kNMax; c8 += 8) {
            if (c8 < n) {
                float p[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    p[q] = have ? tc::ex2(u[c8 + q]) : 0.f;
                    lsum[c8 + q] += p[q];
                }
                uint4 w;
                w.x = tc::f32x2_to_f16x2(p[0], p[1]);
                w.y = tc::f32x2_to_f16x2(p[2], p[3]);
                w.z = tc::f32x2_to_f16x2(p[4], p[5]);
                w.w = tc::f32x2_to_f16x2(p[6], p[7]);
                *reinterpret_cast<uint4 *>(pb + tc::swz_offset(c.tok, c8 * 2, 2 * n)) = w;
            }
        }
        tc::fence_proxy_async();
        tc::mbar_arrive(&sh.p_full[wg]);
    }
    // the group's row sums: per warp by a transposed butterfly, per group in
    // shared memory (added up by the unit's end)
#pragma unroll
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
        float v[16];
        chunk16(lsum, ch, v);
        const float tot = warp_transpose_reduce16<false>(v, c.lane);
        if (c.lane < 16) sh.lsum[wg][c.sw][16 * ch + c.lane] = tot;
    }
    return ok;
}

// End of a unit, both groups: combine the two groups' (offset, O, sum) per
// query column and write the normalised output, or the unit's partial when
// its pair is split.  One thread per column first works out the column's two
// weights and its output row; then group w takes columns [w N/2, (w+1) N/2),
// each thread its d lane.
__device__ __forceinline__ void unit_finish(const Soft &c, const TcArgs &a, const PlanUnit &un, uint32_t gb,
                                            bool ok) {
    Shared &sh = *c.sh;
    const int n = pow2_width(un.nt * a.G), half = n / 2;
    const int rows = un.nt * a.G;
    // blocks of the unit per group: group (gb % 2) has the even positions
    const int first = static_cast<int>(gb & 1u);
    const int n_first = (un.count + 1) / 2, n_second = un.count / 2;
    const int mine = (c.wg == first) ? n_first : n_second;
    if (ok && mine > 0) {
        const uint32_t last = gb + ((c.wg == first) ? 2 * (n_first - 1) : 2 * n_second - 1);
        warp_wait(sh, &sh.pv_done[c.wg], (last >> 1) & 1, c.status);
    }
    tc::tc_fence_before();
    soft_sync();  // both groups' products are complete and their offsets final
    tc::tc_fence_after();
    // per-column weights and output rows, in the P tiles (every product of
    // the unit is done; the next unit's probabilities come after this call)
    float2 *fac = reinterpret_cast<float2 *>(c.smem + kOffP);
    int64_t *orow = reinterpret_cast<int64_t *>(c.smem + kOffP + kNMax * sizeof(float2));
    if (c.st_id < n) {
        const int col = c.st_id;
        const bool has0 = (first == 0 ? n_first : n_second) > 0, has1 = (first == 1 ? n_first : n_second) > 0;
        const float m0 = has0 ? sh.m_run[0][col] : -INFINITY;
        const float m1 = has1 ? sh.m_run[1][col] : -INFINITY;
        const float m = fmaxf(m0, m1);
        float w0 = 0.f, w1 = 0.f;
        if (m0 != -INFINITY) w0 = tc::ex2(m0 - m);
        if (m1 != -INFINITY) w1 = tc::ex2(m1 - m);
        const float l0 = (sh.lsum[0][0][col] + sh.lsum[0][1][col]) + (sh.lsum[0][2][col] + sh.lsum[0][3][col]);
        const float l1 = (sh.lsum[1][0][col] + sh.lsum[1][1][col]) + (sh.lsum[1][2][col] + sh.lsum[1][3][col]);
        const float l = w0 * l0 + w1 * l1;
        int64_t off = -1;  // first element of the column's output (or partial) row; -1 for padding
        if (col < rows) {
            if (un.part_row < 0) {
                const float inv = (l > 0.f) ? a.v_scale / l : 0.f;
                w0 *= inv;
                w1 *= inv;
                const int t = un.t0 + col / a.G, g = col % a.G;
                off = t * a.o_s0 + (un.h * a.G + g) * a.o_s1;
            } else {
                // partial of a split pair: unnormalised O, offset and sum
                off = static_cast<int64_t>(un.part_row + col) * kStride;
                c.partials[off + kD] = m;
                c.partials[off + kD + 1] = l;
            }
        }
        fac[col] = make_float2(w0, w1);
        orow[col] = off;
    }
    soft_sync();
    const int d = c.tok;
    const uint32_t base = c.tmem + c.lane_base;
#pragma unroll 1
    for (int cc = 0; cc < half; cc += 8) {
        const int col0 = c.wg * half + cc;
        float o0[8], o1[8];
        tc::tmem_ld8(base + kColO + col0, o0);
        tc::tmem_ld8(base + kColO + kNMax + col0, o1);
        tc::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int64_t off = orow[col0 + q];
            if (off < 0) continue;
            const float2 f = fac[col0 + q];
            // a group without blocks in this unit has weight 0 and stale O
            const float v = ((f.x != 0.f) ? f.x * o0[q] : 0.f) + ((f.y != 0.f) ? f.y * o1[q] : 0.f);
            if (un.part_row < 0)
                a.out[off + d * a.o_s2] = __float2bfloat16_rn(v);
            else
                c.partials[off + d] = v;
        }
    }
    tc::tc_fence_before();
    soft_sync();  // O may now be overwritten by the next unit's products
}

// The last unit of a split pair to finish merges all of them, both softmax
// groups together: warp w (of 8) takes output rows w and w+8 at once (then
// w+16, w+24, ...), every lane four of their d values.  Each lane reads each
// partial's (offset, sum) -- the same address across the warp -- and its d
// values, four partials of two rows per round with an online maximum, so a
// round costs one round trip to L2.  Partials are read with
// ld.global.cg: other CTAs wrote them during this launch.
__device__ __forceinline__ void merge_partials(const Soft &c_, const TcArgs &a_, const PlanUnit &un_) {
    const Soft c = c_;
    const TcArgs a = a_;
    const PlanUnit un = un_;
    constexpr int kRows = 2, kParts = 4;
    const int rows = un.nt * a.G, ns = un.n_split;
    const int warp8 = c.st_id >> 5;  // 0..7 over both groups
    const float *pbase = c.partials + static_cast<int64_t>(un.part_base) * kStride;
    const int64_t kstep = static_cast<int64_t>(rows) * kStride;
    const int d4 = c.lane * 4;
    for (int r0 = warp8; r0 < rows; r0 += 8 * kRows) {
        float m[kRows], den[kRows];
        float4 acc[kRows];
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            m[j] = -INFINITY;
            den[j] = 0.f;
            acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int k0 = 0; k0 < ns; k0 += kParts) {
            float2 ml[kRows][kParts];
            float4 o[kRows][kParts];
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
                const int r = r0 + 8 * j;
                const float *row = pbase + static_cast<int64_t>(r) * kStride;
#pragma unroll
                for (int q = 0; q < kParts; ++q) {
                    if (r < rows && k0 + q < ns) {
                        ml[j][q] = __ldcg(reinterpret_cast<const float2 *>(row + (k0 + q) * kstep + kD));
                        o[j][q] = __ldcg(reinterpret_cast<const float4 *>(row + (k0 + q) * kstep + d4));
                    } else {
                        ml[j][q] = make_float2(-INFINITY, 0.f);
                        o[j][q] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
                float mc = m[j];
#pragma unroll
                for (int q = 0; q < kParts; ++q) mc = fmaxf(mc, ml[j][q].x);
                if (mc == -INFINITY) continue;
                const float sc = (m[j] == -INFINITY) ? 0.f : tc::ex2(m[j] - mc);
                den[j] *= sc;
                acc[j].x *= sc;
                acc[j].y *= sc;
                acc[j].z *= sc;
                acc[j].w *= sc;
#pragma unroll
                for (int q = 0; q < kParts; ++q) {
                    const float w = (ml[j][q].x == -INFINITY) ? 0.f : tc::ex2(ml[j][q].x - mc);
                    den[j] = fmaf(w, ml[j][q].y, den[j]);
                    acc[j].x = fmaf(w, o[j][q].x, acc[j].x);
                    acc[j].y = fmaf(w, o[j][q].y, acc[j].y);
                    acc[j].z = fmaf(w, o[j][q].z, acc[j].z);
                    acc[j].w = fmaf(w, o[j][q].w, acc[j].w);
                }
                m[j] = mc;
            }
        }
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            const int r = r0 + 8 * j;
            if (r >= rows) continue;
            const float inv = (den[j] > 0.f) ? a.v_scale / den[j] : 0.f;
            const int t = un.t0 + r / a.G, g = r % a.G;
            __nv_bfloat16 *dst = a.out + t * a.o_s0 + (un.h * a.G + g) * a.o_s1;
            dst[(d4 + 0) * a.o_s2] = __float2bfloat16_rn(acc[j].x * inv);
            dst[(d4 + 1) * a.o_s2] = __float2bfloat16_rn(acc[j].y * inv);
            dst[(d4 + 2) * a.o_s2] = __float2bfloat16_rn(acc[j].z * inv);
            dst[(d4 + 3) * a.o_s2] = __float2bfloat16_rn(acc[j].w * inv);
        }
    }
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

__device__ __forceinline__ void resolve_ticket(const Soft &c, const TcArgs &a, PendingMerge &pm) {
    Shared &sh = *c.sh;
    if (pm.un.pair < 0) return;
    if (c.st_id == 0) {
        sh.combine = (pm.ticket == pm.un.n_split - 1);
        if (sh.combine) __threadfence();  // the other units' partials before the merge reads them
    }
    soft_sync();
    if (sh.combine) merge_partials(c, a, pm.un);
    soft_sync();
    pm.un.pair = -1;
}

__global__ void __launch_bounds__(kThreads, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Shared &sh = *reinterpret_cast<Shared *>(smem + kOffShared);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(a.ws + a.lay.header);
    const PlanEntry *lists = reinterpret_cast<const PlanEntry *>(a.ws + a.lay.lists);
    const PlanUnit *units = reinterpret_cast<const PlanUnit *>(a.ws + a.lay.units);

    // prologue (barriers, tensor memory, descriptor prefetch) overlaps the
    // planner; global memory is touched only after pdl_wait
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&sh.kv_full[i], 1);
            tc::mbar_init(&sh.kv_empty[i], kConvThreads + 1);  // V widened + Q K^T done
        }
        for (int i = 0; i < 2; ++i) {
            for (int j = 0; j < 2; ++j) {
                tc::mbar_init(&sh.s_full[i][j], 1);
                tc::mbar_init(&sh.s_empty[i][j], kSoftThreads);
            }
            tc::mbar_init(&sh.p_full[i], kSoftThreads);
            tc::mbar_init(&sh.v_full[i], kConvThreads);
            tc::mbar_init(&sh.pv_done[i], 1);
        }
        tc::mbar_init(&sh.q_full, 1);
        tc::mbar_init(&sh.q_empty, 1);
        for (int i = 0; i < 3; ++i) tc::mbar_init(&sh.drain[i], 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&sh.meta_full[i], 32);
            tc::mbar_init(&sh.meta_empty[i], 2 * kSoftThreads);
        }
        for (int i = 0; i < 4; ++i) {
            tc::mbar_init(&sh.unit_full[i], 1);
            tc::mbar_init(&sh.unit_empty[i], kUnitArrivals);
        }
        sh.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(&sh.tmem_base, kTmemCols);
    if (threadIdx.x == 32) {
        tc::prefetch_tmap(&tmap_k);
        tc::prefetch_tmap(&tmap_v);
        tc::prefetch_tmap(&tmap_q);
    }
    tc::pdl_wait();
    tc::pdl_trigger();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    if (warp < kWarpSoft) {
    tc::regs_dec<kRegsIssue>();
    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        // Metadata is software-pipelined: the next unit record and the next
        // list entry are loaded one step ahead of their use.
        if (lane == 0) {
            const int n_units = hdr->n_units;
            const uint64_t policy = tc::policy_evict_first();
            const uint32_t qbox = static_cast<uint32_t>(a.G * a.gmax * 128);  // one term of a group
            // Units are claimed from the global work counter (in plan order,
            // longest first) and handed to the other roles through a 4-slot
            // ring.  The next unit is claimed only once this unit's loads are
            // all issued, so no CTA holds work it cannot start while others
            // run out; the claim's round trip overlaps the draining stages.
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
            while (!aborted(sh) && un.pair >= 0) {
                // the group's query terms, once the previous unit's last Q K^T is done
                if (uc > 0 && !wait_or_abort(sh, &sh.q_empty, (uc - 1) & 1, &hdr->status)) break;
                if (a.per_token) {
                    // term t of token j at rows t*N + j*G when stacked, else
                    // t*64 + j*G (G >= 8: 1 KiB aligned)
                    const int n = pow2_width(un.nt * a.G);
                    const int tstride = stacked_terms(a.terms, a.per_token, n) ? n : kNMax;
                    tc::mbar_arrive_expect_tx(&sh.q_full, a.terms * un.nt * a.G * 128);
                    for (int term = 0; term < a.terms; ++term)
                        for (int j = 0; j < un.nt; ++j)
                            tc::tma_load_3d(smem + kOffQ + (term * tstride + j * a.G) * 128, &tmap_q, &sh.q_full, 0,
                                            un.h * a.G, term * a.T + un.t0 + j, policy);
                } else {
                    // term t of the group at rows t*64
                    tc::mbar_arrive_expect_tx(&sh.q_full, a.terms * qbox);
                    for (int term = 0; term < a.terms; ++term)
                        tc::tma_load_3d(smem + kOffQ + term * kQBytes, &tmap_q, &sh.q_full, 0, un.h * a.G,
                                        term * a.T + un.t0, policy);
                }
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
                un = claim();
                publish(uc, un);
            }
            // let every issued copy land before the CTA may exit
            if (uc > 0) tc::mbar_wait(&sh.q_full, (uc - 1) & 1);
            const uint32_t first = lb > kStages ? lb - kStages : 0;
            for (uint32_t b = first; b < lb; ++b) tc::mbar_wait(&sh.kv_full[b % kStages], (b / kStages) & 1);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- Q K^T issuer
        // An MMA costs its issuing thread over a hundred cycles however small
        // the tile, so the products are spread over three threads in
        // different warps: this one issues every Q K^T (block order), warps 2
        // and 3 the P V of one softmax group each.  Descriptors are built once
        // and advanced by their 16-byte address field.
        if (lane == 0) {
            uint32_t gb = 0, uc = 0;
            const uint64_t dK0 = tc::smem_desc(tc::smem_u32(smem + kOffK), 16, 1024, tc::kSw128);
            const uint64_t dQ0 = tc::smem_desc(tc::smem_u32(smem + kOffQ), 16, 1024, tc::kSw128);
            int32_t *status = &hdr->status;
            while (!aborted(sh)) {
                const int slot = uc & 3;
                if (!wait_or_abort(sh, &sh.unit_full[slot], (uc >> 2) & 1, status)) break;
                const PlanUnit un = sh.ring[slot];
                if (un.pair < 0) break;
                const int n = pow2_width(un.nt * a.G);
                const bool stacked = stacked_terms(a.terms, a.per_token, n);
                // E4M3 x E4M3, both K-major
                const uint32_t idesc_qk = tc::idesc_m128(stacked ? 2 * n : n, false, false);
                const int tstride = ((a.per_token && stacked) ? n : kNMax) * 128;  // bytes between query terms
                if (!wait_or_abort(sh, &sh.q_full, uc & 1, status)) break;
                tc::tc_fence_after();
                if (un.count == 0) tc::mma_commit(&sh.q_empty);
                bool ok = true;
                for (int i = 0; i < un.count; ++i) {
                    const uint32_t b = gb + i;
                    const int w = b & 1;
                    const uint32_t k = b >> 1;  // the group's block ordinal
                    const int st = b % kStages, sb = k & 1;
                    ok = wait_or_abort(sh, &sh.kv_full[st], (b / kStages) & 1, status);
                    // S buffer sb of group w was read by the group's block before last
                    if (ok && k >= 2) ok = wait_or_abort(sh, &sh.s_empty[w][sb], ((k >> 1) - 1) & 1, status);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint32_t tS = tmem + kColS + (2 * w + sb) * kSCols;
                    const uint64_t dk = dK0 + ((st * kTile) >> 4);
                    if (stacked) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) tc::mma_f8(tS, dk + 2 * ks, dQ0 + 2 * ks, idesc_qk, ks > 0);
                    } else {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            for (int term = 0; term < a.terms; ++term)
                                tc::mma_f8(tS, dk + 2 * ks, dQ0 + ((term * tstride) >> 4) + 2 * ks, idesc_qk,
                                           ks > 0 || term > 0);
                    }
                    tc::mma_commit(&sh.s_full[w][sb]);
                    tc::mma_commit(&sh.kv_empty[st]);
                    if (i + 1 == un.count) tc::mma_commit(&sh.q_empty);  // the unit's last Q K^T
                }
                gb += un.count;
                tc::mbar_arrive(&sh.unit_empty[slot]);
                ++uc;
                if (!ok) break;
            }
            // every issued product completes before tensor memory is released
            tc::mma_commit(&sh.drain[0]);
            tc::mbar_wait(&sh.drain[0], 0);
        }
    } else {
        // ---------------------------------------------- P V issuers (warps 2, 3)
        // O^T[d][n] += V^T[d][tok] P[tok][n] for the blocks of softmax group
        // w = warp - 2: f16 V (two 64-d atoms, 16 KiB apart) and P, 16 tokens
        // per instruction; the group's first block of a unit overwrites.
        if (lane == 0) {
            const int w = warp - 2;
            uint32_t gb = 0, uc = 0;
            const uint64_t dV =
                tc::smem_desc(tc::smem_u32(smem + kOffV16 + w * kV16Tile), 128 * 128, 1024, tc::kSw128);
            const uint32_t tO = tmem + kColO + w * kNMax;
            int32_t *status = &hdr->status;
            while (!aborted(sh)) {
                const int slot = uc & 3;
                if (!wait_or_abort(sh, &sh.unit_full[slot], (uc >> 2) & 1, status)) break;
                const PlanUnit un = sh.ring[slot];
                if (un.pair < 0) break;
                const int n = pow2_width(un.nt * a.G);
                const uint32_t idesc_pv = tc::idesc_m128(n, true, true);  // F16 x F16, both MN-major
                const uint32_t prow = 2 * n;                              // bytes per token row of the P tile
                const uint64_t dP =
                    tc::smem_desc(tc::smem_u32(smem + kOffP + w * kP16Tile), 4096, 8 * prow, p_swizzle(n));
                bool ok = true;
                for (int i = ((gb & 1u) == static_cast<uint32_t>(w)) ? 0 : 1; i < un.count; i += 2) {
                    const uint32_t k = (gb + i) >> 1;
                    ok = wait_or_abort(sh, &sh.p_full[w], k & 1, status) &&
                         wait_or_abort(sh, &sh.v_full[w], k & 1, status);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const bool acc = i >= 2;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_f16(tO, dV + ((ks * 16 * 128) >> 4), dP + ((ks * 16 * prow) >> 4), idesc_pv,
                                    acc || ks > 0);
                    tc::mma_commit(&sh.pv_done[w]);
                }
                gb += un.count;
                tc::mbar_arrive(&sh.unit_empty[slot]);
                ++uc;
                if (!ok) break;
            }
            tc::mma_commit(&sh.drain[1 + w]);
            tc::mbar_wait(&sh.drain[1 + w], 0);
        }
    }
    } else if (warp >= kWarpConv) {
        tc::regs_dec<kRegsConv>();
        // ------------------------------------------------------- V widening
        // E4M3 V rows (128-byte swizzled TMA tile) -> f16 in two 64-d halves
        // with 128-byte swizzle, the A operand of P V, one token row per
        // thread; the E4M3 stage is released once the Q K^T of the same block
        // is done too.
        const int ct = threadIdx.x - kWarpConv * 32;
        const int cw = ct >> 5;
        uint8_t *nvalid = sh.nvalid[cw];
        const float *cfac_g = reinterpret_cast<const float *>(a.ws + a.lay.cfac);
        uint32_t gb = 0, uc = 0;
        for (;;) {
            const int slot = uc & 3;
            if (!wait_or_abort(sh, &sh.unit_full[slot], (uc >> 2) & 1, &hdr->status)) break;
            const PlanUnit un = sh.ring[slot];
            if (un.pair < 0) break;
            // warp 0 also stages the unit's metadata for the softmax groups:
            // block list, key limit per row, logit factor per query column
            const int mb = uc & 1;
            if (cw == 0 && uc >= 2 && !wait_or_abort(sh, &sh.meta_empty[mb], ((uc >> 1) - 1) & 1, &hdr->status))
                break;
            // tokens of each block valid for some row of the unit (each warp
            // its own copy); the rest -- slots no request owns may hold any
            // code, NaN included -- are written as zeros
            int my_lim = 0;
            if (lane < un.nt) {
                int r;
                my_lim = static_cast<int>(token_limit(a.ri, a.ri_s0, a.sl, a.sl_s0, un.t0 + lane, a.R, a.NB, &r));
            }
            for (int i0 = 0; i0 < un.count; i0 += 32) {
                const int i = i0 + lane;
                PlanEntry e{};
                if (i < un.count) e = lists[un.entry + i];
                int m = 0;
                for (int j = 0; j < un.nt; ++j) {
                    const int lj = __shfl_sync(0xffffffffu, my_lim, j);
                    if ((e.mask >> j) & 1) m = max(m, lj);
                }
                if (i < un.count) {
                    nvalid[i] = static_cast<uint8_t>(min(128, max(0, m - e.block * 128)));
                    if (cw == 0) sh.ent[mb][i] = BlockRows{e.block, e.mask};
                }
            }
            if (cw == 0) {
                if (lane < 16) sh.Lj[mb][lane] = (lane < un.nt) ? my_lim : 0;
                for (int r = lane; r < kNMax; r += 32)
                    sh.cfac[mb][r] = (r < un.nt * a.G)
                                         ? cfac_g[static_cast<int64_t>(un.t0 + r / a.G) * a.Hq + un.h * a.G + r % a.G]
                                         : 0.f;
                tc::mbar_arrive(&sh.meta_full[mb]);
            }
            __syncwarp();
            bool ok = true;
            for (int i = 0; i < un.count; ++i) {
                const uint32_t b = gb + i;
                const int stg = b % kStages, vb = b & 1;
                ok = wait_or_abort(sh, &sh.kv_full[stg], (b / kStages) & 1, &hdr->status);
                // the f16 tile vb was read by the product of block b-2
                if (ok && b >= 2) ok = wait_or_abort(sh, &sh.pv_done[vb], ((b >> 1) - 1) & 1, &hdr->status);
                if (!ok) break;
                const int lim = nvalid[i];
                const int tok = ct;
                const uint8_t *vsrc = smem + kOffV + stg * kTile + tok * 128;
                uint8_t *vdst = smem + kOffV16 + vb * kV16Tile + tok * 128;
                const int sw8 = tok & 7;
                // a d-half (64 values: 4 source chunks) at a time, its
                // loads issued together
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint4 x[4];
                    if (tok < lim) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            x[q] = *reinterpret_cast<const uint4 *>(vsrc + (((4 * hh + q) ^ sw8) << 4));
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q) x[q] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    uint8_t *half = vdst + hh * (128 * 128);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t f[8];
                        tc::e4m3x4_to_f16x4(x[q].x, f[0], f[1]);
                        tc::e4m3x4_to_f16x4(x[q].y, f[2], f[3]);
                        tc::e4m3x4_to_f16x4(x[q].z, f[4], f[5]);
                        tc::e4m3x4_to_f16x4(x[q].w, f[6], f[7]);
                        *reinterpret_cast<uint4 *>(half + (((2 * q) ^ sw8) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
                        *reinterpret_cast<uint4 *>(half + (((2 * q + 1) ^ sw8) << 4)) =
                            make_uint4(f[4], f[5], f[6], f[7]);
                    }
                }
                tc::fence_proxy_async();
                tc::mbar_arrive(&sh.kv_empty[stg]);
                tc::mbar_arrive(&sh.v_full[vb]);
            }
            if (!ok) break;
            __syncwarp();  // the counts are rewritten for the next unit
            gb += un.count;
            tc::mbar_arrive(&sh.unit_empty[slot]);
            ++uc;
        }
    } else {
        tc::regs_inc<kRegsSoft>();
        // ------------------------------------------------ softmax / epilogue
        // The eight softmax warps meet at named barriers, so they leave their
        // loops only together: an abort (a timed-out wait anywhere in the
        // CTA) is folded into the per-block vote of each group and into a
        // unit-level vote of both, and acted on after it.
        Soft c;
        c.sh = &sh;
        c.smem = smem;
        c.status = &hdr->status;
        c.counters = reinterpret_cast<int32_t *>(a.ws + a.lay.counters);
        c.partials = reinterpret_cast<float *>(a.ws + a.lay.partials);
        c.st_id = threadIdx.x - kWarpSoft * 32;
        c.wg = (warp - kWarpSoft) >> 2;
        c.lane = lane;
        c.sw = warp & 3;                          // TMEM lane quadrant
        c.tok = c.sw * 32 + lane;                 // token lane of S, d lane of O
        c.lane_base = static_cast<uint32_t>(c.sw * 32) << 16;
        c.tmem = tmem;
        uint32_t gb = 0, uc = 0;
        PendingMerge pending{};
        pending.un.pair = -1;
        // uniform decisions of both groups: bit 0 abort, bit 1 no more units
        auto vote = [&](int mine) -> int {
            if (lane == 0) sh.unit_vote[warp - kWarpSoft] = mine;
            soft_sync();
            int all = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) all |= sh.unit_vote[w];
            soft_sync();
            return all;
        };
        PlanUnit un{};
        un.pair = -1;
        if (wait_or_abort(sh, &sh.unit_full[0], 0, c.status)) un = sh.ring[0];
        int state = vote((aborted(sh) ? 1 : 0) | (un.pair < 0 ? 2 : 0));
        while (state == 0) {
            c.mb = uc & 1;
            wait_or_abort(sh, &sh.meta_full[c.mb], (uc >> 1) & 1, c.status);  // a timeout shows in the votes
            if (c.st_id < 2 * kNMax) {
                const int g = c.st_id / kNMax, col = c.st_id % kNMax;
                sh.m_run[g][col] = -INFINITY;
                sh.m_eff[g][col] = 0.f;
                sh.thr[g][col] = -INFINITY;
            }
            soft_sync();
            const bool ok = unit_blocks(c, a, un, gb);
            unit_finish(c, a, un, gb, ok);
            tc::mbar_arrive(&sh.meta_empty[c.mb]);
            gb += un.count;
            // the next unit's record (published before this unit's loads)
            PlanUnit nx{};
            nx.pair = -1;
            if (wait_or_abort(sh, &sh.unit_full[(uc + 1) & 3], ((uc + 1) >> 2) & 1, c.status))
                nx = sh.ring[(uc + 1) & 3];
            state = vote(((aborted(sh) || !ok) ? 1 : 0) | (nx.pair < 0 ? 2 : 0));
            if (!(state & 1)) {
                resolve_ticket(c, a, pending);
                if (un.part_row >= 0) take_ticket(c, un, pending);
                if (state & 2) resolve_ticket(c, a, pending);
            }
            tc::mbar_arrive(&sh.unit_empty[uc & 3]);
            un = nx;
            ++uc;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
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

// Tensor map of the query terms qterms[term][t][hq][128 bytes]: box = G heads
// x box_rows tokens (one token, or a whole group) of one term, 128-byte
// swizzle.
bool make_tmap_q(CUtensorMap *m, const uint8_t *base, int64_t T, int64_t hq, int g, int box_rows) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(hq),
                          static_cast<cuuint64_t>(kTerms * T)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(hq * kD)};
    cuuint32_t box[3] = {kD, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Query rows of one request that share a unit (a group).  A group reads each
// block of the union of its rows' selections once, but the softmax cost of a
// block grows with the group's width: 16 columns cost about half of 32 or 64
// (measured).  Dense calls and groups no wider than 16 columns always group.
// For sparse calls whose groups would be wider, the union of g independent
// K-of-NB selections is expected to hold NB (1 - (1 - K/NB)^g) blocks; when
// twice that exceeds the g K blocks the rows would read one by one (little
// overlap), each row is a group of its own.
int group_rows(const AttnArgs &a, int G) {
    const int g = std::min(16, kNMax / G);
    if (a.tk == nullptr || g * G <= 16 || a.K >= a.NB || a.NB <= 0) return g;
    const double keep = 1.0 - static_cast<double>(a.K) / a.NB;
    const double uni = a.NB * (1.0 - std::pow(keep, g));
    return (2.0 * uni > static_cast<double>(g) * a.K) ? 1 : g;
}

}  // namespace

// The fast path covers: head dim 128, E4M3 caches whose rows are 16-byte
// aligned, G*gmax <= 64, page tables of at most 256 blocks, at most 4096 rows.
cudaError_t launch_attention_tc(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream, bool *used) {
    *used = false;
    const int G = a.Hq / a.Hkv;
    if (a.kv_dt != SPD_E4M3) return cudaSuccess;
    if (a.D != kD || a.NB > kPlanMaxNB || a.T > kPlanMaxT || G > kNMax) return cudaSuccess;
    if ((a.k_s0 % 16) || (a.k_s1 % 16) || (a.v_s0 % 16) || (a.v_s1 % 16)) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(a.k) % 16) || (reinterpret_cast<uintptr_t>(a.v) % 16)) return cudaSuccess;
    if (a.P * 128 > (int64_t(1) << 31) - 1) return cudaSuccess;
    PlanLayout lay(a.T, a.Hq, a.Hkv, a.D, a.NB);
    if (ws == nullptr || ws_bytes < lay.total) return cudaSuccess;

    CUtensorMap tk, tv;
    if (!make_tmap(&tk, a.k, a.P * 128, a.Hkv, a.k_s0, a.k_s1)) return cudaSuccess;
    if (!make_tmap(&tv, a.v, a.P * 128, a.Hkv, a.v_s0, a.v_s1)) return cudaSuccess;

    const int sms = device_sm_count();
    {
        cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(attention_tc_kernel), kSmemBytes);
        if (e != cudaSuccess) return e;
    }

    PlanArgs p{};
    p.ri = a.ri; p.ri_s0 = a.ri_s0;
    p.sl = a.sl; p.sl_s0 = a.sl_s0;
    p.bt = a.bt; p.bt_s0 = a.bt_s0; p.bt_s1 = a.bt_s1;
    p.tk = a.tk; p.tk_s0 = a.tk_s0; p.tk_s1 = a.tk_s1; p.tk_s2 = a.tk_s2;
    p.T = a.T; p.R = a.R; p.NB = a.NB; p.K = a.K; p.Hkv = a.Hkv; p.G = G;
    p.gmax = group_rows(a, G);
    p.P = a.P;
    p.num_ctas = sms;
    p.ws = static_cast<char *>(ws);
    p.lay = lay;
    p.q = a.q; p.q_s0 = a.q_s0; p.q_s1 = a.q_s1; p.q_s2 = a.q_s2;
    p.q_dt = a.q_dt;
    p.Hq = a.Hq;
    p.zscale = a.sm_scale * a.k_scale * 1.4426950408889634f;
    if (!plan_configure(&p)) return cudaSuccess;

    CUtensorMap tq;
    // with G >= 8 a token's G query rows are 1 KiB, so terms can be loaded
    // (and stacked) token by token
    const bool per_token = G >= 8;
    if (!make_tmap_q(&tq, reinterpret_cast<const uint8_t *>(p.ws + lay.qterms), a.T, a.Hq, G,
                     per_token ? 1 : p.gmax))
        return cudaSuccess;

    const int64_t q_rows = static_cast<int64_t>(a.T) * a.Hq;
    // query conversion: 64 rows per CTA (four per warp), up to two CTAs per SM
    const int conv_ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(2 * sms - 1, (q_rows + 63) / 64)));
    cudaError_t e = launch_prepare(p, conv_ctas, stream);
    if (e != cudaSuccess) return e;

    TcArgs t{};
    t.ri = a.ri; t.ri_s0 = a.ri_s0;
    t.sl = a.sl; t.sl_s0 = a.sl_s0;
    t.out = a.out; t.o_s0 = a.o_s0; t.o_s1 = a.o_s1; t.o_s2 = a.o_s2;
    t.T = a.T; t.Hq = a.Hq; t.Hkv = a.Hkv; t.G = G; t.R = a.R; t.NB = a.NB; t.gmax = p.gmax;
    t.terms = (a.q_dt == SPD_BF16) ? 2 : kTerms;  // bf16 queries are exact in two E4M3 terms
    t.per_token = per_token ? 1 : 0;
    t.v_scale = a.v_scale;
    t.ws = static_cast<char *>(ws);
    t.lay = lay;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attention_tc_kernel, tk, tv, tq, t);
    if (e == cudaSuccess) *used = true;
    return e;
}

}  // namespace spd
