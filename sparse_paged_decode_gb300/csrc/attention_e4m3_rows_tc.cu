// attention_e4m3_rows_tc.cu -- paged sparse / dense GQA decode attention over
// an FP8-E4M3 K/V cache with static scalar scales ("Kernel ABI" --
// attention.decode; "MiniMax-M3 decode through the ATOM kernel library":
// FP8 K/V with one scale each) on the sm_103a tensor cores, for bf16 queries
// of head dim 128, with the query rows on the rows of the MMA.
//
// Work comes from the device planner (plan.cu): a group of consecutive query
// rows of one request (up to 128 / G tokens) and one kv head form a pair
// whose block list is the union of the rows' selections; lists are cut into
// units, a persistent grid of two CTAs per SM claims units from the work
// counter, and a pair split over several units leaves fp32 partials that the
// last unit to finish merges (an atomic ticket, no waiting).  The planner
// also writes each query row as two E4M3 terms (q = 2^-e (t0 + t1), exact
// for a bf16 element within 2^9 of its row's largest magnitude) and the
// row's logit factor c = sm_scale * k_scale * log2(e) * 2^-e.
//
// Per unit, half a page (64 keys) at a time:
//   S  = Q K^T       kind::f8f6f4, M = 128 query rows (token j, head g ->
//                    row j * G + g), N = 64 keys, K = 128 dims; the two query
//                    terms accumulate into the same columns, K as read from
//                    the cache; double-buffered in tensor memory
//   P  = 2^(S c - m) one thread per row: the row's 64 logits stay in its
//                    registers (block max, sum, offset raise need no
//                    exchange); p <= 2^kRaise, stored as f16
//   O += P V         kind::f16, P from tensor memory (written over its own S
//                    buffer), V widened from E4M3 to f16 (exact) by two
//                    warps into one of two tiles, MN-major
// K and V half pages are TMA-gathered straight from the paged cache through
// the block list (64 slots of 128 bytes, 128-byte swizzle).  A CTA takes 112
// KB of shared memory and 256 tensor-memory columns, so two share an SM and
// one's per-block chain runs while the other waits on its own.  With P in
// tensor memory the softmax of a half page no longer waits for the previous
// half page's product (only to rescale O after an offset raise).
//
// Roles (8 warps): warps 0-3 run the softmax and the unit epilogue (warp w
// reads TMEM lanes 32 w .. +31), warp 4 claims units and issues the TMA
// loads, warp 5 owns tensor memory and issues every MMA, warps 6-7 widen V.
// Every wait is bounded: a wait that gives up sets bit 0 of the workspace
// status word and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <set>

#include "plan.cuh"
#include "spd_internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace spd {

cudaError_t launch_attention_e4m3_rows(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream,
                                       bool *used);

namespace {

constexpr int kD = 128;
constexpr int kM = 128;            // query rows of a unit (padded)
constexpr int kKeys = 128;         // slots per page
constexpr int kHalf = 64;          // keys per block of the products: half a page
constexpr int kThreads = 256;      // warps 0-3 softmax / epilogue, 4 TMA, 5 MMA, 6-7 V widening
constexpr int kSoftThreads = 128;
constexpr int kConvThreads = 64;
constexpr int kWarpTma = 4, kWarpMma = 5, kWarpConv = 6;
constexpr int kStages = 3;         // K and V half-page stages of E4M3
constexpr int kTerms = 2;               // E4M3 terms of a bf16 query
constexpr int kQTile = kM * 128;        // one query term: 128 rows x 128 bytes
constexpr int kKVHalf = kHalf * 128;    // E4M3 half page of one kv head: 64 slots x 128 bytes
constexpr int kV16Box = kHalf * 128;    // 64 dims of a widened half page: 64 keys x 128 bytes
constexpr int kV16Tile = 2 * kV16Box;   // 64 keys x 128 dims of f16
constexpr float kRaise = 8.0f;
constexpr int kStride = kD + kPartialStride;  // floats per partial row

// dynamic shared memory (1024-byte aligned tiles): two query terms, three K
// and three V stages of E4M3, two widened V tiles (P lives in tensor memory)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTerms * kQTile;
constexpr int kOffV = kOffK + kStages * kKVHalf;
constexpr int kOffV16 = kOffV + kStages * kKVHalf;
constexpr int kTilesEnd = kOffV16 + 2 * kV16Tile;

struct Shared {
    uint64_t unit_full[4], unit_empty[4];
    uint64_t q_full, q_empty;
    uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
    uint64_t s_full[2], s_free[2];  // S buffer free: the product that read its P is done
    uint64_t v16_free[2];           // widened V tile free: the product that read it is done
    uint64_t v16_full[2];           // widened V tile written
    uint64_t p_full[2];  // P of S buffer b % 2 written (one barrier per buffer: the
                         // softmax may hand off the next buffer's P before the
                         // product of this one is issued)
    uint64_t pv_done, o_free, drain;
    PlanUnit ring[4];
    uint32_t tmem_base;
    int abort;
    int last;     // the unit that took the last ticket of its pair merges
};

// The barriers sit in the padding below the aligned tiles when it is large
// enough, else after them; either way a CTA needs the tiles plus 1023 bytes,
// which lets two CTAs share an SM.
static_assert(sizeof(Shared) <= 511, "barriers fit the alignment padding or after the tiles");
constexpr int kSmemBytes = kTilesEnd + 1023;
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");

// tensor memory: S buffers at columns 0 and 64, O at 128
constexpr uint32_t kColS = 0, kColO = 2 * kHalf, kTmemCols = 256;
// a unit record is released by the MMA issuer, the softmax and the V-widening threads
constexpr uint32_t kUnitArrivals = 1 + kSoftThreads + kConvThreads;
// Registers: the launch gives 128 per thread (two CTAs of 256 threads per
// SM); the softmax warpgroup rises to 184 and the other one (TMA, MMA,
// V widening) drops to 72: 128 x 184 + 128 x 72 = 256 x 128.
constexpr uint32_t kRegsSoft = 184, kRegsOther = 72;
static_assert(128 * kRegsSoft + 128 * kRegsOther <= kThreads * 128, "register split");

struct RowsArgs {
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

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

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

// Warp-uniform wait: the warp goes on only if every lane saw the phase.
__device__ __forceinline__ bool warp_wait(Shared &sh, uint64_t *bar, uint32_t parity, int32_t *status) {
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(bar, parity));
    if (!ok) set_abort(sh, status);
    return ok;
}

// Named barrier of the 128 softmax threads, and the same barrier reducing a
// flag (true if any thread's is).  Every softmax thread reaches every one of
// them: a failed wait never skips one, it only raises the flag of the next
// vote, which all threads then act on together.
__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool soft_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v))
        : "memory");
    return r != 0;
}

// The last unit of a split pair to finish merges every unit's partial: warp w
// of the softmax takes rows w, w + 4, ... two at a time, each lane four head
// dims; the (offset, sum) and output values of two partials of both rows are
// loaded together, then folded with an online maximum.  Partials are read
// with ld.global.cg: other CTAs wrote them during this launch.
__device__ void merge_pair(const RowsArgs &a, const PlanUnit &un, const float *partials, int st_id) {
    constexpr int kParts = 2;
    const int rows = un.nt * a.G, ns = un.n_split;
    const int w = st_id >> 5, d4 = (st_id & 31) * 4;
    const float *pbase = partials + static_cast<int64_t>(un.part_base) * kStride;
    const int64_t kstep = static_cast<int64_t>(rows) * kStride;
    for (int r0 = w; r0 < rows; r0 += 8) {
        float m[2] = {-INFINITY, -INFINITY}, den[2] = {0.f, 0.f};
        float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
        for (int k0 = 0; k0 < ns; k0 += kParts) {
            float2 ml[2][kParts];
            float4 o[2][kParts];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = r0 + 4 * u;
#pragma unroll
                for (int q = 0; q < kParts; ++q) {
                    if (r < rows && k0 + q < ns) {
                        const float *row = pbase + (k0 + q) * kstep + static_cast<int64_t>(r) * kStride;
                        ml[u][q] = __ldcg(reinterpret_cast<const float2 *>(row + kD));
                        o[u][q] = __ldcg(reinterpret_cast<const float4 *>(row + d4));
                    } else {
                        ml[u][q] = make_float2(-INFINITY, 0.f);
                        o[u][q] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float mc = m[u];
#pragma unroll
                for (int q = 0; q < kParts; ++q) mc = fmaxf(mc, ml[u][q].x);
                if (mc == -INFINITY) continue;
                const float sc = (m[u] == -INFINITY) ? 0.f : tc::ex2(m[u] - mc);
                den[u] *= sc;
                acc[u].x *= sc;
                acc[u].y *= sc;
                acc[u].z *= sc;
                acc[u].w *= sc;
#pragma unroll
                for (int q = 0; q < kParts; ++q) {
                    const float wt = (ml[u][q].x == -INFINITY) ? 0.f : tc::ex2(ml[u][q].x - mc);
                    den[u] = fmaf(wt, ml[u][q].y, den[u]);
                    acc[u].x = fmaf(wt, o[u][q].x, acc[u].x);
                    acc[u].y = fmaf(wt, o[u][q].y, acc[u].y);
                    acc[u].z = fmaf(wt, o[u][q].z, acc[u].z);
                    acc[u].w = fmaf(wt, o[u][q].w, acc[u].w);
                }
                m[u] = mc;
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int r = r0 + 4 * u;
            if (r >= rows) continue;
            const float inv = (den[u] > 0.f) ? a.v_scale / den[u] : 0.f;
            __nv_bfloat16 *dst = a.out + static_cast<int64_t>(un.t0 + r / a.G) * a.o_s0 +
                                 static_cast<int64_t>(un.h * a.G + r % a.G) * a.o_s1;
            if (a.o_s2 == 1 && (reinterpret_cast<uintptr_t>(dst + d4) & 7) == 0) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(acc[u].x * inv, acc[u].y * inv);
                __nv_bfloat162 hi = __floats2bfloat162_rn(acc[u].z * inv, acc[u].w * inv);
                uint2 w2;
                w2.x = *reinterpret_cast<uint32_t *>(&lo);
                w2.y = *reinterpret_cast<uint32_t *>(&hi);
                *reinterpret_cast<uint2 *>(dst + d4) = w2;
            } else {
                dst[static_cast<int64_t>(d4 + 0) * a.o_s2] = __float2bfloat16_rn(acc[u].x * inv);
                dst[static_cast<int64_t>(d4 + 1) * a.o_s2] = __float2bfloat16_rn(acc[u].y * inv);
                dst[static_cast<int64_t>(d4 + 2) * a.o_s2] = __float2bfloat16_rn(acc[u].z * inv);
                dst[static_cast<int64_t>(d4 + 3) * a.o_s2] = __float2bfloat16_rn(acc[u].w * inv);
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2)
attention_e4m3_rows_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ RowsArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const bool bar_below = static_cast<size_t>(smem - smem_raw) >= sizeof(Shared);
    Shared &sh = *reinterpret_cast<Shared *>(bar_below ? smem_raw : smem + kTilesEnd);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(a.ws + a.lay.header);
    const PlanEntry *lists = reinterpret_cast<const PlanEntry *>(a.ws + a.lay.lists);
    const PlanUnit *units = reinterpret_cast<const PlanUnit *>(a.ws + a.lay.units);
    int32_t *status = &hdr->status;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) {
            tc::mbar_init(&sh.unit_full[i], 1);
            tc::mbar_init(&sh.unit_empty[i], kUnitArrivals);
        }
        tc::mbar_init(&sh.q_full, 1);
        tc::mbar_init(&sh.q_empty, 1);
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&sh.k_full[i], 1);
            tc::mbar_init(&sh.k_empty[i], 1);
            tc::mbar_init(&sh.v_full[i], 1);
            tc::mbar_init(&sh.v_empty[i], kConvThreads);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&sh.s_full[i], 1);
            tc::mbar_init(&sh.s_free[i], 1);
            tc::mbar_init(&sh.v16_free[i], 1);
            tc::mbar_init(&sh.v16_full[i], kConvThreads);
        }
        tc::mbar_init(&sh.p_full[0], kSoftThreads);
        tc::mbar_init(&sh.p_full[1], kSoftThreads);
        tc::mbar_init(&sh.pv_done, 1);
        tc::mbar_init(&sh.o_free, kSoftThreads);
        tc::mbar_init(&sh.drain, 1);
        sh.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == kWarpMma) tc::tmem_alloc(&sh.tmem_base, kTmemCols);
    if (threadIdx.x == kWarpTma * 32) {
        tc::prefetch_tmap(&tmap_q);
        tc::prefetch_tmap(&tmap_k);
        tc::prefetch_tmap(&tmap_v);
    }
    // the prologue overlaps the planner; global memory only after this wait
    tc::pdl_wait();
    tc::pdl_trigger();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp >= kWarpTma) {
        tc::regs_dec<kRegsOther>();
        if (warp == kWarpTma) {
            // -------------------------------------------------- TMA producer
            if (lane == 0) {
                const int n_units = hdr->n_units;
                const uint64_t policy = tc::policy_evict_first();
                const uint32_t qbytes = static_cast<uint32_t>(kTerms * 128 * a.G * a.gmax);
                uint32_t uc = 0, gb = 0;          // units and half pages claimed by this CTA
                uint32_t nq = 0, nk = 0, nv = 0;  // Q, K and V loads issued
                for (;;) {
                    PlanUnit un{};
                    un.pair = -1;
                    if (!aborted(sh)) {
                        const int uu = atomicAdd(&hdr->next_unit, 1);
                        if (uu < n_units) un = units[uu];
                    }
                    const int slot = uc & 3;
                    if (uc >= 4 && !wait_or_abort(sh, &sh.unit_empty[slot], ((uc >> 2) - 1) & 1, status))
                        un.pair = -1;
                    sh.ring[slot] = un;
                    tc::mbar_arrive(&sh.unit_full[slot]);
                    if (un.pair < 0) break;
                    // the previous unit's last Q K^T has read the query terms
                    if (uc >= 1 && !wait_or_abort(sh, &sh.q_empty, (uc - 1) & 1, status)) break;
                    tc::mbar_arrive_expect_tx(&sh.q_full, qbytes);
                    for (int term = 0; term < kTerms; ++term)
                        tc::tma_load_3d(smem + kOffQ + term * kQTile, &tmap_q, &sh.q_full, 0, un.h * a.G,
                                        term * a.T + un.t0);
                    ++nq;
                    ++uc;
                    bool ok = true;
                    PlanEntry e{};
                    for (int i = 0; i < 2 * un.count; ++i, ++gb) {
                        if ((i & 1) == 0) e = lists[un.entry + (i >> 1)];
                        const int key0 = e.page * kKeys + (i & 1) * kHalf;  // half i & 1 of the page
                        const int st = gb % kStages;
                        const uint32_t ph = ((gb / kStages) - 1) & 1;
                        if (gb >= kStages && !(ok = wait_or_abort(sh, &sh.k_empty[st], ph, status))) break;
                        tc::mbar_arrive_expect_tx(&sh.k_full[st], kKVHalf);
                        tc::tma_load_3d(smem + kOffK + st * kKVHalf, &tmap_k, &sh.k_full[st], 0, un.h, key0, policy);
                        ++nk;
                        if (gb >= kStages && !(ok = wait_or_abort(sh, &sh.v_empty[st], ph, status))) break;
                        tc::mbar_arrive_expect_tx(&sh.v_full[st], kKVHalf);
                        tc::tma_load_3d(smem + kOffV + st * kKVHalf, &tmap_v, &sh.v_full[st], 0, un.h, key0, policy);
                        ++nv;
                    }
                    if (!ok) break;
                }
                // every issued copy lands before the CTA may exit (the last
                // phase of each barrier is the only one still pending)
                if (nq > 0) tc::mbar_wait(&sh.q_full, (nq - 1) & 1);
                for (uint32_t b = (nk > kStages ? nk - kStages : 0); b < nk; ++b)
                    tc::mbar_wait(&sh.k_full[b % kStages], (b / kStages) & 1);
                for (uint32_t b = (nv > kStages ? nv - kStages : 0); b < nv; ++b)
                    tc::mbar_wait(&sh.v_full[b % kStages], (b / kStages) & 1);
            }
        } else if (warp == kWarpMma) {
            // --------------------------------------------------- MMA issuer
            if (lane == 0) {
                const uint32_t idesc_s = tc::idesc_m128(kHalf, false, false);    // E4M3 x E4M3, K-major
                const uint32_t idesc_o = tc::idesc_f16_m128(kD, false) | (1u << 16);  // f16, V MN-major
                const uint32_t aQ = tc::smem_u32(smem + kOffQ), aK0 = tc::smem_u32(smem + kOffK);
                const uint32_t aV0 = tc::smem_u32(smem + kOffV16);
                uint32_t uc = 0, gb = 0;
                bool ok = true;
                while (ok) {
                    const int slot = uc & 3;
                    if (!wait_or_abort(sh, &sh.unit_full[slot], (uc >> 2) & 1, status)) break;
                    const PlanUnit un = sh.ring[slot];
                    tc::mbar_arrive(&sh.unit_empty[slot]);
                    if (un.pair < 0) break;
                    if (!wait_or_abort(sh, &sh.q_full, uc & 1, status)) break;
                    tc::tc_fence_after();
                    const int nblk = 2 * un.count;  // half pages
                    for (int i = 0; ok && i <= nblk; ++i) {
                        if (i < nblk) {
                            const uint32_t b = gb + i;
                            const int st = b % kStages, sb = b & 1;
                            ok = wait_or_abort(sh, &sh.k_full[st], (b / kStages) & 1, status);
                            if (ok && b >= 2) ok = wait_or_abort(sh, &sh.s_free[sb], ((b >> 1) - 1) & 1, status);
                            if (!ok) break;
                            tc::tc_fence_after();
                            const uint32_t aK = aK0 + st * kKVHalf;
                            // 32 dims a step (32 bytes into a 128-byte row), both terms
                            // into the same columns
#pragma unroll
                            for (int term = 0; term < kTerms; ++term)
#pragma unroll
                                for (int ks = 0; ks < kD / 32; ++ks)
                                    tc::mma_f8(tmem + kColS + sb * kHalf,
                                               tc::smem_desc(aQ + term * kQTile + ks * 32, 16, 1024, tc::kSw128),
                                               tc::smem_desc(aK + ks * 32, 16, 1024, tc::kSw128), idesc_s,
                                               term > 0 || ks > 0);
                            tc::mma_commit(&sh.s_full[sb]);
                            tc::mma_commit(&sh.k_empty[st]);
                            if (i + 1 == nblk) tc::mma_commit(&sh.q_empty);
                        }
                        if (i >= 1) {
                            const uint32_t b = gb + i - 1;
                            const int pb = b & 1;
                            // P (in S buffer pb) by the softmax threads, the
                            // widened V of half page b by the V-widening warps
                            ok = wait_or_abort(sh, &sh.p_full[pb], (b >> 1) & 1, status) &&
                                 wait_or_abort(sh, &sh.v16_full[pb], (b >> 1) & 1, status);
                            // the first product of a unit overwrites O: the previous
                            // unit's epilogue must have read it
                            if (ok && i == 1 && uc >= 1) ok = wait_or_abort(sh, &sh.o_free, (uc - 1) & 1, status);
                            if (!ok) break;
                            tc::tc_fence_after();
                            const uint32_t aV = aV0 + pb * kV16Tile;
#pragma unroll
                            for (int ks = 0; ks < kHalf / 16; ++ks) {
                                // P from tensor memory: lane = query row, 16 keys =
                                // 8 columns of f16 pairs per step; V: 16 keys of 128
                                // bytes per step, the second 64 dims one box on
                                tc::mma_f16_tmem_a(tmem + kColO, tmem + kColS + pb * kHalf + ks * 8,
                                                   tc::smem_desc(aV + ks * 2048, kV16Box, 1024, tc::kSw128), idesc_o,
                                                   i > 1 || ks > 0);
                            }
                            tc::mma_commit(&sh.pv_done);
                            tc::mma_commit(&sh.s_free[pb]);
                            tc::mma_commit(&sh.v16_free[pb]);
                        }
                    }
                    if (un.count == 0) tc::mma_commit(&sh.q_empty);
                    gb += nblk;
                    ++uc;
                }
                tc::mma_commit(&sh.drain);
                tc::mbar_wait(&sh.drain, 0);
            }
        } else {
            // ------------------------------------------------ V widening (6-7)
            // Thread ct widens slot ct of each V half page: E4M3 (128-byte
            // swizzled TMA row) -> f16 in two 64-dim halves with 128-byte
            // swizzle, into tile b % 2 once the product of half page b - 2 is
            // done.  Slots past every selecting row's key limit (the tail of a
            // request's last page: they may hold anything, NaN included)
            // become zeros, so that 0-weight keys add exactly nothing.
            const int ct = threadIdx.x - kWarpConv * 32;
            const int sw8 = ct & 7;
            uint32_t uc = 0, gb = 0;
            for (;;) {
                const int slot = uc & 3;
                if (!wait_or_abort(sh, &sh.unit_full[slot], (uc >> 2) & 1, status)) break;
                const PlanUnit un = sh.ring[slot];
                tc::mbar_arrive(&sh.unit_empty[slot]);
                if (un.pair < 0) break;
                // key limit of the unit's token `lane` (every lane of the warp holds them)
                int my_lim = 0;
                if (lane < un.nt) {
                    int r;
                    my_lim = static_cast<int>(token_limit(a.ri, a.ri_s0, a.sl, a.sl_s0, un.t0 + lane, a.R, a.NB, &r));
                }
                bool ok = true;
                PlanEntry e{};
                for (int i = 0; i < 2 * un.count; ++i) {
                    const uint32_t b = gb + i;
                    const int st = b % kStages, x = b & 1;
                    if ((i & 1) == 0) e = lists[un.entry + (i >> 1)];
                    const int bstart = static_cast<int>(e.block) * kKeys + (i & 1) * kHalf;
                    int vlim = 0;
                    for (int j = 0; j < un.nt; ++j) {
                        const int lj = __shfl_sync(0xffffffffu, my_lim, j);
                        if ((e.mask >> j) & 1) vlim = max(vlim, min(kHalf, lj - bstart));
                    }
                    ok = wait_or_abort(sh, &sh.v_full[st], (b / kStages) & 1, status);
                    if (ok && b >= 2) ok = wait_or_abort(sh, &sh.v16_free[x], ((b >> 1) - 1) & 1, status);
                    if (!ok) break;
                    const uint8_t *src = smem + kOffV + st * kKVHalf + ct * 128;
                    uint8_t *dst = smem + kOffV16 + x * kV16Tile + ct * 128;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint4 xv[4];
                        if (ct < vlim) {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                xv[q] = *reinterpret_cast<const uint4 *>(src + (((4 * hh + q) ^ sw8) << 4));
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q) xv[q] = make_uint4(0u, 0u, 0u, 0u);
                        }
                        uint8_t *half = dst + hh * kV16Box;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t f[8];
                            tc::e4m3x4_to_f16x4(xv[q].x, f[0], f[1]);
                            tc::e4m3x4_to_f16x4(xv[q].y, f[2], f[3]);
                            tc::e4m3x4_to_f16x4(xv[q].z, f[4], f[5]);
                            tc::e4m3x4_to_f16x4(xv[q].w, f[6], f[7]);
                            *reinterpret_cast<uint4 *>(half + (((2 * q) ^ sw8) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
                            *reinterpret_cast<uint4 *>(half + (((2 * q + 1) ^ sw8) << 4)) =
                                make_uint4(f[4], f[5], f[6], f[7]);
                        }
                    }
                    tc::fence_proxy_async();
                    tc::mbar_arrive(&sh.v_empty[st]);
                    tc::mbar_arrive(&sh.v16_full[x]);
                }
                if (!ok) break;
                gb += 2 * un.count;
                ++uc;
            }
        }
    } else {
        tc::regs_inc<kRegsSoft>();
        // --------------------------------------------- softmax and epilogue
        const int st_id = threadIdx.x;  // 0..127
        const int r = st_id;            // row of the unit = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        int32_t *counters = reinterpret_cast<int32_t *>(a.ws + a.lay.counters);
        float *partials = reinterpret_cast<float *>(a.ws + a.lay.partials);
        const float *cfac = reinterpret_cast<const float *>(a.ws + a.lay.cfac);
        uint32_t uc = 0, gb = 0;
        bool ok = true;
        // a split unit's ticket, resolved one unit later
        PlanUnit pend{};
        pend.pair = -1;
        int ticket = 0;
        auto resolve = [&]() {
            if (pend.pair < 0) return;
            if (st_id == 0) sh.last = (ticket == pend.n_split - 1);
            soft_sync();
            if (sh.last) {
                __threadfence();  // the other units' partials before the merge reads them
                merge_pair(a, pend, partials, st_id);
            }
            soft_sync();  // sh.last is rewritten by the next resolution
            pend.pair = -1;
        };
        bool finished = false;  // the sentinel unit was reached with no failure
        for (;;) {
            const int slot = uc & 3;
            PlanUnit un{};
            un.pair = -1;
            if (ok && warp_wait(sh, &sh.unit_full[slot], (uc >> 2) & 1, status)) {
                un = sh.ring[slot];
                tc::mbar_arrive(&sh.unit_empty[slot]);
            } else {
                ok = false;
            }
            // leave together: on any failure, or at the sentinel (the same
            // record for every thread)
            if (soft_any(!ok || aborted(sh))) break;
            if (un.pair < 0) {
                finished = true;
                break;
            }
            const int rows = un.nt * a.G;
            const bool active = r < rows;
            const bool warp_active = __any_sync(0xffffffffu, active);
            const int j = active ? r / a.G : 0, g = active ? r % a.G : 0;
            int row_r;
            const int L = active ? static_cast<int>(token_limit(a.ri, a.ri_s0, a.sl, a.sl_s0, un.t0 + j, a.R, a.NB,
                                                                &row_r))
                                 : 0;
            // the row's logit factor: s c is the logit in log2 units
            const float c = active ? cfac[static_cast<int64_t>(un.t0 + j) * a.Hq + un.h * a.G + g] : 0.f;
            float m_run = -INFINITY, l = 0.f;
            PlanEntry e_next{}, e{};
            if (un.count > 0) e_next = lists[un.entry];
            const int nblk = 2 * un.count;  // half pages
            for (int i = 0; i < nblk; ++i) {
                const uint32_t b = gb + i;
                const int sb = b & 1;
                if ((i & 1) == 0) {
                    e = e_next;
                    if ((i >> 1) + 1 < un.count) e_next = lists[un.entry + (i >> 1) + 1];
                }
                const int bstart = static_cast<int>(e.block) * kKeys + (i & 1) * kHalf;  // first key of the half
                const bool sel = active && ((e.mask >> j) & 1);
                const int lim = sel ? min(kHalf, max(0, L - bstart)) : 0;
                ok = warp_wait(sh, &sh.s_full[sb], (b >> 1) & 1, status);
                if (!ok) break;
                tc::tc_fence_after();
                float s[kHalf];
                if (warp_active) {
#pragma unroll
                    for (int ch = 0; ch < kHalf / 32; ++ch)
                        tmem_ld32(tmem + lane_base + kColS + sb * kHalf + ch * 32, s + ch * 32);
                    tc::tmem_wait_ld();
                }
                uint32_t pk[kHalf / 2];
                float alpha = 1.f;
                if (warp_active) {
                    if (lim < kHalf) {
#pragma unroll
                        for (int k = 0; k < kHalf; ++k)
                            if (k >= lim) s[k] = -INFINITY;
                    }
                    // block maximum of s c (c may be negative: then the minimum of s)
                    float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
                    if (c >= 0.f) {
#pragma unroll
                        for (int k = 0; k < kHalf; k += 4) {
                            mx0 = fmaxf(mx0, s[k]);
                            mx1 = fmaxf(mx1, s[k + 1]);
                            mx2 = fmaxf(mx2, s[k + 2]);
                            mx3 = fmaxf(mx3, s[k + 3]);
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < kHalf; k += 4) {
                            mx0 = fmaxf(mx0, s[k] == -INFINITY ? -INFINITY : -s[k]);
                            mx1 = fmaxf(mx1, s[k + 1] == -INFINITY ? -INFINITY : -s[k + 1]);
                            mx2 = fmaxf(mx2, s[k + 2] == -INFINITY ? -INFINITY : -s[k + 2]);
                            mx3 = fmaxf(mx3, s[k + 3] == -INFINITY ? -INFINITY : -s[k + 3]);
                        }
                    }
                    const float mraw = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                    const float bm = (mraw == -INFINITY) ? -INFINITY : mraw * fabsf(c);
                    // raise the offset if the block's maximum runs more than
                    // 2^kRaise above it (or the row had none yet)
                    if (bm != -INFINITY && (m_run == -INFINITY || bm > m_run + kRaise)) {
                        alpha = (m_run == -INFINITY) ? 0.f : tc::ex2(m_run - bm);
                        m_run = bm;
                        l *= alpha;
                    }
                    const float m_eff = (m_run == -INFINITY) ? 0.f : m_run;
                    // p = 2^(s c - m) in [0, 2^kRaise], f16; masked keys take
                    // p = 0 whatever the sign of c
                    if (lim >= kHalf) {
#pragma unroll
                        for (int k = 0; k < kHalf; k += 2) {
                            const float p0 = tc::ex2(fmaf(s[k], c, -m_eff));
                            const float p1 = tc::ex2(fmaf(s[k + 1], c, -m_eff));
                            l += p0 + p1;
                            pk[k / 2] = tc::f32x2_to_f16x2(p0, p1);
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < kHalf; k += 2) {
                            const float p0 = (k < lim) ? tc::ex2(fmaf(s[k], c, -m_eff)) : 0.f;
                            const float p1 = (k + 1 < lim) ? tc::ex2(fmaf(s[k + 1], c, -m_eff)) : 0.f;
                            l += p0 + p1;
                            pk[k / 2] = tc::f32x2_to_f16x2(p0, p1);
                        }
                    }
                }
                // On the unit's last half page L the previous product must be
                // done before P(L) is handed off: the epilogue then waits for
                // product L by parity, which is exact only once L - 1 is done
                // (seeing S(b) guarantees product b - 2 only, since P no longer
                // waits for the product before it)
                if (i == nblk - 1 && b >= 1) {
                    ok = warp_wait(sh, &sh.pv_done, (b - 1) & 1, status);
                    if (!ok) break;
                    tc::tc_fence_after();
                }
                if (warp_active) {
                    // O holds this unit's earlier blocks: rescale rows whose
                    // offset moved (the first block of a unit overwrites O),
                    // once the previous product is done
                    if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                        if (!warp_wait(sh, &sh.pv_done, (b - 1) & 1, status)) {
                            ok = false;
                            break;
                        }
                        tc::tc_fence_after();
#pragma unroll 1
                        for (int ch = 0; ch < kD / 32; ++ch) {
                            float o[32];
                            const uint32_t ta = tmem + lane_base + kColO + ch * 32;
                            tmem_ld32(ta, o);
                            tc::tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 32; ++k) o[k] *= alpha;
                            tmem_st32(ta, o);
                        }
                        tc::tmem_wait_st();
                    }
                    // P over this half page's S (its logits are in registers):
                    // 64 f16 in 32 columns of the row's lane
                    tc::tmem_st32u(tmem + lane_base + kColS + sb * kHalf, pk);
                    tc::tmem_wait_st();
                }
                tc::tc_fence_before();
                tc::mbar_arrive(&sh.p_full[sb]);
            }
            if (soft_any(!ok || aborted(sh))) break;
            // the previous split unit's ticket has had this unit's pages to return
            resolve();
            // ---- unit epilogue: this thread's row of O, 32 dims at a time
            if (un.count > 0) {
                // the unit's last product (the one before it is done: see the
                // last half page's hand-off)
                ok = warp_wait(sh, &sh.pv_done, (gb + nblk - 1) & 1, status);
                tc::tc_fence_after();
            }
            const bool have_o = ok && un.count > 0 && warp_active;
            const bool split = un.part_row >= 0;
            const float inv = (l > 0.f && have_o) ? a.v_scale / l : 0.f;
            __nv_bfloat16 *dst = a.out + static_cast<int64_t>(un.t0 + j) * a.o_s0 +
                                 static_cast<int64_t>(un.h * a.G + g) * a.o_s1;
            const bool vec = a.o_s2 == 1 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0;
            float *prt = partials + static_cast<int64_t>(split ? un.part_row + r : 0) * kStride;
#pragma unroll 1
            for (int ch = 0; ch < kD / 32; ++ch) {
                float o[32];
                __syncwarp();
                if (have_o) {
                    tmem_ld32(tmem + lane_base + kColO + ch * 32, o);
                    tc::tmem_wait_ld();
                }
#pragma unroll
                for (int k = 0; k < 32; ++k) o[k] = have_o ? o[k] : 0.f;
                if (!active) {
                } else if (split) {
                    // partial of a split pair: unnormalised O
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        reinterpret_cast<float4 *>(prt + ch * 32)[q] =
                            make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                } else if (vec) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        __nv_bfloat162 h0 = __floats2bfloat162_rn(o[8 * q + 0] * inv, o[8 * q + 1] * inv);
                        __nv_bfloat162 h1 = __floats2bfloat162_rn(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
                        __nv_bfloat162 h3 = __floats2bfloat162_rn(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
                        w.x = *reinterpret_cast<uint32_t *>(&h0);
                        w.y = *reinterpret_cast<uint32_t *>(&h1);
                        w.z = *reinterpret_cast<uint32_t *>(&h2);
                        w.w = *reinterpret_cast<uint32_t *>(&h3);
                        reinterpret_cast<uint4 *>(dst + ch * 32)[q] = w;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        dst[static_cast<int64_t>(ch * 32 + k) * a.o_s2] = __float2bfloat16_rn(o[k] * inv);
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&sh.o_free);
            if (split) {
                if (active) {
                    prt[kD] = have_o ? m_run : -INFINITY;
                    prt[kD + 1] = have_o ? l : 0.f;
                }
                // every thread's partial row before the ticket; its result is
                // looked at after the next unit's pages
                __threadfence();
                soft_sync();
                if (st_id == 0) ticket = atomicAdd(&counters[un.pair], 1);
                pend = un;
            }
            gb += nblk;
            ++uc;
        }
        if (finished) resolve();
    }

    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == kWarpMma) tc::tmem_dealloc(tmem, kTmemCols);
}

// E4M3 cache [slots, Hkv, 128 bytes] as a 3-D map whose box is 64 slots of
// one kv head (128 bytes each), 128-byte swizzle.
bool make_tmap_kv(CUtensorMap *m, const uint8_t *base, int64_t slots, int64_t hkv, int64_t s0, int64_t s1) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(slots)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(s1), static_cast<cuuint64_t>(s0)};
    cuuint32_t box[3] = {kD, 1, kHalf};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Query terms qterms[term][t][hq][128 bytes] as a 3-D map: box = G heads x
// rows_box tokens of one term (rows token-major, head fastest), 128-byte
// swizzle.
bool make_tmap_terms(CUtensorMap *m, const uint8_t *base, int64_t T, int64_t hq, int g, int rows_box) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(hq),
                          static_cast<cuuint64_t>(kQueryTerms * T)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(hq * kD)};
    cuuint32_t box[3] = {kD, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(rows_box)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The largest shared-memory carveout for the kernel on the current device
// (two CTAs of 113 KB per SM), once per device.
cudaError_t prefer_shared_carveout(const void *func) {
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count(dev)) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e == cudaSuccess) done.insert(dev);
    return e;
}

}  // namespace

// Covers: E4M3 K/V caches with 16-byte aligned rows, bf16 queries of head dim
// 128, G = Hq / Hkv a power of two up to 16, page tables of at most 256
// blocks, at most 4096 rows, a workspace.  Anything else: *used stays false.
cudaError_t launch_attention_e4m3_rows(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream,
                                       bool *used) {
    *used = false;
    const int G = a.Hq / a.Hkv;
    if (a.kv_dt != SPD_E4M3 || a.q_dt != SPD_BF16 || a.D != kD) return cudaSuccess;
    if (a.NB > kPlanMaxNB || a.T > kPlanMaxT || G < 1 || G > 16 || (G & (G - 1)) != 0) return cudaSuccess;
    if ((a.k_s0 % 16) || (a.k_s1 % 16) || (a.v_s0 % 16) || (a.v_s1 % 16)) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(a.k) % 16) || (reinterpret_cast<uintptr_t>(a.v) % 16)) return cudaSuccess;
    if (a.P * kKeys > (int64_t(1) << 31) - 1) return cudaSuccess;
    PlanLayout lay(a.T, a.Hq, a.Hkv, a.D, a.NB);
    if (ws == nullptr || ws_bytes < lay.total) return cudaSuccess;

    // rows of a request share a unit: up to 128 / G tokens (16 at most, the
    // planner's row mask), so one unit fills the M = 128 rows of the MMA
    const int gmax = std::min(16, kM / G);
    CUtensorMap tq, tk, tv;
    if (!make_tmap_kv(&tk, static_cast<const uint8_t *>(a.k), a.P * kKeys, a.Hkv, a.k_s0, a.k_s1)) return cudaSuccess;
    if (!make_tmap_kv(&tv, static_cast<const uint8_t *>(a.v), a.P * kKeys, a.Hkv, a.v_s0, a.v_s1)) return cudaSuccess;
    if (!make_tmap_terms(&tq, reinterpret_cast<const uint8_t *>(static_cast<char *>(ws) + lay.qterms), a.T, a.Hq, G,
                         gmax))
        return cudaSuccess;

    // two persistent CTAs per SM
    const int sms = device_sm_count();
    const int ctas = 2 * sms;
    cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(attention_e4m3_rows_kernel), kSmemBytes);
    if (e == cudaSuccess) e = prefer_shared_carveout(reinterpret_cast<const void *>(attention_e4m3_rows_kernel));
    if (e != cudaSuccess) return e;

    PlanArgs p{};
    p.ri = a.ri; p.ri_s0 = a.ri_s0;
    p.sl = a.sl; p.sl_s0 = a.sl_s0;
    p.bt = a.bt; p.bt_s0 = a.bt_s0; p.bt_s1 = a.bt_s1;
    p.tk = a.tk; p.tk_s0 = a.tk_s0; p.tk_s1 = a.tk_s1; p.tk_s2 = a.tk_s2;
    p.T = a.T; p.R = a.R; p.NB = a.NB; p.K = a.K; p.Hkv = a.Hkv; p.G = G;
    p.gmax = gmax;
    p.P = a.P;
    p.num_ctas = ctas;
    p.ws = static_cast<char *>(ws);
    p.lay = lay;
    p.q = a.q; p.q_s0 = a.q_s0; p.q_s1 = a.q_s1; p.q_s2 = a.q_s2;
    p.q_dt = a.q_dt;
    p.Hq = a.Hq;
    p.zscale = a.sm_scale * a.k_scale * 1.4426950408889634f;
    if (!plan_configure(&p)) return cudaSuccess;
    const int64_t q_rows = static_cast<int64_t>(a.T) * a.Hq;
    // query conversion: 64 rows per CTA (four per warp), up to two CTAs per SM
    const int conv_ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(2 * sms - 1, (q_rows + 63) / 64)));
    e = launch_prepare(p, conv_ctas, stream);
    if (e != cudaSuccess) return e;

    RowsArgs t{};
    t.ri = a.ri; t.ri_s0 = a.ri_s0;
    t.sl = a.sl; t.sl_s0 = a.sl_s0;
    t.out = a.out; t.o_s0 = a.o_s0; t.o_s1 = a.o_s1; t.o_s2 = a.o_s2;
    t.T = a.T; t.Hq = a.Hq; t.Hkv = a.Hkv; t.G = G; t.R = a.R; t.NB = a.NB; t.gmax = gmax;
    t.v_scale = a.v_scale;
    t.ws = static_cast<char *>(ws);
    t.lay = lay;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attention_e4m3_rows_kernel, tq, tk, tv, t);
    if (e == cudaSuccess) *used = true;
    return e;
}

}  // namespace spd
