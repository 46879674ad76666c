// sdpa_tc.cu -- dense GQA attention with a causal flag ("Kernel ABI" --
// attention.sdpa) on the sm_103a tensor cores, for bf16 or f16 q, k and v of
// head dim 128 with a bf16 or f16 output.
//
// A CTA owns one tile of 128 query rows of one kv head: 128 / G consecutive
// query tokens, each with its G q heads (row = token * G + head), so every
// row of the tile reads the same keys.  It streams that kv head's keys 64 at
// a time (one "key block"):
//
//   S  = Q K^T       tcgen05.mma kind::f16, M = 128 rows, N = 64 keys, K = 128
//                    dims, into one of two tensor-memory buffers, so the next
//                    block's product runs while the softmax reads this one
//   P  = 2^(S c - m) one thread per row (its TMEM lane): the row's 64 logits
//                    sit in that thread's registers, so the block maximum and
//                    the row sum need no exchange between threads
//   O += P V         kind::f16, M = 128 rows, N = 128 dims, K = 64 keys, with
//                    P written by the softmax into tensor memory over its own
//                    S buffer (the A operand read from there) and V used as
//                    loaded (MN-major)
//
// Two CTAs share an SM (97 KB of shared memory and 256 tensor-memory
// columns each), so one CTA's softmax runs while the other's products keep
// the tensor pipe busy.  With P in tensor memory a block's softmax does not
// wait for the previous block's product (only to rescale O, and on the last
// block).  Q, K and V arrive by TMA straight from the caller's
// tensors (64-dim boxes, 128-byte swizzle); keys past the end read as zeros
// and are masked.  c = sm_scale * log2(e).  The exponent offset m of a row is
// raised only when a block's maximum exceeds it by more than 2^kRaise (then
// the row's O is rescaled in tensor memory and its sum in a register), so
// every p lies in [0, 2^kRaise] and P can be stored in the inputs' 16-bit
// type.  Under the causal flag query token t reads keys j <= t + S - T; blocks
// past a tile's last readable key are not loaded, and the tiles with the most
// keys are scheduled first.
//
// Roles (6 warps): warp 0 issues the TMA loads, warp 1 owns tensor memory and
// issues every MMA, warps 2-5 run the softmax and the epilogue (warp w reads
// TMEM lanes 32 (w % 4) .. +31, i.e. rows of that quadrant).  Every mbarrier
// wait is bounded; a wait that gives up makes the CTA wind down and write NaN
// into its output rows instead of results.
#include <math.h>

#include <mutex>
#include <set>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sdpa.cuh"
#include "spd.h"
#include "spd_internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace spd {

cudaError_t launch_sdpa_tc(const SdpaArgs &a, cudaStream_t stream, bool *used);

namespace {

constexpr int kD = 128;              // head dim of this path
constexpr int kRowsTile = 128;       // query rows per CTA (M)
constexpr int kKeysBlock = 64;       // keys per block (N of S, K of P V)
constexpr int kThreads = 192;        // warps 0 TMA, 1 MMA, 2-5 softmax
constexpr int kStages = 2;           // K and V stages each
constexpr int kBoxQ = 128 * 128;     // one 64-dim box of 128 query rows, bytes (16-bit elements)
constexpr int kTileQ = 2 * kBoxQ;    // 128 rows x 128 dims
constexpr int kBoxKV = kKeysBlock * 128;  // one 64-dim box of a key block
constexpr int kTileKV = 2 * kBoxKV;       // 64 keys x 128 dims
constexpr float kRaise = 8.0f;       // log2 headroom before a row's offset is raised
constexpr float kLog2e = 1.4426950408889634f;

// dynamic shared memory (1024-byte aligned tiles): Q, K stages, V stages (P
// lives in tensor memory)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileQ;
constexpr int kOffV = kOffK + kStages * kTileKV;
constexpr int kTilesEnd = kOffV + kStages * kTileKV;

struct SdpaShared {
    uint64_t q_full;
    uint64_t k_full[kStages], k_empty[kStages];
    uint64_t v_full[kStages], v_empty[kStages];
    uint64_t s_full[2], s_free[2];  // S buffer free: the product that read its P is done
    uint64_t p_full[2];  // P of S buffer j % 2 written (one barrier per buffer: the
                         // softmax may hand off the next buffer's P before the
                         // product of this one is issued)
    uint64_t pv_done, drain;
    uint32_t tmem_base;
    int abort;
};

// The barriers sit in the padding below the aligned tiles when it is large
// enough, else after them; either way the CTA needs the tiles plus 1023
// bytes, which lets two CTAs share an SM.
static_assert(sizeof(SdpaShared) <= 511, "barriers fit the alignment padding or after the tiles");
constexpr int kSmemBytes = kTilesEnd + 1023;
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");

// tensor memory: S buffers at columns 0 and 64, O at 128
constexpr uint32_t kColS = 0, kColO = 2 * kKeysBlock, kTmemCols = 256;

struct SdpaTcArgs {
    void *out;
    int64_t o_s0, o_s1, o_s2;
    int32_t out_bf16;  // else f16
    int32_t in_bf16;   // else f16
    int32_t T, S, Hq, Hkv, G, tt;  // tt = query tokens per tile (128 / G)
    int32_t n_tiles;
    int32_t causal;
    float c;  // sm_scale * log2(e)
};

// 32 consecutive 32-bit columns of this thread's TMEM lane (warp-collective).
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

// Store 32 consecutive 32-bit columns of this thread's TMEM lane (warp-collective).
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

// Instruction descriptor of kind::f16 with fp32 accumulate, M = 128, the
// given N, A K-major and B MN-major, both bf16 (format code 1) or f16 (0).
__host__ __device__ constexpr uint32_t idesc_f16_m128_bmn(uint32_t n, bool bf16) {
    return tc::idesc_f16_m128(n, bf16) | (1u << 16);
}

__device__ __forceinline__ bool aborted(SdpaShared &sh) { return *reinterpret_cast<volatile int *>(&sh.abort) != 0; }

__device__ __forceinline__ bool wait_or_abort(SdpaShared &sh, uint64_t *bar, uint32_t parity) {
    if (tc::mbar_wait(bar, parity)) return true;
    *reinterpret_cast<volatile int *>(&sh.abort) = 1;
    return false;
}

// Warp-uniform wait (so a warp-collective tcgen05 access that follows is
// uniform): the warp goes on only if every lane saw the phase.
__device__ __forceinline__ bool warp_wait(SdpaShared &sh, uint64_t *bar, uint32_t parity) {
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(bar, parity));
    if (!ok) *reinterpret_cast<volatile int *>(&sh.abort) = 1;
    return ok;
}

// Keys query token t may read.
__device__ __forceinline__ int readable(const SdpaTcArgs &a, int64_t t) {
    if (t >= a.T) return 0;
    if (!a.causal) return a.S;
    const int64_t n = t + (static_cast<int64_t>(a.S) - a.T) + 1;
    return n < 0 ? 0 : (n > a.S ? a.S : static_cast<int>(n));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
    if (bf16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__global__ void __launch_bounds__(kThreads, 2)
sdpa_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
               const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ SdpaTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const bool bar_below = static_cast<size_t>(smem - smem_raw) >= sizeof(SdpaShared);
    SdpaShared &sh = *reinterpret_cast<SdpaShared *>(bar_below ? smem_raw : smem + kTilesEnd);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // heaviest tiles first: under the causal flag later tokens read more keys
    const int h = static_cast<int>(blockIdx.x % a.Hkv);
    const int tile = a.n_tiles - 1 - static_cast<int>(blockIdx.x / a.Hkv);
    const int64_t t0 = static_cast<int64_t>(tile) * a.tt;
    const int64_t t_last = min(t0 + a.tt, static_cast<int64_t>(a.T)) - 1;
    const int n_max = readable(a, t_last);
    const int nb = (n_max + kKeysBlock - 1) / kKeysBlock;  // key blocks of the tile

    if (threadIdx.x == 0) {
        tc::mbar_init(&sh.q_full, 1);
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&sh.k_full[i], 1);
            tc::mbar_init(&sh.k_empty[i], 1);
            tc::mbar_init(&sh.v_full[i], 1);
            tc::mbar_init(&sh.v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&sh.s_full[i], 1);
            tc::mbar_init(&sh.s_free[i], 1);
        }
        tc::mbar_init(&sh.p_full[0], 128);
        tc::mbar_init(&sh.p_full[1], 128);
        tc::mbar_init(&sh.pv_done, 1);
        tc::mbar_init(&sh.drain, 1);
        sh.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(&sh.tmem_base, kTmemCols);
    if (threadIdx.x == 32) {
        tc::prefetch_tmap(&tmap_q);
        tc::prefetch_tmap(&tmap_k);
        tc::prefetch_tmap(&tmap_v);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && nb > 0) {
            uint8_t *sQ = smem + kOffQ;
            tc::mbar_arrive_expect_tx(&sh.q_full, kTileQ);
            tc::tma_load_3d(sQ, &tmap_q, &sh.q_full, 0, h * a.G, static_cast<int>(t0));
            tc::tma_load_3d(sQ + kBoxQ, &tmap_q, &sh.q_full, 64, h * a.G, static_cast<int>(t0));
            int nk = 0, nv = 0;  // K and V blocks issued
            for (int j = 0; j < nb && !aborted(sh); ++j) {
                const int st = j % kStages;
                const uint32_t ph = ((j / kStages) - 1) & 1;
                const int key0 = j * kKeysBlock;
                if (j >= kStages && !wait_or_abort(sh, &sh.k_empty[st], ph)) break;
                uint8_t *sK = smem + kOffK + st * kTileKV;
                tc::mbar_arrive_expect_tx(&sh.k_full[st], kTileKV);
                tc::tma_load_3d(sK, &tmap_k, &sh.k_full[st], 0, h, key0);
                tc::tma_load_3d(sK + kBoxKV, &tmap_k, &sh.k_full[st], 64, h, key0);
                ++nk;
                if (j >= kStages && !wait_or_abort(sh, &sh.v_empty[st], ph)) break;
                uint8_t *sV = smem + kOffV + st * kTileKV;
                tc::mbar_arrive_expect_tx(&sh.v_full[st], kTileKV);
                tc::tma_load_3d(sV, &tmap_v, &sh.v_full[st], 0, h, key0);
                tc::tma_load_3d(sV + kBoxKV, &tmap_v, &sh.v_full[st], 64, h, key0);
                ++nv;
            }
            // every issued copy lands before the CTA may exit (the last use
            // of each stage is the only phase still pending)
            tc::mbar_wait(&sh.q_full, 0);
            for (int b = (nk > kStages ? nk - kStages : 0); b < nk; ++b)
                tc::mbar_wait(&sh.k_full[b % kStages], (b / kStages) & 1);
            for (int b = (nv > kStages ? nv - kStages : 0); b < nv; ++b)
                tc::mbar_wait(&sh.v_full[b % kStages], (b / kStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        // S(j) is issued before P(j-1) V(j-1), so the tensor pipe computes the
        // next block's logits while the softmax works on this one.
        if (lane == 0 && nb > 0) {
            const bool bf16 = a.in_bf16 != 0;
            const uint32_t idesc_s = tc::idesc_f16_m128(kKeysBlock, bf16);
            const uint32_t idesc_o = idesc_f16_m128_bmn(kD, bf16);
            const uint32_t aQ = tc::smem_u32(smem + kOffQ);
            bool ok = wait_or_abort(sh, &sh.q_full, 0);
            tc::tc_fence_after();
            for (int j = 0; ok && j <= nb; ++j) {
                if (j < nb) {
                    const int st = j % kStages, sb = j & 1;
                    ok = wait_or_abort(sh, &sh.k_full[st], (j / kStages) & 1);
                    if (ok && j >= 2) ok = wait_or_abort(sh, &sh.s_free[sb], ((j >> 1) - 1) & 1);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint32_t aK = tc::smem_u32(smem + kOffK + st * kTileKV);
#pragma unroll
                    for (int ks = 0; ks < kD / 16; ++ks) {
                        // 16 dims a step: 32 bytes into a 128-byte row, the
                        // second 64 dims one box on
                        const uint32_t offq = (ks >> 2) * kBoxQ + (ks & 3) * 32;
                        const uint32_t offk = (ks >> 2) * kBoxKV + (ks & 3) * 32;
                        tc::mma_f16(tmem + kColS + sb * kKeysBlock, tc::smem_desc(aQ + offq, 16, 1024, tc::kSw128),
                                    tc::smem_desc(aK + offk, 16, 1024, tc::kSw128), idesc_s, ks > 0);
                    }
                    tc::mma_commit(&sh.s_full[sb]);
                    tc::mma_commit(&sh.k_empty[st]);
                }
                if (j >= 1) {
                    const int i = j - 1, st = i % kStages, pb = i & 1;
                    ok = wait_or_abort(sh, &sh.p_full[pb], (i >> 1) & 1) &&
                         wait_or_abort(sh, &sh.v_full[st], (i / kStages) & 1);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint32_t aV = tc::smem_u32(smem + kOffV + st * kTileKV);
#pragma unroll
                    for (int ks = 0; ks < kKeysBlock / 16; ++ks) {
                        // P from tensor memory (its S buffer): lane = query
                        // row, 16 keys = 8 columns of 16-bit pairs per step;
                        // V: 16 keys = two 8-row groups of 128 bytes per step,
                        // the second 64 dims one box (8 KiB) on
                        tc::mma_f16_tmem_a(tmem + kColO, tmem + kColS + pb * kKeysBlock + ks * 8,
                                           tc::smem_desc(aV + ks * 2048, kBoxKV, 1024, tc::kSw128), idesc_o,
                                           i > 0 || ks > 0);
                    }
                    tc::mma_commit(&sh.pv_done);
                    tc::mma_commit(&sh.v_empty[st]);
                    tc::mma_commit(&sh.s_free[pb]);
                }
            }
            // every issued product completes before tensor memory is released
            tc::mma_commit(&sh.drain);
            tc::mbar_wait(&sh.drain, 0);
        }
    } else {
        // --------------------------------------------- softmax and epilogue
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // row of the tile = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const int64_t t = t0 + r / a.G;
        const int g = r % a.G;
        const int n_row = readable(a, t);
        const bool bf16 = a.in_bf16 != 0;
        const float c = a.c;
        float m_run = -INFINITY;  // offset of the row's exponents (log2 units)
        float l = 0.f;            // row sum of 2^(s c - m_run)
        bool ok = true;
        for (int j = 0; j < nb; ++j) {
            const int sb = j & 1;
            ok = warp_wait(sh, &sh.s_full[sb], (j >> 1) & 1);
            if (!ok) break;
            tc::tc_fence_after();
            float s[kKeysBlock];
#pragma unroll
            for (int ch = 0; ch < kKeysBlock / 32; ++ch)
                tmem_ld32(tmem + lane_base + kColS + sb * kKeysBlock + ch * 32, s + ch * 32);
            tc::tmem_wait_ld();
            // keys at or past the row's limit (and past S) take no weight
            const int lim = n_row - j * kKeysBlock;
            if (lim < kKeysBlock) {
#pragma unroll
                for (int i = 0; i < kKeysBlock; ++i)
                    if (i >= lim) s[i] = -INFINITY;
            }
            // block maximum of s c (c may be negative: then the minimum of s)
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
            if (c >= 0.f) {
#pragma unroll
                for (int i = 0; i < kKeysBlock; i += 4) {
                    mx0 = fmaxf(mx0, s[i]);
                    mx1 = fmaxf(mx1, s[i + 1]);
                    mx2 = fmaxf(mx2, s[i + 2]);
                    mx3 = fmaxf(mx3, s[i + 3]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < kKeysBlock; i += 4) {
                    const float n0 = s[i] == -INFINITY ? -INFINITY : -s[i];
                    const float n1 = s[i + 1] == -INFINITY ? -INFINITY : -s[i + 1];
                    const float n2 = s[i + 2] == -INFINITY ? -INFINITY : -s[i + 2];
                    const float n3 = s[i + 3] == -INFINITY ? -INFINITY : -s[i + 3];
                    mx0 = fmaxf(mx0, n0);
                    mx1 = fmaxf(mx1, n1);
                    mx2 = fmaxf(mx2, n2);
                    mx3 = fmaxf(mx3, n3);
                }
            }
            const float mraw = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
            const float bm = (mraw == -INFINITY) ? -INFINITY : mraw * fabsf(c);
            // raise the offset if the block's maximum runs more than 2^kRaise
            // above it (or the row had none yet)
            float alpha = 1.f;
            if (bm != -INFINITY && (m_run == -INFINITY || bm > m_run + kRaise)) {
                alpha = (m_run == -INFINITY) ? 0.f : tc::ex2(m_run - bm);
                m_run = bm;
                l *= alpha;
            }
            const float m_eff = (m_run == -INFINITY) ? 0.f : m_run;
            // p = 2^(s c - m) in [0, 2^kRaise], packed in the inputs' type;
            // masked keys take p = 0 whatever the sign of c
            uint32_t pk[kKeysBlock / 2];
            if (lim >= kKeysBlock) {
#pragma unroll
                for (int i = 0; i < kKeysBlock; i += 2) {
                    const float p0 = tc::ex2(fmaf(s[i], c, -m_eff));
                    const float p1 = tc::ex2(fmaf(s[i + 1], c, -m_eff));
                    l += p0 + p1;
                    pk[i / 2] = pack2(p0, p1, bf16);
                }
            } else {
#pragma unroll
                for (int i = 0; i < kKeysBlock; i += 2) {
                    const float p0 = (i < lim) ? tc::ex2(fmaf(s[i], c, -m_eff)) : 0.f;
                    const float p1 = (i + 1 < lim) ? tc::ex2(fmaf(s[i + 1], c, -m_eff)) : 0.f;
                    l += p0 + p1;
                    pk[i / 2] = pack2(p0, p1, bf16);
                }
            }
            // Seeing S(j) means the product of block j - 2 is done (S(j) waited
            // for it), so a parity wait for product j - 1 is exact here.  It is
            // made to rescale O after an offset raise, and on the last block
            // (so that the epilogue's wait for the last product is exact too)
            if (j > 0 && (j == nb - 1 || __any_sync(0xffffffffu, alpha != 1.f))) {
                ok = warp_wait(sh, &sh.pv_done, (j - 1) & 1);
                if (!ok) break;
                tc::tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int ch = 0; ch < kD / 32; ++ch) {
                        float o[32];
                        const uint32_t ta = tmem + lane_base + kColO + ch * 32;
                        tmem_ld32(ta, o);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(ta, o);
                    }
                    tc::tmem_wait_st();
                }
            }
            // the row's P over this block's S (its logits are in registers):
            // 64 16-bit values in 32 columns of the row's lane
            tc::tmem_st32u(tmem + lane_base + kColS + sb * kKeysBlock, pk);
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(&sh.p_full[sb]);
        }
        // epilogue: O / l for rows that read keys, zeros for rows that read
        // none, NaN if the CTA gave up.  The tensor-memory loads are
        // warp-collective, so every lane of a warp takes them (rows past T
        // included) and only the stores are per row.
        bool have_o = __all_sync(0xffffffffu, ok && nb > 0 && !aborted(sh));
        if (have_o) {
            have_o = warp_wait(sh, &sh.pv_done, (nb - 1) & 1);
            tc::tc_fence_after();
        }
        const bool bad = !ok || aborted(sh);
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        const int64_t obase = t * a.o_s0 + static_cast<int64_t>(h * a.G + g) * a.o_s1;
        const bool vec = a.o_s2 == 1 && ((reinterpret_cast<uintptr_t>(a.out) + obase * 2) & 15) == 0;
        for (int ch = 0; ch < kD / 32; ++ch) {
            float o[32];
            if (have_o) {
                tmem_ld32(tmem + lane_base + kColO + ch * 32, o);
                tc::tmem_wait_ld();
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = bad ? NAN : (l > 0.f && have_o) ? o[i] * inv : 0.f;
            if (t < a.T) {
                if (vec) {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + obase + ch * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack2(o[8 * q + 0], o[8 * q + 1], a.out_bf16 != 0);
                        w.y = pack2(o[8 * q + 2], o[8 * q + 3], a.out_bf16 != 0);
                        w.z = pack2(o[8 * q + 4], o[8 * q + 5], a.out_bf16 != 0);
                        w.w = pack2(o[8 * q + 6], o[8 * q + 7], a.out_bf16 != 0);
                        dst[q] = w;
                    }
                } else {
                    for (int i = 0; i < 32; ++i) {
                        const int64_t off = obase + static_cast<int64_t>(ch * 32 + i) * a.o_s2;
                        if (a.out_bf16)
                            static_cast<__nv_bfloat16 *>(a.out)[off] = __float2bfloat16_rn(o[i]);
                        else
                            static_cast<__half *>(a.out)[off] = __float2half_rn(o[i]);
                    }
                }
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// [rows, heads, 128] 16-bit tensor as a 3-D map whose box is 64 dims x
// `heads_box` heads x `rows_box` rows, 128-byte swizzle.
bool make_tmap_16(CUtensorMap *m, const void *base, int64_t rows, int64_t heads, int64_t s0, int64_t s1,
                  int heads_box, int rows_box) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(s1) * 2, static_cast<cuuint64_t>(s0) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(heads_box), static_cast<cuuint32_t>(rows_box)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tma_strides_ok(const void *base, int64_t s0, int64_t s1, int64_t s2, int64_t n0, int64_t n1) {
    if (s2 != 1 || (reinterpret_cast<uintptr_t>(base) % 16) != 0) return false;
    // strides of dims with more than one element must be positive multiples of 16 bytes
    if (n1 > 1 && (s1 <= 0 || (s1 * 2) % 16 != 0)) return false;
    if (n0 > 1 && (s0 <= 0 || (s0 * 2) % 16 != 0)) return false;
    return true;
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

// Covers: q, k, v all bf16 or all f16 with head dim 128 and 16-byte aligned
// rows; a bf16 or f16 output (any strides); G = Hq / Hkv a power of two up to
// 128.  Anything else: *used stays false.
cudaError_t launch_sdpa_tc(const SdpaArgs &a, cudaStream_t stream, bool *used) {
    *used = false;
    if (a.in_dt != SPD_BF16 && a.in_dt != SPD_F16) return cudaSuccess;
    if (a.out_dt != SPD_BF16 && a.out_dt != SPD_F16) return cudaSuccess;
    if (a.D != kD || a.S <= 0 || a.T <= 0) return cudaSuccess;
    const int G = a.Hq / a.Hkv;
    if (G < 1 || G > kRowsTile || (G & (G - 1)) != 0) return cudaSuccess;
    if (!tma_strides_ok(a.q, a.q_s0, a.q_s1, a.q_s2, a.T, a.Hq)) return cudaSuccess;
    if (!tma_strides_ok(a.k, a.k_s0, a.k_s1, a.k_s2, a.S, a.Hkv)) return cudaSuccess;
    if (!tma_strides_ok(a.v, a.v_s0, a.v_s1, a.v_s2, a.S, a.Hkv)) return cudaSuccess;
    const int tt = kRowsTile / G;
    const int64_t n_tiles = (static_cast<int64_t>(a.T) + tt - 1) / tt;
    if (n_tiles * a.Hkv > INT32_MAX) return cudaSuccess;

    CUtensorMap tq, tk, tv;
    // strides of extent-1 dims are never stepped over; give the map a legal value
    const int64_t qs1 = a.Hq > 1 ? a.q_s1 : kD, qs0 = a.T > 1 ? a.q_s0 : static_cast<int64_t>(a.Hq) * qs1;
    const int64_t ks1 = a.Hkv > 1 ? a.k_s1 : kD, ks0 = a.S > 1 ? a.k_s0 : static_cast<int64_t>(a.Hkv) * ks1;
    const int64_t vs1 = a.Hkv > 1 ? a.v_s1 : kD, vs0 = a.S > 1 ? a.v_s0 : static_cast<int64_t>(a.Hkv) * vs1;
    if (!make_tmap_16(&tq, a.q, a.T, a.Hq, qs0, qs1, G, tt)) return cudaSuccess;
    if (!make_tmap_16(&tk, a.k, a.S, a.Hkv, ks0, ks1, 1, kKeysBlock)) return cudaSuccess;
    if (!make_tmap_16(&tv, a.v, a.S, a.Hkv, vs0, vs1, 1, kKeysBlock)) return cudaSuccess;

    cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(sdpa_tc_kernel), kSmemBytes);
    if (e == cudaSuccess) e = prefer_shared_carveout(reinterpret_cast<const void *>(sdpa_tc_kernel));
    if (e != cudaSuccess) return e;

    SdpaTcArgs t{};
    t.out = a.out; t.o_s0 = a.o_s0; t.o_s1 = a.o_s1; t.o_s2 = a.o_s2;
    t.out_bf16 = a.out_dt == SPD_BF16;
    t.in_bf16 = a.in_dt == SPD_BF16;
    t.T = a.T; t.S = a.S; t.Hq = a.Hq; t.Hkv = a.Hkv; t.G = G; t.tt = tt;
    t.n_tiles = static_cast<int32_t>(n_tiles);
    t.causal = a.causal;
    t.c = a.sm_scale * kLog2e;
    sdpa_tc_kernel<<<static_cast<unsigned>(n_tiles * a.Hkv), kThreads, kSmemBytes, stream>>>(tq, tk, tv, t);
    e = cudaGetLastError();
    if (e == cudaSuccess) *used = true;
    return e;
}

}  // namespace spd
