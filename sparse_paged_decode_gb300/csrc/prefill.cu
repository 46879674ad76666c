// prefill.cu -- fused prefill score-to-selection ("Kernel ABI" --
// attention.msa_prefill_block_score): one call scores and selects key blocks
// per query head and per query block of block_size_q tokens for a ragged
// batch of prefill chunks.
//
// Three kernels on the caller's stream, no host synchronisation:
//   1. token_limits_kernel: each query token's sequence (a search of
//      cu_seqlens), its query block, and the key limit that block sees
//      (prefix_lens + qb * block_size_q + 1, clipped to seq_lens), written
//      with the token's page-table row to the workspace;
//   2. the decode score-sheet kernels (tensor-core score_tc_kernel where the
//      layout allows it) over all query tokens with those limits: a
//      token-level block-max sheet [Hi, total_q, NB] in the workspace.  Every
//      token of a query block shares the block's limit, so the query block's
//      score of key block kb is the maximum of its tokens' cells;
//   3. prefill_select_kernel: one CTA per (query block, head) reduces its
//      tokens' rows, places the initial and local policy blocks first
//      (ascending id) and ranks the other visible candidates (descending
//      score, ties to the lower id) into the rest of the row; unused cells
//      are -1.
#include <math.h>

#include "prefill.cuh"
#include "spd_dispatch.h"
#include "spd_internal.cuh"

namespace spd {

namespace {

constexpr int kLimitThreads = 256;
constexpr int kSelectThreads = 128;

struct PrefillWs {
    float *sheet;  // [Hi, total_q, NB]
    int32_t *sl;   // [total_q] key limit of each token's query block
    int32_t *ri;   // [total_q] page-table row of each token
};

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

PrefillWs carve(void *ws, int64_t total_q, int64_t Hi, int64_t NB) {
    char *p = static_cast<char *>(ws);
    PrefillWs w;
    w.sheet = reinterpret_cast<float *>(p);
    p += align256(static_cast<size_t>(Hi * total_q * NB) * sizeof(float));
    w.sl = reinterpret_cast<int32_t *>(p);
    p += align256(static_cast<size_t>(total_q) * sizeof(int32_t));
    w.ri = reinterpret_cast<int32_t *>(p);
    return w;
}

// Largest b in [0, B) with cu[b] <= x, or -1 (cu is read at stride s).
__device__ __forceinline__ int owner(const int32_t *cu, int64_t s, int B, int64_t x) {
    int lo = 0, hi = B - 1, found = -1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid * s] <= x) {
            found = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    return found;
}

// Keys visible to query block qb of sequence b: through the block's first
// token's own position, clipped to the sequence and the page table; 0 when
// the sequence's page-table row is outside the table.
__device__ __forceinline__ int32_t block_limit(const PrefillArgs &a, int b, int64_t qb) {
    const int32_t r = a.slot_ids[b * a.sid_s0];
    int64_t L = static_cast<int64_t>(a.prefix[b * a.pre_s0]) + qb * a.bsq + 1;
    const int64_t sl = a.seq_lens[b * a.sl_s0];
    if (L > sl) L = sl;
    const int64_t cap = static_cast<int64_t>(a.NB) * kBlock;
    if (L > cap) L = cap;
    if (r < 0 || r >= a.R || L < 0) L = 0;
    return static_cast<int32_t>(L);
}

__global__ void __launch_bounds__(kLimitThreads) token_limits_kernel(const PrefillArgs a, PrefillWs w) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kLimitThreads + threadIdx.x;
    if (i >= a.total_q) return;
    const int b = owner(a.cu_q, a.cuq_s0, a.B, i);
    int32_t L = 0, r = -1;
    if (b >= 0 && i < a.cu_q[(b + 1) * a.cuq_s0]) {
        const int64_t qb = (i - a.cu_q[b * a.cuq_s0]) / a.bsq;
        L = block_limit(a, b, qb);
        r = a.slot_ids[b * a.sid_s0];
    }
    w.sl[i] = L;
    w.ri[i] = r;
}

__global__ void __launch_bounds__(kSelectThreads) prefill_select_kernel(const PrefillArgs a, PrefillWs w) {
    __shared__ float comb[kMaxNB];
    const int64_t row = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    int32_t *o = a.out + h * a.o_s0 + row * a.o_s1;
    for (int k = tid; k < a.topk; k += kSelectThreads) o[k * a.o_s2] = -1;

    const int b = owner(a.cu_b, a.cub_s0, a.B, row);
    if (b < 0 || row >= a.cu_b[(b + 1) * a.cub_s0]) return;  // a row no sequence owns stays -1
    const int64_t qb = row - a.cu_b[b * a.cub_s0];
    const int32_t L = block_limit(a, b, qb);
    const int nvis = (L + kBlock - 1) / kBlock;

    // the query block's tokens, clipped to its chunk and to the batch
    int64_t t0 = static_cast<int64_t>(a.cu_q[b * a.cuq_s0]) + qb * a.bsq;
    int64_t t1 = t0 + a.bsq;
    const int64_t end = a.cu_q[(b + 1) * a.cuq_s0];
    if (t1 > end) t1 = end;
    if (t0 < 0) t0 = 0;
    if (t1 > a.total_q) t1 = a.total_q;

    // block scores of the query block: the maximum of its tokens' cells
    const float *sheet = w.sheet + static_cast<int64_t>(h) * a.total_q * a.NB;
    for (int kb = tid; kb < a.NB; kb += kSelectThreads) {
        float best = -INFINITY;
        if (kb < nvis)
            for (int64_t t = t0; t < t1; ++t) best = fmaxf(best, sheet[t * a.NB + kb]);
        comb[kb] = best;
    }
    __syncthreads();  // also orders the -1 fill before the writes below

    // policy blocks [0, n_init) and [c_local, nvis), ascending
    const int n_init = a.init_blocks < nvis ? a.init_blocks : nvis;
    const int c_local = a.local_blocks < nvis ? nvis - a.local_blocks : 0;
    const int n_forced = c_local <= n_init ? nvis : n_init + (nvis - c_local);
    for (int kb = tid; kb < nvis; kb += kSelectThreads) {
        const bool forced = kb < n_init || kb >= c_local;
        if (forced) {
            const int pos = (kb < n_init || c_local <= n_init) ? kb : n_init + (kb - c_local);
            if (pos < a.topk) o[pos * a.o_s2] = kb;
            continue;
        }
        const float s = comb[kb];
        if (isnan(s) || s == -INFINITY) continue;
        // rank among the other candidates: higher score first, ties to the lower id
        int rank = 0;
        for (int c = n_init; c < c_local; ++c) {
            const float x = comb[c];
            rank += (x > s) || (x == s && c < kb);
        }
        const int64_t pos = static_cast<int64_t>(n_forced) + rank;
        if (pos < a.topk) o[pos * a.o_s2] = kb;
    }
}

}  // namespace

size_t prefill_workspace_bytes(int64_t total_q, int64_t Hi, int64_t NB) {
    return align256(static_cast<size_t>(Hi * total_q * NB) * sizeof(float)) +
           2 * align256(static_cast<size_t>(total_q) * sizeof(int32_t));
}

cudaError_t launch_prefill(const PrefillArgs &a, void *ws, cudaStream_t stream) {
    const PrefillWs w = carve(ws, a.total_q, a.Hi, a.NB);
    if (a.total_q > 0) {
        const unsigned nblk = static_cast<unsigned>((static_cast<int64_t>(a.total_q) + kLimitThreads - 1) /
                                                    kLimitThreads);
        count_launches(1);
        token_limits_kernel<<<nblk, kLimitThreads, 0, stream>>>(a, w);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;

        ScoreArgs s{};
        s.q = a.q; s.q_s0 = a.q_s0; s.q_s1 = a.q_s1; s.q_s2 = a.q_s2;
        s.k = a.k; s.k_s0 = a.k_s0; s.k_s2 = a.k_s2;
        s.bt = a.bt; s.bt_s0 = a.bt_s0; s.bt_s1 = a.bt_s1;
        s.sl = w.sl; s.sl_s0 = 1;
        s.ri = w.ri; s.ri_s0 = 1;
        s.out = w.sheet; s.o_s0 = static_cast<int64_t>(a.total_q) * a.NB; s.o_s1 = a.NB; s.o_s2 = 1;
        s.q_dt = a.q_dt; s.k_dt = a.k_dt;
        s.T = a.total_q; s.Hi = a.Hi; s.Di = a.Di; s.R = a.R; s.NB = a.NB;
        s.P = a.P;
        s.idx_scale = a.scale;
        e = dispatch_score(s, stream);
        if (e != cudaSuccess) return e;
    }
    if (a.n_rows == 0) return cudaSuccess;
    count_launches(1);
    prefill_select_kernel<<<dim3(static_cast<unsigned>(a.n_rows), static_cast<unsigned>(a.Hi)), kSelectThreads, 0,
                            stream>>>(a, w);
    return cudaGetLastError();
}

}  // namespace spd
