/*
 * spd.h -- C ABI of the sparse paged decode library (libspd.so, sm_103a).
 *
 * Three stages of the decode-time attention boundary of an LLM serving engine:
 *   1. msa_block_score                block-max score sheet over a paged index cache
 *   2. msa_select_topk                top-k block ids per query row
 *   3. paged_sparse_decode_attention  paged GQA attention over the selected blocks
 *      paged_decode_attention         the same over every block (dense decode)
 * and, beside them, for prefill: msa_prefill_block_score, the fused
 * score-to-selection of a ragged batch of chunks per query block, and
 * attention_sdpa, dense (not paged) GQA attention with a causal flag.
 *
 * Contract shared by every entry point ("Kernel ABI" -- Core rules; "Slot
 * contract" -- 1. The validator owns the boundary):
 *   - The caller allocates every output (and the workspace) and owns all
 *     memory; the library allocates nothing, keeps no pointer after a call
 *     returns and never synchronises the host with the device.
 *   - Each call writes every logical cell of every output, honouring the
 *     output's shape, dtype and strides (outputs need not be contiguous), and
 *     leaves every input unchanged.
 *   - Work is enqueued on the supplied stream (NULL = the legacy default
 *     stream) and completes asynchronously; inputs must stay valid until it
 *     has run.  No device data is read on the host, so a call can be captured
 *     in a CUDA graph and replayed with new input values at the same
 *     addresses.
 *   - Entry points return nothing.  A call that fails host-side validation
 *     (bad dtype, rank, shape, stride, alignment, an output that overlaps an
 *     input or itself, a workspace that is too small, a shape outside the
 *     capability domain) launches nothing and records an error;
 *     spd_last_error() reports the last call's status on the calling thread.
 *     Device code never traps: metadata outside its range is excluded as
 *     described for each call.
 *
 * Tensors are passed as spd_tensor descriptors of device memory.  Strides are
 * in elements and may be any value for inputs (0 broadcasts); outputs need
 * strictly positive strides that map distinct cells to distinct elements.
 *
 * Paged addressing (shared by all calls): the caches hold P pages of
 * block_size = 128 token slots; logical token tau of request row r lives in
 * slot block_size * block_table[r][tau / block_size] + tau % block_size.
 * This page-granular table plays the part of the token-granular
 * req_to_token + req_pool_indices pair of "Kernel ABI" -- attention.decode:
 * query token t belongs to request row req_idx[t].  Tokens at or beyond
 * seq_lens[t] are excluded; seq_lens[t] <= 0 or a req_idx outside [0, R)
 * gives the token no keys; blocks whose page id lies outside [0, P) are
 * excluded; seq_lens beyond NB * block_size are clipped to it.
 */
#ifndef SPD_H
#define SPD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SPD_API __attribute__((visibility("default")))
#else
#define SPD_API
#endif

/* cudaStream_t without pulling in the CUDA headers */
typedef struct CUstream_st *spd_stream_t;

typedef enum {
    SPD_F32 = 0,  /* IEEE binary32                         */
    SPD_BF16 = 1, /* bfloat16                              */
    SPD_F16 = 2,  /* IEEE binary16                         */
    SPD_E4M3 = 3, /* OCP FP8 E4M3 ("e4m3fn"), max 448      */
    SPD_I32 = 4   /* int32                                 */
} spd_dtype;

typedef struct {
    void *data;        /* device address of element [0, ..., 0]        */
    int32_t dtype;     /* spd_dtype                                   */
    int32_t ndim;      /* number of dimensions used, 1..4             */
    int64_t shape[4];  /* extents of dims 0..ndim-1                   */
    int64_t stride[4]; /* element strides of dims 0..ndim-1           */
} spd_tensor;

typedef enum {
    SPD_OK = 0,
    SPD_ERR_INVALID_ARGUMENT = 1, /* malformed descriptor or inconsistent shapes     */
    SPD_ERR_UNSUPPORTED = 2,      /* well formed but outside the capability domain   */
    SPD_ERR_WORKSPACE = 3,        /* workspace missing, misaligned or too small      */
    SPD_ERR_ALIASING = 4,         /* an output overlaps an input or itself           */
    SPD_ERR_CUDA = 5              /* the CUDA runtime refused the launch             */
} spd_status;

/*
 * Stage 1 -- block-max score sheet.
 * "Kernel ABI" -- attention.msa_block_score (the decode score-sheet slot:
 * "per-request block-max scores"; the validator-side top-k consumes it) and
 * attention.msa_prefill_block_score (paged index cache "(slots, 1, D)";
 * queries see keys up to their own position).
 *
 *   scores[h][t][b] = max over valid tokens tau of block b of
 *                     (sum_d q_idx[t][h][d] * k_idx_cache[slot(tau)][0][d]) * idx_scale
 *   and -inf where block b of token t holds no valid token (including every
 *   b whose page id is outside the pool).
 *
 * q_idx        [T, Hi, Di]  f32 | bf16 | f16   query index heads
 * k_idx_cache  [P*128, 1, Di] same dtype as q_idx, or e4m3 (an FP8 index
 *              cache: its values enter as the E4M3 numbers they encode; a
 *              static scalar dequantisation scale is folded into idx_scale
 *              by the caller); one index key head
 * block_table  [R, NB] i32  page id of each logical block
 * seq_lens     [T] i32      valid keys of each query token (prefill: position + 1)
 * req_idx      [T] i32      block_table row of each query token
 * block_size   must be 128
 * scores       OUT [Hi, T, NB] f32
 * idx_scale    finite and > 0 (so the max commutes with the scaling)
 * Domain: Di in [1, 512], Hi >= 1, NB in [1, 1024].  Accumulation is fp32.
 */
SPD_API void msa_block_score(const spd_tensor *q_idx, const spd_tensor *k_idx_cache,
                     const spd_tensor *block_table, const spd_tensor *seq_lens,
                     const spd_tensor *req_idx, int32_t block_size,
                     const spd_tensor *scores, float idx_scale, spd_stream_t stream);

/*
 * Stage 2 -- top-k block selection.
 * "Kernel ABI" -- attention.decode ("topk_idx: (Hkv,B,K) block IDs"; -1
 * entries select nothing) and attention.msa_prefill_block_score ("unused
 * output cells must be -1"); "Slot contract" -- 2. (selection graded by set
 * overlap).
 *
 * For each row (h, t): the K largest candidate cells of scores[h][t][:], in
 * descending score order with ties broken toward the lower block id; a
 * candidate is a cell that is neither NaN nor -inf; rows with fewer than K
 * candidates are padded with -1.  Comparisons are exact on the fp32 values.
 *
 * scores    [Hi, T, NB] f32
 * topk_idx  OUT [Hi, T, K] i32 (K >= 1 taken from its shape; K may exceed NB)
 * Domain: NB in [1, 1024].
 */
SPD_API void msa_select_topk(const spd_tensor *scores, const spd_tensor *topk_idx, spd_stream_t stream);

/*
 * Stage 3 -- paged sparse GQA decode attention.
 * "Kernel ABI" -- attention.decode: a query row reads the given block ids
 * that are >= 0 and nothing else; a -1 id selects nothing, and keys at
 * positions >= seq_lens are left out; the K/V tensors are described at this
 * boundary, dense BF16 for the commissioned cache.  "Kernel ABI" --
 * attention.sdpa: Hq divisible by Hkv; q head g reads kv head g / (Hq / Hkv).
 * "MiniMax-M3 decode through the ATOM kernel library" -- static scalar K/V
 * scales on FP8 caches.
 *
 *   z_tau = sm_scale * k_scale * (q[t][g] . k_cache[slot(tau)][h])
 *   out[t][g] = sum_tau softmax(z)_tau * v_scale * v_cache[slot(tau)][h]
 * over the union of the valid tokens of the blocks listed in
 * topk_idx[h][t][:].  A selection is a set: repeated ids count once; ids
 * that are negative or >= NB select nothing.  A query row with no valid key
 * writes zeros.  Logits, softmax and accumulation are fp32; the output is
 * rounded to bf16 (nearest even).
 *
 * q          [T, Hq, D] f32 | bf16 | f16
 * k_cache    [P*128, Hkv, D] e4m3 | bf16 } innermost stride 1
 * v_cache    [P*128, Hkv, D] the dtype and shape of k_cache
 *            (the scales multiply the decoded values either way; pass 1.0
 *            for a BF16 cache stored unscaled)
 * block_table [R, NB] i32, seq_lens [T] i32, req_idx [T] i32 (see above)
 * topk_idx   [Hkv, T, K] i32; a stride of 0 on dim 0 shares one selection
 *            across kv heads (the usual case: one index head)
 * out        OUT [T, Hq, D] bf16
 * sm_scale, k_scale, v_scale  finite fp32 scalars
 * block_size must be 128
 * workspace  device scratch of at least spd_decode_workspace_bytes(...)
 *            bytes, 256-byte aligned; contents need no initialisation and
 *            are overwritten; it must not be shared by calls that may run
 *            concurrently
 * Domain: D in [1, 256], Hq / Hkv <= 16, NB in [1, 1024], K >= 1.
 * Query rows of one request that sit next to each other (the draft tokens
 * of a verification row) share each K/V page read.
 */
SPD_API void paged_sparse_decode_attention(const spd_tensor *q, const spd_tensor *k_cache,
                                   const spd_tensor *v_cache, const spd_tensor *block_table,
                                   const spd_tensor *seq_lens, const spd_tensor *req_idx,
                                   const spd_tensor *topk_idx, const spd_tensor *out,
                                   float sm_scale, int32_t block_size, float k_scale,
                                   float v_scale, void *workspace, size_t workspace_bytes,
                                   spd_stream_t stream);

/*
 * Dense paged decode attention: paged_sparse_decode_attention with every
 * block selected (the degenerate case of "Kernel ABI" -- attention.decode
 * whose selection lists all blocks below ceil(seq_len / 128)).  Same
 * arguments without topk_idx.
 */
SPD_API void paged_decode_attention(const spd_tensor *q, const spd_tensor *k_cache,
                            const spd_tensor *v_cache, const spd_tensor *block_table,
                            const spd_tensor *seq_lens, const spd_tensor *req_idx,
                            const spd_tensor *out, float sm_scale, int32_t block_size,
                            float k_scale, float v_scale, void *workspace,
                            size_t workspace_bytes, spd_stream_t stream);

/*
 * Fused prefill score-to-selection for a ragged batch of prefill chunks.
 * "Kernel ABI" -- attention.msa_prefill_block_score (the V2 call: one call
 * scores and selects for the whole ragged batch; a query block may pick only
 * key blocks it can see from position prefix_lens[b] + qb * block_size_q;
 * the init/local arguments fix blocks that are always taken; ids count the
 * blocks of the request's own key sequence; leftover cells hold -1).
 *
 * Sequence b owns query tokens cu_seqlens[b] .. cu_seqlens[b+1]-1, whose
 * first token sits at key position prefix_lens[b]; it has seq_lens[b] keys
 * in total, read through row slot_ids[b] of block_table; its query blocks of
 * block_size_q tokens are output rows cu_seqblocks_q[b] + qb.  For query
 * block qb and index head h:
 *   L     = min(prefix_lens[b] + qb * block_size_q + 1, seq_lens[b], NB * 128)
 *           visible keys (through the block's first token's own position;
 *           0 if slot_ids[b] is outside the table); nvis = ceil(L / 128)
 *   S[kb] = max over the block's tokens t and keys tau < L of key block kb of
 *           (q[t][h] . index_k_cache[slot(tau)][0]) * scale   (kb < nvis)
 *   row   = the policy blocks (the first init_blocks and the last
 *           local_blocks visible blocks) in ascending id, then the other
 *           visible blocks whose S is neither NaN nor -inf in descending S
 *           (ties to the lower id), truncated to topk, padded with -1.
 * Output rows that no sequence owns are all -1.  With block_size_q = 1 and
 * no policy blocks a row is msa_select_topk of msa_block_score for one token
 * with seq_len = its position + 1.
 *
 * q              [total_q, Hi, Di] f32 | bf16 | f16 index queries (Hi heads)
 * index_k_cache  [P*128, 1, Di] the dtype of q, or e4m3 (values as encoded)
 * block_table    [R, NB] i32 page ids (stands in for req_to_token)
 * slot_ids       [B] i32 page-table row of each sequence
 * cu_seqlens     [B+1] i32 nondecreasing query token offsets
 * seq_lens       [B] i32, prefix_lens [B] i32
 * block_size_q >= 1; block_size_k must be 128; init_blocks, local_blocks >= 0
 * scale          finite and > 0
 * cu_seqblocks_q [B+1] i32 nondecreasing output row offsets
 *                (normally cu_seqblocks_q[b+1] - cu_seqblocks_q[b] =
 *                ceil(chunk_b / block_size_q))
 * out_topk       OUT [Hi, all_seqblock_q, topk] i32 (topk >= 1 from its shape)
 * workspace      device scratch of at least spd_prefill_workspace_bytes(
 *                total_q, Hi, NB) bytes, 256-byte aligned, no initialisation
 *                needed, not shared by calls that may run concurrently
 * The pages' max_seqlen_q, max_seqlen_k, topk, max_seqblock_q and
 * all_seqblock_q arguments are not taken: the launch is sized from the
 * tensors' shapes, so the call reads no device data on the host.
 * Domain: Di in [1, 512], Hi <= 65535, NB in [1, 1024].  Accumulation is fp32.
 */
SPD_API void msa_prefill_block_score(const spd_tensor *q, const spd_tensor *index_k_cache,
                                     const spd_tensor *block_table, const spd_tensor *slot_ids,
                                     const spd_tensor *cu_seqlens, const spd_tensor *seq_lens,
                                     const spd_tensor *prefix_lens, int32_t block_size_q, int32_t block_size_k,
                                     int32_t init_blocks, int32_t local_blocks, float scale,
                                     const spd_tensor *cu_seqblocks_q, const spd_tensor *out_topk,
                                     void *workspace, size_t workspace_bytes, spd_stream_t stream);

/*
 * Workspace bytes msa_prefill_block_score needs for total_q query tokens, Hi
 * index heads and a page table of NB blocks (0 for invalid sizes).
 */
SPD_API size_t spd_prefill_workspace_bytes(int64_t total_q, int64_t Hi, int64_t NB);

/*
 * Dense GQA attention with a causal flag.
 * "Kernel ABI" -- attention.sdpa (q, k, v, out, a softmax scale and a
 * causal flag; softmax attention where each kv head serves Hq / Hkv query
 * heads, Hq a multiple of Hkv).
 *
 *   z_j = sm_scale * (q[t][g] . k[j][h]),  h = g / (Hq / Hkv)
 *   out[t][g] = sum_j softmax(z)_j * v[j][h]
 * over the keys j that query token t may read: all S keys, or, when causal
 * is nonzero, the keys j <= t + S - T (the T query tokens are the last T
 * positions of the key sequence -- a prefill chunk after S - T cached
 * tokens; for T == S the usual lower-triangular mask).  A query token that
 * may read no key (causal with t < T - S, or S == 0) writes zeros.  The page
 * fixes the flag, not its alignment; this bottom-right alignment is the
 * reading taken here.
 *
 * q    [T, Hq, D]   f32 | bf16 | f16, any strides
 * k, v [S, Hkv, D]  the dtype of q, any strides (keys are not paged)
 * out  OUT [T, Hq, D] f32 | bf16 | f16 (rounded to nearest even)
 * sm_scale finite fp32 scalar
 * Logits, softmax and accumulation are fp32.  No workspace.
 * Domain: D in [1, 256], Hq a positive multiple of Hkv, Hkv <= 65535,
 * T * Hq and S below 2^30.
 */
SPD_API void attention_sdpa(const spd_tensor *q, const spd_tensor *k, const spd_tensor *v, const spd_tensor *out,
                            float sm_scale, int32_t causal, spd_stream_t stream);

/*
 * paged_sparse_decode_attention without a caller-provided workspace.
 *
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory -- for example a kernel slot inside a host
 * engine that hands it only its input and output buffers and keeps every
 * device allocation to its own memory planner, or code that must not call an
 * allocator on its decode path.  Such a caller passes the same inputs and
 * output as to paged_sparse_decode_attention and gets the same result; the
 * scratch comes from a 16 MiB device array built into the library instead of
 * the workspace argument.  The call allocates nothing.
 *
 * - Limit: shapes whose spd_decode_workspace_bytes(...) exceeds 16 MiB are
 *   rejected with SPD_ERR_UNSUPPORTED (use the workspace entry point).
 * - The array is part of the library's device code: it is created on a GPU
 *   when that code is loaded there and held until the process exits.  With
 *   CUDA's default lazy module loading that is the first use of this call on
 *   the GPU; under CUDA_MODULE_LOADING=EAGER every GPU on which the process
 *   creates a context holds the 16 MiB, whether or not the call is used.
 * - The first call on a device looks up the array's device address, with
 *   that device current; make that first call before any stream capture.
 * - Every call shares the one array and it keeps the last call's contents
 *   (each call rewrites whatever it needs zeroed).  Calls that could run on
 *   the GPU at the same time -- on different streams, or from different host
 *   threads -- race on it: serialise them.
 * - A device-side wait that timed out is recorded in the array's status
 *   word, not in a caller buffer: spd_workspace_status(NULL, stream) reads it
 *   for the current device.
 */
SPD_API void paged_sparse_decode_attention_noalloc(const spd_tensor *q, const spd_tensor *k_cache,
                                                   const spd_tensor *v_cache, const spd_tensor *block_table,
                                                   const spd_tensor *seq_lens, const spd_tensor *req_idx,
                                                   const spd_tensor *topk_idx, const spd_tensor *out,
                                                   float sm_scale, int32_t block_size, float k_scale,
                                                   float v_scale, spd_stream_t stream);

/*
 * Workspace bytes the two attention calls need for T query rows, Hq q heads,
 * Hkv kv heads, head dim D and a page table of NB blocks.  Depends on these
 * capacities only (never on seq_lens or topk_idx), so one allocation serves
 * every replay of a captured graph.  Returns 0 for shapes outside the domain.
 */
SPD_API size_t spd_decode_workspace_bytes(int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t NB,
                                  int32_t block_size);

/*
 * Status of the last call made on this thread: SPD_OK or an spd_status code.
 * When msg is not NULL, up to cap-1 bytes of a NUL-terminated description
 * are copied into it.
 */
SPD_API int spd_last_error(char *msg, size_t cap);

/*
 * Diagnostics: number of CUDA kernels this library has enqueued in this
 * process so far (all threads, all streams).  Benchmarks difference it
 * around a timed region to count their launches.
 */
SPD_API uint64_t spd_launch_count(void);

/*
 * Diagnostics: kernel selection for the attention calls on this thread's
 * subsequent calls.  0 (default) picks the tensor-core kernel whenever the
 * shapes and layouts allow it and the general-layout kernel otherwise; 1
 * always uses the general-layout kernel (for cross-checking the two).
 * Returns the previous setting.  Results agree within the stated tolerance
 * either way.
 */
SPD_API int spd_set_attention_kernel(int policy);

/*
 * Diagnostics: kernel selection per stage on this thread's subsequent calls.
 * stage 1 = msa_block_score, 2 = msa_select_topk, 3 = the attention calls
 * (the same setting as spd_set_attention_kernel), 4 = attention_sdpa.  policy
 * 0 (default) picks the specialised kernel whenever the shapes and layouts
 * allow it, 1 always the general-layout kernel; for stage 2, policy 2 picks
 * the shared-memory rank kernel (the default sorts rows of up to 256 blocks
 * in registers and ranks longer ones); for stage 3 and an FP8-E4M3 cache,
 * policy 2 picks the keys-on-lanes tensor-core kernel and 3 the query-rows
 * one (the default takes the query-rows kernel for bf16 queries of head dim
 * 128, G <= 16 and on average at least 48 query rows per request and kv
 * head, the keys-on-lanes one otherwise; a shape the picked kernel does not
 * cover runs on the general-layout kernel).  All give identical selections, and
 * attention results that agree within the stated tolerance.  Returns the
 * previous setting, or -1 for an unknown stage.
 */
SPD_API int spd_set_kernel_policy(int stage, int policy);

/*
 * Diagnostics: status word an attention call left in its workspace (0 = ok;
 * bit 0 = a device-side wait timed out and the call's output is not valid).
 * workspace = NULL reads the built-in scratch of
 * paged_sparse_decode_attention_noalloc on the current device.
 * Synchronises with `stream` to read it -- never call it on a hot path.
 * Returns -1 when the status cannot be read.  Leaves spd_last_error alone.
 */
SPD_API int spd_workspace_status(const void *workspace, spd_stream_t stream);

/* Library version string, e.g. "spd 0.1 sm_103a". */
SPD_API const char *spd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPD_H */
