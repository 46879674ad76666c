"""GPU parity: each stage through the C ABI against the CPU oracle.

Every call gets NaN / sentinel-poisoned outputs and its inputs are hashed
before and after ("Kernel ABI" -- Why the ABI is shaped this way: poisoning
and input-mutation checks).  Small cases compare every output cell; the
full-size decode configurations compare every cell of the score sheet, the
top-k and the attention output: each output row depends only on its own
query row, so the single-threaded oracle runs on disjoint sets of rows in
several host threads at once (ctypes releases the interpreter lock during a
call; the oracle keeps no state between calls).  Attention is checked with
the oracle's top-k fed to both sides, and end to end from the GPU's own
selection.  After every attention call the workspace's status word must be 0
(no device-side wait timed out).
"""
import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from parity import check_attention, check_scores, check_topk, digest, nan_like
from sparse_paged_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu
BS = 128
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def spd():
    import sparse_paged_decode_gb300 as m

    return m


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


# ------------------------------------------------------------------ runners

def gpu_scores(spd, g, Hi=None):
    T, NB = g.seq_lens.shape[0], g.block_table.shape[1]
    Hi = g.q_idx.shape[1] if Hi is None else Hi
    out = nan_like((Hi, T, NB), torch.float32, DEV)
    before = digest(g.q_idx, g.k_idx_cache, g.block_table, g.seq_lens, g.req_idx)
    spd.msa_block_score(g.q_idx, g.k_idx_cache, g.block_table, g.seq_lens, g.req_idx, BS, out, g.idx_scale)
    torch.cuda.synchronize()
    assert digest(g.q_idx, g.k_idx_cache, g.block_table, g.seq_lens, g.req_idx) == before, "inputs mutated"
    return out


def gpu_topk(spd, scores, K):
    out = nan_like((scores.shape[0], scores.shape[1], K), torch.int32, DEV)
    before = digest(scores)
    spd.msa_select_topk(scores, out)
    torch.cuda.synchronize()
    assert digest(scores) == before, "scores mutated"
    return out


def gpu_attention(spd, g, topk):
    T = g.q.shape[0]
    out = nan_like((T, g.Hq, g.D), torch.bfloat16, DEV)
    # zeroed, so the status word reads 0 after the general-layout kernel too
    # (only the tensor-core path's planner writes the workspace header)
    ws = torch.zeros(spd.decode_workspace_bytes(T, g.Hq, g.Hkv, g.D, g.NB), dtype=torch.uint8, device=DEV)
    ins = (g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, g.req_idx, topk)
    before = digest(*ins)
    if topk is None:
        spd.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, g.req_idx, out,
                                   g.sm_scale, BS, g.k_scale, g.v_scale, ws)
    else:
        spd.paged_sparse_decode_attention(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, g.req_idx,
                                          topk, out, g.sm_scale, BS, g.k_scale, g.v_scale, ws)
    torch.cuda.synchronize()
    assert digest(*ins) == before, "inputs mutated"
    assert spd.workspace_status(ws) == 0, "a device-side wait timed out (workspace status bit 0)"
    return out


def f32(x):
    return float(np.float32(x))


ORACLE_THREADS = max(1, os.cpu_count() or 1)


def _oracle_chunk(orc, w, rows, topk_np):
    idx = torch.tensor(rows, dtype=torch.int64)
    tk = None if topk_np is None else np.ascontiguousarray(topk_np[:, rows, :])
    return orc.paged_attention(w.q[idx], w.k_cache, w.v_cache, w.block_table, w.req_idx[idx],
                               w.seq_lens[idx], tk, f32(w.sm_scale), f32(w.k_scale), f32(w.v_scale))


def oracle_rows(orc, w, rows, topk_np):
    """Oracle attention for the query rows ``rows`` only, the rows dealt out
    round-robin to ORACLE_THREADS host threads (each thread a separate call
    of the single-threaded oracle on its own rows)."""
    rows = list(rows)
    n = min(ORACLE_THREADS, len(rows))
    if n <= 1:
        return _oracle_chunk(orc, w, rows, topk_np)
    parts = [rows[i::n] for i in range(n)]
    with ThreadPoolExecutor(max_workers=n) as ex:
        outs = list(ex.map(lambda part: _oracle_chunk(orc, w, part, topk_np), parts))
    ref = np.empty((len(rows),) + outs[0].shape[1:], dtype=np.float64)
    for i, o in enumerate(outs):
        ref[i::n] = o
    return ref


class _policy:
    """Stage-3 kernel policy for the duration of a block (None: as set)."""

    def __init__(self, spd, pol):
        self.spd, self.pol, self.old = spd, pol, None

    def __enter__(self):
        if self.pol is not None:
            self.old = self.spd.set_kernel_policy(3, self.pol)

    def __exit__(self, *exc):
        if self.pol is not None:
            self.spd.set_kernel_policy(3, self.old)


def full_check(spd, orc, w, attn_rows=None, score_rows=None, per_head_topk=False, policies=(None,)):
    """Score + select + sparse attention + dense attention against the oracle;
    the attention calls run once per stage-3 kernel policy in ``policies``
    (None: the policy as set), all against the same oracle outputs."""
    g = w.to(DEV)
    res = {}
    full_s = None
    if w.q_idx is not None:
        s = gpu_scores(spd, g)
        rows = list(range(w.T)) if score_rows is None else score_rows
        ridx = torch.tensor(rows, dtype=torch.int64)
        ref_s = orc.block_score(w.q_idx[ridx], w.k_idx_cache, w.block_table, w.req_idx[ridx], w.seq_lens[ridx],
                                f32(w.idx_scale))
        if score_rows is None:
            full_s = ref_s
        res["score_err"] = check_scores(s.cpu().numpy()[:, rows], ref_s)
        tk = gpu_topk(spd, s, w.K)
        res["overlap"] = check_topk(tk.cpu().numpy()[:, rows], ref_s, w.K)
    if w.q is None:
        return res
    rows = list(range(w.T)) if attn_rows is None else attn_rows
    pad = [i for i, t in enumerate(rows) if int(w.seq_lens[t]) <= 0]
    if w.K > 0 and w.q_idx is not None:
        # oracle selection for every token, fed to both sides
        if full_s is None:
            full_s = orc.block_score(w.q_idx, w.k_idx_cache, w.block_table, w.req_idx, w.seq_lens,
                                     f32(w.idx_scale))
        ref_tk = orc.select_topk(full_s, w.K)  # [1, T, K]
        if per_head_topk:
            ref_tk = np.concatenate([np.roll(ref_tk, h, axis=2) for h in range(w.Hkv)], axis=0)
            tk_dev = torch.from_numpy(ref_tk).to(DEV)
        else:
            tk_dev = torch.from_numpy(ref_tk).to(DEV).expand(w.Hkv, -1, -1)
        ref = oracle_rows(orc, w, rows, ref_tk)
        # end to end: the GPU's own selection feeds the GPU attention
        ref_e2e = oracle_rows(orc, w, rows, tk.cpu().numpy())
        for pol in policies:
            with _policy(spd, pol):
                out = gpu_attention(spd, g, tk_dev)
                res["sparse"] = check_attention(out.float().cpu().numpy()[rows], ref,
                                                "sparse attention (policy %s)" % pol, pad)
                out_e2e = gpu_attention(spd, g, tk.expand(w.Hkv, -1, -1))
                res["e2e"] = check_attention(out_e2e.float().cpu().numpy()[rows], ref_e2e,
                                             "end-to-end attention (policy %s)" % pol, pad)
    ref_d = oracle_rows(orc, w, rows, None)
    for pol in policies:
        with _policy(spd, pol):
            out_d = gpu_attention(spd, g, None)
            res["dense"] = check_attention(out_d.float().cpu().numpy()[rows], ref_d,
                                           "dense attention (policy %s)" % pol, pad)
    return res


# --------------------------------------------------------------- small cases

SMALL = {
    "g8_d128_bf16_mixed": dict(lengths=[1500, 700, 129, 2048, 1], tokens_per_request=[4, 4, 1, 16, 1], Hq=64, Hkv=8,
                               D=128, Di=128, NB=16, P=96, K=5),
    "g4_d64_f32": dict(lengths=[300, 512, 77], tokens_per_request=[1, 2, 3], Hq=8, Hkv=2, D=64, Di=32, NB=4, P=16,
                       K=2, dtype=torch.float32),
    "g16_d128_f16": dict(lengths=[1000, 257], tokens_per_request=[3, 8], Hq=32, Hkv=2, D=128, Di=64, NB=8, P=24,
                         K=3, dtype=torch.float16),
    "g1_d96_mha": dict(lengths=[640, 90], tokens_per_request=[2, 1], Hq=4, Hkv=4, D=96, Di=16, NB=6, P=12, K=4),
    "padded_t3": dict(lengths=[1200, 3000, 400], tokens_per_request=[8, 16, 4], Hq=64, Hkv=8, D=128, Di=128, NB=32,
                      P=64, K=8, q_dist="student_t3", padded_tail=[3, 16, 0]),
    "k_above_nb": dict(lengths=[200, 384], tokens_per_request=[1, 4], Hq=16, Hkv=2, D=128, Di=128, NB=3, P=8, K=7),
}


@pytest.fixture(params=[0, 1], ids=["auto_kernel", "general_kernel"])
def kernel_policy(request, spd):
    """Run a test through the default kernel choice and through the
    general-layout kernels, for every stage."""
    old = [spd.set_kernel_policy(stage, request.param) for stage in (1, 2, 3)]
    yield request.param
    for stage, o in zip((1, 2, 3), old):
        spd.set_kernel_policy(stage, o)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases(spd, orc, name, kernel_policy):
    w = W.make_decode(name, seed=zlib.crc32(name.encode()) % 1000, **SMALL[name])
    full_check(spd, orc, w)


# stage-3 policies that force one of the two FP8-cache tensor-core kernels
FP8_KERNELS = (2, 3)  # keys on the TMEM lanes, query rows on the MMA rows


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases_both_fp8_kernels(spd, orc, name):
    """Each small case through each of the two FP8-cache kernels (a shape a
    kernel does not cover runs on the general-layout kernel)."""
    w = W.make_decode(name, seed=zlib.crc32(name.encode()) % 1000, **SMALL[name])
    full_check(spd, orc, w, policies=FP8_KERNELS)


def test_large_logits(spd, orc, kernel_policy):
    """Heavy-tailed queries scaled up: logits of tens of units and outputs
    dominated by a few keys, where rounding of the queries or of the
    probabilities shows first."""
    w = W.make_decode("large", lengths=[3000, 1700, 600], tokens_per_request=[4, 8, 1], Hq=64, Hkv=8, D=128,
                      Di=128, NB=32, P=64, K=8, seed=21, q_dist="student_t3")
    w.q = (w.q.float() * 4.0).to(w.q.dtype)
    res = full_check(spd, orc, w)
    assert res["dense"][1] >= 0.9999


def test_tiny_sparse_decode(spd, orc):
    full_check(spd, orc, W.config(1))


SELECT_SHAPES = [(1, 1), (5, 3), (31, 16), (32, 32), (33, 7), (64, 64), (100, 16), (128, 32), (128, 64),
                 (129, 32), (200, 50), (256, 128), (256, 300), (257, 16), (300, 64)]


def edge_score_rows(rng, T, NB):
    """Score rows that stress the ordering: random values, heavy ties, signed
    zeros, NaN / -inf (not candidates), +inf, rows with fewer candidates than
    K and rows with none."""
    s = rng.standard_normal((T, NB)).astype(np.float32)
    for t in range(T):
        kind = t % 8
        if kind == 1:
            s[t] = rng.choice(np.array([-1.0, 0.0, 1.0, 2.0], np.float32), NB)
        elif kind == 2:
            s[t] = rng.choice(np.array([0.0, -0.0, -np.inf, 0.5], np.float32), NB)
        elif kind == 3:
            s[t, rng.random(NB) < 0.3] = np.nan
        elif kind == 4:
            s[t, rng.random(NB) < 0.2] = np.inf
        elif kind == 5:
            s[t] = rng.choice(np.array([np.nan, -np.inf], np.float32), NB)
        elif kind == 6:
            s[t] = 0.25
        elif kind == 7:
            s[t, rng.random(NB) < 0.9] = -np.inf
    return s


@pytest.mark.parametrize("NB,K", SELECT_SHAPES)
def test_select_kernels_agree_on_edge_rows(spd, orc, NB, K):
    """Top-k ("attention.msa_select_topk"): every selection kernel (register
    sort, shared-memory ranks, general layout) gives the oracle's ids exactly
    -- ties to the lower block id, -0 equal to +0, NaN and -inf never
    selected, -1 padding -- on contiguous and strided sheets."""
    rng = np.random.default_rng(NB * 1000 + K)
    Hi, T = 2, 16
    sheet = np.stack([edge_score_rows(rng, T, NB) for _ in range(Hi)])
    ref = orc.select_topk(sheet, K)
    dense = torch.from_numpy(sheet).to(DEV)
    wide = torch.full((Hi, T, 2 * NB), 77.0, device=DEV)
    wide[:, :, ::2] = dense
    for scores in (dense, wide[:, :, ::2]):
        for policy in (0, 2, 1):
            old = spd.set_kernel_policy(2, policy)
            try:
                got = gpu_topk(spd, scores, K).cpu().numpy()
            finally:
                spd.set_kernel_policy(2, old)
            assert np.array_equal(got, ref), f"policy {policy}, stride {scores.stride()}"


def test_per_head_selection_and_bad_metadata(spd, orc):
    w = W.make_decode("meta", lengths=[900, 300, 1700], tokens_per_request=[2, 3, 4], Hq=32, Hkv=4, D=128,
                      Di=128, NB=16, P=48, K=6, seed=77)
    # pages outside the pool, a request row outside the table, negative and
    # over-long seq_lens: excluded, never trapped
    w.block_table[0, 2] = -1
    w.block_table[1, 0] = w.P + 5
    w.req_idx[4] = 9
    w.seq_lens[5] = -3
    w.seq_lens[0] = w.NB * BS + 50
    full_check(spd, orc, w, per_head_topk=True)


def test_many_rows_planner_rounds(spd, orc):
    """More query rows than one planner round (512) and more lists than one
    list CTA's warps, with per-kv-head selection: the group scan carries run
    starts and group counts across rounds, and lists spread over CTAs."""
    rng = np.random.default_rng(404)
    n_req = 170
    toks = rng.choice([1, 2, 3, 4, 8], size=n_req).tolist()
    lengths = rng.integers(1, 500, size=n_req).tolist()
    w = W.make_decode("rows", lengths=lengths, tokens_per_request=toks, Hq=16, Hkv=2, D=128, Di=64, NB=4,
                      P=4 * n_req + 8, K=2, seed=404)
    assert w.T > 512
    full_check(spd, orc, w, per_head_topk=True)


def test_duplicate_and_out_of_range_ids(spd, orc):
    w = W.make_decode("dup", lengths=[1000, 600], tokens_per_request=[2, 1], Hq=16, Hkv=2, D=128, Di=128, NB=8,
                      P=20, K=4, seed=5)
    tk = np.array([[[3, 3, -1, 0, 99, -7, 5, 3], [1, 2, 2, 2, -1, -1, 7, 0], [4, -1, 4, 0, 1, 1, 1, 1]]],
                  dtype=np.int32)
    g = w.to(DEV)
    out = gpu_attention(spd, g, torch.from_numpy(tk).to(DEV).expand(w.Hkv, -1, -1))
    ref = orc.paged_attention(w.q, w.k_cache, w.v_cache, w.block_table, w.req_idx, w.seq_lens, tk,
                              f32(w.sm_scale), f32(w.k_scale), f32(w.v_scale))
    check_attention(out.float().cpu().numpy(), ref)


def test_nan_poison_pages_never_leak(spd, orc):
    w = W.make_decode("nanpoison", lengths=[700, 333], tokens_per_request=[4, 2], Hq=16, Hkv=2, D=128, Di=128,
                      NB=8, P=20, K=3, seed=6)
    owned = set()
    for r, L in enumerate(w.request_lengths):
        for tau in range(L):
            owned.add(int(w.block_table[r, tau // BS]) * BS + tau % BS)
    mask = torch.ones(w.P * BS, dtype=torch.bool)
    mask[torch.tensor(sorted(owned))] = False
    for c in (w.k_cache, w.v_cache):
        c.view(torch.uint8)[mask] = 0x7F  # NaN codes everywhere no valid token lives
    kmask = mask.clone()
    w.k_idx_cache[kmask] = float("nan")
    res = full_check(spd, orc, w)
    assert res["dense"][1] >= 0.9999


def test_strided_inputs_and_outputs(spd, orc):
    w = W.make_decode("strided", lengths=[800, 250], tokens_per_request=[3, 2], Hq=16, Hkv=2, D=128, Di=64, NB=8,
                      P=20, K=3, seed=9)
    g = w.to(DEV)
    # q stored head-major and viewed token-major; index queries with a gap
    q_hm = g.q.transpose(0, 1).contiguous().transpose(0, 1)
    qi_big = torch.zeros((w.T, 1, w.Di * 2), dtype=g.q_idx.dtype, device=DEV)
    qi_big[:, :, ::2] = g.q_idx
    qi = qi_big[:, :, ::2]
    # outputs are views inside larger poisoned buffers
    s_big = torch.full((1, w.T, w.NB + 3), 123.0, device=DEV)
    s_view = s_big[:, :, 1:1 + w.NB]
    spd.msa_block_score(qi, g.k_idx_cache, g.block_table, g.seq_lens, g.req_idx, BS, s_view, g.idx_scale)
    tk_big = torch.full((1, w.T, 2 * w.K), 4242, dtype=torch.int32, device=DEV)
    tk_view = tk_big[:, :, ::2]
    spd.msa_select_topk(s_view, tk_view)
    o_big = torch.full((w.T, w.Hq, w.D + 8), 7.0, dtype=torch.bfloat16, device=DEV)
    o_view = o_big[:, :, 4:4 + w.D]
    ws = torch.empty(spd.decode_workspace_bytes(w.T, w.Hq, w.Hkv, w.D, w.NB), dtype=torch.uint8, device=DEV)
    spd.paged_sparse_decode_attention(q_hm, g.k_cache, g.v_cache, g.block_table, g.seq_lens, g.req_idx,
                                      tk_view.expand(w.Hkv, -1, -1), o_view, g.sm_scale, BS, g.k_scale,
                                      g.v_scale, ws)
    torch.cuda.synchronize()
    ref_s = orc.block_score(w.q_idx, w.k_idx_cache, w.block_table, w.req_idx, w.seq_lens, f32(w.idx_scale))
    check_scores(s_view.cpu().numpy(), ref_s)
    assert torch.all(s_big[:, :, 0] == 123.0) and torch.all(s_big[:, :, -2:] == 123.0)
    check_topk(tk_view.cpu().numpy(), ref_s, w.K)
    assert torch.all(tk_big[:, :, 1::2] == 4242)
    ref = orc.paged_attention(w.q, w.k_cache, w.v_cache, w.block_table, w.req_idx, w.seq_lens,
                              tk_view.cpu().numpy(), f32(w.sm_scale), f32(w.k_scale), f32(w.v_scale))
    check_attention(o_view.float().cpu().numpy(), ref)
    assert torch.all(o_big[:, :, :4] == 7.0) and torch.all(o_big[:, :, -4:] == 7.0)


@pytest.mark.parametrize("kv,policy", [("e4m3", None), ("e4m3", 3), ("bf16", None)],
                         ids=["e4m3", "e4m3_query_rows_kernel", "bf16"])
def test_graph_capture_and_replay_with_new_inputs(spd, orc, kv, policy):
    """"Slot contract" -- CUDA graph contract: capture, mutate every dynamic
    input in place, replay, re-verify (FP8 and BF16 caches; for FP8 the
    default kernel choice and the query-rows kernel forced at capture)."""
    w = W.make_decode("graph", lengths=[1500, 900], tokens_per_request=[4, 2], Hq=16, Hkv=2, D=128, Di=128,
                      NB=16, P=40, K=4, seed=13, kv_dtype=kv)
    g = w.to(DEV)
    s = torch.empty((1, w.T, w.NB), device=DEV)
    tk = torch.empty((1, w.T, w.K), dtype=torch.int32, device=DEV)
    out = torch.empty((w.T, w.Hq, w.D), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(spd.decode_workspace_bytes(w.T, w.Hq, w.Hkv, w.D, w.NB), dtype=torch.uint8, device=DEV)

    def step():
        spd.msa_block_score(g.q_idx, g.k_idx_cache, g.block_table, g.seq_lens, g.req_idx, BS, s, g.idx_scale)
        spd.msa_select_topk(s, tk)
        spd.paged_sparse_decode_attention(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, g.req_idx,
                                          tk.expand(w.Hkv, -1, -1), out, g.sm_scale, BS, g.k_scale, g.v_scale, ws)

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with _policy(spd, policy):
        with torch.cuda.stream(stream):
            step()  # warm up outside capture
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
    for it in range(3):
        gen = torch.Generator().manual_seed(100 + it)
        w.q.copy_(torch.randn(w.q.shape, generator=gen).to(w.q.dtype))
        w.q_idx.copy_(torch.randn(w.q_idx.shape, generator=gen).to(w.q_idx.dtype))
        w.seq_lens.copy_(torch.clamp(w.seq_lens - 37 * (it + 1), min=0))
        g.q.copy_(w.q)
        g.q_idx.copy_(w.q_idx)
        g.seq_lens.copy_(w.seq_lens)
        s.fill_(float("nan"))
        tk.fill_(0x7FFFFFF0)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ref_s = orc.block_score(w.q_idx, w.k_idx_cache, w.block_table, w.req_idx, w.seq_lens, f32(w.idx_scale))
        check_scores(s.cpu().numpy(), ref_s, "replay %d scores" % it)
        check_topk(tk.cpu().numpy(), ref_s, w.K, "replay %d topk" % it)
        ref = orc.paged_attention(w.q, w.k_cache, w.v_cache, w.block_table, w.req_idx, w.seq_lens,
                                  tk.cpu().numpy(), f32(w.sm_scale), f32(w.k_scale), f32(w.v_scale))
        check_attention(out.float().cpu().numpy(), ref, "replay %d attention" % it)


def test_empty_batch(spd):
    q = torch.empty((0, 8, 64), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((128, 1, 64), dtype=torch.float8_e4m3fn, device=DEV)
    bt = torch.zeros((1, 1), dtype=torch.int32, device=DEV)
    z = torch.empty((0,), dtype=torch.int32, device=DEV)
    out = torch.empty((0, 8, 64), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(spd.decode_workspace_bytes(0, 8, 1, 64, 1), dtype=torch.uint8, device=DEV)
    spd.paged_decode_attention(q, k, k, bt, z, z, out, 0.1, BS, 1.0, 1.0, ws)
    torch.cuda.synchronize()


# ------------------------------------------------------ FP8 index cache

FP8_INDEX = {
    # bf16 queries of 128 dims: the tensor-core f8 product
    "di128": dict(lengths=[1500, 700, 300], tokens_per_request=[4, 2, 1], Di=128, NB=16, P=40, K=4),
    # 64 dims: the general-layout kernel
    "di64": dict(lengths=[900, 200], tokens_per_request=[3, 1], Di=64, NB=8, P=16, K=3),
    # two index heads (64 lanes of tokens per tile)
    "hi2": dict(lengths=[1300, 600], tokens_per_request=[5, 2], Di=128, Hi=2, NB=16, P=32, K=3),
}


@pytest.mark.parametrize("name", sorted(FP8_INDEX))
def test_fp8_index_cache(spd, orc, name, kernel_policy):
    """An FP8-E4M3 index cache (its static scale folded into idx_scale):
    the score sheet and top-k against the oracle on the same E4M3 codes."""
    w = W.with_fp8_index(W.make_decode("fp8idx_" + name, Hq=16, Hkv=2, D=128, seed=zlib.crc32(name.encode()) % 1000,
                                       with_kv=False, **FP8_INDEX[name]))
    g = w.to(DEV)
    s = gpu_scores(spd, g)
    ref = orc.block_score(w.q_idx, w.k_idx_cache, w.block_table, w.req_idx, w.seq_lens, f32(w.idx_scale))
    check_scores(s.cpu().numpy(), ref, name + " scores")
    check_topk(gpu_topk(spd, s, w.K).cpu().numpy(), ref, w.K, name + " topk")


def test_fp8_index_cache_strided_queries(spd, orc):
    """Queries viewed inside a wider buffer (16-byte aligned rows) still take
    the f8 product; the result matches the contiguous call."""
    w = W.with_fp8_index(W.make_decode("fp8idx_strided", lengths=[1100, 500], tokens_per_request=[3, 3], Hq=16,
                                       Hkv=2, D=128, Di=128, NB=16, P=24, K=4, seed=77, with_kv=False))
    g = w.to(DEV)
    wide = torch.zeros((w.T, 1, 2 * w.Di), dtype=g.q_idx.dtype, device=DEV)
    wide[:, :, 8:8 + w.Di] = g.q_idx
    view = wide[:, :, 8:8 + w.Di]
    T, NB = g.seq_lens.shape[0], g.block_table.shape[1]
    out = nan_like((1, T, NB), torch.float32, DEV)
    spd.msa_block_score(view, g.k_idx_cache, g.block_table, g.seq_lens, g.req_idx, BS, out, g.idx_scale)
    torch.cuda.synchronize()
    ref = orc.block_score(w.q_idx, w.k_idx_cache, w.block_table, w.req_idx, w.seq_lens, f32(w.idx_scale))
    check_scores(out.cpu().numpy(), ref, "strided fp8 index scores")


def test_fp8_index_cache_full_size(spd, orc):
    """The verification-decode and prefill index shapes with an FP8 index
    cache: the verification decode's whole sheet, sampled prefill rows."""
    w = W.with_fp8_index(W.config(2))
    g = w.to(DEV)
    s = gpu_scores(spd, g)
    ref = orc.block_score(w.q_idx, w.k_idx_cache, w.block_table, w.req_idx, w.seq_lens, f32(w.idx_scale))
    check_scores(s.cpu().numpy(), ref, "verification decode fp8 index scores")
    check_topk(gpu_topk(spd, s, w.K).cpu().numpy(), ref, w.K, "verification decode fp8 index topk")
    w = W.with_fp8_index(W.config(4))
    g = w.to(DEV)
    s = gpu_scores(spd, g)
    rows = [0, 1, 511, 512, 2047, w.T - 1]
    ridx = torch.tensor(rows)
    ref = orc.block_score(w.q_idx[ridx], w.k_idx_cache, w.block_table, w.req_idx[ridx], w.seq_lens[ridx],
                          f32(w.idx_scale))
    check_scores(s.cpu().numpy()[:, rows], ref, "prefill fp8 index scores")


# ------------------------------------------------------ dense BF16 K/V cache

BF16_KV = {
    # tensor-core path (bf16 queries, D = 128): GQA 8, multi-token rows (a
    # 16-token request fills the 128 MMA rows), ragged tails
    "g8_d128": dict(lengths=[1500, 700, 129, 2048, 1], tokens_per_request=[4, 4, 1, 16, 1], Hq=64, Hkv=8, D=128,
                    Di=128, NB=16, P=96, K=5),
    # tensor-core path: group 16 (8 tokens per unit), long rows split over
    # several units and merged, heavy-tailed queries
    "g16_d128_split": dict(lengths=[7000, 5000, 300], tokens_per_request=[8, 3, 1], Hq=32, Hkv=2, D=128, Di=128,
                           NB=64, P=128, K=40, q_dist="student_t3"),
    # tensor-core path: MHA (G = 1, 16 tokens per unit)
    "g1_d128": dict(lengths=[2000, 640], tokens_per_request=[5, 2], Hq=4, Hkv=4, D=128, Di=64, NB=16, P=32, K=6),
    # head dim 64, fp32 queries, group 4
    "g4_d64_f32q": dict(lengths=[300, 512, 77], tokens_per_request=[1, 2, 3], Hq=8, Hkv=2, D=64, Di=32, NB=4, P=16,
                        K=2, dtype=torch.float32),
    # group 16, f16 queries, heavy-tailed
    "g16_d128_f16q": dict(lengths=[900, 2600], tokens_per_request=[3, 2], Hq=32, Hkv=2, D=128, Di=64, NB=24, P=48,
                          K=7, dtype=torch.float16, q_dist="student_t3"),
}


@pytest.mark.parametrize("name", sorted(BF16_KV))
def test_bf16_kv_cache_small(spd, orc, name, kernel_policy):
    """Paged attention over a dense BF16 K/V cache (scale 1, unowned slots
    poisoned with +/-448): sparse with the oracle's selection, end to end and
    dense, every cell against the oracle's BF16 path."""
    w = W.make_decode("bf16kv_" + name, seed=zlib.crc32(name.encode()) % 1000, kv_dtype="bf16", **BF16_KV[name])
    assert w.k_cache.dtype == torch.bfloat16
    full_check(spd, orc, w)


def test_bf16_kv_cache_full_size(spd, orc):
    """The verification-decode and dense-decode shapes over BF16 caches:
    every row of each."""
    full_check(spd, orc, W.config(2, kv_dtype="bf16"))
    w = W.config(3, kv_dtype="bf16")
    out = gpu_attention(spd, w.to(DEV), None)
    ref = oracle_rows(orc, w, list(range(w.T)), None)
    check_attention(out.float().cpu().numpy(), ref, "dense decode, BF16 cache")


def test_bf16_kv_nan_slots_never_leak(spd, orc, kernel_policy):
    """A BF16 cache whose unowned slots (unused pages and the tails of the
    requests' last pages) hold NaN: no output cell may see them."""
    w = W.make_decode("bf16nan", lengths=[700, 333, 129], tokens_per_request=[4, 2, 3], Hq=16, Hkv=2, D=128,
                      Di=128, NB=8, P=24, K=3, seed=16, kv_dtype="bf16")
    owned = set()
    for r, L in enumerate(w.request_lengths):
        for tau in range(L):
            owned.add(int(w.block_table[r, tau // BS]) * BS + tau % BS)
    mask = torch.ones(w.P * BS, dtype=torch.bool)
    mask[torch.tensor(sorted(owned))] = False
    for c in (w.k_cache, w.v_cache):
        c[mask] = float("nan")
    w.k_idx_cache[mask] = float("nan")
    full_check(spd, orc, w)


def test_kv_cache_dtypes_must_match(spd):
    from sparse_paged_decode_gb300.binding import SpdError

    w = W.make_decode("kvmix", lengths=[300], tokens_per_request=[1], Hq=8, Hkv=1, D=64, Di=32, NB=4, P=8, K=2,
                      seed=3).to(DEV)
    out = torch.empty((w.T, w.Hq, w.D), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(spd.decode_workspace_bytes(w.T, w.Hq, w.Hkv, w.D, w.NB), dtype=torch.uint8, device=DEV)
    with pytest.raises(SpdError):
        spd.paged_decode_attention(w.q, w.k_cache.to(torch.bfloat16), w.v_cache, w.block_table, w.seq_lens,
                                   w.req_idx, out, w.sm_scale, BS, 1.0, 1.0, ws)


# ------------------------------------------------- capability-domain edges

def test_domain_edges_head_dim_256_index_dim_512_and_1024_blocks(spd, orc):
    """The largest shapes the calls declare: head dim 256, index dim 512, a
    page table of 1024 blocks with one request using all of them (131072
    tokens), a top-k wider than one selection kernel's register row (the
    rank kernel takes rows of more than 256 blocks).  Every cell of the score
    sheet, the top-k and the sparse, end-to-end and dense attention
    outputs."""
    w = W.make_decode("edges", lengths=[1024 * BS, 2000], tokens_per_request=[1, 3], Hq=4, Hkv=1, D=256, Di=512,
                      NB=1024, P=1056, K=40, seed=1024)
    assert w.NB == 1024 and w.D == 256 and w.Di == 512 and int(w.seq_lens.max()) == 1024 * BS
    full_check(spd, orc, w)


# --------------------------------------------------------- full-size configs

def test_verification_decode_full(spd, orc):
    full_check(spd, orc, W.config(2), policies=(None,) + FP8_KERNELS)


def test_dense_decode_full(spd, orc):
    """Dense decode at full size (16 rows of 16384 tokens): every row, through
    the default kernel choice and each of the two FP8-cache kernels."""
    w = W.config(3)
    g = w.to(DEV)
    rows = list(range(w.T))
    ref = oracle_rows(orc, w, rows, None)
    for pol in (None,) + FP8_KERNELS:
        with _policy(spd, pol):
            out = gpu_attention(spd, g, None)
        check_attention(out.float().cpu().numpy(), ref, "dense decode (policy %s)" % pol)


def test_prefill_score_select_full_sampled(spd, orc):
    w = W.config(4)
    g = w.to(DEV)
    s = gpu_scores(spd, g)
    tk = gpu_topk(spd, s, w.K)
    rng = np.random.default_rng(4)
    rows = sorted(set(rng.integers(0, w.T, 24).tolist()) | {0, 511, 512, w.T - 1})
    ridx = torch.tensor(rows)
    ref_s = orc.block_score(w.q_idx[ridx], w.k_idx_cache, w.block_table, w.req_idx[ridx], w.seq_lens[ridx],
                            f32(w.idx_scale))
    check_scores(s.cpu().numpy()[:, rows], ref_s, "prefill scores")
    check_topk(tk.cpu().numpy()[:, rows], ref_s, w.K, "prefill topk")
    # causal visibility: no token selects a block past its own position
    pos_block = ((g.seq_lens - 1) // BS).view(1, -1, 1)
    assert torch.all((tk < 0) | (tk <= pos_block))


def test_stress_decode_full(spd, orc):
    """The stress configuration at full size: every cell of the score sheet,
    the top-k and the sparse (oracle selection), end-to-end (GPU selection)
    and dense attention outputs of every query row -- all four bucket sizes,
    every group the planner forms, every pair it splits and merges, the
    padded rows (exact zeros) and the longest row; through the default
    kernel choice and each of the two FP8-cache tensor-core kernels."""
    w = W.config(5)
    assert set(w.tokens_per_request) == {1, 4, 8, 16}
    assert any(int(x) == 0 for x in w.seq_lens), "the configuration has padded rows"
    full_check(spd, orc, w, policies=(None,) + FP8_KERNELS)
