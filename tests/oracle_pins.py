"""Pins of the CPU oracle against things other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when
the oracle disagrees with what the pages and the mathematics fix:

  * the FP8-E4M3 / BF16 / F16 decoders against torch's and numpy's casts of
    every code;
  * the block-score sheet against a numpy brute force (gather the request's
    logical keys through the page table, one matrix product, mask, per-block
    max; bf16, fp32 and FP8-E4M3 index caches) and against a hand-worked
    fixture and a closed-form ramp;
  * top-k against numpy's lexicographic sort, ties and padding included;
  * attention against torch's fp64 ``scaled_dot_product_attention`` with GQA
    expansion on gathered, torch-dequantised keys and values (FP8-E4M3
    caches, and dense BF16 caches, which must also reproduce the E4M3 path
    bit for bit when they hold its decoded values), against a
    hand-worked fixture and closed forms (uniform logits -> mean of V, one key
    -> that key's value), and the invariants "selecting every block equals
    dense decode", "a one-block context is that block's softmax", "permuting
    pool pages changes nothing", "a selection is a set";
  * dense GQA attention against torch's fp64 ``scaled_dot_product_attention``
    (explicit bottom-right causal mask, and its own ``is_causal`` flag on a
    square case), a closed form (two keys give tanh(q/2)), uniform logits,
    one key, and the invariants "a causal row is non-causal attention over
    its prefix", "GQA equals MHA on repeated kv heads", "key order does not
    matter without the flag";
  * the fused prefill score-to-selection against a numpy brute force
    (gathered keys, one product per sequence, masked maxima, policy blocks,
    lexicographic sort; bad metadata included), its reduction to the decode
    score sheet and top-k when query blocks are single tokens, and the
    invariants "positive scale changes nothing", "page permutation changes
    nothing", "a wide enough selection takes every visible block, policy
    blocks first".

``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutants.py``
runs them on copies of the oracle with planted mistakes and checks that each
mistake is caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

from sparse_paged_decode_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
BS = W.BLOCK_SIZE


# ----------------------------------------------------------------- helpers

def tiny_decode(seed, *, lengths=(300, 130, 1, 511), tpr=(2, 1, 1, 3), Hq=4, Hkv=2, D=8, Di=8,
                NB=4, P=24, K=3, dtype=torch.float32, idx_dtype=None, pad=None, q_dist="normal"):
    return W.make_decode("tiny", lengths=list(lengths), tokens_per_request=list(tpr), Hq=Hq, Hkv=Hkv,
                         D=D, Hi=1, Di=Di, NB=NB, P=P, K=K, dtype=dtype, idx_dtype=idx_dtype,
                         seed=seed, padded_tail=pad, q_dist=q_dist)


def corrupt_metadata(w, seed=None):
    """Add the out-of-domain metadata cases the oracle defines: page ids
    outside the pool, request rows outside the table, seq_len past the
    table, negative seq_len."""
    bt = w.block_table.clone()
    bt[0, 1] = -1
    bt[min(1, w.R - 1), 0] = w.P + 3
    ri = w.req_idx.clone()
    sl = w.seq_lens.clone()
    if w.T >= 3:
        ri[w.T - 1] = w.R + 5
        sl[w.T - 2] = -7
    sl[0] = w.NB * BS + 100
    return bt, ri, sl


def e4m3_to_f64(codes: torch.Tensor) -> torch.Tensor:
    return codes.view(torch.float8_e4m3fn).to(torch.float32).to(torch.float64)


def cache_to_f64(cache: torch.Tensor) -> torch.Tensor:
    """A K or V cache's values: torch's own decoding of E4M3 codes, or of bf16."""
    return cache.to(torch.float64) if cache.dtype == torch.bfloat16 else e4m3_to_f64(cache)


def np_valid_slots(bt, r, L, NB, P, blocks=None):
    """Logical tokens 0..L-1 of request r (optionally only in ``blocks``),
    ascending, as (tau, slot) pairs; tokens whose page is outside the pool are
    dropped.  Written independently of the oracle."""
    R = bt.shape[0]
    if r < 0 or r >= R or L <= 0:
        return []
    L = min(L, NB * BS)
    out = []
    for tau in range(L):
        b = tau // BS
        if blocks is not None and b not in blocks:
            continue
        page = int(bt[r, b])
        if 0 <= page < P:
            out.append((tau, page * BS + tau % BS))
    return out


def np_block_score(q_idx, k_idx, bt, ri, sl, idx_scale, NB, P):
    q = q_idx.to(torch.float64).numpy()
    k = k_idx.to(torch.float64).numpy()[:, 0, :]
    T, Hi, _ = q.shape
    out = np.full((Hi, T, NB), -np.inf)
    for t in range(T):
        pairs = np_valid_slots(bt, int(ri[t]), int(sl[t]), NB, P)
        if not pairs:
            continue
        taus = np.array([p[0] for p in pairs])
        slots = np.array([p[1] for p in pairs])
        dots = (k[slots] @ q[t].T) * idx_scale  # [n, Hi]
        blocks = taus // BS
        for b in np.unique(blocks):
            out[:, t, b] = dots[blocks == b].max(axis=0)
    return out


def sdpa_reference(w, topk, bt=None, ri=None, sl=None):
    """torch fp64 SDPA per query token over its selected valid keys."""
    bt = w.block_table if bt is None else bt
    ri = w.req_idx if ri is None else ri
    sl = w.seq_lens if sl is None else sl
    G = w.Hq // w.Hkv
    kf = cache_to_f64(w.k_cache) * w.k_scale
    vf = cache_to_f64(w.v_cache) * w.v_scale
    q = w.q.to(torch.float64)
    out = torch.zeros((w.T, w.Hq, w.D), dtype=torch.float64)
    for t in range(w.T):
        for h in range(w.Hkv):
            if topk is None:
                blocks = None
            else:
                blocks = {int(b) for b in topk[min(h, topk.shape[0] - 1), t] if 0 <= int(b) < w.NB}
            pairs = np_valid_slots(bt, int(ri[t]), int(sl[t]), w.NB, w.P, blocks)
            if not pairs:
                continue
            slots = torch.tensor([p[1] for p in pairs])
            kk = kf[slots, h, :][None, None]  # [1,1,n,D]
            vv = vf[slots, h, :][None, None]
            qq = q[t, h * G:(h + 1) * G, :][None, :, None, :]  # [1,G,1,D]
            o = torch.nn.functional.scaled_dot_product_attention(
                qq, kk.expand(1, G, -1, -1), vv.expand(1, G, -1, -1), scale=w.sm_scale)
            out[t, h * G:(h + 1) * G, :] = o[0, :, 0, :]
    return out.numpy()


def assert_close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    ninf_a, ninf_b = np.isneginf(a), np.isneginf(b)
    assert np.array_equal(ninf_a, ninf_b), "%s: -inf pattern differs" % what
    fa, fb = a[~ninf_a], b[~ninf_b]
    assert np.all(np.isfinite(fa)) and np.all(np.isfinite(fb)), "%s: non-finite values" % what
    err = np.abs(fa - fb)
    assert np.all(err <= atol + rtol * np.abs(fb)), "%s: max err %g" % (what, err.max() if err.size else 0)


# ------------------------------------------------------------ the decoders

def pin_e4m3_decoder(o):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = np.array([o.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "E4M3 NaN codes"
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m]), "E4M3 values"
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def pin_bf16_decoder(o):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([o.bf16_value(b) for b in range(0, 65536)])
    m = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "BF16 NaN codes"
    assert np.array_equal(got[m], ref[m]), "BF16 values"


def pin_f16_decoder(o):
    ref = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([o.f16_value(b) for b in range(0, 65536)])
    m = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "F16 NaN codes"
    assert np.array_equal(got[m], ref[m]), "F16 values"


# ------------------------------------------------------------ block score

def pin_block_score_bruteforce(o):
    for seed, dt in ((11, torch.float32), (12, torch.bfloat16)):
        w = tiny_decode(seed, idx_dtype=dt)
        bt, ri, sl = corrupt_metadata(w, seed)
        got = o.block_score(w.q_idx, w.k_idx_cache, bt, ri, sl, w.idx_scale)
        ref = np_block_score(w.q_idx, w.k_idx_cache, bt, ri, sl, w.idx_scale, w.NB, w.P)
        assert_close(got, ref, what="block score seed %d" % seed)
    # an FP8-E4M3 index cache: the oracle decodes the codes itself; the brute
    # force takes torch's decoding of the same codes
    w = W.with_fp8_index(tiny_decode(14, idx_dtype=torch.bfloat16))
    got = o.block_score(w.q_idx, w.k_idx_cache, w.block_table, w.req_idx, w.seq_lens, w.idx_scale)
    ref = np_block_score(w.q_idx, e4m3_to_f64(w.k_idx_cache.view(torch.uint8)), w.block_table, w.req_idx,
                         w.seq_lens, w.idx_scale, w.NB, w.P)
    assert_close(got, ref, what="block score, E4M3 index cache")
    # two query index heads sharing the single index key head
    w = tiny_decode(13)
    q2 = torch.randn((w.T, 2, w.Di), generator=torch.Generator().manual_seed(5))
    got = o.block_score(q2, w.k_idx_cache, w.block_table, w.req_idx, w.seq_lens, 0.3)
    ref = np_block_score(q2, w.k_idx_cache, w.block_table, w.req_idx, w.seq_lens, 0.3, w.NB, w.P)
    assert_close(got, ref, what="block score Hi=2")


def pin_block_score_golden(o):
    with open(os.path.join(GOLDEN, "block_score_ramp.json")) as f:
        fx = json.load(f)
    P, NB = fx["pool_pages"], len(fx["block_table"][0])
    bt = torch.tensor(fx["block_table"], dtype=torch.int32)
    kidx = torch.full((P * BS, 1, 2), 64.0)
    for r, sign in ((0, 1.0), (1, -1.0)):
        n_tok = 300 if r == 0 else 256
        for tau in range(n_tok):
            page = int(bt[r, tau // BS])
            kidx[page * BS + tau % BS, 0, 0] = sign * tau
            kidx[page * BS + tau % BS, 0, 1] = 0.0
    q = torch.tensor([[[1.0, 0.0]]] * 3)
    got = o.block_score(q, kidx, bt, torch.tensor(fx["req_idx"], dtype=torch.int32),
                        torch.tensor(fx["seq_lens"], dtype=torch.int32), fx["idx_scale"])
    exp = np.array([[float(v) for v in row] for row in fx["expected"]])[None]
    assert got.shape == exp.shape
    assert np.array_equal(got, exp), (got, exp)


def pin_block_score_closed_form(o):
    """q_idx = e0 and key tau = [tau, ...]: every block scores the position of
    its last valid token times idx_scale."""
    w = tiny_decode(21, lengths=(333, 129, 512), tpr=(2, 1, 1), NB=4, P=16)
    kidx = torch.full_like(w.k_idx_cache, 64.0)
    for r, L in enumerate(w.request_lengths):
        for tau in range(L):
            page = int(w.block_table[r, tau // BS])
            kidx[page * BS + tau % BS, 0, :] = 0.0
            kidx[page * BS + tau % BS, 0, 0] = float(tau)
    q = torch.zeros_like(w.q_idx)
    q[:, 0, 0] = 1.0
    got = o.block_score(q, kidx, w.block_table, w.req_idx, w.seq_lens, 0.25)
    for t in range(w.T):
        L = int(w.seq_lens[t])
        for b in range(w.NB):
            exp = -math.inf if b * BS >= L else (min(BS * (b + 1), L) - 1) * 0.25
            assert got[0, t, b] == exp, (t, b, got[0, t, b], exp)


# ------------------------------------------------------------------ top-k

def np_topk(scores, K):
    s = np.asarray(scores, dtype=np.float64)
    lead, NB = s.shape[:-1], s.shape[-1]
    flat = s.reshape(-1, NB)
    out = np.full((flat.shape[0], K), -1, dtype=np.int32)
    for i, row in enumerate(flat):
        cand = [b for b in range(NB) if not (np.isnan(row[b]) or row[b] == -np.inf)]
        order = np.lexsort((np.array(cand), -row[cand])) if cand else []
        picked = [cand[j] for j in order][:K]
        out[i, :len(picked)] = picked
    return out.reshape(lead + (K,))


def pin_topk_sort(o):
    g = np.random.default_rng(3)
    s = g.standard_normal((3, 17, 40))
    s[0, :, 5:9] = 0.5  # ties
    s[1, 3, :] = -np.inf  # no candidate
    s[1, 4, ::3] = np.nan
    s[2, :, 20:] = -np.inf  # short rows
    s[2, 5, 7] = np.inf
    for K in (1, 4, 16, 40, 45):
        assert np.array_equal(o.select_topk(s, K), np_topk(s, K)), "top-%d" % K


def pin_topk_closed_form(o):
    NB = 128
    desc = -np.arange(NB, dtype=np.float64)[None, :]  # score decreasing in block id
    assert np.array_equal(o.select_topk(desc, 5)[0], np.arange(5))
    flat = np.zeros((1, NB))  # all tied -> lowest ids
    assert np.array_equal(o.select_topk(flat, 7)[0], np.arange(7))
    none = np.full((1, NB), -np.inf)
    assert np.array_equal(o.select_topk(none, 4)[0], -np.ones(4))
    inc = np.arange(NB, dtype=np.float64)[None, :]
    assert np.array_equal(o.select_topk(inc, 3)[0], [127, 126, 125])
    # positive rescaling of the sheet does not change the selection
    g = np.random.default_rng(9)
    s = g.standard_normal((50, NB))
    assert np.array_equal(o.select_topk(s, 16), o.select_topk(s * 0.37, 16))


# -------------------------------------------------------------- attention

def pin_attention_vs_sdpa(o):
    for seed, dt, qd in ((31, torch.float32, "normal"), (32, torch.bfloat16, "student_t3")):
        w = tiny_decode(seed, dtype=dt, q_dist=qd)
        bt, ri, sl = corrupt_metadata(w, seed)
        s = o.block_score(w.q_idx, w.k_idx_cache, bt, ri, sl, w.idx_scale)
        topk = o.select_topk(s, w.K)
        topk_h = np.concatenate([topk, np.roll(topk, 1, axis=2)], axis=0)  # distinct per kv head
        got = o.paged_attention(w.q, w.k_cache, w.v_cache, bt, ri, sl, topk_h,
                                w.sm_scale, w.k_scale, w.v_scale)
        ref = sdpa_reference(w, topk_h, bt, ri, sl)
        assert_close(got, ref, rtol=1e-11, atol=1e-12, what="sparse vs sdpa seed %d" % seed)
        got_d = o.paged_attention(w.q, w.k_cache, w.v_cache, bt, ri, sl, None,
                                  w.sm_scale, w.k_scale, w.v_scale)
        ref_d = sdpa_reference(w, None, bt, ri, sl)
        assert_close(got_d, ref_d, rtol=1e-11, atol=1e-12, what="dense vs sdpa seed %d" % seed)


def bf16_cache_copy(w, seed):
    """The workload with dense BF16 K/V caches of fresh N(0, 1) values (not
    quantised), unit scales and the same finite poison in unowned slots."""
    g = torch.Generator().manual_seed(seed)
    out = W.Workload(**{f: getattr(w, f) for f in w.__dataclass_fields__})
    owned = torch.zeros(w.k_cache.shape[0], dtype=torch.bool)  # slots of the requests' tokens
    for r, L in enumerate(w.request_lengths):
        for tau in range(L):
            owned[int(w.block_table[r, tau // BS]) * BS + tau % BS] = True
    for name in ("k_cache", "v_cache"):
        fresh = torch.randn(w.k_cache.shape, generator=g, dtype=torch.float64)
        setattr(out, name, torch.where(owned[:, None, None], fresh, torch.full_like(fresh, 448.0)).to(torch.bfloat16))
    out.k_scale = out.v_scale = 1.0
    return out


def pin_attention_bf16_cache(o):
    w = tiny_decode(61, dtype=torch.bfloat16)
    topk = o.select_topk(o.block_score(w.q_idx, w.k_idx_cache, w.block_table, w.req_idx, w.seq_lens,
                                       w.idx_scale), w.K)
    # BF16 caches holding the E4M3-decoded values give the E4M3 path's result bit for bit
    same = W.Workload(**{f: getattr(w, f) for f in w.__dataclass_fields__})
    same.k_cache = e4m3_to_f64(w.k_cache).to(torch.bfloat16)
    same.v_cache = e4m3_to_f64(w.v_cache).to(torch.bfloat16)
    for sel in (topk, None):
        a = o.paged_attention(w.q, w.k_cache, w.v_cache, w.block_table, w.req_idx, w.seq_lens, sel,
                              w.sm_scale, w.k_scale, w.v_scale)
        b = o.paged_attention(same.q, same.k_cache, same.v_cache, w.block_table, w.req_idx, w.seq_lens, sel,
                              w.sm_scale, w.k_scale, w.v_scale)
        assert np.array_equal(a, b), "bf16 copy of the E4M3 cache differs"
    # fresh BF16 values against torch's fp64 SDPA over the same selections
    wb = bf16_cache_copy(w, 62)
    for sel in (topk, None):
        got = o.paged_attention(wb.q, wb.k_cache, wb.v_cache, wb.block_table, wb.req_idx, wb.seq_lens, sel,
                                wb.sm_scale, 1.0, 1.0)
        assert_close(got, sdpa_reference(wb, sel), rtol=1e-11, atol=1e-12, what="bf16 cache vs sdpa")


def pin_attention_golden(o):
    with open(os.path.join(GOLDEN, "attention_two_tokens.json")) as f:
        fx = json.load(f)
    P, page, D = fx["pool_pages"], fx["page"], 4
    k = torch.full((P * BS, 1, D), 448.0)
    v = torch.full((P * BS, 1, D), 448.0)
    for i in range(2):
        k[page * BS + i, 0] = torch.tensor(fx["k_tokens"][i])
        v[page * BS + i, 0] = torch.tensor(fx["v_tokens"][i])
    k8, v8 = k.to(torch.float8_e4m3fn), v.to(torch.float8_e4m3fn)
    q = torch.tensor(fx["q"]).view(1, 1, D)
    bt = torch.tensor([[page]], dtype=torch.int32)
    ri = torch.tensor([0], dtype=torch.int32)
    sl = torch.tensor([fx["seq_len"]], dtype=torch.int32)
    kscale = math.log(3.0)
    exp = np.array(fx["expected"])
    dense = o.paged_attention(q, k8, v8, bt, ri, sl, None, fx["sm_scale"], kscale, fx["v_scale"])
    assert np.allclose(dense[0, 0], exp, rtol=1e-14, atol=1e-14), dense
    sparse = o.paged_attention(q, k8, v8, bt, ri, sl, np.array([[[-1, 0]]], dtype=np.int32),
                               fx["sm_scale"], kscale, fx["v_scale"])
    assert np.array_equal(sparse, dense)
    empty = o.paged_attention(q, k8, v8, bt, ri, sl, np.array([[[-1, -1]]], dtype=np.int32),
                              fx["sm_scale"], kscale, fx["v_scale"])
    assert np.array_equal(empty, np.zeros_like(empty))


def pin_attention_closed_forms(o):
    w = tiny_decode(41)
    # uniform logits (q = 0): every head returns the mean of its valid values
    qz = torch.zeros_like(w.q)
    got = o.paged_attention(qz, w.k_cache, w.v_cache, w.block_table, w.req_idx, w.seq_lens, None,
                            w.sm_scale, w.k_scale, w.v_scale)
    vf = e4m3_to_f64(w.v_cache).numpy() * w.v_scale
    G = w.Hq // w.Hkv
    for t in range(w.T):
        pairs = np_valid_slots(w.block_table, int(w.req_idx[t]), int(w.seq_lens[t]), w.NB, w.P)
        slots = [p[1] for p in pairs]
        for g in range(w.Hq):
            exp = vf[slots, g // G, :].mean(axis=0)
            assert np.allclose(got[t, g], exp, rtol=1e-12, atol=1e-13), (t, g)
    # one valid key: the output is that key's value, exactly
    sl1 = torch.ones_like(w.seq_lens)
    got1 = o.paged_attention(w.q, w.k_cache, w.v_cache, w.block_table, w.req_idx, sl1, None,
                             w.sm_scale, w.k_scale, w.v_scale)
    for t in range(w.T):
        slot = int(w.block_table[int(w.req_idx[t]), 0]) * BS
        for g in range(w.Hq):
            assert np.array_equal(got1[t, g], vf[slot, g // G, :]), (t, g)
    # padding token: zeros
    sl0 = w.seq_lens.clone()
    sl0[:] = 0
    got0 = o.paged_attention(w.q, w.k_cache, w.v_cache, w.block_table, w.req_idx, sl0, None,
                             w.sm_scale, w.k_scale, w.v_scale)
    assert not np.any(got0)


def pin_attention_invariants(o):
    w = tiny_decode(51, lengths=(400, 257, 90), tpr=(3, 2, 1), K=4)
    args = (w.block_table, w.req_idx, w.seq_lens)
    dense = o.paged_attention(w.q, w.k_cache, w.v_cache, *args, None, w.sm_scale, w.k_scale, w.v_scale)
    # selecting every block (any order, with repeats and -1) equals dense, bit for bit
    allb = np.tile(np.array([3, -1, 0, 2, 1, 2, -5, 9], dtype=np.int32), (1, w.T, 1))
    sparse = o.paged_attention(w.q, w.k_cache, w.v_cache, *args, allb, w.sm_scale, w.k_scale, w.v_scale)
    assert np.array_equal(sparse, dense), "select-all != dense"
    # a selection is a set: repeats and out-of-range ids change nothing
    sel = np.tile(np.array([2, 0], dtype=np.int32), (1, w.T, 1))
    sel_rep = np.tile(np.array([2, 0, 0, -1, 2, 17], dtype=np.int32), (1, w.T, 1))
    a = o.paged_attention(w.q, w.k_cache, w.v_cache, *args, sel, w.sm_scale, w.k_scale, w.v_scale)
    b = o.paged_attention(w.q, w.k_cache, w.v_cache, *args, sel_rep, w.sm_scale, w.k_scale, w.v_scale)
    assert np.array_equal(a, b), "repeated ids changed the result"
    # permuting pool pages (and the table with them) changes nothing
    perm = torch.randperm(w.P, generator=torch.Generator().manual_seed(8))
    inv_slots = (perm.to(torch.int64)[:, None] * BS + torch.arange(BS)[None]).reshape(-1)
    k2 = torch.empty_like(w.k_cache.view(torch.uint8))
    v2 = torch.empty_like(w.v_cache.view(torch.uint8))
    k2[inv_slots] = w.k_cache.view(torch.uint8)
    v2[inv_slots] = w.v_cache.view(torch.uint8)
    bt2 = perm[w.block_table.to(torch.int64)].to(torch.int32)
    c = o.paged_attention(w.q, k2, v2, bt2, w.req_idx, w.seq_lens, sel, w.sm_scale, w.k_scale, w.v_scale)
    assert np.array_equal(a, c), "page permutation changed the result"
    # one-block context: selecting block 1 alone equals dense decode of a
    # request whose whole context is that block's valid tokens
    one = np.tile(np.array([1], dtype=np.int32), (1, w.T, 1))
    r1 = o.paged_attention(w.q, w.k_cache, w.v_cache, *args, one, w.sm_scale, w.k_scale, w.v_scale)
    bt1 = w.block_table[:, 1:2].contiguous()
    sl1 = (w.seq_lens - BS).clamp(min=0, max=BS)
    r2 = o.paged_attention(w.q, w.k_cache, w.v_cache, bt1, w.req_idx, sl1, None,
                           w.sm_scale, w.k_scale, w.v_scale)
    assert np.array_equal(r1, r2), "one-block context != that block's softmax"
    # linearity in v_scale
    d2 = o.paged_attention(w.q, w.k_cache, w.v_cache, *args, None, w.sm_scale, w.k_scale, 2 * w.v_scale)
    assert np.allclose(d2, 2 * dense, rtol=1e-14, atol=0)


# ---------------------------------------------------------- dense attention

def np_causal_mask(T, S):
    """[T, S] booleans: query t reads key j iff j <= t + S - T (the query
    tokens are the last T positions of the key sequence)."""
    t = np.arange(T)[:, None]
    j = np.arange(S)[None, :]
    return j <= t + (S - T)


def torch_sdpa_f64(q, k, v, sm_scale, causal):
    """torch's fp64 ``scaled_dot_product_attention`` with the kv heads
    repeated for GQA and the causal mask given explicitly; rows with no
    readable key (which torch leaves NaN) are set to zero."""
    qf, kf, vf = (x.to(torch.float64) for x in (q, k, v))
    T, Hq, D = qf.shape
    S, Hkv, _ = kf.shape
    G = Hq // Hkv
    qh = qf.permute(1, 0, 2)
    kh = kf.repeat_interleave(G, dim=1).permute(1, 0, 2)
    vh = vf.repeat_interleave(G, dim=1).permute(1, 0, 2)
    mask = torch.from_numpy(np_causal_mask(T, S)) if causal else torch.ones((T, S), dtype=torch.bool)
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask, scale=sm_scale)
    out = out.permute(1, 0, 2).numpy().copy()
    empty = ~mask.numpy().any(axis=1)
    out[empty] = 0.0
    return out


def pin_sdpa_vs_torch(o):
    cases = [  # T, S, Hq, Hkv, D, causal, dtype
        (5, 9, 4, 2, 8, True, torch.float32),
        (5, 9, 4, 2, 8, False, torch.bfloat16),
        (7, 7, 6, 3, 5, True, torch.float16),
        (9, 4, 4, 1, 16, True, torch.bfloat16),  # T > S: the first rows read nothing
        (1, 13, 8, 8, 4, True, torch.float32),
        (3, 0, 2, 1, 4, False, torch.float32),  # no keys at all
    ]
    for i, (T, S, Hq, Hkv, D, causal, dt) in enumerate(cases):
        w = W.make_dense("pin", T=T, S=S, Hq=Hq, Hkv=Hkv, D=D, causal=causal, seed=60 + i, dtype=dt,
                         q_dist="student_t3" if i % 2 else "normal")
        got = o.sdpa(w.q, w.k, w.v, w.sm_scale, causal)
        ref = torch_sdpa_f64(w.q, w.k, w.v, w.sm_scale, causal)
        assert_close(got, ref, rtol=1e-11, atol=1e-12, what="sdpa case %d" % i)
    # square causal case against torch's own causal flag (no explicit mask)
    w = W.make_dense("pin", T=6, S=6, Hq=4, Hkv=2, D=8, causal=True, seed=70, dtype=torch.float32)
    qf, kf, vf = (x.to(torch.float64) for x in (w.q, w.k, w.v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        qf.permute(1, 0, 2), kf.repeat_interleave(2, dim=1).permute(1, 0, 2),
        vf.repeat_interleave(2, dim=1).permute(1, 0, 2), is_causal=True, scale=w.sm_scale)
    got = o.sdpa(w.q, w.k, w.v, w.sm_scale, True)
    assert_close(got, ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12, what="sdpa is_causal")


def pin_sdpa_closed_forms(o):
    # two keys, one dim: weights e^{q} and 1, values +1 and -1, so the row
    # that reads both keys is tanh(q / 2); the causal first row reads key 0
    qv = float(np.float32(math.log(3.0)))
    q = torch.tensor([[[qv]], [[qv]]], dtype=torch.float32)
    k = torch.tensor([[[1.0]], [[0.0]]], dtype=torch.float32)
    v = torch.tensor([[[1.0]], [[-1.0]]], dtype=torch.float32)
    full = o.sdpa(q, k, v, 1.0, False)
    assert np.allclose(full[:, 0, 0], math.tanh(qv / 2), rtol=1e-14, atol=1e-15), full
    causal = o.sdpa(q, k, v, 1.0, True)
    assert causal[0, 0, 0] == 1.0 and abs(causal[1, 0, 0] - math.tanh(qv / 2)) < 1e-15, causal
    # q = 0: every row is the mean of the values it may read
    w = W.make_dense("pin", T=5, S=8, Hq=4, Hkv=2, D=6, causal=True, seed=71, dtype=torch.float32)
    got = o.sdpa(torch.zeros_like(w.q), w.k, w.v, w.sm_scale, True)
    vf = w.v.to(torch.float64).numpy()
    for t in range(5):
        n = t + 8 - 5 + 1
        for g in range(4):
            assert np.allclose(got[t, g], vf[:n, g // 2].mean(axis=0), rtol=1e-13, atol=1e-14), (t, g)
    # one key: the output is that key's value, exactly
    got1 = o.sdpa(w.q, w.k[:1], w.v[:1], w.sm_scale, False)
    for g in range(4):
        assert np.array_equal(got1[:, g], np.broadcast_to(vf[0, g // 2], (5, 6))), g


def pin_sdpa_invariants(o):
    w = W.make_dense("pin", T=4, S=11, Hq=6, Hkv=2, D=7, causal=True, seed=72, dtype=torch.bfloat16)
    causal = o.sdpa(w.q, w.k, w.v, w.sm_scale, True)
    full = o.sdpa(w.q, w.k, w.v, w.sm_scale, False)
    # causal row t equals non-causal attention over the keys it may read
    for t in range(4):
        n = t + 11 - 4 + 1
        pre = o.sdpa(w.q[t:t + 1], w.k[:n], w.v[:n], w.sm_scale, False)
        assert np.array_equal(causal[t], pre[0]), t
    # the last row reads every key under either flag
    assert np.array_equal(causal[3], full[3])
    # GQA equals multi-head attention on kv heads repeated explicitly
    mha = o.sdpa(w.q, w.k.repeat_interleave(3, dim=1), w.v.repeat_interleave(3, dim=1), w.sm_scale, True)
    assert np.array_equal(mha, causal)
    # without the flag, permuting the keys (values with them) changes only rounding
    perm = torch.randperm(11, generator=torch.Generator().manual_seed(5))
    fp = o.sdpa(w.q, w.k[perm], w.v[perm], w.sm_scale, False)
    assert_close(fp, full, rtol=1e-12, atol=1e-13, what="key permutation")
    # scaling V scales the output
    f2 = o.sdpa(w.q, w.k, (w.v.float() * 2).to(w.v.dtype), w.sm_scale, False)
    assert np.allclose(f2, 2 * full, rtol=1e-14, atol=0)


# ----------------------------------------- prefill score-to-selection (V2)

def np_prefill(pb, bt=None, slot_ids=None, seq_lens=None, n_rows=None, topk=None):
    """Brute force of the fused prefill call with numpy, written from the
    rule without the oracle's loops: gather each sequence's keys through its
    page-table row, one matrix product per sequence, mask, reduce each
    (query block, key block) cell with a max, then the policy blocks and a
    lexicographic sort.  Returns (ids [Hi, n_rows, topk], scores)."""
    bt = (pb.block_table if bt is None else bt).numpy()
    sid = (pb.slot_ids if slot_ids is None else slot_ids).numpy()
    sl = (pb.seq_lens if seq_lens is None else seq_lens).numpy()
    cu, cub, pre = pb.cu_seqlens.numpy(), pb.cu_seqblocks_q.numpy(), pb.prefix_lens.numpy()
    n_rows = pb.n_rows if n_rows is None else n_rows
    topk = pb.topk if topk is None else topk
    q = pb.q_idx.to(torch.float64).numpy()
    k = pb.k_idx_cache.to(torch.float64).numpy()[:, 0, :]
    R, NB = bt.shape
    Hi = q.shape[1]
    ids = np.full((Hi, n_rows, topk), -1, dtype=np.int32)
    sc = np.full((Hi, n_rows, NB), -np.inf)
    for b in range(pb.B):
        r = int(sid[b])
        for qb in range(int(cub[b + 1] - cub[b])):
            row = int(cub[b]) + qb
            if not 0 <= row < n_rows:
                continue
            L = min(int(pre[b]) + qb * pb.block_size_q + 1, int(sl[b]), NB * BS)
            if not 0 <= r < R:
                L = 0
            L = max(L, 0)
            nvis = -(-L // BS)
            toks = list(range(int(cu[b]) + qb * pb.block_size_q,
                              min(int(cu[b]) + (qb + 1) * pb.block_size_q, int(cu[b + 1]))))
            taus = np.arange(L)
            pages = bt[r, taus // BS] if L else np.zeros(0, dtype=np.int64)
            ok = (pages >= 0) & (pages < pb.P)
            slots = pages.astype(np.int64) * BS + taus % BS
            for h in range(Hi):
                z = q[toks, h, :] @ k[np.where(ok, slots, 0)].T * pb.scale if toks else np.zeros((0, L))
                z = np.where(ok[None, :], z, -np.inf)
                for kb in range(nvis):
                    cell = z[:, kb * BS:min((kb + 1) * BS, L)]
                    sc[h, row, kb] = cell.max() if cell.size else -np.inf
                forced = [kb for kb in range(nvis) if kb < pb.init_blocks or kb >= nvis - pb.local_blocks]
                rest = np.array([kb for kb in range(nvis) if kb not in forced and np.isfinite(sc[h, row, kb])],
                                dtype=np.int64)
                rest = rest[np.lexsort((rest, -sc[h, row, rest]))] if len(rest) else rest
                sel = (forced + rest.tolist())[:topk]
                ids[h, row, :len(sel)] = sel
    return ids, sc


def tiny_prefill(seed, **kw):
    args = dict(offsets=[130, 0, 250], chunks=[5, 1, 9], block_size_q=4, topk=3, init_blocks=1, local_blocks=1,
                Hi=2, Di=8, NB=4, P=24, seed=seed, idx_dtype=torch.float32)
    args.update(kw)
    return W.make_prefill_batch("tiny", **args)


def run_prefill(o, pb, bt=None, slot_ids=None, seq_lens=None, n_rows=None, topk=None, scale=None):
    return o.prefill_topk(pb.q_idx, pb.k_idx_cache, pb.block_table if bt is None else bt,
                          pb.slot_ids if slot_ids is None else slot_ids, pb.cu_seqlens,
                          pb.seq_lens if seq_lens is None else seq_lens, pb.prefix_lens, pb.cu_seqblocks_q,
                          pb.block_size_q, pb.init_blocks, pb.local_blocks, pb.scale if scale is None else scale,
                          pb.n_rows if n_rows is None else n_rows, pb.topk if topk is None else topk)


def pin_prefill_bruteforce(o):
    cases = [dict(), dict(block_size_q=1, init_blocks=0, local_blocks=0),
             dict(topk=6), dict(topk=1, init_blocks=2, local_blocks=2),
             dict(block_size_q=3, idx_dtype=torch.bfloat16, Hi=1, local_blocks=0),
             dict(offsets=[0, 0, 380], chunks=[130, 7, 4], block_size_q=32, init_blocks=0, local_blocks=2)]
    for i, kw in enumerate(cases):
        pb = tiny_prefill(90 + i, **kw)
        got, gs = run_prefill(o, pb)
        ref, rs = np_prefill(pb)
        assert np.array_equal(got, ref), "prefill ids, case %d" % i
        assert_close(gs, rs, rtol=1e-12, atol=1e-12, what="prefill scores, case %d" % i)
    # out-of-domain metadata: a sequence outside the table, a page outside
    # the pool, seq_lens short of the chunk, rows that no sequence owns
    pb = tiny_prefill(97)
    bt = pb.block_table.clone()
    bt[int(pb.slot_ids[2]), 1] = pb.P + 5
    sid = pb.slot_ids.clone()
    sid[1] = bt.shape[0] + 3
    sl = pb.seq_lens.clone()
    sl[0] = int(pb.prefix_lens[0]) + 2
    got, gs = run_prefill(o, pb, bt=bt, slot_ids=sid, seq_lens=sl, n_rows=pb.n_rows + 2)
    ref, rs = np_prefill(pb, bt=bt, slot_ids=sid, seq_lens=sl, n_rows=pb.n_rows + 2)
    assert np.array_equal(got, ref), "prefill ids, bad metadata"
    assert np.all(got[:, pb.n_rows:] == -1)
    assert_close(gs, rs, rtol=1e-12, atol=1e-12, what="prefill scores, bad metadata")


def pin_prefill_golden(o):
    with open(os.path.join(GOLDEN, "prefill_policy.json")) as f:
        fx = json.load(f)
    P, pages = fx["pool_pages"], fx["pages"]
    NB = len(pages)
    k = torch.full((P * BS, 1, 1), 64.0)
    L = fx["prefix"] + fx["chunk"]
    for tau in range(L):
        k[pages[tau // BS] * BS + tau % BS, 0, 0] = fx["block_values"][tau // BS]
    for tau, val in fx["spikes"]:
        k[pages[tau // BS] * BS + tau % BS, 0, 0] = val
    q = torch.ones((fx["chunk"], 1, 1))
    q[fx["negated_token"], 0, 0] = -1.0
    bt = torch.tensor([[2] * NB, pages], dtype=torch.int32)
    n_q = -(-fx["chunk"] // fx["block_size_q"])
    i32 = lambda v: torch.tensor(v, dtype=torch.int32)  # noqa: E731
    for K, key in ((4, "expected_top4"), (6, "expected_top6")):
        ids, _ = o.prefill_topk(q, k, bt, i32([1]), i32([0, fx["chunk"]]), i32([L]), i32([fx["prefix"]]),
                                i32([0, n_q]), fx["block_size_q"], fx["init_blocks"], fx["local_blocks"],
                                fx["scale"], n_q, K)
        assert ids[0].tolist() == fx[key], (K, ids[0].tolist())


def pin_prefill_reduces_to_decode(o):
    """Query blocks of one token and no policy blocks: each row is the decode
    top-k of its token with seq_len = position + 1 (the pinned score sheet
    and selection)."""
    pb = tiny_prefill(98, block_size_q=1, init_blocks=0, local_blocks=0, topk=3)
    got, _ = run_prefill(o, pb)
    cu = pb.cu_seqlens.tolist()
    ri, sl = [], []
    for b in range(pb.B):
        for j in range(cu[b + 1] - cu[b]):
            ri.append(int(pb.slot_ids[b]))
            sl.append(int(pb.prefix_lens[b]) + j + 1)
    s = o.block_score(pb.q_idx, pb.k_idx_cache, pb.block_table, torch.tensor(ri, dtype=torch.int32),
                      torch.tensor(sl, dtype=torch.int32), pb.scale)
    assert np.array_equal(got, o.select_topk(s, pb.topk))


def pin_prefill_invariants(o):
    pb = tiny_prefill(99, topk=4, init_blocks=1, local_blocks=1)
    base, _ = run_prefill(o, pb)
    # selection does not depend on the (positive) scale
    assert np.array_equal(run_prefill(o, pb, scale=3.5 * pb.scale)[0], base)
    # permuting pool pages (and the table with them) changes nothing
    perm = torch.randperm(pb.P, generator=torch.Generator().manual_seed(3))
    slots = (perm.to(torch.int64)[:, None] * BS + torch.arange(BS)[None]).reshape(-1)
    k2 = torch.empty_like(pb.k_idx_cache)
    k2[slots] = pb.k_idx_cache
    pb2 = W.PrefillBatch(**{f: getattr(pb, f) for f in pb.__dataclass_fields__})
    pb2.k_idx_cache = k2
    pb2.block_table = perm[pb.block_table.to(torch.int64)].to(torch.int32)
    assert np.array_equal(run_prefill(o, pb2)[0], base)
    # a selection at least as wide as the visible blocks takes them all, and
    # the policy blocks always lead
    wide, _ = run_prefill(o, pb, topk=8)
    cub, pre = pb.cu_seqblocks_q.tolist(), pb.prefix_lens.tolist()
    for b in range(pb.B):
        for qb in range(cub[b + 1] - cub[b]):
            L = min(pre[b] + qb * pb.block_size_q + 1, int(pb.seq_lens[b]))
            nvis = -(-L // BS)
            for h in range(pb.Hi):
                row = wide[h, cub[b] + qb]
                assert sorted(row[row >= 0].tolist()) == list(range(nvis)), (b, qb, h, row)
                forced = sorted({0, nvis - 1})
                assert row[:len(forced)].tolist() == forced, (b, qb, h, row)


PINS = [
    pin_e4m3_decoder,
    pin_bf16_decoder,
    pin_f16_decoder,
    pin_block_score_bruteforce,
    pin_block_score_golden,
    pin_block_score_closed_form,
    pin_topk_sort,
    pin_topk_closed_form,
    pin_attention_vs_sdpa,
    pin_attention_bf16_cache,
    pin_attention_golden,
    pin_attention_closed_forms,
    pin_attention_invariants,
    pin_sdpa_vs_torch,
    pin_sdpa_closed_forms,
    pin_sdpa_invariants,
    pin_prefill_bruteforce,
    pin_prefill_golden,
    pin_prefill_reduces_to_decode,
    pin_prefill_invariants,
]
