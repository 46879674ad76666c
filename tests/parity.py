"""Comparators and stage runners for the GPU-vs-oracle parity tests.

Tolerances (written here, applied by every GPU test):
  * score sheet: -inf cells identical; finite cells within relative error
    1e-3, the relative error of a cell taken against
    max(|oracle|, 1e-2 * max |oracle| of its row) so that cells near zero are
    judged on the row's scale;
  * top-k: ranked against the oracle's fp64 scores, candidates whose scores
    lie within 1e-3 (same guarded relative measure) of their sorted
    neighbours form a tie cluster; each output position must hold a member of
    the oracle's cluster at that position (so positions outside any near-tie
    are bit-exact), padding -1 must match exactly, ids must be distinct, and
    the set overlap over all rows must be >= 0.99;
  * attention: max absolute error <= 2e-2 and cosine similarity >= 0.9999
    against the fp64 oracle; rows with no valid key exactly zero.
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch

SCORE_RTOL = 1e-3
TIE_RTOL = 1e-3
ATTN_ATOL = 2e-2
ATTN_COS = 0.9999
TOPK_OVERLAP = 0.99


def guarded_rel_err(got, ref):
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    fin = np.isfinite(ref)
    row_scale = np.max(np.where(fin, np.abs(ref), 0.0), axis=-1, keepdims=True)
    denom = np.maximum(np.abs(ref), 1e-2 * row_scale)
    denom = np.where(denom > 0, denom, 1.0)
    return np.where(fin, np.abs(got - ref) / denom, 0.0)


def check_scores(got, ref, what="scores"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert not np.any(np.isnan(got)), "%s: NaN in output (unwritten cell?)" % what
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "%s: -inf pattern differs" % what
    err = guarded_rel_err(got, ref)
    assert err.max() <= SCORE_RTOL, "%s: max relative error %.3g" % (what, err.max())
    return float(err.max())


def check_topk(got, ref_scores, K, what="topk"):
    """``got`` [rows..., K] int; ``ref_scores`` [rows..., NB] fp64 oracle sheet."""
    got = np.asarray(got).reshape(-1, K)
    s = np.asarray(ref_scores, dtype=np.float64).reshape(got.shape[0], -1)
    matched = total = 0
    for row in range(got.shape[0]):
        r = s[row]
        cand = np.flatnonzero(np.isfinite(r) | np.isposinf(r))
        order = cand[np.lexsort((cand, -r[cand]))]
        n = len(order)
        g = got[row]
        assert np.all(g[min(n, K):] == -1), "%s row %d: padding differs" % (what, row)
        sel = g[:min(n, K)]
        assert np.all(sel >= 0) and len(set(sel.tolist())) == len(sel), "%s row %d: bad ids %s" % (what, row, sel)
        scale = max(np.max(np.abs(r[cand])) if n else 1.0, 1e-30)
        vals = r[order]
        # tie clusters over the sorted candidates
        cluster = np.zeros(n, dtype=np.int64)
        for i in range(1, n):
            gap = abs(vals[i - 1] - vals[i]) / max(abs(vals[i - 1]), 1e-2 * scale)
            cluster[i] = cluster[i - 1] + (gap > TIE_RTOL)
        cl_of = {int(b): int(c) for b, c in zip(order, cluster)}
        for k, b in enumerate(sel):
            assert int(b) in cl_of, "%s row %d: id %d is not a candidate" % (what, row, b)
            assert cl_of[int(b)] == cluster[k], (
                "%s row %d pos %d: got block %d, oracle %d (scores %.9g vs %.9g)"
                % (what, row, k, b, order[k], r[b], vals[k]))
        ref_set = set(order[:K].tolist())
        matched += len(ref_set & set(sel.tolist()))
        total += len(ref_set)
    overlap = matched / total if total else 1.0
    assert overlap >= TOPK_OVERLAP, "%s: overlap %.4f" % (what, overlap)
    return overlap


def check_attention(got, ref, what="attention", zero_rows=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite output (unwritten cell?)" % what
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    num = float((got * ref).sum())
    den = float(np.sqrt((got ** 2).sum() * (ref ** 2).sum()))
    cos = num / den if den > 0 else (1.0 if not got.any() and not ref.any() else 0.0)
    assert err <= ATTN_ATOL, "%s: max abs err %.4g" % (what, err)
    assert cos >= ATTN_COS, "%s: cosine %.7f" % (what, cos)
    if zero_rows is not None:
        for t in zero_rows:
            assert not np.any(got[t]), "%s: padding row %d not zero" % (what, t)
    return err, cos


def digest(*tensors) -> str:
    h = hashlib.sha256()
    for t in tensors:
        if t is None:
            continue
        t = t.detach()
        h.update(str((t.shape, t.stride(), t.dtype)).encode())
        h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes() if t.numel() else b"")
    return h.hexdigest()


def nan_like(shape, dtype, device):
    if dtype == torch.int32:
        return torch.full(shape, 0x7FFFFFF0, dtype=dtype, device=device)
    return torch.full(shape, float("nan"), dtype=dtype, device=device)


def check_prefill_rows(got, ref_ids, ref_scores, n_forced, what="prefill"):
    """Rows of the fused prefill selection.  ``got``/``ref_ids`` [rows, topk]
    int; ``ref_scores`` [rows, NB] fp64 oracle block scores; ``n_forced[row]``
    the number of policy blocks the row leads with.  The policy blocks must
    match exactly; the rest of each row is held to the top-k rule above
    (tie clusters of the oracle's scores over the row's other visible
    candidates, exact padding, distinct ids), the set overlap taken over all
    rows together."""
    got = np.asarray(got)
    ref_ids = np.asarray(ref_ids)
    s = np.asarray(ref_scores, dtype=np.float64)
    matched = total = 0
    for row in range(got.shape[0]):
        K = got.shape[1]
        nf = min(int(n_forced[row]), K)
        assert np.array_equal(got[row, :nf], ref_ids[row, :nf]), (
            "%s row %d: policy blocks %s, oracle %s" % (what, row, got[row, :nf], ref_ids[row, :nf]))
        forced = set(ref_ids[row, :nf].tolist())
        r = s[row].copy()
        r[list(forced)] = -np.inf
        # the other candidates (blocks that are not visible score -inf)
        cand = np.flatnonzero(np.isfinite(r) | np.isposinf(r))
        order = cand[np.lexsort((cand, -r[cand]))]
        Kr = K - nf
        n = min(len(order), Kr)
        g = got[row, nf:]
        assert np.all(g[n:] == -1), "%s row %d: padding differs (%s)" % (what, row, g)
        sel = g[:n]
        assert np.all(sel >= 0) and len(set(sel.tolist()) | forced) == len(sel) + len(forced), (
            "%s row %d: bad or repeated ids %s" % (what, row, got[row]))
        if n == 0:
            continue
        vals = r[order]
        scale = max(np.max(np.abs(vals[np.isfinite(vals)])) if np.any(np.isfinite(vals)) else 1.0, 1e-30)
        cluster = np.zeros(len(order), dtype=np.int64)
        for i in range(1, len(order)):
            gap = abs(vals[i - 1] - vals[i]) / max(abs(vals[i - 1]), 1e-2 * scale)
            cluster[i] = cluster[i - 1] + (gap > TIE_RTOL)
        cl_of = {int(b): int(c) for b, c in zip(order, cluster)}
        for k, b in enumerate(sel):
            assert int(b) in cl_of, "%s row %d: id %d is not a candidate" % (what, row, b)
            assert cl_of[int(b)] == cluster[k], (
                "%s row %d pos %d: got block %d, oracle %d" % (what, row, nf + k, b, order[k]))
        ref_set = set(order[:Kr].tolist())
        matched += len(ref_set & set(sel.tolist()))
        total += len(ref_set)
    overlap = matched / total if total else 1.0
    assert overlap >= TOPK_OVERLAP, "%s: overlap %.4f" % (what, overlap)
    return overlap
