"""GPU parity of the dense GQA attention call (attention_sdpa) against the
CPU oracle, through the C ABI.

Outputs are NaN-poisoned before each call and the inputs hashed before and
after.  Small cases compare every cell; they span several 64-row CTAs and
64-key tiles with ragged tails, every head-dim specialisation (D up to 32,
64, 128, 256, and a D that is none of these), group sizes 1 to 16, all input
and output dtypes, arbitrary strides, and the degenerate cases (no keys,
query tokens that may read nothing under the causal flag, no query tokens).
The full-size prefill chunk is checked on sampled query tokens: under the
causal flag, token t of the chunk is non-causal attention over the first
t + S - T + 1 keys (an invariant the oracle's pins establish), so the oracle
runs on those tokens alone.

Tolerance: bf16 / f16 outputs as for the paged attention (max absolute
error 2e-2, cosine >= 0.9999 against fp64); f32 outputs max absolute error
1e-4 (fp32 logits, softmax and sums over at most a few thousand keys of
unit-scale values, well inside it).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import check_attention, digest, nan_like
from sparse_paged_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
F32_ATOL = 1e-4


@pytest.fixture(scope="module")
def spd():
    import sparse_paged_decode_gb300 as m

    return m


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def run(spd, q, k, v, sm_scale, causal, out_dtype=torch.bfloat16, out=None):
    if out is None:
        out = nan_like(tuple(q.shape), out_dtype, DEV)
    before = digest(q, k, v)
    spd.attention_sdpa(q, k, v, out, sm_scale, causal)
    torch.cuda.synchronize()
    assert digest(q, k, v) == before, "inputs mutated"
    return out


def check(got, ref, what):
    g = got.float().cpu().numpy()
    if got.dtype == torch.float32:
        assert np.all(np.isfinite(g)), "%s: non-finite output (unwritten cell?)" % what
        err = float(np.max(np.abs(g - ref))) if g.size else 0.0
        assert err <= F32_ATOL, "%s: max abs err %.3g" % (what, err)
    else:
        check_attention(g, ref, what)


CASES = [
    # T, S, Hq, Hkv, D, causal, in dtype, out dtype, q distribution
    (37, 300, 8, 1, 64, True, torch.bfloat16, torch.bfloat16, "normal"),
    (37, 300, 8, 1, 64, False, torch.bfloat16, torch.bfloat16, "student_t3"),
    (50, 20, 4, 2, 72, True, torch.float16, torch.float32, "normal"),  # T > S: first rows read nothing
    (24, 1000, 32, 2, 128, False, torch.bfloat16, torch.bfloat16, "student_t3"),  # group of 16
    (9, 200, 4, 4, 256, True, torch.float32, torch.bfloat16, "normal"),
    (129, 129, 6, 3, 32, True, torch.float32, torch.float32, "normal"),  # square causal
    (5, 7, 2, 1, 1, True, torch.bfloat16, torch.float16, "normal"),
    (3, 0, 4, 2, 16, False, torch.bfloat16, torch.bfloat16, "normal"),  # no keys
]


@pytest.mark.parametrize("case", CASES, ids=["T%d_S%d_H%d_%d_D%d_%s_%s_%s_%s" % (
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full", str(c[6])[6:], str(c[7])[6:], c[8])
    for c in CASES])
def test_sdpa_small(spd, orc, case):
    T, S, Hq, Hkv, D, causal, dt, odt, qd = case
    w = W.make_dense("t", T=T, S=S, Hq=Hq, Hkv=Hkv, D=D, causal=causal, seed=300 + T + S + D, dtype=dt,
                     q_dist=qd)
    ref = orc.sdpa(w.q, w.k, w.v, w.sm_scale, causal)
    g = w.to(DEV)
    got = run(spd, g.q, g.k, g.v, w.sm_scale, causal, odt)
    check(got, ref, "sdpa %s" % (case,))
    if causal and T > S:
        assert not got[:T - S].float().any(), "rows that read no key must be zero"


def test_sdpa_strided_inputs_and_output(spd, orc):
    """q inside a packed [T, 3, Hq, D] tensor, k and v as head-major caches
    viewed [S, Hkv, D], the output a strided window of a larger buffer whose
    other elements must stay untouched."""
    T, S, Hq, Hkv, D = 21, 150, 8, 2, 64
    gen = torch.Generator().manual_seed(77)
    qkv = torch.randn((T, 3, Hq, D), generator=gen).to(torch.bfloat16)
    kh = torch.randn((Hkv, S, D), generator=gen).to(torch.bfloat16)
    vh = torch.randn((Hkv, S, D), generator=gen).to(torch.bfloat16)
    sm = 0.11
    ref = orc.sdpa(qkv[:, 0].contiguous(), kh.permute(1, 0, 2).contiguous(), vh.permute(1, 0, 2).contiguous(),
                   sm, True)
    qkv_d, kh_d, vh_d = qkv.to(DEV), kh.to(DEV), vh.to(DEV)
    big = torch.full((T, Hq + 3, 2 * D), -7.0, dtype=torch.float32, device=DEV)
    out = big[:, 1:Hq + 1, ::2]
    out.fill_(float("nan"))
    run(spd, qkv_d[:, 0], kh_d.permute(1, 0, 2), vh_d.permute(1, 0, 2), sm, True, out=out)
    check(out, ref, "strided")
    mask = torch.ones_like(big, dtype=torch.bool)
    mask[:, 1:Hq + 1, ::2] = False
    assert torch.all(big[mask] == -7.0), "wrote outside the output's cells"


def test_sdpa_empty_batch(spd):
    q = torch.empty((0, 4, 8), dtype=torch.bfloat16, device=DEV)
    k = torch.randn((5, 2, 8), device=DEV).to(torch.bfloat16)
    out = torch.empty((0, 4, 8), dtype=torch.bfloat16, device=DEV)
    spd.attention_sdpa(q, k, k.clone(), out, 0.3, True)
    torch.cuda.synchronize()


def test_sdpa_full_size_sampled(spd, orc):
    """The benchmarked prefill chunk (512 query tokens after 7680 cached
    tokens, 64/8 heads, D=128, bf16), in the benchmark's launch
    configuration, checked on sampled query tokens with all their heads."""
    w = W.dense_prefill()
    g = w.to(DEV)
    got = run(spd, g.q, g.k, g.v, w.sm_scale, True).float().cpu().numpy()
    for t in (0, 1, 63, 64, 200, 255, 256, 511):
        n = t + w.S - w.T + 1
        ref = orc.sdpa(w.q[t:t + 1], w.k[:n], w.v[:n], w.sm_scale, False)
        check_attention(got[t:t + 1], ref, "dense prefill token %d" % t)
