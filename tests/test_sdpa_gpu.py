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


# The tensor-core kernel's domain (16-bit q, k, v of head dim 128, 16-bit
# output, G a power of two): each case runs on it (policy 0) and on the
# CUDA-core kernel (policy 1), both against the oracle.
TC_CASES = [
    # T, S, Hq, Hkv, causal, in dtype, out dtype, q distribution, sm_scale factor
    (64, 1000, 64, 8, True, torch.bfloat16, torch.bfloat16, "normal", 1.0),     # tiles of 16 tokens, ragged keys
    (77, 300, 16, 8, False, torch.float16, torch.float16, "student_t3", 1.0),   # G = 2, ragged token tail
    (200, 200, 4, 4, True, torch.bfloat16, torch.float16, "normal", 1.0),       # MHA, square causal, 2 tiles
    (50, 20, 16, 1, True, torch.bfloat16, torch.bfloat16, "normal", 1.0),      # G = 16, T > S: rows read nothing
    (33, 700, 32, 2, True, torch.bfloat16, torch.bfloat16, "student_t3", -1.0),  # negative scale
    (9, 129, 128, 1, False, torch.float16, torch.bfloat16, "normal", 3.0),     # G = 128: one token per tile
]


@pytest.mark.parametrize("policy", [0, 1], ids=["tensor_core", "cuda_core"])
@pytest.mark.parametrize("case", TC_CASES, ids=["T%d_S%d_H%d_%d_%s_%s_%s_%s_x%g" % (
    c[0], c[1], c[2], c[3], "causal" if c[4] else "full", str(c[5])[6:], str(c[6])[6:], c[7], c[8])
    for c in TC_CASES])
def test_sdpa_tensor_core_domain(spd, orc, case, policy):
    T, S, Hq, Hkv, causal, dt, odt, qd, fac = case
    w = W.make_dense("tc", T=T, S=S, Hq=Hq, Hkv=Hkv, D=128, causal=causal, seed=900 + T + S, dtype=dt, q_dist=qd)
    sm = w.sm_scale * fac
    ref = orc.sdpa(w.q, w.k, w.v, sm, causal)
    g = w.to(DEV)
    old = spd.set_kernel_policy(4, policy)
    try:
        got = run(spd, g.q, g.k, g.v, sm, causal, odt)
    finally:
        spd.set_kernel_policy(4, old)
    check(got, ref, "sdpa %s policy %d" % (case, policy))
    if causal and T > S:
        assert not got[:T - S].float().any(), "rows that read no key must be zero"


def test_sdpa_tensor_core_strided_views(spd, orc):
    """q inside a packed [T, 3, Hq, 128] tensor and k, v as head-major caches
    viewed [S, Hkv, 128] (16-byte aligned rows, so the tensor-core kernel
    takes them through its TMA maps); the output a strided window whose
    other elements stay untouched."""
    T, S, Hq, Hkv, D = 40, 500, 16, 2, 128
    gen = torch.Generator().manual_seed(78)
    qkv = torch.randn((T, 3, Hq, D), generator=gen).to(torch.bfloat16)
    kh = torch.randn((Hkv, S, D), generator=gen).to(torch.bfloat16)
    vh = torch.randn((Hkv, S, D), generator=gen).to(torch.bfloat16)
    sm = 0.09
    ref = orc.sdpa(qkv[:, 1].contiguous(), kh.permute(1, 0, 2).contiguous(), vh.permute(1, 0, 2).contiguous(),
                   sm, True)
    qkv_d, kh_d, vh_d = qkv.to(DEV), kh.to(DEV), vh.to(DEV)
    big = torch.full((T, Hq + 2, 2 * D), -5.0, dtype=torch.bfloat16, device=DEV)
    out = big[:, 1:Hq + 1, ::2]
    out.fill_(float("nan"))
    run(spd, qkv_d[:, 1], kh_d.permute(1, 0, 2), vh_d.permute(1, 0, 2), sm, True, out=out)
    check(out, ref, "tensor-core strided")
    mask = torch.ones_like(big, dtype=torch.bool)
    mask[:, 1:Hq + 1, ::2] = False
    assert torch.all(big[mask] == -5.0), "wrote outside the output's cells"


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


def test_sdpa_full_size(spd, orc):
    """The benchmarked prefill chunk (512 query tokens after 7680 cached
    tokens, 64/8 heads, D=128, bf16), in the benchmark's launch
    configuration, checked on every query token with all its heads: under
    the causal flag token t is non-causal attention over its first
    t + S - T + 1 keys, so the oracle runs token by token, from one host
    thread per core."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    w = W.dense_prefill()
    g = w.to(DEV)
    got = run(spd, g.q, g.k, g.v, w.sm_scale, True).float().cpu().numpy()

    def one(t):
        n = t + w.S - w.T + 1
        return orc.sdpa(w.q[t:t + 1], w.k[:n], w.v[:n], w.sm_scale, False)

    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        ref = np.concatenate(list(ex.map(one, range(w.T))), axis=0)
    check_attention(got, ref, "dense prefill chunk")
