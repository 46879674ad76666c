"""paged_sparse_decode_attention_noalloc: the attention entry point for
callers that cannot allocate device memory (it uses the library's built-in
scratch instead of a caller workspace).

It must give the same result as paged_sparse_decode_attention on the same
inputs, call after call, while the built-in scratch keeps the previous call's
contents.  Both entry points run the same kernels on the same inputs, so the
outputs must agree bit for bit.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
BS = 128


def _run_both(spd, g, w, topk):
    dev = g.q.device
    ref = torch.full((w.T, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(spd.decode_workspace_bytes(w.T, w.Hq, w.Hkv, w.D, w.NB), dtype=torch.uint8, device=dev)
    spd.paged_sparse_decode_attention(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, g.req_idx, topk, ref,
                                      g.sm_scale, BS, g.k_scale, g.v_scale, ws)
    got = torch.full_like(ref, float("nan"))
    spd.paged_sparse_decode_attention_noalloc(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, g.req_idx,
                                              topk, got, g.sm_scale, BS, g.k_scale, g.v_scale)
    torch.cuda.synchronize()
    # neither call saw a device-side wait time out: the workspace's status
    # word, and the built-in scratch's (workspace None)
    assert spd.workspace_status(ws) == 0
    assert spd.workspace_status(None) == 0
    return got.cpu(), ref.cpu()


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    import sparse_paged_decode_gb300 as spd
    from sparse_paged_decode_gb300 import workloads as W

    dev = torch.device("cuda:0")
    # two different batches back to back: the second call runs on scratch the
    # first one left behind
    batches = [
        W.make_decode("noalloc_a", lengths=[2500, 900, 4096, 130], tokens_per_request=[4, 4, 1, 8], Hq=64, Hkv=8,
                      D=128, Di=128, NB=64, P=128, K=12, seed=501),
        W.make_decode("noalloc_b", lengths=[700, 3000], tokens_per_request=[2, 4], Hq=32, Hkv=4, D=128, Di=128,
                      NB=32, P=64, K=6, seed=502),
        # wide groups (24 rows of 8 q heads over 2 requests): the query-rows
        # FP8 kernel by default, where the first two take the keys-on-lanes one
        W.make_decode("noalloc_c", lengths=[3000, 1200], tokens_per_request=[16, 8], Hq=64, Hkv=8, D=128,
                      Di=128, NB=32, P=64, K=10, seed=503),
    ]
    for w in batches:
        g = w.to(dev)
        gen = torch.Generator().manual_seed(w.T)
        topk = torch.stack([torch.randperm(w.NB, generator=gen)[:w.K] for _ in range(w.T)]).to(torch.int32)
        topk = topk.view(1, w.T, w.K).to(dev).expand(w.Hkv, -1, -1)
        got, ref = _run_both(spd, g, w, topk)
        assert torch.isfinite(ref.float()).all(), "unwritten output cells"
        assert np.array_equal(got.view(torch.int16).numpy(), ref.view(torch.int16).numpy()), \
            "noalloc output differs from the workspace entry point's (bits)"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import sparse_paged_decode_gb300 as spd
    from sparse_paged_decode_gb300.binding import SpdError

    dev = torch.device("cuda:0")
    T, Hq, Hkv, D, NB = 4096, 64, 8, 128, 128
    assert spd.decode_workspace_bytes(T, Hq, Hkv, D, NB) > (16 << 20)
    q = torch.zeros((T, Hq, D), dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((128, Hkv, D), dtype=torch.float8_e4m3fn, device=dev)
    bt = torch.zeros((1, NB), dtype=torch.int32, device=dev)
    z = torch.zeros((T,), dtype=torch.int32, device=dev)
    tk = torch.zeros((1, T, 4), dtype=torch.int32, device=dev).expand(Hkv, -1, -1)
    out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    with pytest.raises(SpdError) as err:
        spd.paged_sparse_decode_attention_noalloc(q, kv, kv, bt, z, z, tk, out, 0.1, BS, 1.0, 1.0)
    assert err.value.code == 2 and "scratch" in str(err.value)
