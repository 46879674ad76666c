"""The benchmark's work accounting on the host (no GPU): the algorithmic
FLOP counts behind the dense-attention and fused-prefill roofline lines are
checked against closed forms and against the oracle's own visibility rule,
so a miscounted roofline cannot pass unnoticed.
"""
import numpy as np
import torch

import bench
import oracle
from sparse_paged_decode_gb300 import workloads as W


def test_dense_flops_closed_forms():
    # square causal: query t reads t + 1 keys
    w = W.make_dense("x", T=9, S=9, Hq=4, Hkv=2, D=8, causal=True, seed=1)
    assert bench.dense_flops(w) == 4 * 8 * 4 * (9 * 10 // 2)
    # without the flag every query reads every key
    w = W.make_dense("x", T=5, S=13, Hq=6, Hkv=3, D=16, causal=False, seed=1)
    assert bench.dense_flops(w) == 4 * 16 * 6 * 5 * 13
    # a chunk after a prefix: query t reads S - T + t + 1 keys
    w = W.make_dense("x", T=4, S=10, Hq=2, Hkv=1, D=4, causal=True, seed=1)
    assert bench.dense_flops(w) == 4 * 4 * 2 * (7 + 8 + 9 + 10)
    # more queries than keys: the first T - S read nothing
    w = W.make_dense("x", T=6, S=2, Hq=2, Hkv=1, D=4, causal=True, seed=1)
    assert bench.dense_flops(w) == 4 * 4 * 2 * (1 + 2)


def test_dense_workload_flops():
    w = W.dense_prefill()
    n_keys = sum(7680 + t + 1 for t in range(512))
    assert bench.dense_flops(w) == 4 * 128 * 64 * n_keys == 133152374784


def test_prefill_limits_match_the_oracle_visibility():
    """The benchmark's per-query-block (tokens, visible keys) against the
    oracle: on a batch with every page in the pool, the visible blocks
    ceil(L / 128) are exactly the blocks the oracle scores finite."""
    pb = W.make_prefill_batch("x", offsets=[300, 0, 1000, 77], chunks=[70, 5, 130, 1], block_size_q=16, topk=4,
                              init_blocks=0, local_blocks=0, Hi=1, Di=16, NB=16, P=96, seed=3,
                              idx_dtype=torch.float32)
    lim = bench.prefill_limits(pb)
    assert len(lim) == pb.n_rows
    assert sum(n for n, _ in lim) == pb.q_idx.shape[0]
    _, sc = oracle.default().prefill_topk(pb.q_idx, pb.k_idx_cache, pb.block_table, pb.slot_ids, pb.cu_seqlens,
                                          pb.seq_lens, pb.prefix_lens, pb.cu_seqblocks_q, pb.block_size_q, 0, 0,
                                          pb.scale, pb.n_rows, pb.topk)
    for row, (n, L) in enumerate(lim):
        assert int(np.isfinite(sc[0, row]).sum()) == -(-L // 128), (row, n, L)
    assert bench.prefill_flops(pb) == 2 * 16 * sum(n * L for n, L in lim)


def test_prefill_workload_shape():
    pb = W.prefill_batch()
    assert pb.B == 8 and pb.q_idx.shape == (4096, 1, 128)
    assert pb.n_rows == 64 and pb.cu_seqblocks_q.tolist() == [8 * i for i in range(9)]
    assert pb.seq_lens.tolist() == [o + 512 for o in pb.prefix_lens.tolist()]
    # the same sequences as the per-token prefill configuration
    w4 = W.config(4)
    assert [w4.request_lengths[i] for i in range(8)] == pb.seq_lens.tolist()


def test_reference_arms_run_on_rank_zero_only():
    """Under torchrun the oracle arm of every workload runs on rank 0 alone;
    the other ranks return without work (and print nothing)."""
    import types

    args = types.SimpleNamespace(steps=1, warmup=3, config=2, index_cache="native", cpu_seconds=1.0)
    for arm in (bench.run_reference, bench.run_dense_reference, bench.run_prefill_reference):
        assert arm(args, 1, 2) is None


def test_oracle_rate_threads_take_disjoint_rows():
    """The CPU baseline's threaded oracle: each row is taken once, and with a
    budget large enough every non-padding row of the workload is done."""
    w = W.make_decode("rate", lengths=[300, 129, 0], tokens_per_request=[2, 1, 1], Hq=8, Hkv=2, D=64, Di=32, NB=4,
                      P=16, K=2, seed=5, dtype=torch.float32)
    n_valid = int((w.seq_lens > 0).sum())
    rate, done, dt = bench.oracle_rate(w, budget_s=60.0, threads=3)
    assert done == n_valid and rate > 0 and dt > 0
    rate1, done1, _ = bench.oracle_rate(w, budget_s=60.0, max_rows=2, threads=1)
    assert done1 == 2 and rate1 > 0
    assert bench.host_cores() >= 1
