"""GPU parity of the fused prefill score-to-selection call
(msa_prefill_block_score) against the CPU oracle, through the C ABI.

Outputs are poisoned before each call and the inputs hashed before and
after.  Small ragged batches compare every row: query blocks of 1, 3, 4, 64
and 100 tokens (some not dividing the chunk), policy blocks from none to more
than the selection holds, selections wider than the visible blocks, one and
two index heads, bf16 index tensors (tensor-core score kernel), fp32 (general
kernel) and an FP8-E4M3 index cache, a strided query and output window,
sequences outside the page table, pages outside the pool, seq_lens short of
the chunk, and rows no sequence owns.  At full size (the batched prefill
sequences, 8 x 512 tokens) the rows of the longest and the shortest
sequence are checked against the oracle run on that sequence alone, and
single-token query blocks without policy blocks must equal, bit for bit,
the decode score sheet and top-k calls on the same tokens.

Tolerance: the policy blocks exactly; the other ids by the top-k rule of the
decode selection (exact outside near-ties of the oracle's scores, within
1e-3 relative; overlap >= 0.99).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import check_prefill_rows, digest, nan_like
from sparse_paged_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
BS = 128


@pytest.fixture(scope="module")
def spd():
    import sparse_paged_decode_gb300 as m

    return m


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def n_forced(pb, slot_ids=None, seq_lens=None):
    """Policy blocks each output row leads with (from the metadata)."""
    sid = (pb.slot_ids if slot_ids is None else slot_ids).tolist()
    sl = (pb.seq_lens if seq_lens is None else seq_lens).tolist()
    cub, pre = pb.cu_seqblocks_q.tolist(), pb.prefix_lens.tolist()
    R = pb.block_table.shape[0]
    out = [0] * pb.n_rows
    for b in range(pb.B):
        for qb in range(cub[b + 1] - cub[b]):
            L = min(pre[b] + qb * pb.block_size_q + 1, sl[b], pb.NB * BS)
            L = 0 if not 0 <= sid[b] < R else max(L, 0)
            nvis = -(-L // BS)
            out[cub[b] + qb] = len({k for k in range(nvis) if k < pb.init_blocks or k >= nvis - pb.local_blocks})
    return out


def gpu_prefill(spd, g, n_rows=None, topk=None, out=None, q=None, slot_ids=None, seq_lens=None, bt=None):
    n_rows = g.n_rows if n_rows is None else n_rows
    topk = g.topk if topk is None else topk
    q = g.q_idx if q is None else q
    sid = g.slot_ids if slot_ids is None else slot_ids
    sl = g.seq_lens if seq_lens is None else seq_lens
    bt = g.block_table if bt is None else bt
    if out is None:
        out = nan_like((g.Hi, n_rows, topk), torch.int32, DEV)
    ws = torch.empty(spd.prefill_workspace_bytes(q.shape[0], g.Hi, g.NB), dtype=torch.uint8, device=DEV)
    ins = (q, g.k_idx_cache, bt, sid, g.cu_seqlens, sl, g.prefix_lens, g.cu_seqblocks_q)
    before = digest(*ins)
    spd.msa_prefill_block_score(q, g.k_idx_cache, bt, sid, g.cu_seqlens, sl, g.prefix_lens, g.block_size_q, BS,
                                g.init_blocks, g.local_blocks, g.scale, g.cu_seqblocks_q, out, ws)
    torch.cuda.synchronize()
    assert digest(*ins) == before, "inputs mutated"
    return out


def oracle_prefill(orc, pb, n_rows=None, topk=None, slot_ids=None, seq_lens=None, bt=None):
    return orc.prefill_topk(pb.q_idx, pb.k_idx_cache, pb.block_table if bt is None else bt,
                            pb.slot_ids if slot_ids is None else slot_ids, pb.cu_seqlens,
                            pb.seq_lens if seq_lens is None else seq_lens, pb.prefix_lens, pb.cu_seqblocks_q,
                            pb.block_size_q, pb.init_blocks, pb.local_blocks, pb.scale,
                            pb.n_rows if n_rows is None else n_rows, pb.topk if topk is None else topk)


def compare(got, ref, sc, nf, what):
    got = got.cpu().numpy()
    for h in range(got.shape[0]):
        check_prefill_rows(got[h], ref[h], sc[h], nf, "%s head %d" % (what, h))


CASES = [
    # offsets, chunks, block_size_q, topk, init, local, Hi, Di, index dtype
    ([300, 0, 1000, 77], [70, 5, 130, 1], 4, 8, 1, 2, 1, 128, torch.bfloat16),
    ([300, 0, 1000, 77], [70, 5, 130, 1], 1, 8, 0, 0, 2, 64, torch.bfloat16),
    ([1500, 20, 900], [200, 64, 33], 64, 4, 0, 8, 1, 128, torch.bfloat16),  # policy fills the row
    ([1500, 20, 900], [200, 64, 33], 100, 40, 2, 1, 2, 128, torch.bfloat16),  # wider than the visible blocks
    ([640, 3, 1200, 0, 256], [90, 17, 40, 128, 9], 3, 6, 4, 0, 1, 64, torch.float32),
    ([640, 3, 1200, 0, 256], [90, 17, 40, 128, 9], 16, 5, 1, 1, 1, 128, "e4m3"),
]


@pytest.mark.parametrize("case", CASES, ids=["bsq%d_top%d_init%d_local%d_H%d_D%d_%s" % (
    c[2], c[3], c[4], c[5], c[6], c[7], "e4m3" if c[8] == "e4m3" else str(c[8])[6:]) for c in CASES])
def test_prefill_small(spd, orc, case):
    offsets, chunks, bsq, topk, init, local, Hi, Di, dt = case
    pb = W.make_prefill_batch("t", offsets=offsets, chunks=chunks, block_size_q=bsq, topk=topk, init_blocks=init,
                              local_blocks=local, Hi=Hi, Di=Di, NB=16, P=96, seed=500 + bsq + topk,
                              idx_dtype=torch.bfloat16 if dt == "e4m3" else dt)
    if dt == "e4m3":
        codes, s8 = W._to_e4m3(pb.k_idx_cache.float())
        pb.k_idx_cache = codes
        pb.scale = pb.scale * s8
    ref, sc = oracle_prefill(orc, pb)
    got = gpu_prefill(spd, pb.to(DEV))
    compare(got, ref, sc, n_forced(pb), "case %s" % (case[2:],))


def test_prefill_bad_metadata_and_layouts(spd, orc):
    pb = W.make_prefill_batch("t", offsets=[300, 0, 1000, 77], chunks=[70, 5, 130, 1], block_size_q=8, topk=6,
                              init_blocks=1, local_blocks=1, Hi=2, Di=128, NB=16, P=96, seed=610)
    bt = pb.block_table.clone()
    bt[int(pb.slot_ids[2]), 3] = pb.P + 11  # a page outside the pool
    sid = pb.slot_ids.clone()
    sid[1] = bt.shape[0] + 4  # a sequence outside the table
    sl = pb.seq_lens.clone()
    sl[0] = int(pb.prefix_lens[0]) + 20  # seq_lens short of the chunk
    rows = pb.n_rows + 3  # rows that no sequence owns
    ref, sc = oracle_prefill(orc, pb, n_rows=rows, slot_ids=sid, seq_lens=sl, bt=bt)
    g = pb.to(DEV)
    # a strided query (one head of a wider tensor) and a strided output window
    wide_q = torch.zeros((pb.q_idx.shape[0], pb.Hi, 2, pb.Di), dtype=pb.q_idx.dtype, device=DEV)
    wide_q[:, :, 1] = g.q_idx
    big = torch.full((pb.Hi, rows, 2 * pb.topk + 3), -9, dtype=torch.int32, device=DEV)
    out = big[:, :, 1:1 + 2 * pb.topk:2]
    out.fill_(0x7FFFFFF0)
    gpu_prefill(spd, g, n_rows=rows, out=out, q=wide_q[:, :, 1], slot_ids=sid.to(DEV), seq_lens=sl.to(DEV),
                bt=bt.to(DEV))
    nf = n_forced(pb, slot_ids=sid, seq_lens=sl) + [0, 0, 0]
    compare(out, ref, sc, nf, "bad metadata")
    assert torch.all(out[:, pb.n_rows:] == -1)
    mask = torch.ones_like(big, dtype=torch.bool)
    mask[:, :, 1:1 + 2 * pb.topk:2] = False
    assert torch.all(big[mask] == -9), "wrote outside the output's cells"


def sub_batch(pb, b):
    """Sequence b of a batch as a batch of its own (same keys and table)."""
    cu, cub = pb.cu_seqlens.tolist(), pb.cu_seqblocks_q.tolist()
    one = W.PrefillBatch(**{f: getattr(pb, f) for f in pb.__dataclass_fields__})
    one.B = 1
    one.q_idx = pb.q_idx[cu[b]:cu[b + 1]]
    one.slot_ids = pb.slot_ids[b:b + 1]
    one.seq_lens = pb.seq_lens[b:b + 1]
    one.prefix_lens = pb.prefix_lens[b:b + 1]
    one.cu_seqlens = torch.tensor([0, cu[b + 1] - cu[b]], dtype=torch.int32)
    one.cu_seqblocks_q = torch.tensor([0, cub[b + 1] - cub[b]], dtype=torch.int32)
    one.n_rows = cub[b + 1] - cub[b]
    return one


def test_prefill_full_size_sampled(spd, orc):
    """The batched prefill sequences (8 x 512 tokens, offsets up to 15872,
    query blocks of 64, 1 initial + 2 local blocks, top-32), as the
    benchmark launches them; the longest and the shortest sequence's rows
    against the oracle."""
    pb = W.prefill_batch()
    got = gpu_prefill(spd, pb.to(DEV)).cpu()
    nf = n_forced(pb)
    cub = pb.cu_seqblocks_q.tolist()
    lens = pb.seq_lens.tolist()
    for b in (int(np.argmax(lens)), int(np.argmin(lens))):
        one = sub_batch(pb, b)
        ref, sc = oracle_prefill(orc, one)
        compare(got[:, cub[b]:cub[b + 1]], ref, sc, nf[cub[b]:cub[b + 1]], "full size sequence %d" % b)


def test_prefill_single_token_blocks_equal_decode_calls(spd):
    """Query blocks of one token and no policy blocks: the fused call's rows
    are, bit for bit, msa_select_topk of msa_block_score for the same tokens
    with seq_len = position + 1 (the per-token prefill configuration)."""
    pb = W.prefill_batch(block_size_q=1, init_blocks=0, local_blocks=0, topk=32)
    g = pb.to(DEV)
    fused = gpu_prefill(spd, g)
    cu = pb.cu_seqlens.tolist()
    ri, sl = [], []
    for b in range(pb.B):
        for j in range(cu[b + 1] - cu[b]):
            ri.append(int(pb.slot_ids[b]))
            sl.append(int(pb.prefix_lens[b]) + j + 1)
    ri = torch.tensor(ri, dtype=torch.int32, device=DEV)
    sl = torch.tensor(sl, dtype=torch.int32, device=DEV)
    T = pb.q_idx.shape[0]
    scores = torch.empty((pb.Hi, T, pb.NB), device=DEV)
    topk = torch.empty((pb.Hi, T, pb.topk), dtype=torch.int32, device=DEV)
    spd.msa_block_score(g.q_idx, g.k_idx_cache, g.block_table, sl, ri, BS, scores, pb.scale)
    spd.msa_select_topk(scores, topk)
    torch.cuda.synchronize()
    assert torch.equal(fused, topk)
