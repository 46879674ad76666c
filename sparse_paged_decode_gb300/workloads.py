"""Seeded synthetic inputs for the sparse paged decode path.

This module only draws and lays out input tensors; it holds none of the
method's arithmetic, so the oracle tests, the GPU tests and the benchmark can
all use it.  Everything is drawn on the CPU from a ``torch.Generator`` seeded
with ``1000 + config`` unless a seed is given.

Shapes follow the serving setup of "MiniMax-M3 decode through the ATOM kernel
library" -- Supported experiment: 128-token pages, maximum model length 16384
(so a page table holds at most 128 blocks), a 1024-block pool, decode and
verification buckets of 1, 4, 8 and 16 query tokens, FP8 main and index caches
with static scalar K/V scales.

Recipe shared by every workload
  * Pool pages are handed out from a seeded permutation of the pool, so a
    request's pages are scattered (the block table is a true indirection).
  * Page-table entries past a request's last block point at pages that no
    request owns.  Every slot that no request owns -- unused pages and the
    tail of a request's last page -- holds finite poison: E4M3 +/-448 in the
    K/V caches, +64 in the index cache, so that a read past ``seq_lens`` or of
    an unselected block dominates the result and fails parity.
  * Query token j of an n-token request of length L has ``seq_len = L - (n-1-j)``
    (causal among the draft tokens of a verification row).
  * K and V are drawn in fp32 and stored as FP8-E4M3 with one static scalar
    scale each: ``scale = max|x| / 448`` over the stored (valid) values, codes
    ``= e4m3(x / scale)`` (round to nearest even, via torch's cast).  With
    ``kv_dtype="bf16"`` they are stored as dense BF16 instead (rounded to
    nearest even, scale 1.0; unowned slots hold the poison +/-448.0).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

BLOCK_SIZE = 128
E4M3_POS_MAX = 0x7E  # +448
E4M3_NEG_MAX = 0xFE  # -448
INDEX_POISON = 64.0


@dataclass
class Workload:
    """One batch of inputs for the three stages (CPU tensors)."""

    name: str
    T: int
    R: int
    Hq: int
    Hkv: int
    D: int
    Hi: int
    Di: int
    NB: int
    P: int
    K: int
    block_size: int
    dense: bool
    block_table: torch.Tensor  # int32 [R, NB]
    req_idx: torch.Tensor  # int32 [T]
    seq_lens: torch.Tensor  # int32 [T]
    q: Optional[torch.Tensor] = None  # [T, Hq, D] f32 | bf16
    k_cache: Optional[torch.Tensor] = None  # float8_e4m3fn [P*BS, Hkv, D]
    v_cache: Optional[torch.Tensor] = None
    k_scale: float = 1.0
    v_scale: float = 1.0
    q_idx: Optional[torch.Tensor] = None  # [T, Hi, Di] f32 | bf16
    k_idx_cache: Optional[torch.Tensor] = None  # [P*BS, 1, Di] f32 | bf16
    sm_scale: float = 1.0
    idx_scale: float = 1.0
    tokens_per_request: List[int] = field(default_factory=list)
    request_lengths: List[int] = field(default_factory=list)

    @property
    def n_valid_tokens(self) -> int:
        """Query rows that are not padding (seq_len > 0): the unit of the metric."""
        return int((self.seq_lens > 0).sum())

    def to(self, device) -> "Workload":
        out = Workload(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("block_table", "req_idx", "seq_lens", "q", "k_cache", "v_cache", "q_idx", "k_idx_cache"):
            v = getattr(out, k)
            if v is not None:
                setattr(out, k, v.to(device))
        return out


def _pages_for(lengths: Sequence[int], P: int, NB: int, g: torch.Generator):
    """Scatter each request's blocks over a seeded permutation of the pool."""
    perm = torch.randperm(P, generator=g)
    need = [max(1, math.ceil(L / BLOCK_SIZE)) for L in lengths]
    if sum(need) > P:
        raise ValueError("pool of %d pages too small for %d blocks" % (P, sum(need)))
    if max(need) > NB:
        raise ValueError("a request needs more than NB=%d blocks" % NB)
    owned, pos = [], 0
    for n in need:
        owned.append(perm[pos:pos + n])
        pos += n
    spare = perm[pos:]
    table = torch.empty((len(lengths), NB), dtype=torch.int32)
    for r, pages in enumerate(owned):
        table[r, :len(pages)] = pages.to(torch.int32)
        tail = NB - len(pages)
        if tail:
            if len(spare):
                fill = spare[torch.randint(0, len(spare), (tail,), generator=g)]
            else:  # every page is owned: point past-the-end entries at random pages
                fill = torch.randint(0, P, (tail,), generator=g)
            table[r, len(pages):] = fill.to(torch.int32)
    return table, owned


def _request_slots(pages: torch.Tensor, L: int) -> torch.Tensor:
    slots = (pages.to(torch.int64)[:, None] * BLOCK_SIZE + torch.arange(BLOCK_SIZE)[None, :]).reshape(-1)
    return slots[:L]


def _to_e4m3(x: torch.Tensor):
    """Static scalar scale max|x|/448 and E4M3 codes of x/scale."""
    amax = float(x.abs().max()) if x.numel() else 1.0
    scale = amax / 448.0 if amax > 0 else 1.0
    codes = (x / scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    return codes, scale


def _poison_e4m3(shape, g: torch.Generator) -> torch.Tensor:
    sign = torch.randint(0, 2, shape, generator=g, dtype=torch.uint8)
    codes = torch.where(sign.bool(), torch.tensor(E4M3_NEG_MAX, dtype=torch.uint8),
                        torch.tensor(E4M3_POS_MAX, dtype=torch.uint8))
    return codes.view(torch.float8_e4m3fn)


def _student_t3(shape, g: torch.Generator) -> torch.Tensor:
    z = torch.randn(shape, generator=g)
    chi2 = torch.randn(shape + (3,), generator=g).square().sum(-1)
    return z / torch.sqrt(chi2 / 3.0)


def make_decode(name: str, *, lengths: Sequence[int], tokens_per_request: Sequence[int],
                Hq: int, Hkv: int, D: int, Hi: int = 1, Di: int = 128, NB: int = 128, P: int,
                K: int, dtype: torch.dtype = torch.bfloat16, idx_dtype: Optional[torch.dtype] = None,
                seed: int, dense: bool = False, q_dist: str = "normal",
                padded_tail: Optional[Sequence[int]] = None, with_index: bool = True,
                with_kv: bool = True, kv_dtype: str = "e4m3") -> Workload:
    """A decode/verification batch: request r owns ``tokens_per_request[r]``
    consecutive query rows and has total length ``lengths[r]``.
    ``padded_tail[r]`` trailing rows of request r get ``seq_len = 0``.
    ``kv_dtype`` is "e4m3" (static scalar scales) or "bf16" (dense, scale 1)."""
    if kv_dtype not in ("e4m3", "bf16"):
        raise ValueError("kv_dtype must be 'e4m3' or 'bf16'")
    g = torch.Generator().manual_seed(seed)
    idx_dtype = idx_dtype or dtype
    R = len(lengths)
    table, owned = _pages_for(lengths, P, NB, g)

    req_idx, seq_lens = [], []
    for r, (L, n) in enumerate(zip(lengths, tokens_per_request)):
        pad = padded_tail[r] if padded_tail is not None else 0
        for j in range(n):
            req_idx.append(r)
            seq_lens.append(0 if j >= n - pad else max(0, L - (n - 1 - j)))
    T = len(req_idx)
    w = Workload(name=name, T=T, R=R, Hq=Hq, Hkv=Hkv, D=D, Hi=Hi, Di=Di, NB=NB, P=P, K=K,
                 block_size=BLOCK_SIZE, dense=dense, block_table=table,
                 req_idx=torch.tensor(req_idx, dtype=torch.int32),
                 seq_lens=torch.tensor(seq_lens, dtype=torch.int32),
                 sm_scale=1.0 / math.sqrt(D), idx_scale=1.0 / math.sqrt(Di),
                 tokens_per_request=list(tokens_per_request), request_lengths=list(lengths))
    n_slots = P * BLOCK_SIZE
    all_slots = torch.cat([_request_slots(pages, L) for pages, L in zip(owned, lengths)])

    if with_kv:
        if q_dist == "student_t3":
            q = _student_t3((T, Hq, D), g)
        else:
            q = torch.randn((T, Hq, D), generator=g)
        w.q = q.to(dtype)
        for name_, attr in (("k", "k_cache"), ("v", "v_cache")):
            vals = torch.randn((all_slots.numel(), Hkv, D), generator=g)
            if kv_dtype == "bf16":
                cache = _poison_e4m3((n_slots, Hkv, D), g).to(torch.bfloat16)  # +/-448.0
                cache.index_copy_(0, all_slots, vals.to(torch.bfloat16))
                scale = 1.0
            else:
                codes, scale = _to_e4m3(vals)
                cache = _poison_e4m3((n_slots, Hkv, D), g)
                cache.view(torch.uint8).index_copy_(0, all_slots, codes.view(torch.uint8))
            del vals
            setattr(w, attr, cache)
            setattr(w, name_ + "_scale", scale)

    if with_index:
        w.q_idx = torch.randn((T, Hi, Di), generator=g).to(idx_dtype)
        kidx = torch.full((n_slots, 1, Di), INDEX_POISON, dtype=idx_dtype)
        kidx.index_copy_(0, all_slots, torch.randn((all_slots.numel(), 1, Di), generator=g).to(idx_dtype))
        w.k_idx_cache = kidx
    return w


def make_prefill(name: str, *, offsets: Sequence[int], chunk: int, Di: int = 128, Hi: int = 1,
                 NB: int = 128, P: int, K: int, seed: int,
                 idx_dtype: torch.dtype = torch.bfloat16) -> Workload:
    """Prefill score-to-selection batch: sequence s has ``chunk`` query tokens at
    absolute positions ``offsets[s] .. offsets[s]+chunk-1``; query token at
    position p sees keys 0..p (``seq_len = p + 1``)."""
    g = torch.Generator().manual_seed(seed)
    lengths = [o + chunk for o in offsets]
    table, owned = _pages_for(lengths, P, NB, g)
    req_idx, seq_lens = [], []
    for s, o in enumerate(offsets):
        for i in range(chunk):
            req_idx.append(s)
            seq_lens.append(o + i + 1)
    T = len(req_idx)
    w = Workload(name=name, T=T, R=len(offsets), Hq=0, Hkv=0, D=0, Hi=Hi, Di=Di, NB=NB, P=P, K=K,
                 block_size=BLOCK_SIZE, dense=False, block_table=table,
                 req_idx=torch.tensor(req_idx, dtype=torch.int32),
                 seq_lens=torch.tensor(seq_lens, dtype=torch.int32),
                 idx_scale=1.0 / math.sqrt(Di), tokens_per_request=[chunk] * len(offsets),
                 request_lengths=lengths)
    n_slots = P * BLOCK_SIZE
    all_slots = torch.cat([_request_slots(pages, L) for pages, L in zip(owned, lengths)])
    w.q_idx = torch.randn((T, Hi, Di), generator=g).to(idx_dtype)
    kidx = torch.full((n_slots, 1, Di), INDEX_POISON, dtype=idx_dtype)
    kidx.index_copy_(0, all_slots, torch.randn((all_slots.numel(), 1, Di), generator=g).to(idx_dtype))
    w.k_idx_cache = kidx
    return w


# ----------------------------------------------------------------- configs

# descriptions of the five workloads, by the number bench.py --config takes
CONFIG_NAMES = {
    1: "tiny sparse decode (B=1, 8/1 heads, D=64, Di=32, L=512, top-2, fp32 inputs)",
    2: "EAGLE-style verification decode (4 rows x 4 tokens, 64/8 heads, D=128, L~U[2048,16384], top-16)",
    3: "dense paged decode (16 rows x 1 token, 64/8 heads, D=128, L=16384, all blocks)",
    4: "batched paged prefill score-to-selection (8 x 512 tokens, Di=128, causal, top-32)",
    5: "stress sparse decode (64 rows x {1,4,8,16} tokens, L log-uniform [256,16384], top-64, t3 queries)",
}
WORKLOAD_NAMES = {1: "tiny_sparse_decode", 2: "verification_decode", 3: "dense_decode", 4: "prefill_score_select",
                  5: "stress_decode"}


def with_fp8_index(w: Workload) -> Workload:
    """The same batch with its index cache stored as FP8-E4M3 under a static
    scalar scale max|x|/448; the scale is folded into idx_scale, as a caller
    of msa_block_score does for an FP8 index cache."""
    out = Workload(**{k: getattr(w, k) for k in w.__dataclass_fields__})
    codes, scale = _to_e4m3(w.k_idx_cache.float())
    out.k_idx_cache = codes
    out.idx_scale = w.idx_scale * scale
    return out


def config(cfg: int, seed: Optional[int] = None, kv_dtype: str = "e4m3") -> Workload:
    """The five benchmark configurations, full size (``kv_dtype="bf16"``: the
    same batch shapes over a dense BF16 K/V cache)."""
    seed = 1000 + cfg if seed is None else seed
    if kv_dtype != "e4m3" and cfg in (1, 4):
        raise ValueError("configuration %d has no BF16 K/V variant" % cfg)
    if cfg == 1:
        return make_decode("tiny_sparse_decode", lengths=[512], tokens_per_request=[1], Hq=8, Hkv=1, D=64,
                           Hi=1, Di=32, NB=4, P=16, K=2, dtype=torch.float32, seed=seed)
    if cfg == 2:
        g = torch.Generator().manual_seed(seed + 7919)
        lengths = torch.randint(2048, 16385, (4,), generator=g).tolist()
        return make_decode("verification_decode", lengths=lengths, tokens_per_request=[4] * 4, Hq=64, Hkv=8, D=128,
                           Di=128, NB=128, P=1024, K=16, seed=seed, kv_dtype=kv_dtype)
    if cfg == 3:
        return make_decode("dense_decode", lengths=[16384] * 16, tokens_per_request=[1] * 16, Hq=64, Hkv=8,
                           D=128, NB=128, P=2048, K=0, seed=seed, dense=True, with_index=False, kv_dtype=kv_dtype)
    if cfg == 4:
        g = torch.Generator().manual_seed(seed + 7919)
        offsets = torch.randint(0, 15873, (8,), generator=g).tolist()
        return make_prefill("prefill_score_select", offsets=offsets, chunk=512, P=1024, K=32, seed=seed)
    if cfg == 5:
        return stress(seed=seed, kv_dtype=kv_dtype)
    raise ValueError("unknown config %r" % cfg)


def stress(seed: int = 1005, rows: int = 64, P: int = 8192, K: int = 64,
           min_len: int = 256, max_len: int = 16384, kv_dtype: str = "e4m3") -> Workload:
    """Config 5 recipe, parameterised so tests can draw smaller copies."""
    g = torch.Generator().manual_seed(seed + 7919)
    buckets = torch.tensor([1, 4, 8, 16])
    n = buckets[torch.randint(0, 4, (rows,), generator=g)].tolist()
    u = torch.rand((rows,), generator=g, dtype=torch.float64)
    lengths = torch.exp(math.log(min_len) + u * (math.log(max_len) - math.log(min_len)))
    lengths = [max(int(L), nr) for L, nr in zip(lengths.round().tolist(), n)]
    n_pad = max(1, round(0.05 * rows))
    pad_rows = torch.randperm(rows, generator=g)[:n_pad].tolist()
    padded = [0] * rows
    for r in pad_rows:
        padded[r] = int(torch.randint(1, n[r] + 1, (1,), generator=g))
    return make_decode("stress_decode" if rows == 64 else "stress%d" % rows, lengths=lengths,
                       tokens_per_request=n, Hq=64, Hkv=8, D=128, Di=128, NB=128, P=P, K=K,
                       seed=seed, q_dist="student_t3", padded_tail=padded, kv_dtype=kv_dtype)


# ------------------------------------------------------- dense attention

@dataclass
class DenseAttention:
    """Inputs of one dense GQA attention call (CPU tensors): T query tokens
    over S keys that are not paged."""

    name: str
    T: int
    S: int
    Hq: int
    Hkv: int
    D: int
    causal: bool
    q: torch.Tensor  # [T, Hq, D]
    k: torch.Tensor  # [S, Hkv, D]
    v: torch.Tensor  # [S, Hkv, D]
    sm_scale: float

    def to(self, device) -> "DenseAttention":
        out = DenseAttention(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for name in ("q", "k", "v"):
            setattr(out, name, getattr(self, name).to(device))
        return out


def make_dense(name: str, *, T: int, S: int, Hq: int, Hkv: int, D: int, causal: bool, seed: int,
               dtype: torch.dtype = torch.bfloat16, q_dist: str = "normal") -> DenseAttention:
    """q, k, v drawn N(0, 1) (q optionally Student-t with 3 degrees of
    freedom), cast to ``dtype``; ``sm_scale = 1/sqrt(D)``."""
    g = torch.Generator().manual_seed(seed)
    q = _student_t3((T, Hq, D), g) if q_dist == "student_t3" else torch.randn((T, Hq, D), generator=g)
    k = torch.randn((S, Hkv, D), generator=g)
    v = torch.randn((S, Hkv, D), generator=g)
    return DenseAttention(name=name, T=T, S=S, Hq=Hq, Hkv=Hkv, D=D, causal=causal, q=q.to(dtype),
                          k=k.to(dtype), v=v.to(dtype), sm_scale=1.0 / math.sqrt(D))


DENSE_NAME = ("dense causal GQA prefill chunk (512 query tokens after a 7680-token prefix, S=8192, "
              "64/8 heads, D=128, bf16)")


def dense_prefill(seed: int = 1006) -> DenseAttention:
    """Dense-attention workload: one 512-token prefill chunk of a sequence
    whose first 7680 tokens are already cached (the chunk length and head
    shape of the prefill and decode configurations above)."""
    return make_dense("dense_prefill", T=512, S=8192, Hq=64, Hkv=8, D=128, causal=True, seed=seed)


# ------------------------------------------- prefill score-to-selection (V2)

@dataclass
class PrefillBatch:
    """Inputs of one fused prefill score-to-selection call (CPU tensors):
    a ragged batch of query chunks over a paged index cache."""

    name: str
    B: int
    Hi: int
    Di: int
    NB: int
    P: int
    topk: int
    block_size_q: int
    init_blocks: int
    local_blocks: int
    scale: float
    n_rows: int  # query blocks over the batch (all_seqblock_q)
    q_idx: torch.Tensor  # [total_q, Hi, Di]
    k_idx_cache: torch.Tensor  # [P*BS, 1, Di]
    block_table: torch.Tensor  # int32 [R, NB] (R >= B; rows in shuffled order)
    slot_ids: torch.Tensor  # int32 [B]: page-table row of each sequence
    cu_seqlens: torch.Tensor  # int32 [B+1]: query token offsets
    seq_lens: torch.Tensor  # int32 [B]: keys of each sequence, chunk included
    prefix_lens: torch.Tensor  # int32 [B]: keys before the chunk
    cu_seqblocks_q: torch.Tensor  # int32 [B+1]: query block offsets

    def to(self, device) -> "PrefillBatch":
        out = PrefillBatch(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for name in ("q_idx", "k_idx_cache", "block_table", "slot_ids", "cu_seqlens", "seq_lens", "prefix_lens",
                     "cu_seqblocks_q"):
            setattr(out, name, getattr(self, name).to(device))
        return out


def make_prefill_batch(name: str, *, offsets: Sequence[int], chunks: Sequence[int], block_size_q: int,
                       topk: int, init_blocks: int = 0, local_blocks: int = 0, Hi: int = 1, Di: int = 128,
                       NB: int = 128, P: int = 1024, spare_rows: int = 2, seed: int,
                       idx_dtype: torch.dtype = torch.bfloat16) -> PrefillBatch:
    """Sequence b has ``chunks[b]`` query tokens at positions ``offsets[b]`` ..
    ``offsets[b] + chunks[b] - 1`` and ``offsets[b] + chunks[b]`` keys; its
    page-table row is drawn from a shuffled table with ``spare_rows`` rows
    that no sequence owns (their entries point at unowned pages).  Index
    queries and keys are N(0, 1); unowned index slots hold the finite poison.
    ``scale = 1/sqrt(Di)``."""
    g = torch.Generator().manual_seed(seed)
    B = len(offsets)
    lengths = [o + c for o, c in zip(offsets, chunks)]
    table, owned = _pages_for(lengths + [0] * spare_rows, P, NB, g)
    perm = torch.randperm(B + spare_rows, generator=g)
    block_table = table[perm].contiguous()
    slot_ids = torch.argsort(perm)[:B].to(torch.int32)  # row of sequence b in the shuffled table
    cu = [0]
    cub = [0]
    for c in chunks:
        cu.append(cu[-1] + c)
        cub.append(cub[-1] + (c + block_size_q - 1) // block_size_q)
    total_q = cu[-1]
    n_slots = P * BLOCK_SIZE
    all_slots = torch.cat([_request_slots(pages, L) for pages, L in zip(owned[:B], lengths)])
    q_idx = torch.randn((total_q, Hi, Di), generator=g).to(idx_dtype)
    kidx = torch.full((n_slots, 1, Di), INDEX_POISON, dtype=idx_dtype)
    kidx.index_copy_(0, all_slots, torch.randn((all_slots.numel(), 1, Di), generator=g).to(idx_dtype))
    return PrefillBatch(name=name, B=B, Hi=Hi, Di=Di, NB=NB, P=P, topk=topk, block_size_q=block_size_q,
                        init_blocks=init_blocks, local_blocks=local_blocks, scale=1.0 / math.sqrt(Di),
                        n_rows=cub[-1], q_idx=q_idx, k_idx_cache=kidx, block_table=block_table,
                        slot_ids=slot_ids, cu_seqlens=torch.tensor(cu, dtype=torch.int32),
                        seq_lens=torch.tensor(lengths, dtype=torch.int32),
                        prefix_lens=torch.tensor(list(offsets), dtype=torch.int32),
                        cu_seqblocks_q=torch.tensor(cub, dtype=torch.int32))


PREFILL_BATCH_NAME = ("batched paged prefill score-to-selection, one call (8 x 512-token chunks at offsets "
                      "~U[0,15872], Di=128, query blocks of 64 tokens, 1 initial + 2 local blocks, top-32)")


def prefill_batch(seed: int = 1004, block_size_q: int = 64, init_blocks: int = 1, local_blocks: int = 2,
                  topk: int = 32) -> PrefillBatch:
    """The batched prefill configuration's sequences (same offsets as the
    per-token score-to-selection workload) as one fused call."""
    g = torch.Generator().manual_seed(seed + 7919)
    offsets = torch.randint(0, 15873, (8,), generator=g).tolist()
    return make_prefill_batch("prefill_batch", offsets=offsets, chunks=[512] * 8, block_size_q=block_size_q,
                              topk=topk, init_blocks=init_blocks, local_blocks=local_blocks, seed=seed)
