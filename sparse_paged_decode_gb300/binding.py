"""Thin ctypes binding of libspd.so: torch tensors in, C ABI call, error check.

Argument marshalling only -- every step of every call runs in the CUDA
library.  Importing this module loads ``libspd.so`` (built in-tree by
``sparse_paged_decode_gb300.build``) and raises if it is missing: there is no
CPU or PyTorch fallback.  Each function enqueues on the current torch CUDA
stream unless a stream is given, returns None, and raises ``SpdError`` when
the library rejects the call (see ``include/spd.h``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB_PATH

__all__ = [
    "SpdError",
    "msa_block_score",
    "msa_select_topk",
    "paged_sparse_decode_attention",
    "paged_decode_attention",
    "paged_sparse_decode_attention_noalloc",
    "attention_sdpa",
    "msa_prefill_block_score",
    "prefill_workspace_bytes",
    "decode_workspace_bytes",
    "launch_count",
    "set_attention_kernel",
    "set_kernel_policy",
    "workspace_status",
    "library_path",
    "lib",
]

SPD_F32, SPD_BF16, SPD_F16, SPD_E4M3, SPD_I32 = 0, 1, 2, 3, 4
_DTYPES = {
    torch.float32: SPD_F32,
    torch.bfloat16: SPD_BF16,
    torch.float16: SPD_F16,
    torch.float8_e4m3fn: SPD_E4M3,
    torch.int32: SPD_I32,
}


class SpdError(RuntimeError):
    """A call rejected by libspd (validation failure or launch error)."""

    def __init__(self, code: int, msg: str):
        super().__init__("spd error %d: %s" % (code, msg))
        self.code = code


class SpdTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 4),
        ("stride", ctypes.c_int64 * 4),
    ]


def library_path() -> str:
    return LIB_PATH


def _load():
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            "libspd.so is not built (%s); run `python -m sparse_paged_decode_gb300.build` "
            "or __graft_entry__.build() -- there is no fallback implementation" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(SpdTensor)
    vp, f32, i32, sz = ctypes.c_void_p, ctypes.c_float, ctypes.c_int32, ctypes.c_size_t
    L.msa_block_score.argtypes = [P, P, P, P, P, i32, P, f32, vp]
    L.msa_block_score.restype = None
    L.msa_select_topk.argtypes = [P, P, vp]
    L.msa_select_topk.restype = None
    L.paged_sparse_decode_attention.argtypes = [P, P, P, P, P, P, P, P, f32, i32, f32, f32, vp, sz, vp]
    L.paged_sparse_decode_attention.restype = None
    L.paged_sparse_decode_attention_noalloc.argtypes = [P, P, P, P, P, P, P, P, f32, i32, f32, f32, vp]
    L.paged_sparse_decode_attention_noalloc.restype = None
    L.paged_decode_attention.argtypes = [P, P, P, P, P, P, P, f32, i32, f32, f32, vp, sz, vp]
    L.paged_decode_attention.restype = None
    L.msa_prefill_block_score.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, f32, P, P, vp, sz, vp]
    L.msa_prefill_block_score.restype = None
    L.spd_prefill_workspace_bytes.argtypes = [ctypes.c_int64] * 3
    L.spd_prefill_workspace_bytes.restype = sz
    L.attention_sdpa.argtypes = [P, P, P, P, f32, i32, vp]
    L.attention_sdpa.restype = None
    L.spd_decode_workspace_bytes.argtypes = [ctypes.c_int64] * 5 + [i32]
    L.spd_decode_workspace_bytes.restype = sz
    L.spd_last_error.argtypes = [ctypes.c_char_p, sz]
    L.spd_last_error.restype = ctypes.c_int
    L.spd_set_attention_kernel.argtypes = [ctypes.c_int]
    L.spd_set_attention_kernel.restype = ctypes.c_int
    L.spd_set_kernel_policy.argtypes = [ctypes.c_int, ctypes.c_int]
    L.spd_set_kernel_policy.restype = ctypes.c_int
    L.spd_workspace_status.argtypes = [vp, vp]
    L.spd_workspace_status.restype = ctypes.c_int
    L.spd_launch_count.argtypes = []
    L.spd_launch_count.restype = ctypes.c_uint64
    L.spd_version.argtypes = []
    L.spd_version.restype = ctypes.c_char_p
    return L


lib = _load()


def _desc(t: Optional[torch.Tensor], name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype not in _DTYPES:
        raise TypeError("%s: dtype %s is not supported by libspd" % (name, t.dtype))
    if t.numel() > 0 and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dim() > 4:
        raise ValueError("%s has more than 4 dims" % name)
    d = SpdTensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return ctypes.byref(d)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check():
    buf = ctypes.create_string_buffer(512)
    code = lib.spd_last_error(buf, 512)
    if code != 0:
        raise SpdError(code, buf.value.decode(errors="replace"))


def msa_block_score(q_idx, k_idx_cache, block_table, seq_lens, req_idx, block_size, scores,
                    idx_scale, stream=None) -> None:
    """Stage 1: fill ``scores`` [Hi, T, NB] with block-max index scores."""
    lib.msa_block_score(_desc(q_idx, "q_idx"), _desc(k_idx_cache, "k_idx_cache"),
                        _desc(block_table, "block_table"), _desc(seq_lens, "seq_lens"),
                        _desc(req_idx, "req_idx"), int(block_size), _desc(scores, "scores"),
                        float(idx_scale), _stream(stream))
    _check()


def msa_select_topk(scores, topk_idx, stream=None) -> None:
    """Stage 2: fill ``topk_idx`` [Hi, T, K] with the top-K block ids per row."""
    lib.msa_select_topk(_desc(scores, "scores"), _desc(topk_idx, "topk_idx"), _stream(stream))
    _check()


def paged_sparse_decode_attention(q, k_cache, v_cache, block_table, seq_lens, req_idx, topk_idx, out,
                                  sm_scale, block_size, k_scale, v_scale, workspace, stream=None) -> None:
    """Stage 3: fill ``out`` [T, Hq, D] (bf16) with attention over the selected blocks.

    ``workspace`` is a CUDA uint8 tensor of at least ``decode_workspace_bytes`` bytes."""
    ws_ptr, ws_bytes = _workspace(workspace)
    lib.paged_sparse_decode_attention(
        _desc(q, "q"), _desc(k_cache, "k_cache"), _desc(v_cache, "v_cache"), _desc(block_table, "block_table"),
        _desc(seq_lens, "seq_lens"), _desc(req_idx, "req_idx"), _desc(topk_idx, "topk_idx"), _desc(out, "out"),
        float(sm_scale), int(block_size), float(k_scale), float(v_scale), ws_ptr, ws_bytes, _stream(stream))
    _check()


def paged_sparse_decode_attention_noalloc(q, k_cache, v_cache, block_table, seq_lens, req_idx, topk_idx, out,
                                          sm_scale, block_size, k_scale, v_scale, stream=None) -> None:
    """Stage 3 for callers that cannot allocate: no workspace argument, the
    library's built-in 16 MiB scratch is used instead (see include/spd.h for
    its limit and its sharing rules)."""
    lib.paged_sparse_decode_attention_noalloc(
        _desc(q, "q"), _desc(k_cache, "k_cache"), _desc(v_cache, "v_cache"), _desc(block_table, "block_table"),
        _desc(seq_lens, "seq_lens"), _desc(req_idx, "req_idx"), _desc(topk_idx, "topk_idx"), _desc(out, "out"),
        float(sm_scale), int(block_size), float(k_scale), float(v_scale), _stream(stream))
    _check()


def paged_decode_attention(q, k_cache, v_cache, block_table, seq_lens, req_idx, out, sm_scale, block_size,
                           k_scale, v_scale, workspace, stream=None) -> None:
    """Dense paged decode: attention over every block of each row."""
    ws_ptr, ws_bytes = _workspace(workspace)
    lib.paged_decode_attention(
        _desc(q, "q"), _desc(k_cache, "k_cache"), _desc(v_cache, "v_cache"), _desc(block_table, "block_table"),
        _desc(seq_lens, "seq_lens"), _desc(req_idx, "req_idx"), _desc(out, "out"), float(sm_scale),
        int(block_size), float(k_scale), float(v_scale), ws_ptr, ws_bytes, _stream(stream))
    _check()


def msa_prefill_block_score(q, index_k_cache, block_table, slot_ids, cu_seqlens, seq_lens, prefix_lens,
                            block_size_q, block_size_k, init_blocks, local_blocks, scale, cu_seqblocks_q, out_topk,
                            workspace, stream=None) -> None:
    """Fused prefill score-to-selection: fill ``out_topk`` [Hi, rows, topk]
    with the selected key blocks of every query block of a ragged batch.

    ``workspace`` is a CUDA uint8 tensor of at least
    ``prefill_workspace_bytes(total_q, Hi, NB)`` bytes."""
    ws_ptr, ws_bytes = _workspace(workspace)
    lib.msa_prefill_block_score(
        _desc(q, "q"), _desc(index_k_cache, "index_k_cache"), _desc(block_table, "block_table"),
        _desc(slot_ids, "slot_ids"), _desc(cu_seqlens, "cu_seqlens"), _desc(seq_lens, "seq_lens"),
        _desc(prefix_lens, "prefix_lens"), int(block_size_q), int(block_size_k), int(init_blocks),
        int(local_blocks), float(scale), _desc(cu_seqblocks_q, "cu_seqblocks_q"), _desc(out_topk, "out_topk"),
        ws_ptr, ws_bytes, _stream(stream))
    _check()


def prefill_workspace_bytes(total_q: int, Hi: int, NB: int) -> int:
    """Workspace bytes msa_prefill_block_score needs for these sizes."""
    return int(lib.spd_prefill_workspace_bytes(total_q, Hi, NB))


def attention_sdpa(q, k, v, out, sm_scale, causal, stream=None) -> None:
    """Dense GQA attention: fill ``out`` [T, Hq, D] from q [T, Hq, D] and
    k, v [S, Hkv, D]; with ``causal`` query t reads keys j <= t + S - T."""
    lib.attention_sdpa(_desc(q, "q"), _desc(k, "k"), _desc(v, "v"), _desc(out, "out"), float(sm_scale),
                       1 if causal else 0, _stream(stream))
    _check()


def _workspace(ws):
    if ws is None:
        return None, 0
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    return ws.data_ptr(), ws.numel() * ws.element_size()


def set_attention_kernel(policy: int) -> int:
    """0 = tensor-core kernel where it applies (default), 1 = general-layout
    kernel always.  Applies to this thread; returns the previous policy."""
    return int(lib.spd_set_attention_kernel(int(policy)))


STAGE_SCORE, STAGE_SELECT, STAGE_ATTENTION, STAGE_SDPA = 1, 2, 3, 4


def set_kernel_policy(stage: int, policy: int) -> int:
    """Kernel choice of one stage (1 score, 2 select, 3 attention, 4 dense
    attention) on this thread: 0 = specialised kernel where it applies
    (default), 1 = general-layout kernel always.  Returns the previous
    policy."""
    old = int(lib.spd_set_kernel_policy(int(stage), int(policy)))
    if old < 0:
        raise ValueError("unknown stage %r" % (stage,))
    return old


def workspace_status(workspace, stream=None) -> int:
    """Status word an attention call left in ``workspace`` (synchronises):
    0 ok, bit 0 a device-side wait timed out.  ``workspace=None`` reads the
    built-in scratch that paged_sparse_decode_attention_noalloc uses on the
    current device."""
    ptr = None if workspace is None else workspace.data_ptr()
    return int(lib.spd_workspace_status(ptr, _stream(stream)))


def launch_count() -> int:
    """Kernels enqueued by libspd in this process so far."""
    return int(lib.spd_launch_count())


def decode_workspace_bytes(T: int, Hq: int, Hkv: int, D: int, NB: int, block_size: int = 128) -> int:
    """Workspace bytes the attention calls need for these capacities."""
    return int(lib.spd_decode_workspace_bytes(T, Hq, Hkv, D, NB, block_size))
