"""CPU oracle for the sparse paged decode path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and shares no code
with it: the oracle is plain C (``oracle.c``), compiled with gcc, evaluated in
fp64, with its own FP8-E4M3 and BF16 decoders.

What each function computes, and the page passage it follows, is written in
``oracle.c``.  This module only marshals arrays: it copies inputs into
contiguous buffers of their raw element bits (bf16 -> uint16, e4m3 -> uint8)
and lets the C code decode them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
DEFAULT_LIB = os.path.join(_HERE, "liboracle.so")

# element type codes understood by oracle.c
OR_F32, OR_BF16, OR_F16, OR_E4M3, OR_I32 = 0, 1, 2, 3, 4

_CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(out_path: str = DEFAULT_LIB, source: str = SOURCE) -> str:
    """Compile ``source`` into a shared library at ``out_path`` with gcc."""
    tmp = out_path + ".tmp%d" % os.getpid()
    cmd = ["gcc", *_CFLAGS, source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def _needs_build(lib_path: str, source: str) -> bool:
    return (not os.path.exists(lib_path)) or os.path.getmtime(lib_path) < os.path.getmtime(source)


def _raw(x, kind: str):
    """(contiguous numpy buffer of raw element bits, dtype code) for a tensor/array."""
    try:
        import torch
    except ImportError:  # pragma: no cover - torch is always present here
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().to("cpu")
        if x.dtype == torch.bfloat16:
            return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16)), OR_BF16
        if x.dtype == torch.float16:
            return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16)), OR_F16
        if x.dtype == torch.float8_e4m3fn:
            return np.ascontiguousarray(x.contiguous().view(torch.uint8).numpy()), OR_E4M3
        if x.dtype == torch.uint8 and kind == "e4m3":
            return np.ascontiguousarray(x.contiguous().numpy()), OR_E4M3
        if x.dtype == torch.float32:
            return np.ascontiguousarray(x.contiguous().numpy()), OR_F32
        if x.dtype == torch.int32:
            return np.ascontiguousarray(x.contiguous().numpy()), OR_I32
        raise TypeError("oracle: unsupported tensor dtype %s" % x.dtype)
    a = np.asarray(x)
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), OR_F32
    if a.dtype == np.uint8 and kind == "e4m3":
        return np.ascontiguousarray(a), OR_E4M3
    if a.dtype == np.int32:
        return np.ascontiguousarray(a), OR_I32
    raise TypeError("oracle: unsupported array dtype %s" % a.dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes front end of one compiled copy of ``oracle.c``."""

    def __init__(self, lib_path: str = DEFAULT_LIB, source: str = SOURCE):
        if lib_path == DEFAULT_LIB and _needs_build(lib_path, source):
            build(lib_path, source)
        self.lib = ctypes.CDLL(lib_path)
        L = self.lib
        i64, vp, dbl, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_value.restype = dbl
        L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_value.restype = dbl
        L.oracle_f16_value.argtypes = [ctypes.c_uint16]
        L.oracle_f16_value.restype = dbl
        L.oracle_block_score.argtypes = [vp, c_int, i64, i64, i64, vp, c_int, i64, vp, i64, i64,
                                         vp, vp, dbl, i64, vp]
        L.oracle_block_score.restype = c_int
        L.oracle_select_topk.argtypes = [vp, i64, i64, i64, vp]
        L.oracle_select_topk.restype = c_int
        L.oracle_paged_attention.argtypes = [vp, c_int, i64, i64, i64, vp, vp, c_int, i64, i64, vp, i64, i64,
                                             vp, vp, vp, i64, dbl, dbl, dbl, i64, vp]
        L.oracle_paged_attention.restype = c_int
        L.oracle_sdpa.argtypes = [vp, vp, vp, c_int, i64, i64, i64, i64, i64, dbl, c_int, vp]
        L.oracle_sdpa.restype = c_int
        L.oracle_prefill_topk.argtypes = [vp, c_int, i64, i64, i64, vp, c_int, i64, vp, i64, i64,
                                          vp, vp, vp, vp, vp, i64, i64, i64, i64, dbl, i64, i64, i64, vp, vp]
        L.oracle_prefill_topk.restype = c_int

    # -- decoders ----------------------------------------------------------
    def e4m3_value(self, code: int) -> float:
        return self.lib.oracle_e4m3_value(int(code) & 0xFF)

    def bf16_value(self, bits: int) -> float:
        return self.lib.oracle_bf16_value(int(bits) & 0xFFFF)

    def f16_value(self, bits: int) -> float:
        return self.lib.oracle_f16_value(int(bits) & 0xFFFF)

    # -- stage 1 -----------------------------------------------------------
    def block_score(self, q_idx, k_idx_cache, block_table, req_idx, seq_lens,
                    idx_scale: float, block_size: int = 128) -> np.ndarray:
        """Score sheet [Hi, T, NB] (fp64); see oracle_block_score in oracle.c."""
        q, qdt = _raw(q_idx, "float")
        k, kdt = _raw(k_idx_cache, "float")
        bt, _ = _raw(block_table, "int")
        ri, _ = _raw(req_idx, "int")
        sl, _ = _raw(seq_lens, "int")
        T, Hi, Di = q.shape
        n_slots = k.shape[0]
        if k.ndim != 3 or k.shape[1] != 1 or k.shape[2] != Di:
            raise ValueError("oracle: index cache must be [slots, 1, Di]")
        R, NB = bt.shape
        out = np.empty((Hi, T, NB), dtype=np.float64)
        rc = self.lib.oracle_block_score(_ptr(q), qdt, T, Hi, Di, _ptr(k), kdt, n_slots,
                                         _ptr(bt), R, NB, _ptr(ri), _ptr(sl),
                                         float(idx_scale), int(block_size), _ptr(out))
        if rc:
            raise RuntimeError("oracle_block_score failed")
        return out

    # -- stage 2 -----------------------------------------------------------
    def select_topk(self, scores, K: int) -> np.ndarray:
        """Top-K block ids per row of ``scores[..., NB]`` (int32, padded with -1)."""
        s = np.ascontiguousarray(np.asarray(scores, dtype=np.float64))
        lead = s.shape[:-1]
        NB = s.shape[-1]
        rows = int(np.prod(lead)) if lead else 1
        out = np.empty(lead + (K,), dtype=np.int32)
        rc = self.lib.oracle_select_topk(_ptr(s), rows, NB, int(K), _ptr(out))
        if rc:
            raise RuntimeError("oracle_select_topk failed")
        return out

    # -- stage 3 -----------------------------------------------------------
    def paged_attention(self, q, k_cache, v_cache, block_table, req_idx, seq_lens,
                        topk_idx, sm_scale: float, k_scale: float, v_scale: float,
                        block_size: int = 128) -> np.ndarray:
        """Attention output [T, Hq, D] (fp64); ``topk_idx=None`` means dense.
        The caches are FP8-E4M3 (float8 or uint8 codes) or BF16."""
        qa, qdt = _raw(q, "float")
        k8, kdt = _raw(k_cache, "e4m3")
        v8, vdt = _raw(v_cache, "e4m3")
        if kdt != vdt or kdt not in (OR_E4M3, OR_BF16):
            raise ValueError("oracle: K/V caches must both be E4M3 or both BF16")
        bt, _ = _raw(block_table, "int")
        ri, _ = _raw(req_idx, "int")
        sl, _ = _raw(seq_lens, "int")
        T, Hq, D = qa.shape
        n_slots, Hkv, Dk = k8.shape
        if Dk != D or v8.shape != k8.shape:
            raise ValueError("oracle: K/V cache shapes do not match q")
        R, NB = bt.shape
        if topk_idx is None:
            tk, K, tk_ptr = None, 0, None
        else:
            try:
                import torch
                if isinstance(topk_idx, torch.Tensor):
                    topk_idx = topk_idx.detach().cpu().numpy()
            except ImportError:  # pragma: no cover
                pass
            tk = np.asarray(topk_idx, dtype=np.int32)
            if tk.ndim != 3 or tk.shape[1] != T:
                raise ValueError("oracle: topk_idx must be [Hkv or 1, T, K]")
            tk = np.ascontiguousarray(np.broadcast_to(tk, (Hkv, T, tk.shape[2])))
            K = tk.shape[2]
            tk_ptr = _ptr(tk)
        out = np.empty((T, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_paged_attention(_ptr(qa), qdt, T, Hq, D, _ptr(k8), _ptr(v8), kdt, n_slots, Hkv,
                                             _ptr(bt), R, NB, _ptr(ri), _ptr(sl), tk_ptr, K,
                                             float(sm_scale), float(k_scale), float(v_scale),
                                             int(block_size), _ptr(out))
        if rc:
            raise RuntimeError("oracle_paged_attention failed")
        return out

    # -- dense attention ---------------------------------------------------
    def sdpa(self, q, k, v, sm_scale: float, causal: bool) -> np.ndarray:
        """Dense GQA attention output [T, Hq, D] (fp64); see oracle_sdpa."""
        qa, qdt = _raw(q, "float")
        ka, kdt = _raw(k, "float")
        va, vdt = _raw(v, "float")
        if not (qdt == kdt == vdt):
            raise ValueError("oracle: q, k and v must share one dtype")
        T, Hq, D = qa.shape
        S, Hkv, Dk = ka.shape
        if Dk != D or va.shape != ka.shape or Hkv < 1 or Hq % Hkv:
            raise ValueError("oracle: k/v must be [S, Hkv, D] with Hq divisible by Hkv")
        out = np.empty((T, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_sdpa(_ptr(qa), _ptr(ka), _ptr(va), qdt, T, S, Hq, Hkv, D,
                                  float(sm_scale), int(bool(causal)), _ptr(out))
        if rc:
            raise RuntimeError("oracle_sdpa failed")
        return out

    # -- prefill score-to-selection ------------------------------------------
    def prefill_topk(self, q_idx, k_idx_cache, block_table, slot_ids, cu_seqlens, seq_lens, prefix_lens,
                     cu_seqblocks_q, block_size_q: int, init_blocks: int, local_blocks: int, scale: float,
                     n_rows: int, topk: int, block_size: int = 128):
        """(topk ids [Hi, n_rows, topk] int32, block scores [Hi, n_rows, NB]
        fp64); see oracle_prefill_topk in oracle.c."""
        q, qdt = _raw(q_idx, "float")
        k, kdt = _raw(k_idx_cache, "float")
        bt, _ = _raw(block_table, "int")
        arrs = [_raw(x, "int")[0] for x in (slot_ids, cu_seqlens, seq_lens, prefix_lens, cu_seqblocks_q)]
        T, Hi, Di = q.shape
        if k.ndim != 3 or k.shape[1] != 1 or k.shape[2] != Di:
            raise ValueError("oracle: index cache must be [slots, 1, Di]")
        R, NB = bt.shape
        B = arrs[0].shape[0]
        if arrs[1].shape[0] != B + 1 or arrs[4].shape[0] != B + 1:
            raise ValueError("oracle: cu_seqlens and cu_seqblocks_q need B + 1 entries")
        out = np.empty((Hi, n_rows, topk), dtype=np.int32)
        sc = np.empty((Hi, n_rows, NB), dtype=np.float64)
        rc = self.lib.oracle_prefill_topk(_ptr(q), qdt, T, Hi, Di, _ptr(k), kdt, k.shape[0], _ptr(bt), R, NB,
                                          *[_ptr(a) for a in arrs], B, int(block_size_q), int(init_blocks),
                                          int(local_blocks), float(scale), int(block_size), int(n_rows),
                                          int(topk), _ptr(out), _ptr(sc))
        if rc:
            raise RuntimeError("oracle_prefill_topk failed")
        return out, sc


_default: Optional[Oracle] = None


def default() -> Oracle:
    """The oracle compiled from ``oracle.c`` next to this file (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def mutant(source_text: str, workdir: Optional[str] = None) -> Oracle:
    """An Oracle compiled from modified source text (for planted-mistake tests)."""
    d = workdir or tempfile.mkdtemp(prefix="oracle_mutant_")
    src = os.path.join(d, "oracle_mutant.c")
    with open(src, "w") as f:
        f.write(source_text)
    lib = os.path.join(d, "liboracle_mutant.so")
    build(lib, src)
    return Oracle(lib, src)
