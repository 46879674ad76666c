"""The C ABI library on the host (no GPU needed).

* libspd.so loads and exports every function that include/spd.h declares;
* host-side validation rejects malformed calls before any launch, with the
  error code the header documents.  Descriptors here carry fake device
  addresses: validation never dereferences them, and a call that passes
  validation is only enqueued, so without a GPU it reports SPD_ERR_CUDA.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spd.h")

SPD_OK, SPD_ERR_INVALID_ARGUMENT, SPD_ERR_UNSUPPORTED, SPD_ERR_WORKSPACE, SPD_ERR_ALIASING, SPD_ERR_CUDA = range(6)
F32, BF16, F16, E4M3, I32 = range(5)
ES = {F32: 4, BF16: 2, F16: 2, E4M3: 1, I32: 4}


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^SPD_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)


@pytest.fixture(scope="module")
def spd():
    from sparse_paged_decode_gb300 import binding

    return binding


def test_exports_every_declared_symbol(spd):
    names = declared_functions()
    assert set(names) >= {"msa_block_score", "msa_select_topk", "paged_sparse_decode_attention",
                          "paged_decode_attention", "spd_decode_workspace_bytes", "spd_last_error",
                          "spd_version"}
    for n in names:
        assert hasattr(spd.lib, n), n
    assert spd.lib.spd_version().startswith(b"spd ")


class Fake:
    """Descriptor with a fake, aligned device address and contiguous strides."""

    next_addr = 1 << 40

    def __init__(self, shape, dtype, strides=None, addr=None):
        from sparse_paged_decode_gb300.binding import SpdTensor

        self.d = SpdTensor()
        n = 1
        for s in shape:
            n *= s
        if addr is None:
            addr = Fake.next_addr
            Fake.next_addr += ((n * ES[dtype] + 4095) // 4096 + 1) * 4096
        self.d.data = addr
        self.d.dtype = dtype
        self.d.ndim = len(shape)
        if strides is None:
            strides, acc = [], 1
            for s in reversed(shape):
                strides.insert(0, acc)
                acc *= s
        for i, (s, st) in enumerate(zip(shape, strides)):
            self.d.shape[i] = s
            self.d.stride[i] = st

    def ref(self):
        return ctypes.byref(self.d)


def status(spd):
    buf = ctypes.create_string_buffer(512)
    return spd.lib.spd_last_error(buf, 512), buf.value.decode()


def attn_call(spd, T=4, Hq=8, Hkv=2, D=64, NB=4, P=8, K=2, q_dtype=BF16, out=None, ws_bytes=None,
              block_size=128, tk=True, k_strides=None, sm_scale=0.125, k_dtype=E4M3, v_dtype=E4M3):
    q = Fake((T, Hq, D), q_dtype)
    k = Fake((P * 128, Hkv, D), k_dtype, strides=k_strides)
    v = Fake((P * 128, Hkv, D), v_dtype)
    bt = Fake((2, NB), I32)
    sl = Fake((T,), I32)
    ri = Fake((T,), I32)
    topk = Fake((Hkv, T, K), I32, strides=(0, K, 1)) if tk else None
    o = out or Fake((T, Hq, D), BF16)
    need = spd.lib.spd_decode_workspace_bytes(T, Hq, Hkv, D, NB, 128)
    ws = Fake((need + 256,), E4M3)
    nb = need if ws_bytes is None else ws_bytes
    if tk:
        spd.lib.paged_sparse_decode_attention(q.ref(), k.ref(), v.ref(), bt.ref(), sl.ref(), ri.ref(), topk.ref(),
                                              o.ref(), sm_scale, block_size, 1.0, 1.0, ws.d.data, nb, None)
    else:
        spd.lib.paged_decode_attention(q.ref(), k.ref(), v.ref(), bt.ref(), sl.ref(), ri.ref(), o.ref(),
                                       sm_scale, block_size, 1.0, 1.0, ws.d.data, nb, None)
    return status(spd)


def test_valid_attention_call_reaches_launch(spd):
    for tk in (True, False):
        for kv in (E4M3, BF16):
            code, msg = attn_call(spd, tk=tk, k_dtype=kv, v_dtype=kv)
            # validation passed; the launch itself needs a GPU
            assert code in (SPD_OK, SPD_ERR_CUDA), msg


def test_attention_rejections(spd):
    assert attn_call(spd, block_size=64)[0] == SPD_ERR_UNSUPPORTED
    assert attn_call(spd, Hq=6, Hkv=4)[0] == SPD_ERR_UNSUPPORTED  # not divisible
    assert attn_call(spd, Hq=64, Hkv=2)[0] == SPD_ERR_UNSUPPORTED  # group of 32
    assert attn_call(spd, D=512)[0] == SPD_ERR_UNSUPPORTED
    assert attn_call(spd, q_dtype=I32)[0] == SPD_ERR_UNSUPPORTED
    # K and V caches must share their dtype; F16 / F32 caches are outside the domain
    assert attn_call(spd, k_dtype=BF16, v_dtype=E4M3)[0] == SPD_ERR_INVALID_ARGUMENT
    assert attn_call(spd, k_dtype=F16, v_dtype=F16)[0] == SPD_ERR_UNSUPPORTED
    assert attn_call(spd, ws_bytes=16)[0] == SPD_ERR_WORKSPACE
    assert attn_call(spd, k_strides=(2 * 64 * 2, 64 * 2, 2))[0] == SPD_ERR_UNSUPPORTED  # D not contiguous
    assert attn_call(spd, sm_scale=float("nan"))[0] == SPD_ERR_INVALID_ARGUMENT
    # an output whose strides make two cells share one element
    assert attn_call(spd, out=Fake((4, 8, 64), BF16, strides=(64, 8, 1)))[0] == SPD_ERR_ALIASING
    # wrong output shape
    assert attn_call(spd, out=Fake((4, 8, 32), BF16))[0] == SPD_ERR_INVALID_ARGUMENT


def sdpa_call(spd, T=5, S=9, Hq=8, Hkv=2, D=64, dtype=BF16, kv_dtype=None, out=None, sm_scale=0.125,
              causal=1, v_shape=None):
    q = Fake((T, Hq, D), dtype)
    k = Fake((S, Hkv, D), kv_dtype if kv_dtype is not None else dtype)
    v = Fake(v_shape or (S, Hkv, D), kv_dtype if kv_dtype is not None else dtype)
    o = out or Fake((T, Hq, D), BF16)
    spd.lib.attention_sdpa(q.ref(), k.ref(), v.ref(), o.ref(), sm_scale, causal, None)
    return status(spd)


def test_sdpa_validation(spd):
    for dt in (F32, BF16, F16):
        code, msg = sdpa_call(spd, dtype=dt)
        assert code in (SPD_OK, SPD_ERR_CUDA), msg
    assert sdpa_call(spd, T=0)[0] == SPD_OK  # nothing to write, nothing launched
    assert sdpa_call(spd, Hq=6, Hkv=4)[0] == SPD_ERR_UNSUPPORTED  # not divisible
    assert sdpa_call(spd, D=300)[0] == SPD_ERR_UNSUPPORTED
    assert sdpa_call(spd, dtype=E4M3)[0] == SPD_ERR_UNSUPPORTED
    assert sdpa_call(spd, kv_dtype=F16)[0] == SPD_ERR_UNSUPPORTED  # k/v dtype != q dtype
    assert sdpa_call(spd, v_shape=(8, 2, 64))[0] == SPD_ERR_INVALID_ARGUMENT
    assert sdpa_call(spd, sm_scale=float("inf"))[0] == SPD_ERR_INVALID_ARGUMENT
    assert sdpa_call(spd, out=Fake((5, 8, 32), BF16))[0] == SPD_ERR_INVALID_ARGUMENT
    assert sdpa_call(spd, out=Fake((5, 8, 64), BF16, strides=(64, 8, 1)))[0] == SPD_ERR_ALIASING
    q = Fake((5, 8, 64), BF16)
    k = Fake((9, 2, 64), BF16)
    v = Fake((9, 2, 64), BF16)
    spd.lib.attention_sdpa(q.ref(), k.ref(), v.ref(), Fake((5, 8, 64), BF16, addr=q.d.data).ref(), 0.1, 0, None)
    assert status(spd)[0] == SPD_ERR_ALIASING


def prefill_call(spd, total_q=20, Hi=2, Di=64, B=3, NB=4, P=8, rows=7, topk=4, q_dtype=BF16, k_dtype=None,
                 bsq=4, bsk=128, init=1, local=1, scale=0.125, ws_bytes=None, cu_len=None, out=None):
    q = Fake((total_q, Hi, Di), q_dtype)
    k = Fake((P * 128, 1, Di), k_dtype if k_dtype is not None else q_dtype)
    bt = Fake((B + 1, NB), I32)
    sid, sl, pre = Fake((B,), I32), Fake((B,), I32), Fake((B,), I32)
    cu_q = Fake(((B + 1) if cu_len is None else cu_len,), I32)
    cu_b = Fake((B + 1,), I32)
    o = out or Fake((Hi, rows, topk), I32)
    need = spd.lib.spd_prefill_workspace_bytes(total_q, Hi, NB)
    ws = Fake((need + 256,), E4M3)
    spd.lib.msa_prefill_block_score(q.ref(), k.ref(), bt.ref(), sid.ref(), cu_q.ref(), sl.ref(), pre.ref(), bsq, bsk,
                                    init, local, scale, cu_b.ref(), o.ref(), ws.d.data,
                                    need if ws_bytes is None else ws_bytes, None)
    return status(spd)


def test_prefill_validation(spd):
    for kd in (None, E4M3):
        code, msg = prefill_call(spd, k_dtype=kd)
        assert code in (SPD_OK, SPD_ERR_CUDA), msg
    assert prefill_call(spd, rows=0)[0] == SPD_OK  # no rows: nothing to write
    assert prefill_call(spd, bsk=64)[0] == SPD_ERR_UNSUPPORTED
    assert prefill_call(spd, bsq=0)[0] == SPD_ERR_INVALID_ARGUMENT
    assert prefill_call(spd, init=-1)[0] == SPD_ERR_INVALID_ARGUMENT
    assert prefill_call(spd, scale=-0.5)[0] == SPD_ERR_UNSUPPORTED
    assert prefill_call(spd, NB=2000)[0] == SPD_ERR_UNSUPPORTED
    assert prefill_call(spd, k_dtype=F16)[0] == SPD_ERR_UNSUPPORTED  # bf16 queries, f16 keys
    assert prefill_call(spd, cu_len=3)[0] == SPD_ERR_INVALID_ARGUMENT  # cu_seqlens needs B + 1 entries
    assert prefill_call(spd, topk=0)[0] == SPD_ERR_INVALID_ARGUMENT
    assert prefill_call(spd, ws_bytes=64)[0] == SPD_ERR_WORKSPACE
    assert prefill_call(spd, out=Fake((2, 7, 4), I32, strides=(4, 4, 1)))[0] == SPD_ERR_ALIASING
    assert prefill_call(spd, out=Fake((3, 7, 4), I32))[0] == SPD_ERR_INVALID_ARGUMENT  # Hi mismatch
    assert spd.lib.spd_prefill_workspace_bytes(4096, 1, 128) >= 4096 * 128 * 4 + 2 * 4096 * 4


def test_output_overlapping_input_rejected(spd):
    q = Fake((2, 1, 32), BF16)
    k = Fake((128, 1, 32), BF16)
    bt = Fake((1, 1), I32)
    sl = Fake((2,), I32)
    ri = Fake((2,), I32)
    out = Fake((1, 2, 1), F32, addr=k.d.data + 64)  # lands inside the index cache
    spd.lib.msa_block_score(q.ref(), k.ref(), bt.ref(), sl.ref(), ri.ref(), 128, out.ref(), 0.5, None)
    assert status(spd)[0] == SPD_ERR_ALIASING


def test_score_and_select_rejections(spd):
    q = Fake((3, 1, 32), BF16)
    k = Fake((256, 1, 32), BF16)
    bt = Fake((2, 2), I32)
    sl = Fake((3,), I32)
    ri = Fake((3,), I32)
    out = Fake((1, 3, 2), F32)

    def score(qq=q, kk=k, o=out, scale=0.5, bs=128, sll=sl):
        spd.lib.msa_block_score(qq.ref(), kk.ref(), bt.ref(), sll.ref(), ri.ref(), bs, o.ref(), scale, None)
        return status(spd)[0]

    assert score() in (SPD_OK, SPD_ERR_CUDA)
    assert score(scale=-1.0) == SPD_ERR_UNSUPPORTED
    assert score(scale=0.0) == SPD_ERR_UNSUPPORTED
    assert score(bs=256) == SPD_ERR_UNSUPPORTED
    assert score(kk=Fake((256, 2, 32), BF16)) == SPD_ERR_UNSUPPORTED  # two index key heads
    assert score(kk=Fake((256, 1, 32), F32)) == SPD_ERR_UNSUPPORTED  # dtype mismatch
    # an E4M3 index cache goes with any query dtype (validation passes; the launch needs a GPU)
    assert score(kk=Fake((256, 1, 32), E4M3)) in (SPD_OK, SPD_ERR_CUDA)
    assert score(qq=Fake((3, 1, 32), F32), kk=Fake((256, 1, 32), E4M3)) in (SPD_OK, SPD_ERR_CUDA)
    assert score(o=Fake((1, 3, 3), F32)) == SPD_ERR_INVALID_ARGUMENT
    assert score(sll=Fake((2,), I32)) == SPD_ERR_INVALID_ARGUMENT
    # select
    s = Fake((1, 3, 2), F32)
    tk = Fake((1, 3, 5), I32)
    spd.lib.msa_select_topk(s.ref(), tk.ref(), None)
    assert status(spd)[0] in (SPD_OK, SPD_ERR_CUDA)
    spd.lib.msa_select_topk(s.ref(), Fake((1, 3, 0), I32).ref(), None)
    assert status(spd)[0] == SPD_ERR_INVALID_ARGUMENT
    spd.lib.msa_select_topk(Fake((1, 3, 2000), F32).ref(), tk.ref(), None)
    assert status(spd)[0] == SPD_ERR_UNSUPPORTED


def test_null_descriptor_and_empty_batch(spd):
    spd.lib.msa_select_topk(None, None, None)
    assert status(spd)[0] == SPD_ERR_INVALID_ARGUMENT
    # T = 0: nothing to write, nothing launched, success
    code, msg = attn_call(spd, T=0)
    assert code == SPD_OK, msg


def test_workspace_size_depends_on_capacities_only(spd):
    f = spd.lib.spd_decode_workspace_bytes
    a = f(16, 64, 8, 128, 128, 128)
    assert a > 0 and a % 256 == 0
    assert f(32, 64, 8, 128, 128, 128) >= a
    assert f(16, 64, 8, 128, 128, 64) == 0


def test_binding_refuses_host_tensors_and_raises_library_errors(spd):
    """The Python binding never computes on the host: non-empty CPU tensors
    are refused before the library is called, and a call the library rejects
    raises SpdError carrying the documented code (empty tensors carry no
    device address, so validation runs without a GPU)."""
    import torch

    q = torch.zeros((2, 4, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        spd.attention_sdpa(q, q.clone(), q.clone(), q.clone(), 0.3, True, stream=0)
    e = lambda *shape, dt=torch.bfloat16: torch.empty(shape, dtype=dt)  # noqa: E731
    with pytest.raises(spd.SpdError) as err:  # Hq = 6 is not a multiple of Hkv = 4
        spd.attention_sdpa(e(0, 6, 8), e(0, 4, 8), e(0, 4, 8), e(0, 6, 8), 0.3, False, stream=0)
    assert err.value.code == SPD_ERR_UNSUPPORTED
    # a valid empty batch is accepted and launches nothing (stream 0: the
    # legacy default stream, never touched)
    with pytest.raises(ValueError, match="CUDA tensor"):  # k and v hold data: refused on the host
        spd.attention_sdpa(e(0, 8, 8), e(3, 2, 8), e(3, 2, 8), e(0, 8, 8), 0.3, True, stream=0)
    spd.attention_sdpa(e(0, 8, 8), e(0, 2, 8), e(0, 2, 8), e(0, 8, 8), 0.3, True, stream=0)


def test_status_query_without_a_gpu_keeps_the_last_error(spd):
    """spd_workspace_status is a diagnostic: with no device to read (here: no
    GPU, for a caller workspace and for the built-in scratch alike) it returns
    -1 and leaves the last call's recorded status untouched."""
    q = Fake((4, 8, 64), BF16)
    spd.lib.paged_decode_attention(q.ref(), None, None, None, None, None, None, ctypes.c_float(0.1), 128,
                                   ctypes.c_float(1.0), ctypes.c_float(1.0), None, ctypes.c_size_t(0), None)
    before = status(spd)
    assert before[0] == SPD_ERR_INVALID_ARGUMENT
    assert spd.lib.spd_workspace_status(None, None) == -1
    assert spd.lib.spd_workspace_status(ctypes.c_void_p(1 << 40), None) == -1
    assert status(spd) == before
