"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Every mutation below is a plausible slip in ``oracle.c`` (a dropped scale, a
wrong GQA index, an off-by-one on ``seq_lens``, a reversed tie rule, a wrong
E4M3 bias ...).  The test compiles the mutated copy in a temporary directory
and runs the pins against it; a mutation that no pin catches would mean the
pins leave that part of the oracle unchecked.
"""
import os

import pytest

import oracle
from oracle_pins import PINS

MUTATIONS = [
    ("gqa index", "int64_t h = g / G;", "int64_t h = g % Hkv;"),
    ("score seq_len off by one", "if (tau >= L)\n                            break;",
     "if (tau > L)\n                            break;"),
    ("score drops idx_scale", "double s = dot * idx_scale;", "double s = dot;"),
    ("score min instead of max", "if (s > best)", "if (s < best || best == -INFINITY)"),
    ("attention seq_len off by one", "b * block_size + i < L; ++i)", "b * block_size + i <= L; ++i)"),
    ("attention drops k_scale", "z[j] = sm_scale * k_scale * dot;", "z[j] = sm_scale * dot;"),
    ("attention drops v_scale", "o[d] += w * v_scale *", "o[d] += w *"),
    ("attention ignores selection", "if (!selected[b] || b * block_size >= L)", "if (b * block_size >= L)"),
    ("top-k tie to higher id", "return (a->block > b->block) - (a->block < b->block);",
     "return (a->block < b->block) - (a->block > b->block);"),
    ("top-k pads with 0", "? cells[k].block : -1;", "? cells[k].block : 0;"),
    ("top-k keeps -inf", "if (!isnan(s) && s != -INFINITY) {", "if (!isnan(s)) {"),
    ("e4m3 bias", "mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);", "mag = ldexp(1.0 + (double)mant / 8.0, expo - 8);"),
    ("e4m3 subnormal scale", "mag = ldexp((double)mant / 8.0, -6);", "mag = ldexp((double)mant / 8.0, -7);"),
    ("bf16 shift", "uint32_t word = (uint32_t)bits << 16;", "uint32_t word = (uint32_t)bits << 15;"),
    ("clip to one block short", "L = NB * bs;", "L = (NB - 1) * bs;"),
    ("dense skips last block", "for (int64_t b = 0; b < NB && L > 0; ++b) {", "for (int64_t b = 0; b + 1 < NB && L > 0; ++b) {"),
    ("no max subtraction guard on empty", "if (n == 0) {", "if (n < 0) {"),
    ("attention reads every cache as e4m3", "load(k8, kv_dtype,", "load(k8, OR_E4M3,"),
    ("sdpa causal off by one", "n = t + (S - T) + 1;", "n = t + (S - T);"),
    ("sdpa causal aligned top-left", "n = t + (S - T) + 1;", "n = t + 1;"),
    ("sdpa gqa index", "int64_t kvh = g / G;", "int64_t kvh = g % Hkv;"),
    ("sdpa drops sm_scale", "z[j] = sm_scale * dot;", "z[j] = dot;"),
    ("sdpa ignores the causal flag", "if (causal) {", "if (0) {"),
    ("prefill visibility excludes the own position", "int64_t L = (int64_t)prefix_lens[b] + qb * block_size_q + 1;",
     "int64_t L = (int64_t)prefix_lens[b] + qb * block_size_q;"),
    ("prefill visibility through the block end", "int64_t L = (int64_t)prefix_lens[b] + qb * block_size_q + 1;",
     "int64_t L = (int64_t)prefix_lens[b] + (qb + 1) * block_size_q;"),
    ("prefill local blocks off by one", "kb >= nvis - local_blocks);", "kb > nvis - local_blocks);"),
    ("prefill init ignores visibility", "forced[kb] = kb < nvis && (kb < init_blocks || kb >= nvis - local_blocks);",
     "forced[kb] = kb < init_blocks || (kb < nvis && kb >= nvis - local_blocks);"),
    ("prefill query block is its first token", "int64_t t1 = t0 + block_size_q;", "int64_t t1 = t0 + 1;"),
    ("prefill ranks the policy blocks again", "if (forced[kb] || isnan(s[kb]) || s[kb] == -INFINITY)",
     "if (isnan(s[kb]) || s[kb] == -INFINITY)"),
    ("prefill ignores slot_ids", "int64_t r = slot_ids[b];", "int64_t r = b;"),
    ("sdpa drops the first value", "o[d] += w * load(v, dtype,", "o[d] += (j > 0) * w * load(v, dtype,"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(tmp_path, name, old, new):
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, "mutation anchor not found exactly once: %r" % old
    m = oracle.mutant(src.replace(old, new), workdir=str(tmp_path))
    caught = []
    for pin in PINS:
        try:
            pin(m)
        except (AssertionError, ValueError, RuntimeError) as e:  # noqa: PERF203
            caught.append(pin.__name__)
    assert caught, "planted mistake %r passed every pin" % name
