"""The CPU oracle against its pins, and copies of the oracle with a planted
mistake against the same pins (each mistake must fail at least one)."""
import os

import pytest

import oracle
from oracle import build_oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle)


# (description, text in pkv_oracle.c, replacement).  Each text occurs once.
MISTAKES = [
    ("GQA head mapping", "int32_t g = h / (J->Hq / J->Hkv);", "int32_t g = h % J->Hkv;"),
    ("causal position off by one", "int64_t p = n_s - q_s + i;          /*",
     "int64_t p = n_s - q_s + i - 1;      /*"),
    ("dropped softmax scale", "scores[j] = J->scale * dot;", "scores[j] = dot;"),
    ("sign of the exponent", "double w = exp(scores[j] - m);", "double w = exp(m - scores[j]);"),
    ("page offset index", "  int64_t offset = j % J->block_size;\n  return",
     "  int64_t offset = j / J->block_size;\n  return"),
    ("slot formula operands", "slot[cu_seqlens_q[s] + i] = physical_block * block_size + offset;",
     "slot[cu_seqlens_q[s] + i] = offset * block_size + physical_block;"),
    ("V read from the K cache", "o[d] += w * load_cache(J->v_cache,", "o[d] += w * load_cache(J->k_cache,"),
    ("missing normalisation", "for (int32_t d = 0; d < J->D; ++d) o[d] /= l;", ""),
    ("e4m3 rounding mode", "double q = nearbyint(a / ldexp(1.0, e - 3));",
     "double q = floor(a / ldexp(1.0, e - 3));"),
    ("e4m3 exponent bias", "mag = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("append scale not inverted", "float inv_scale = 1.0f / scale;", "float inv_scale = scale;"),
    ("q/k operand transposed", "load_src(J->q, J->q_dtype, qbase + d) *",
     "load_src(J->q, J->q_dtype, qbase + (J->D - 1 - d)) *"),
    ("max over keys skipped", "if (scores[j] > m) m = scores[j];", "m = scores[0];"),
    ("sliding window off by one", "lo = p - J->window_left;", "lo = p - J->window_left + 1;"),
    ("soft cap on the unscaled dot", "scores[j] = J->soft_cap * tanh(scores[j] / J->soft_cap);",
     "scores[j] = J->soft_cap * tanh(dot / J->soft_cap);"),
]


@pytest.mark.parametrize("desc,old,new", MISTAKES, ids=[m[0] for m in MISTAKES])
def test_planted_mistake_is_caught(desc, old, new, tmp_path):
    src = open(build_oracle.SRC).read()
    assert src.count(old) == 1, desc
    lib = build_oracle.build_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    prev = oracle.use_library(lib)
    caught = []
    try:
        for pin in pins.ALL_PINS:
            try:
                pin(oracle)
            except Exception as e:  # AssertionError or a refused input
                caught.append((pin.__name__, type(e).__name__))
    finally:
        oracle.restore_library(prev)
    assert caught, f"no pin catches: {desc}"
