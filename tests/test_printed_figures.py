"""The figures the pages print that fix parts of the format and of the
workloads (tests/golden/printed_figures.txt, each line with its passage),
checked against the oracle's byte accounting and the input recipe."""
import os
from fractions import Fraction

import numpy as np

from bit_kv_cache_13_gb300 import inputs
from oracle import bgtq, int2

HERE = os.path.dirname(os.path.abspath(__file__))


def _figures():
    out = {}
    with open(os.path.join(HERE, "golden", "printed_figures.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = (x.strip() for x in line.split("="))
                out[key] = Fraction(val)
    return out


def test_int2_codes_are_an_eighth_of_bf16_and_half_of_int4():
    fig = _figures()
    acc = int2.storage_bytes_per_token_head()
    d = 128
    assert Fraction(acc["k_codes"], d * 2) == fig["int2_code_fraction_of_bf16"]   # bf16: 2 bytes per channel
    assert Fraction(acc["k_codes"], d // 2) == fig["int2_code_fraction_of_int4"]  # int4: half a byte
    assert Fraction(acc["k_codes"] + acc["v_codes"], acc["bf16_kv"]) == fig["int2_code_fraction_of_bf16"]


def test_block_gtq_budget_is_the_printed_average_width():
    fig = _figures()
    extra = inputs.SPECS["bgtq"].extra
    assert Fraction(extra["avg_bits"]) == fig["bgtq_average_bits"]
    # the greedy allocation spends avg_bits per dimension: 64 blocks of 2 dims
    rng = np.random.default_rng(0)
    w = bgtq.greedy_allocate(rng.lognormal(0, 2, 64), extra["b_min"], extra["b_max"], 64 * extra["avg_bits"])
    assert Fraction(int(2 * w.sum()), 128) == fig["bgtq_average_bits"]


def test_window_workload_is_the_printed_protection():
    fig = _figures()
    assert inputs.WINDOW_SINK == fig["window_sink_tokens"]
    assert inputs.WINDOW_RECENT == fig["window_recent_tokens"]
