"""The C-ABI library builds, loads and exports every entry point that
include/kvq.h declares; host-only entry points work without a GPU."""
import os

import numpy as np
import pytest

from bit_kv_cache_13_gb300 import _lib, build
from oracle import bgtq


@pytest.fixture(scope="module")
def cpu_lib():
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


def test_exports_every_declared_symbol(cpu_lib):
    names = _lib.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(cpu_lib, n), n
    assert set(names) == set(_lib._SIGS), set(names) ^ set(_lib._SIGS)


def test_sizes(cpu_lib):
    assert _lib.kvq_int2_tile_bytes(128) == 1536
    assert _lib.kvq_int2_tile_bytes(64) == 0
    assert _lib.bgtq_tile_bytes(192, 3) == 16 * (48 + 16 + 48 + 2)
    assert _lib.bgtq_tile_bytes(192, 3) == bgtq.tile_layout(192, 3)["tile"]
    ws = _lib.kvq_decode_workspace_bytes(2, 8, 2, 100, 3)
    assert ws >= 2 * 8 * 3 * 132 * 4
    assert _lib.kvq_decode_workspace_bytes(0, 8, 2, 100, 3) == 0


@pytest.mark.parametrize("B,H_kv,pages,want", [
    (1, 8, 8192, 19),      # 128K batch 1: 8 x 19 = 152 CTAs, one wave
    (8, 8, 2048, 2),       # 32K batch 8: 64 (sequence, KV head) units, 128 CTAs
    (8, 8, 8192, 2),
    (64, 8, 256, 1),       # more units than SMs: one split each
    (1, 1, 16, 1),         # at least 32 pages per split
    (1, 1, 64, 2),
    (1, 1, 100000, 152),   # bounded by the SM count, then by 256
    (1, 2, 4096, 76),
])
def test_auto_splits_fill_one_wave(cpu_lib, B, H_kv, pages, want):
    s = _lib.kvq_decode_auto_splits(B, 4 * H_kv, H_kv, pages)
    assert s == want
    assert s * B * H_kv <= max(152, B * H_kv)          # never a second wave of CTAs of its own
    assert 1 <= s <= min(max(1, (pages + 31) // 32), 256)


def test_workspace_with_auto_splits_holds_every_entry_point(cpu_lib):
    """num_splits = 0 sizes the partials for the automatic choice of every
    decode call: the INT2 decode's slots (one per unit and page CTA, at most
    units + C - 1 with C = one CTA per SM (152 where no device is visible),
    at least one per unit and at most one per 32 pages), the BF16-window
    form's (whose units carry up to 256 more virtual pages, and one more
    slot each for the window), the decode step's (whose units carry up to 96
    more virtual pages) and Block-GTQ's per-unit splits."""
    nsm = 152
    for B, H_kv, pages in [(1, 8, 8192), (8, 8, 2048), (3, 2, 40), (64, 8, 256), (1, 1, 17)]:
        H_q = 4 * H_kv
        units = B * H_kv
        V = units * pages
        c_plain = min(max(min(nsm, -(-V // 32)), units), V)
        vw = units * (pages + (0 if pages < 96 else 256))  # the window's virtual pages, at most
        c_win = min(max(min(nsm, -(-vw // 32)), units), vw)
        vs = units * (pages + (0 if pages < 96 else 96))  # a decode step's virtual pages
        c_step = min(max(min(nsm, -(-vs // 32)), units), vs)
        slots = max(units + c_plain, 2 * units + c_win, units + c_step,
                    units * _lib.kvq_decode_auto_splits(B, H_q, H_kv, pages))
        header = 256 + -(-units * 4 // 256) * 256
        ws0 = _lib.kvq_decode_workspace_bytes(B, H_q, H_kv, pages, 0)
        assert ws0 == header + slots * 4 * 132 * 4
        # an explicit split count covers the plain and the window form
        for S in (1, 3, 40):
            assert _lib.kvq_decode_workspace_bytes(B, H_q, H_kv, pages, S) == header + (S + 2) * units * 4 * 132 * 4


def test_allocator_matches_oracle(cpu_lib):
    rng = np.random.default_rng(0)
    for trial in range(50):
        s = rng.lognormal(0, 2, 64)
        if trial % 5 == 0:
            s[rng.integers(0, 64, 8)] = s[0]          # ties
        bmin, bmax = [(1, 8), (2, 4), (1, 3)][trial % 3]
        total = int(rng.integers(64 * bmin, 64 * bmax + 10))
        got = _lib.bgtq_allocate(s, bmin, bmax, total)
        assert np.array_equal(got, bgtq.greedy_allocate(s, bmin, bmax, total))


def test_allocator_rejects_bad_arguments(cpu_lib):
    with pytest.raises(_lib.KvqError):
        _lib.bgtq_allocate(np.ones(4), 3, 2, 20)
    with pytest.raises(_lib.KvqError):
        _lib.bgtq_allocate(np.ones(4), 1, 8, 3)
    with pytest.raises(_lib.KvqError):
        _lib.bgtq_allocate(np.array([1.0, np.nan]), 1, 8, 4)


def test_codebooks_match_oracle(cpu_lib):
    table = bgtq.lloyd_max_table()
    for b in range(1, 9):
        got = _lib.bgtq_lloyd_max_codebook(b)
        want = table[b - 1, : 2 ** b]
        assert np.max(np.abs(got - want)) <= 1e-9, b
        # the fp32 tables both sides quantise against agree bit for bit
        for n in range(2, 129, 2):
            assert np.array_equal((got / np.sqrt(n)).astype(np.float32), (want / np.sqrt(n)).astype(np.float32)), (b, n)


def test_device_calls_reject_bad_arguments_before_launch(cpu_lib):
    L = cpu_lib
    # d != 128 and null pointers are refused on the host
    assert L.kvq_append_int2(None, None, 1, 1, 64, None, None, None, None, None, 1, None, None, None, None) == -2
    assert L.kvq_append_int2(None, None, 1, 1, 128, None, None, None, None, None, 1, None, None, None, None) == -1
    assert L.kvq_decode_attn_int2(None, 1, 12, 1, 128, None, 1, None, 1, None, None, None, 0.1, None, None, 0, 0,
                                  None) == -2
    assert L.kvq_decode_attn_int2(None, 1, 6, 4, 128, None, 1, None, 1, None, None, None, 0.1, None, None, 0, 0,
                                  None) == -1
    assert b"GQA" in L.kvq_last_error() or b"H_q" in L.kvq_last_error()
