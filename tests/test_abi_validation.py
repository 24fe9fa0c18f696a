"""Argument checks of the C ABI, on the host (no GPU needed).

Every decode and append entry point validates its arguments before it
touches CUDA and returns a status code, with the reason in
kvq_last_error(). These calls pass placeholder addresses that are never
dereferenced: each case fails validation first, so nothing is launched.
"""
import os

import pytest
import torch

from bit_kv_cache_13_gb300 import _lib, build

# Placeholder addresses must never reach a launch: on a machine with a GPU
# these host-side checks are skipped (the GPU tests cover the same paths
# with real buffers).
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="host-only checks with placeholder addresses")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, -1, -2, -3
A = 0x10000          # a 16-byte-aligned placeholder address
MIS = 0x10004        # not 16-byte aligned


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


def _err(lib) -> str:
    return lib.kvq_last_error().decode()


def _decode(lib, q=A, B=1, H_q=4, H_kv=1, d=128, cache=A, num_pages=10, bt=A, max_pages=4, ctx=A, rk=A, rv=A,
            out=A, ws=A, ws_bytes=1 << 20, splits=0):
    return lib.kvq_decode_attn_int2(q, B, H_q, H_kv, d, cache, num_pages, bt, max_pages, ctx, rk, rv, 0.1, out, ws,
                                    ws_bytes, splits, None)


@pytest.mark.parametrize("kw,status,text", [
    (dict(d=64), UNSUPPORTED, "d=64"),
    (dict(H_q=6, H_kv=4), INVALID, "H_q=6"),
    (dict(B=0), INVALID, "B=0"),
    (dict(num_pages=0), INVALID, "num_pages=0"),
    (dict(splits=-1), INVALID, "splits=-1"),
    (dict(H_q=16, H_kv=1), UNSUPPORTED, "group 16"),
    (dict(B=70000), UNSUPPORTED, "65535"),
    (dict(max_pages=(1 << 28) + 1), UNSUPPORTED, "above 2^28"),
    (dict(q=None), INVALID, "null pointer"),
    (dict(out=None), INVALID, "null pointer"),
    (dict(cache=MIS), INVALID, "alignment"),
    (dict(ws=MIS), INVALID, "alignment"),
    (dict(rv=MIS), INVALID, "alignment"),
    (dict(splits=300), INVALID, "300"),
    (dict(ws_bytes=64), WORKSPACE, "workspace"),
])
def test_decode_rejects_before_launch(lib, kw, status, text):
    assert _decode(lib, **kw) == status
    assert text in _err(lib)


def test_window_decode_needs_its_window_arguments(lib):
    args = [A, 1, 4, 1, 128, A, 10, A, 4, A, A, A, A]
    # win_k given, win_v missing
    st = lib.kvq_decode_attn_int2_window(*args, A, None, A, 8, 0.1, A, A, 1 << 20, 0, None)
    assert st == INVALID and "window needs" in _err(lib)
    st = lib.kvq_decode_attn_int2_window(*args, MIS, A, A, 8, 0.1, A, A, 1 << 20, 0, None)
    assert st == INVALID and "win_k and win_v" in _err(lib)
    st = lib.kvq_decode_attn_int2_window(*args, A, A, A, 0, 0.1, A, A, 1 << 20, 0, None)
    assert st == INVALID and "win_max" in _err(lib)


def _append(lib, n=4, H_kv=1, d=128, k=A, cache=A, num_pages=4, clip=None):
    if clip is None:
        return lib.kvq_append_int2(k, A, n, H_kv, d, A, A, A, A, cache, num_pages, None, None, None, None)
    return lib.kvq_append_int2_clip(k, A, n, H_kv, d, A, A, A, A, clip, cache, num_pages, None, None, None, None)


@pytest.mark.parametrize("kw,status,text", [
    (dict(d=96), UNSUPPORTED, "d=96"),
    (dict(n=-1), INVALID, "n_tok=-1"),
    (dict(H_kv=0), INVALID, "H_kv=0"),
    (dict(num_pages=0), INVALID, "num_pages=0"),
    (dict(H_kv=70000), UNSUPPORTED, "too large"),
    (dict(clip=0.0), INVALID, "clip ratio"),
    (dict(clip=1.5), INVALID, "clip ratio"),
    (dict(k=None), INVALID, "null pointer"),
    (dict(cache=MIS), INVALID, "16-byte"),
])
def test_append_rejects_before_launch(lib, kw, status, text):
    assert _append(lib, **kw) == status
    assert text in _err(lib)


def test_empty_append_is_a_no_op(lib):
    # no tokens: success without touching any pointer or the GPU
    assert lib.kvq_append_int2(None, None, 0, 1, 128, None, None, None, None, None, 4, None, None, None, None) == OK


def _bgtq_decode(lib, total_bits=192, v_bits=3, H_q=4, H_kv=1, q=A, ws_bytes=1 << 20, splits=0):
    return lib.bgtq_decode_attn(q, 1, H_q, H_kv, 128, A, 10, A, 4, A, A, total_bits, v_bits, A, A, A, 0.1, A, A,
                                ws_bytes, splits, None)


@pytest.mark.parametrize("kw,status,text", [
    (dict(v_bits=9), INVALID, "v_bits=9"),
    (dict(v_bits=0), INVALID, "v_bits=0"),
    (dict(total_bits=10), INVALID, "total_bits=10"),
    (dict(H_q=36, H_kv=4), UNSUPPORTED, "group 9"),
    (dict(q=None), INVALID, "null pointer"),
    (dict(splits=257), INVALID, "257"),
    (dict(ws_bytes=16), WORKSPACE, "workspace"),
])
def test_bgtq_decode_rejects_before_launch(lib, kw, status, text):
    assert _bgtq_decode(lib, **kw) == status
    assert text in _err(lib)
