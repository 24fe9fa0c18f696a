"""ctypes binding of libkvq.so (include/kvq.h), same names as the C ABI.

Argument marshalling only: tensors are checked for device, dtype and
contiguity, their device pointers and the current CUDA stream are passed to
the library, and a non-zero status raises KvqError with the library's error
text.  Every step of the path runs in the library's kernels; there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvq.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "kvq.h")

_lib = None

P, I, I64, SZ, F, D = C.c_void_p, C.c_int, C.c_int64, C.c_size_t, C.c_float, C.c_double

_SIGS = {
    "kvq_last_error": ([], C.c_char_p),
    "kvq_int2_tile_bytes": ([I], SZ),
    "kvq_append_int2": ([P, P, I, I, I, P, P, P, P, P, I64, P, P, P, P], I),
    "kvq_decode_workspace_bytes": ([I, I, I, I, I], SZ),
    "kvq_decode_auto_splits": ([I, I, I, I], I),
    "kvq_decode_attn_int2": ([P, I, I, I, I, P, I64, P, I, P, P, P, F, P, P, SZ, I, P], I),
    "kvq_decode_attn_int2_window": ([P, I, I, I, I, P, I64, P, I, P, P, P, P, P, P, P, I, F, P, P, SZ, I, P], I),
    "kvq_workspace_status": ([P, P], I),
    "kvq_append_int2_clip": ([P, P, I, I, I, P, P, P, P, F, P, I64, P, P, P, P], I),
    "kvq_dequant_int2": ([P, I64, I, I, P, I, P, P, P], I),
    "bgtq_energy_scores": ([P, P, I, I, I, I, P, P, P], I),
    "kvq_decode_attn_int2_noalloc": ([P, I, I, I, I, P, I64, P, I, P, P, P, F, P, I, P], I),
    "kvq_debug_drop_next_copy": ([], None),
    "kvq_decode_step_int2": ([P, P, P, I, I, I, I, P, I64, P, I, P, P, P, P, F, P, P, SZ, I, I, P], I),
    "bgtq_lloyd_max_codebook": ([I, P], I),
    "bgtq_allocate": ([P, I, I, I, I64, P], I),
    "bgtq_tile_bytes": ([I, I], SZ),
    "bgtq_append": ([P, P, I, I, I, P, P, I, I, P, P, P, P, I64, P, P], I),
    "bgtq_decode_attn": ([P, I, I, I, I, P, I64, P, I, P, P, I, I, P, P, P, F, P, P, SZ, I, P], I),
}

STATUS = {0: "KVQ_OK", -1: "KVQ_ERR_INVALID_ARG", -2: "KVQ_ERR_UNSUPPORTED", -3: "KVQ_ERR_WORKSPACE",
          -4: "KVQ_ERR_CUDA", -5: "KVQ_ERR_BAD_BLOCK_TABLE"}


class KvqError(RuntimeError):
    def __init__(self, status: int, text: str):
        super().__init__(f"{STATUS.get(status, status)}: {text}")
        self.status = status


def header_functions() -> list[str]:
    """Names of the functions include/kvq.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"\b(kvq_\w+|bgtq_\w+)\s*\(", src)


def load():
    """Loads the in-tree library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with bit_kv_cache_13_gb300.build.build()")
        lib = C.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _check(status: int):
    if status != 0:
        raise KvqError(status, load().kvq_last_error().decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(x: torch.Tensor | None, dtype, name: str):
    if x is None:
        return None
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {x.dtype}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return x.data_ptr()


# ------------------------------------------------------------------- INT2

def kvq_int2_tile_bytes(d: int = 128) -> int:
    return load().kvq_int2_tile_bytes(d)


def kvq_append_int2(k, v, slot_mapping, mu_k, R_k, R_v, cache, num_pages: int,
                    dbg_rot_k=None, dbg_rot_v=None, err_count=None, stream=None):
    n_tok, h_kv, d = k.shape
    _check(load().kvq_append_int2(
        _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"), n_tok, h_kv, d,
        _dev(slot_mapping, torch.int32, "slot_mapping"), _dev(mu_k, torch.float32, "mu_k"),
        _dev(R_k, torch.float32, "R_k"), _dev(R_v, torch.float32, "R_v"),
        _dev(cache, torch.uint8, "cache"), int(num_pages),
        _dev(dbg_rot_k, torch.float32, "dbg_rot_k"), _dev(dbg_rot_v, torch.float32, "dbg_rot_v"),
        _dev(err_count, torch.int32, "err_count"), _stream(stream)))


def kvq_append_int2_clip(k, v, slot_mapping, mu_k, R_k, R_v, clip: float, cache, num_pages: int,
                         dbg_rot_k=None, dbg_rot_v=None, err_count=None, stream=None):
    """kvq_append_int2 with clip ratio c in (0, 1] (c = 1: the plain call)."""
    n_tok, h_kv, d = k.shape
    _check(load().kvq_append_int2_clip(
        _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"), n_tok, h_kv, d,
        _dev(slot_mapping, torch.int32, "slot_mapping"), _dev(mu_k, torch.float32, "mu_k"),
        _dev(R_k, torch.float32, "R_k"), _dev(R_v, torch.float32, "R_v"), float(clip),
        _dev(cache, torch.uint8, "cache"), int(num_pages),
        _dev(dbg_rot_k, torch.float32, "dbg_rot_k"), _dev(dbg_rot_v, torch.float32, "dbg_rot_v"),
        _dev(err_count, torch.int32, "err_count"), _stream(stream)))


def kvq_dequant_int2(cache, num_pages: int, H_kv: int, slot_mapping, k_rot=None, v_rot=None, stream=None):
    """Dequantised rotated vectors [n, H_kv, d] fp32 of the cached tokens at
    slot_mapping [n]."""
    n = slot_mapping.shape[0]
    _check(load().kvq_dequant_int2(
        _dev(cache, torch.uint8, "cache"), int(num_pages), H_kv, 128, _dev(slot_mapping, torch.int32, "slot_mapping"),
        n, _dev(k_rot, torch.float32, "k_rot"), _dev(v_rot, torch.float32, "v_rot"), _stream(stream)))


def kvq_decode_workspace_bytes(B: int, H_q: int, H_kv: int, max_pages_per_seq: int, num_splits: int = 0) -> int:
    return load().kvq_decode_workspace_bytes(B, H_q, H_kv, max_pages_per_seq, num_splits)


def kvq_decode_auto_splits(B: int, H_q: int, H_kv: int, max_pages_per_seq: int) -> int:
    return load().kvq_decode_auto_splits(B, H_q, H_kv, max_pages_per_seq)


def kvq_decode_attn_int2(q, cache, num_pages: int, block_table, context_lens, R_k, R_v, scale: float,
                         out, workspace, num_splits: int = 0, H_kv: int | None = None, stream=None):
    B, H_q, d = q.shape
    h_kv = R_k.shape[0] if H_kv is None else H_kv
    _check(load().kvq_decode_attn_int2(
        _dev(q, torch.bfloat16, "q"), B, H_q, h_kv, d, _dev(cache, torch.uint8, "cache"), int(num_pages),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
        _dev(context_lens, torch.int32, "context_lens"), _dev(R_k, torch.float32, "R_k"),
        _dev(R_v, torch.float32, "R_v"), float(scale), _dev(out, torch.float32, "out"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), int(num_splits), _stream(stream)))


KVQ_STEP_INPUTS_READY = 1


def kvq_decode_step_int2(q, k_new, v_new, cache, num_pages: int, block_table, context_lens, mu_k, R_k, R_v,
                         scale: float, out, workspace, num_splits: int = 0, flags: int = 0, stream=None):
    """One decode step in one launch: the new token k_new, v_new [B, H_kv, d]
    bf16 is appended at position context_lens[b] - 1 of each sequence, then
    the context_lens[b] tokens are attended.  flags = KVQ_STEP_INPUTS_READY
    declares the rotations, key centre, block table, context lengths and
    cache untouched by the kernel just before (read early)."""
    B, H_q, d = q.shape
    h_kv = k_new.shape[1]
    _check(load().kvq_decode_step_int2(
        _dev(q, torch.bfloat16, "q"), _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        B, H_q, h_kv, d, _dev(cache, torch.uint8, "cache"), int(num_pages),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
        _dev(context_lens, torch.int32, "context_lens"), _dev(mu_k, torch.float32, "mu_k"),
        _dev(R_k, torch.float32, "R_k"), _dev(R_v, torch.float32, "R_v"), float(scale),
        _dev(out, torch.float32, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        int(num_splits), int(flags), _stream(stream)))


def kvq_decode_attn_int2_window(q, cache, num_pages: int, block_table, context_lens, R_k, R_v, mu_k, win_k, win_v,
                                win_lens, scale: float, out, workspace, num_splits: int = 0, H_kv: int | None = None,
                                stream=None):
    """kvq_decode_attn_int2 over the cache plus a BF16 window (win_k, win_v:
    [B, win_max, H_kv, d] bf16; win_lens: [B] int32)."""
    B, H_q, d = q.shape
    h_kv = R_k.shape[0] if H_kv is None else H_kv
    _check(load().kvq_decode_attn_int2_window(
        _dev(q, torch.bfloat16, "q"), B, H_q, h_kv, d, _dev(cache, torch.uint8, "cache"), int(num_pages),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
        _dev(context_lens, torch.int32, "context_lens"), _dev(R_k, torch.float32, "R_k"),
        _dev(R_v, torch.float32, "R_v"), _dev(mu_k, torch.float32, "mu_k"), _dev(win_k, torch.bfloat16, "win_k"),
        _dev(win_v, torch.bfloat16, "win_v"), _dev(win_lens, torch.int32, "win_lens"), win_k.shape[1], float(scale),
        _dev(out, torch.float32, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        int(num_splits), _stream(stream)))


def kvq_decode_attn_int2_noalloc(q, cache, num_pages: int, block_table, context_lens, R_k, R_v, scale: float,
                                 out, num_splits: int = 0, H_kv: int | None = None, stream=None):
    """kvq_decode_attn_int2 with the library's fixed scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    B, H_q, d = q.shape
    h_kv = R_k.shape[0] if H_kv is None else H_kv
    _check(load().kvq_decode_attn_int2_noalloc(
        _dev(q, torch.bfloat16, "q"), B, H_q, h_kv, d, _dev(cache, torch.uint8, "cache"), int(num_pages),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
        _dev(context_lens, torch.int32, "context_lens"), _dev(R_k, torch.float32, "R_k"),
        _dev(R_v, torch.float32, "R_v"), float(scale), _dev(out, torch.float32, "out"), int(num_splits),
        _stream(stream)))


def kvq_debug_drop_next_copy() -> None:
    """Test hook: the next INT2 decode launch leaves one bulk copy unissued
    so a bounded wait runs out (the call then reports KVQ_ERR_CUDA)."""
    load().kvq_debug_drop_next_copy()


def kvq_workspace_status(workspace, stream=None) -> int:
    """Returns the status code recorded in a decode workspace (0 = OK) and
    clears it."""
    return load().kvq_workspace_status(_dev(workspace, torch.uint8, "workspace"), _stream(stream))


# -------------------------------------------------------------- Block-GTQ

def bgtq_energy_scores(q, k, H_kv: int, scores, paired=None, stream=None):
    """Calibration block energy scores (and the paired AM-GM estimate) of
    q [T, H_q, d] and k [T, H_kv, d] bf16 into fp64 [H_kv, d/2] tensors."""
    T, H_q, d = q.shape
    _check(load().bgtq_energy_scores(
        _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), T, H_q, H_kv, d,
        _dev(scores, torch.float64, "scores"), None if paired is None else _dev(paired, torch.float64, "paired"),
        _stream(stream)))

def bgtq_lloyd_max_codebook(b: int):
    import numpy as np
    out = np.zeros(1 << b, dtype=np.float64)
    _check(load().bgtq_lloyd_max_codebook(b, out.ctypes.data))
    return out


def bgtq_allocate(scores, b_min: int, b_max: int, total_bits: int):
    import numpy as np
    s = np.ascontiguousarray(scores, dtype=np.float64)
    w = np.zeros(s.shape[0], dtype=np.int8)
    _check(load().bgtq_allocate(s.ctypes.data, s.shape[0], b_min, b_max, int(total_bits), w.ctypes.data))
    return w


def bgtq_tile_bytes(total_bits: int, v_bits: int) -> int:
    return load().bgtq_tile_bytes(total_bits, v_bits)


def bgtq_append(k, v, slot_mapping, widths, total_bits: int, v_bits: int, pi_table, pi_offsets, codebooks,
                cache, num_pages: int, err_count=None, stream=None):
    n_tok, h_kv, d = k.shape
    _check(load().bgtq_append(
        _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"), n_tok, h_kv, d,
        _dev(slot_mapping, torch.int32, "slot_mapping"), _dev(widths, torch.int8, "widths"), int(total_bits),
        int(v_bits), _dev(pi_table, torch.float32, "pi_table"), _dev(pi_offsets, torch.int64, "pi_offsets"),
        _dev(codebooks, torch.float64, "codebooks"), _dev(cache, torch.uint8, "cache"), int(num_pages),
        _dev(err_count, torch.int32, "err_count"), _stream(stream)))


def bgtq_decode_attn(q, cache, num_pages: int, block_table, context_lens, widths, total_bits: int, v_bits: int,
                     pi_table, pi_offsets, codebooks, scale: float, out, workspace, num_splits: int = 0,
                     stream=None):
    B, H_q, d = q.shape
    h_kv = widths.shape[0]
    _check(load().bgtq_decode_attn(
        _dev(q, torch.bfloat16, "q"), B, H_q, h_kv, d, _dev(cache, torch.uint8, "cache"), int(num_pages),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
        _dev(context_lens, torch.int32, "context_lens"), _dev(widths, torch.int8, "widths"), int(total_bits),
        int(v_bits), _dev(pi_table, torch.float32, "pi_table"), _dev(pi_offsets, torch.int64, "pi_offsets"),
        _dev(codebooks, torch.float64, "codebooks"), float(scale), _dev(out, torch.float32, "out"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), int(num_splits), _stream(stream)))
