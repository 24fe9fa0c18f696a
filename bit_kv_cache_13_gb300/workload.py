"""Device-side set-up of a synthetic decode workload for the INT2 and
Block-GTQ caches: parameters, paged cache, prefill through the library's own
append call, and the per-step inputs (new key/value token, query).

Only the seeded input generators and the C-ABI binding are used here.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import _lib, inputs
from .inputs import PAGE_SIZE, Spec


def history_positions(spec: Spec) -> torch.Tensor:
    """Positions of the cached tokens before the decode step (ctx - 1 of them)."""
    return torch.arange(spec.ctx - 1, dtype=torch.int64)


class Int2Layer:
    """One attention layer's INT2 cache and parameters on `device`."""

    def __init__(self, spec: Spec, layer: int, device="cuda", block_table=None, extra_pages: int = 0):
        self.spec, self.layer, self.device = spec, layer, device
        d = spec.d
        self.R_k64 = np.stack([inputs.head_rotation(d, spec.name, layer, h, "Rk") for h in range(spec.h_kv)])
        self.R_v64 = np.stack([inputs.head_rotation(d, spec.name, layer, h, "Rv") for h in range(spec.h_kv)])
        self.R_k = torch.as_tensor(self.R_k64, dtype=torch.float32, device=device).contiguous()
        self.R_v = torch.as_tensor(self.R_v64, dtype=torch.float32, device=device).contiguous()
        bt = inputs.block_tables(spec, device="cpu") if block_table is None else block_table.cpu()
        self.block_table = bt.to(device=device, dtype=torch.int32).contiguous()
        self.num_pages = int(bt.max().item()) + 1 + extra_pages
        self.tile = _lib.kvq_int2_tile_bytes(d)
        self.cache = torch.zeros((self.num_pages, spec.h_kv, self.tile), dtype=torch.uint8, device=device)
        self.context_lens = torch.full((spec.batch,), spec.ctx, dtype=torch.int32, device=device)
        self.mu = None
        self.scale = 1.0 / math.sqrt(d)

    # inputs ---------------------------------------------------------------
    def history_kv(self, b: int, device=None):
        dev = self.device if device is None else device
        pos = history_positions(self.spec).to(dev)
        k = inputs.gen_keys(self.spec, self.layer, b, pos, device=dev)
        v = inputs.gen_values(self.spec, self.layer, b, pos.numel(), device=dev)
        return k, v

    def new_kv(self, device=None):
        """The decode-step token of every sequence: [B, H_kv, d] each."""
        dev = self.device if device is None else device
        pos = torch.tensor([self.spec.ctx - 1], device=dev)
        k = torch.cat([inputs.gen_keys(self.spec, self.layer, b, pos, device=dev, tag="new")
                       for b in range(self.spec.batch)])
        v = torch.cat([inputs.gen_values(self.spec, self.layer, b, 1, device=dev, tag="new")
                       for b in range(self.spec.batch)])
        return k.contiguous(), v.contiguous()

    def queries(self, device=None):
        return inputs.gen_queries(self.spec, self.layer, device=self.device if device is None else device)

    def slots(self, b: int, positions: torch.Tensor) -> torch.Tensor:
        return inputs.slot_mapping(self.block_table[b].cpu(), positions.cpu()).to(self.device)

    def new_slots(self) -> torch.Tensor:
        pos = torch.tensor([self.spec.ctx - 1])
        return torch.cat([self.slots(b, pos) for b in range(self.spec.batch)]).contiguous()

    # prefill --------------------------------------------------------------
    def prefill(self, chunk: int = 1 << 16):
        """Appends every sequence's history through kvq_append_int2; the key
        centre is taken from sequence 0 (first 512 keys) before that."""
        pos = history_positions(self.spec)
        for b in range(self.spec.batch):
            k, v = self.history_kv(b)
            if self.mu is None:
                self.mu = inputs.key_centre(k).to(self.device).contiguous()
            sl = self.slots(b, pos)
            for s in range(0, k.shape[0], chunk):
                e = min(k.shape[0], s + chunk)
                _lib.kvq_append_int2(k[s:e].contiguous(), v[s:e].contiguous(), sl[s:e].contiguous(), self.mu,
                                     self.R_k, self.R_v, self.cache, self.num_pages)
            del k, v
        if self.mu is None:
            self.mu = torch.zeros((self.spec.h_kv, self.spec.d), dtype=torch.float32, device=self.device)

    def workspace(self, num_splits: int = 0) -> torch.Tensor:
        n = _lib.kvq_decode_workspace_bytes(self.spec.batch, self.spec.h_q, self.spec.h_kv,
                                            self.block_table.shape[1], num_splits)
        return torch.zeros(n, dtype=torch.uint8, device=self.device)

    def packed_bytes_per_decode(self) -> int:
        """Algorithmic cache bytes one decode reads: 96 B per attended
        token-head (codes + fp16 scale/min of K and V)."""
        return int(self.context_lens.sum().item()) * self.spec.h_kv * 96


class BgtqLayer:
    """One attention layer's Block-GTQ cache and parameters on `device`:
    per-head widths from the greedy allocator (library, host) over the
    per-block energy scores, shared TQ rotations, Lloyd-Max codebooks from
    the library, paged cache filled with bgtq_append."""

    def __init__(self, spec: Spec, layer: int, device="cuda", block_table=None, extra_pages: int = 0,
                 codebooks=None):
        self.spec, self.layer, self.device = spec, layer, device
        ex = spec.extra
        self.avg_bits, self.v_bits = int(ex.get("avg_bits", 3)), int(ex.get("v_bits", 3))
        self.b_min, self.b_max = int(ex.get("b_min", 1)), int(ex.get("b_max", 8))
        self.total_bits = self.avg_bits * (spec.d // 2)
        self.scores = np.stack([inputs.block_energies(spec, layer, h) for h in range(spec.h_kv)])
        w = np.stack([_lib.bgtq_allocate(self.scores[h], self.b_min, self.b_max, self.total_bits)
                      for h in range(spec.h_kv)])
        self.widths_np = w
        self.widths = torch.as_tensor(w, dtype=torch.int8, device=device).contiguous()
        table64, offsets = inputs.tq_rotations(spec.d, "tq", spec.name)
        self.pi_table64, self.pi_offsets_np = table64, offsets
        self.pi_table = torch.as_tensor(table64, dtype=torch.float32, device=device).contiguous()
        self.pi_offsets = torch.as_tensor(offsets, dtype=torch.int64, device=device).contiguous()
        if codebooks is None:
            cb = np.zeros((8, 256))
            for b in range(1, 9):
                cb[b - 1, : 2 ** b] = _lib.bgtq_lloyd_max_codebook(b)
            codebooks = cb
        self.codebooks_np = np.asarray(codebooks, dtype=np.float64)
        self.codebooks = torch.as_tensor(self.codebooks_np, dtype=torch.float64, device=device).contiguous()
        bt = inputs.block_tables(spec, device="cpu") if block_table is None else block_table.cpu()
        self.block_table = bt.to(device=device, dtype=torch.int32).contiguous()
        self.num_pages = int(bt.max().item()) + 1 + extra_pages
        self.tile = _lib.bgtq_tile_bytes(self.total_bits, self.v_bits)
        self.cache = torch.zeros((self.num_pages, spec.h_kv, self.tile), dtype=torch.uint8, device=device)
        self.context_lens = torch.full((spec.batch,), spec.ctx, dtype=torch.int32, device=device)
        self.scale = 1.0 / math.sqrt(spec.d)

    history_kv = Int2Layer.history_kv
    new_kv = Int2Layer.new_kv
    queries = Int2Layer.queries
    slots = Int2Layer.slots
    new_slots = Int2Layer.new_slots
    workspace = Int2Layer.workspace

    def append(self, k, v, slots, err_count=None):
        _lib.bgtq_append(k, v, slots, self.widths, self.total_bits, self.v_bits, self.pi_table, self.pi_offsets,
                         self.codebooks, self.cache, self.num_pages, err_count)

    def prefill(self, chunk: int = 1 << 16):
        pos = history_positions(self.spec)
        for b in range(self.spec.batch):
            k, v = self.history_kv(b)
            sl = self.slots(b, pos)
            for s in range(0, k.shape[0], chunk):
                e = min(k.shape[0], s + chunk)
                self.append(k[s:e].contiguous(), v[s:e].contiguous(), sl[s:e].contiguous())
            del k, v

    def decode(self, q, out, ws, num_splits: int = 0, context_lens=None):
        _lib.bgtq_decode_attn(q, self.cache, self.num_pages, self.block_table,
                              self.context_lens if context_lens is None else context_lens, self.widths,
                              self.total_bits, self.v_bits, self.pi_table, self.pi_offsets, self.codebooks,
                              self.scale, out, ws, num_splits)

    def bytes_per_token_head(self) -> int:
        """Algorithmic bytes of one cached token for one KV head."""
        return self.tile // PAGE_SIZE
