"""Head and batch sharding of the INT2 decode across devices (host side).

Every (sequence, KV head) unit of the decode is independent: the rotations
R_k, R_v and the key centre mu are per KV head, and a GQA group never spans
two KV heads.  A decode therefore splits, without any exchange, into shards
of KV heads (tensor-parallel style: each rank owns the cache, rotations and
query heads of its KV heads) or of sequences (each rank owns its sequences'
block-table rows; the pages may live in one shared pool).  Each shard is the
same kvq_decode_attn_int2 call on its slice; concatenating the shards'
outputs along the head (or batch) axis gives the unsharded output.  With an
explicit split count every unit is cut into the same page shares whatever
the shard holds, so the concatenation equals the unsharded call bit for bit.

The "RoPE-Aware Bit Allocation for KV-Cache Quantization" page names
multi-GPU decode an open direction (limitations); this is the plain
partition, with no collective on the data path.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib


def ranges(n: int, parts: int) -> list[tuple[int, int]]:
    """Split range(n) into `parts` contiguous pieces, sizes within one,
    larger pieces first; empty pieces when parts > n."""
    if n < 0 or parts <= 0:
        raise ValueError("n >= 0 and parts > 0 required")
    base, extra = divmod(n, parts)
    out, start = [], 0
    for i in range(parts):
        size = base + (1 if i < extra else 0)
        out.append((start, start + size))
        start += size
    return out


@dataclass
class Int2DecodeInputs:
    """The tensors of one INT2 decode call (kvq_decode_attn_int2)."""
    q: torch.Tensor              # [B, H_q, d] bf16
    cache: torch.Tensor          # [num_pages, H_kv, 1536] uint8
    block_table: torch.Tensor    # [B, max_pages] int32
    context_lens: torch.Tensor   # [B] int32
    R_k: torch.Tensor            # [H_kv, d, d] fp32
    R_v: torch.Tensor            # [H_kv, d, d] fp32
    scale: float

    @property
    def h_kv(self) -> int:
        return self.R_k.shape[0]

    @property
    def group(self) -> int:
        return self.q.shape[1] // self.h_kv


def head_shard(x: Int2DecodeInputs, h0: int, h1: int) -> Int2DecodeInputs:
    """KV heads h0..h1-1 and their query heads: the cache slice is copied
    into its own [num_pages, h1 - h0, 1536] tensor (as a rank owning those
    heads would hold it); the rotations are row slices."""
    g = x.group
    return Int2DecodeInputs(q=x.q[:, h0 * g:h1 * g].contiguous(), cache=x.cache[:, h0:h1].contiguous(),
                            block_table=x.block_table, context_lens=x.context_lens,
                            R_k=x.R_k[h0:h1], R_v=x.R_v[h0:h1], scale=x.scale)


def batch_shard(x: Int2DecodeInputs, b0: int, b1: int) -> Int2DecodeInputs:
    """Sequences b0..b1-1: their queries, block-table rows and context
    lengths; the page pool (cache) is shared."""
    return Int2DecodeInputs(q=x.q[b0:b1].contiguous(), cache=x.cache, block_table=x.block_table[b0:b1].contiguous(),
                            context_lens=x.context_lens[b0:b1].contiguous(), R_k=x.R_k, R_v=x.R_v, scale=x.scale)


def decode(x: Int2DecodeInputs, num_splits: int = 0, stream=None) -> torch.Tensor:
    """kvq_decode_attn_int2 on one (possibly sharded) set of inputs; returns
    the [B, H_q, d] fp32 output."""
    B, H_q, d = x.q.shape
    out = torch.empty((B, H_q, d), dtype=torch.float32, device=x.q.device)
    if B == 0 or x.h_kv == 0:
        return out
    nbytes = _lib.kvq_decode_workspace_bytes(B, H_q, x.h_kv, x.block_table.shape[1], num_splits)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=x.q.device)
    _lib.kvq_decode_attn_int2(x.q, x.cache, x.cache.shape[0], x.block_table, x.context_lens, x.R_k, x.R_v, x.scale,
                              out, ws, num_splits, stream=stream)
    return out


def sharded_decode(x: Int2DecodeInputs, shards: int, by: str = "head", num_splits: int = 1) -> torch.Tensor:
    """The decode cut into `shards` pieces by KV head or by sequence, run one
    after the other here (on one device; across ranks each runs its own) and
    concatenated."""
    if by == "head":
        parts = [decode(head_shard(x, h0, h1), num_splits) for h0, h1 in ranges(x.h_kv, shards) if h1 > h0]
        return torch.cat(parts, dim=1)
    if by == "batch":
        parts = [decode(batch_shard(x, b0, b1), num_splits) for b0, b1 in ranges(x.q.shape[0], shards) if b1 > b0]
        return torch.cat(parts, dim=0)
    raise ValueError(f"by must be 'head' or 'batch', not {by!r}")
