"""Head and batch sharding of the INT2 decode on one GPU: the shards'
concatenated outputs equal the unsharded call bit for bit (explicit split
count, so every (sequence, KV head) unit gets the same page shares in every
shard), and the sharded result matches the fp64 oracle."""
import numpy as np
import pytest
import torch

from bit_kv_cache_13_gb300 import inputs, shard
from bit_kv_cache_13_gb300.workload import Int2Layer

pytestmark = pytest.mark.gpu


def _inputs(name, h_q, h_kv, batch, ctx):
    spec = inputs.small_spec(name, h_q=h_q, h_kv=h_kv, batch=batch, ctx=ctx, permute=True)
    layer = Int2Layer(spec, 0)
    layer.prefill()
    cl = torch.tensor([ctx - 37 * b for b in range(batch)], dtype=torch.int32, device="cuda")   # ragged
    return shard.Int2DecodeInputs(q=layer.queries(), cache=layer.cache, block_table=layer.block_table,
                                  context_lens=cl, R_k=layer.R_k, R_v=layer.R_v, scale=layer.scale)


@pytest.mark.parametrize("h_q,h_kv,batch,ctx,splits", [(32, 8, 3, 2000, 3), (64, 8, 2, 1500, 2), (12, 3, 4, 500, 1)])
def test_shards_equal_the_unsharded_decode_bit_for_bit(h_q, h_kv, batch, ctx, splits):
    x = _inputs(f"shard{h_q}{h_kv}", h_q, h_kv, batch, ctx)
    full = shard.decode(x, splits)
    for n in (2, 3, h_kv):
        assert torch.equal(shard.sharded_decode(x, n, "head", splits), full), ("head", n)
    for n in (2, batch):
        assert torch.equal(shard.sharded_decode(x, n, "batch", splits), full), ("batch", n)
    torch.cuda.synchronize()
    assert torch.isfinite(full).all()
