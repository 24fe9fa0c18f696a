"""GPU parity of the Block-GTQ calibration energy scores (method step (1)
of "RoPE-Aware Bit Allocation for KV-Cache Quantization") against the fp64
oracle, and the widths the greedy allocator gives from them.

Bars: scores <= 1e-12 relative (exact squares, fp64 sums in another order);
the paired estimate <= 1e-6 relative (fp32 square roots) and never above
the scores (AM-GM, technical novelty (2)).
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_13_gb300 import _lib, inputs
from oracle import bgtq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("h_q,h_kv,T", [(32, 8, 1000), (64, 8, 257), (4, 4, 1), (8, 2, 4096), (16, 1, 0)])
def test_energy_scores_match_oracle(h_q, h_kv, T):
    spec = inputs.small_spec(f"cal{h_q}_{h_kv}", h_q=h_q, h_kv=h_kv, batch=1, ctx=max(T, 1), k_kind="energy_rope")
    pos = torch.arange(T)
    q = inputs.gen_prefix_queries(spec, 0, pos, device="cuda")
    k = inputs.gen_keys(spec, 0, 0, pos, device="cuda")
    s = torch.full((h_kv, 64), float("nan"), dtype=torch.float64, device="cuda")
    p = torch.full_like(s, float("nan"))
    _lib.bgtq_energy_scores(q, k, h_kv, s, p)
    torch.cuda.synchronize()
    want_s, want_p = bgtq.energy_scores(q.float().cpu().numpy(), k.float().cpu().numpy(), h_kv)
    got_s, got_p = s.cpu().numpy(), p.cpu().numpy()
    if T == 0:
        assert np.all(got_s == 0) and np.all(got_p == 0)
        return
    assert np.max(np.abs(got_s - want_s) / want_s) <= 1e-12
    assert np.max(np.abs(got_p - want_p) / want_p) <= 1e-6
    assert np.all(got_p <= got_s * (1 + 1e-6))


def test_widths_from_gpu_scores_match_the_oracle_allocation():
    # Greedy widths (b in [1, 8], sum 192 per head) from the GPU scores equal
    # the oracle's from the oracle scores; the scores agree to ~1e-15, far
    # inside the gaps between competing marginal gains of this seeded draw.
    spec = inputs.small_spec("calw", h_q=32, h_kv=8, batch=1, ctx=2048, k_kind="energy_rope")
    pos = torch.arange(2048)
    q = inputs.gen_prefix_queries(spec, 0, pos, device="cuda")
    k = inputs.gen_keys(spec, 0, 0, pos, device="cuda")
    s = torch.zeros((8, 64), dtype=torch.float64, device="cuda")
    _lib.bgtq_energy_scores(q, k, 8, s)
    want_s, _ = bgtq.energy_scores(q.float().cpu().numpy(), k.float().cpu().numpy(), 8)
    for h in range(8):
        got = _lib.bgtq_allocate(s[h].cpu().numpy(), 1, 8, 192)
        want = bgtq.greedy_allocate(want_s[h], 1, 8, 192)
        assert np.array_equal(np.asarray(got), np.asarray(want))
        assert int(np.sum(got)) == 192
