"""The failure path of the tensor-core attention kernel, driven without a GPU
fault: a test hook makes the MMA-issuing thread of every CTA wait on a barrier
that nothing arrives on. Its bounded wait runs out, the CTA's other roles see
the abort flag in their own bounded waits and leave their loops, the copies
and MMAs in flight are drained, tensor memory is released, and the kernel
returns with DSV4_STATUS_TIMEOUT in the cache's status word. The test checks
that status, that the call came back within its bound, and that the context
is still usable: with the hook off, the same call gives bit for bit what it
gave before, and that matches the oracle."""
import time

import numpy as np
import pytest
import torch

from compressed_sparse_kv_05_b300 import dsv4, synth
from compressed_sparse_kv_05_b300 import workloads as W

from .gpu_util import gpu_cache_from_planes, oracle_attend_planes, oracle_direct_planes, row_rel_err, to_dev, to_host

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def _call(desc, cache, layer, q, sel):
    B, H = layer.batch, layer.heads
    out = torch.full((B, H, layer.dim), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = dsv4.workspace(desc, H, layer.idx_heads, max(layer.topk, 1))
    if sel is None:
        dsv4.dsv4_hca_decode(desc, cache, H, to_dev(q), layer.sm_scale, out, lse, ws)
    else:
        dsv4.dsv4_csa_decode(desc, cache, H, to_dev(q), layer.sm_scale, to_dev(sel), layer.topk, out, lse, ws)
    torch.cuda.synchronize()
    return to_host(out), to_host(lse)


@pytest.mark.parametrize("kind", ["hca", "csa"])
def test_attention_wait_runs_out_and_context_survives(kind):
    base = W.STACK_HCA if kind == "hca" else W.STACK_CSA
    n = base.ratio * 1200 + 3
    layer = W.scaled(base, batch=2, n_tokens=n)
    planes = oracle_direct_planes(layer, "timeout", 0, range(layer.batch))
    desc, cache = gpu_cache_from_planes(layer, planes)
    q = synth.decode_inputs("timeout", 0, layer)["q"]
    sel = None
    if kind == "csa":
        rng = np.random.default_rng(5)
        sel = np.stack([np.sort(rng.choice(layer.n_comp, layer.topk, replace=False)).astype(np.int32)
                        for _ in range(layer.batch)])

    ref_out, ref_lse = _call(desc, cache, layer, q, sel)
    assert dsv4.dsv4_read_status(cache) == 0

    dsv4.dsv4_debug_force_timeout(True)
    try:
        t0 = time.perf_counter()
        _call(desc, cache, layer, q, sel)
        elapsed = time.perf_counter() - t0
    finally:
        dsv4.dsv4_debug_force_timeout(False)
    status = dsv4.dsv4_read_status(cache)
    assert status & dsv4.STATUS_TIMEOUT, status
    assert elapsed < 20.0   # every wait is bounded (the forced one by 50 ms, the rest by 2 s)
    assert dsv4.dsv4_read_status(cache) == 0   # reading cleared it

    # the context still works: a torch kernel, and the same call as before
    x = torch.arange(1 << 20, device="cuda", dtype=torch.float64)
    assert x.sum().item() == float((1 << 20) * ((1 << 20) - 1) // 2)
    out, lse = _call(desc, cache, layer, q, sel)
    assert dsv4.dsv4_read_status(cache) == 0
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)
    for b in range(layer.batch):
        o_out, o_lse = oracle_attend_planes(layer, planes[b], q[b], None if sel is None else sel[b])
        assert row_rel_err(out[b], o_out).max() <= 2e-3
        assert np.abs(lse[b] - o_lse).max() <= 1e-3
