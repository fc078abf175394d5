"""dsv4_hca_decode_static: HCA decode for callers that cannot allocate device
memory (for example code running under CUDA graph capture, or engines whose
device memory is owned by a planning allocator). Its split partials live in a
static device array inside the library instead of a caller workspace.

Checked through the C ABI against dsv4_hca_decode on the same cache: two calls
in a row with different queries (the static array keeps the previous call's
contents), on a separate-K/V layer and on a shared-entry layer that spans
several tiles and splits (there also against the float64 oracle); and an
oversized call is refused on the host.

This file is named to be collected last, so a failure here never hides the
other GPU tests when pytest stops at the first failure."""
import numpy as np
import pytest
import torch

from compressed_sparse_kv_05_b300 import dsv4, synth
from compressed_sparse_kv_05_b300 import workloads as W

from .gpu_util import (gpu_cache_from_planes, gpu_stream_cache, oracle_attend_planes, oracle_direct_planes,
                       row_rel_err, to_dev, to_host)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

TOL = 2e-3


def _both(desc, cache, layer, q):
    H, D, B = layer.heads, layer.dim, layer.batch
    ws = dsv4.workspace(desc, H)
    ref = torch.zeros((B, H, D), dtype=torch.float32, device="cuda")
    ref_lse = torch.zeros((B, H), dtype=torch.float32, device="cuda")
    got = torch.full((B, H, D), float("nan"), dtype=torch.float32, device="cuda")
    got_lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    dsv4.dsv4_hca_decode(desc, cache, H, q, layer.sm_scale, ref, ref_lse, ws)
    dsv4.dsv4_hca_decode_static(desc, cache, H, q, layer.sm_scale, got, got_lse)
    torch.cuda.synchronize()
    return to_host(got), to_host(got_lse), to_host(ref), to_host(ref_lse)


def _check_two_calls(desc, cache, layer, tag, planes=None):
    need = dsv4.dsv4_workspace_size(desc, layer.heads, 0, 0)
    assert 0 < need <= dsv4.STATIC_SCRATCH_BYTES
    for call in range(2):
        q_host = synth.decode_inputs(f"{tag}{call}", 0, layer)["q"]
        got, got_lse, ref, ref_lse = _both(desc, cache, layer, to_dev(q_host))
        assert np.isfinite(got).all() and np.isfinite(got_lse).all()
        assert row_rel_err(got, ref).max() <= TOL
        assert np.abs(got_lse - ref_lse).max() <= 1e-3
        for b, p in enumerate(planes or ()):
            # and against the float64 oracle on the same cache planes
            o_out, o_lse = oracle_attend_planes(layer, p, q_host[b], None)
            assert row_rel_err(got[b], o_out).max() <= TOL
            assert np.abs(got_lse[b] - o_lse).max() <= 1e-3
    assert dsv4.dsv4_read_status(cache) == 0


def test_static_scratch_matches_workspace_separate_kv():
    layer = W.scaled(W.HCA_128K, n_tokens=128 * 300)
    desc, cache = gpu_stream_cache(layer, "static", 0, layer.n_tokens, (4096,))
    _check_two_calls(desc, cache, layer, "static-sep")


def test_static_scratch_matches_workspace_shared_entry():
    layer = W.scaled(W.STACK_HCA, batch=2, n_tokens=128 * 1500)
    planes = oracle_direct_planes(layer, "static", 1, range(layer.batch))
    desc, cache = gpu_cache_from_planes(layer, planes)
    _check_two_calls(desc, cache, layer, "static-shared", planes)


def test_static_scratch_refuses_oversized_calls():
    layer = W.scaled(W.STACK_HCA, batch=64)
    desc = dsv4.layer_desc(layer, layer.capacity())
    assert dsv4.dsv4_workspace_size(desc, layer.heads, 0, 0) > dsv4.STATIC_SCRATCH_BYTES
    small = W.scaled(W.HCA_128K, n_tokens=1024)
    cache = dsv4.Cache(dsv4.layer_desc(small, 16))        # never read: the call fails on the host
    q = torch.zeros((64, layer.heads, layer.dim), dtype=torch.int16, device="cuda")
    out = torch.zeros((64, layer.heads, layer.dim), dtype=torch.float32, device="cuda")
    with pytest.raises(dsv4.Dsv4Error) as e:
        dsv4.dsv4_hca_decode_static(desc, cache, layer.heads, q, layer.sm_scale, out, None)
    assert e.value.code == dsv4.ERR_SCRATCH
