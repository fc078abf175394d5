"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/dsv4.h declares, sizes workspaces, and rejects bad
arguments before any launch. Every call here fails validation by construction
(null, misaligned or out-of-range arguments), so no kernel can be reached."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsv4.h")


@pytest.fixture(scope="module")
def dsv4():
    from compressed_sparse_kv_05_b300 import build
    build.build()
    from compressed_sparse_kv_05_b300 import dsv4 as mod
    return mod


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t)\s+(dsv4_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_four_calls():
    fns = declared_functions()
    for name in ("dsv4_compress_append", "dsv4_index_topk", "dsv4_csa_decode", "dsv4_hca_decode"):
        assert name in fns


def test_library_exports_every_declared_symbol(dsv4):
    lib = ctypes.CDLL(dsv4._LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(dsv4.EXPORTED)


def _desc(dsv4, **kw):
    base = dict(batch=4, d_nope=448, d_rope=64, ratio=4, window=128, separate_v=0, idx_dim=128, capacity=1000)
    base.update(kw)
    return dsv4.LayerDesc(*[base[f] for f, _ in dsv4.LayerDesc._fields_])


def test_workspace_size(dsv4):
    d = _desc(dsv4)
    n = dsv4.dsv4_workspace_size(d, 64, 64, 512)
    assert n >= 4 * 1000 * 4 + 4 * 64 * 128 * 4            # scores + decoded indexer query
    assert n >= 4 * 64 * (512 + 1) * 4                      # at least one split partial per head
    assert dsv4.dsv4_workspace_size(d, 0, 64, 512) == 0
    assert dsv4.dsv4_workspace_size(d, 129, 64, 512) == 0
    assert dsv4.dsv4_workspace_size(_desc(dsv4, d_nope=40), 64, 64, 512) == 0


FAKE = 0x10000000          # 16-byte aligned fake address: never dereferenced (validation fails first)


def _cache(dsv4, **kw):
    c = dsv4.CacheStruct()
    for name in ("idx_codes", "idx_scales", "win_k", "win_v", "pend_k", "pend_v", "pend_z", "pend_u", "pend_zu",
                 "n_tokens", "status"):
        setattr(c, name, kw.get(name, FAKE))
    c.k = dsv4.KvPlanes(kw.get("k_nope", FAKE), FAKE, FAKE)
    c.v = dsv4.KvPlanes(FAKE, FAKE, FAKE)
    return c


def _hca(dsv4, d, c, H=64, q=FAKE, out=FAKE, ws=FAKE, ws_bytes=1 << 40):
    return dsv4.lib.dsv4_hca_decode(ctypes.byref(d), ctypes.byref(c), H, q, 0.1, out, None, ws, ws_bytes, None)


def test_decode_rejects_bad_arguments_on_host(dsv4):
    d = _desc(dsv4)
    c = _cache(dsv4)
    assert _hca(dsv4, d, c, H=0) == dsv4.ERR_INVALID_ARG
    assert _hca(dsv4, d, c, H=129) == dsv4.ERR_UNSUPPORTED
    assert _hca(dsv4, d, c, q=None) == dsv4.ERR_INVALID_ARG
    assert _hca(dsv4, d, c, q=FAKE + 2) == dsv4.ERR_MISALIGNED
    assert _hca(dsv4, d, c, ws_bytes=16) == dsv4.ERR_WORKSPACE
    assert _hca(dsv4, d, _cache(dsv4, k_nope=0)) == dsv4.ERR_INVALID_ARG
    assert _hca(dsv4, d, _cache(dsv4, n_tokens=FAKE + 8)) == dsv4.ERR_MISALIGNED
    for bad in (dict(d_nope=40), dict(d_rope=12), dict(ratio=300), dict(window=5000), dict(idx_dim=48),
                dict(d_nope=512, d_rope=128)):
        assert _hca(dsv4, _desc(dsv4, **bad), c) == dsv4.ERR_UNSUPPORTED, bad
    for bad in (dict(batch=0), dict(capacity=0), dict(ratio=0), dict(window=-1)):
        assert _hca(dsv4, _desc(dsv4, **bad), c) == dsv4.ERR_INVALID_ARG, bad
    assert dsv4.lib.dsv4_hca_decode(None, ctypes.byref(c), 64, FAKE, 0.1, FAKE, None, FAKE, 1 << 40, None) == \
        dsv4.ERR_INVALID_ARG


def test_csa_and_index_reject_bad_arguments_on_host(dsv4):
    d = _desc(dsv4)
    c = _cache(dsv4)
    L = dsv4.lib
    assert L.dsv4_csa_decode(ctypes.byref(d), ctypes.byref(c), 64, FAKE, 0.1, FAKE, -1, FAKE, None, FAKE, 1 << 40,
                             None) == dsv4.ERR_INVALID_ARG
    assert L.dsv4_csa_decode(ctypes.byref(d), ctypes.byref(c), 64, FAKE, 0.1, None, 0, None, None, FAKE, 1 << 40,
                             None) == dsv4.ERR_INVALID_ARG           # window-only call: out still required
    assert L.dsv4_csa_decode(ctypes.byref(d), ctypes.byref(c), 64, FAKE, 0.1, FAKE, 4096, FAKE, None, FAKE, 1 << 40,
                             None) == dsv4.ERR_UNSUPPORTED
    assert L.dsv4_csa_decode(ctypes.byref(d), ctypes.byref(c), 64, FAKE, 0.1, FAKE + 4, 512, FAKE, None, FAKE,
                             1 << 40, None) == dsv4.ERR_MISALIGNED
    assert L.dsv4_index_topk(ctypes.byref(_desc(dsv4, idx_dim=0)), ctypes.byref(c), 64, FAKE, FAKE, 512, FAKE,
                             None, FAKE, 1 << 40, None) == dsv4.ERR_INVALID_ARG
    assert L.dsv4_index_topk(ctypes.byref(d), ctypes.byref(c), 64, FAKE, FAKE, 512, FAKE, None, FAKE, 8,
                             None) == dsv4.ERR_WORKSPACE
    assert L.dsv4_index_topk(ctypes.byref(d), ctypes.byref(c), 200, FAKE, FAKE, 512, FAKE, None, FAKE, 1 << 40,
                             None) == dsv4.ERR_UNSUPPORTED
    assert L.dsv4_index_topk(ctypes.byref(d), ctypes.byref(c), 64, FAKE, FAKE, 512, None, None, FAKE, 1 << 40,
                             None) == dsv4.ERR_INVALID_ARG


def test_append_rejects_bad_arguments_on_host(dsv4):
    d = _desc(dsv4)
    L = dsv4.lib
    c = _cache(dsv4)
    assert L.dsv4_compress_append(ctypes.byref(d), ctypes.byref(c), -1, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  None) == dsv4.ERR_INVALID_ARG
    assert L.dsv4_compress_append(ctypes.byref(d), ctypes.byref(c), 8, FAKE, None, FAKE, FAKE, None, FAKE, FAKE,
                                  None) == dsv4.ERR_INVALID_ARG          # indexer stream missing
    assert L.dsv4_compress_append(ctypes.byref(d), ctypes.byref(_cache(dsv4, pend_z=0)), 8, FAKE, None, FAKE, FAKE,
                                  FAKE, FAKE, FAKE, None) == dsv4.ERR_INVALID_ARG
    assert L.dsv4_compress_append(ctypes.byref(d), ctypes.byref(c), 8, FAKE + 2, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  None) == dsv4.ERR_MISALIGNED


def test_quantizers_and_pool_reject_bad_arguments_on_host(dsv4):
    L = dsv4.lib
    assert L.dsv4_quantize_kv_rows(FAKE, 10, 40, 64, FAKE, FAKE, FAKE, None) == dsv4.ERR_UNSUPPORTED
    assert L.dsv4_quantize_kv_rows(FAKE, -1, 448, 64, FAKE, FAKE, FAKE, None) == dsv4.ERR_INVALID_ARG
    assert L.dsv4_quantize_kv_rows(None, 10, 448, 64, FAKE, FAKE, FAKE, None) == dsv4.ERR_INVALID_ARG
    assert L.dsv4_quantize_kv_rows(FAKE, 0, 448, 64, None, None, None, None) == dsv4.OK     # nothing to do
    assert L.dsv4_quantize_fp4_rows(FAKE, 10, 48, FAKE, FAKE, None) == dsv4.ERR_UNSUPPORTED
    assert L.dsv4_quantize_fp4_rows(FAKE, 10, 128, FAKE + 1, FAKE, None) == dsv4.ERR_MISALIGNED
    assert L.dsv4_quantize_kv_rows(FAKE + 2, 10, 448, 64, FAKE, FAKE, FAKE, None) == dsv4.ERR_MISALIGNED
    assert L.dsv4_pool_rows(FAKE, FAKE, FAKE, 10, 0, 128, FAKE, None) == dsv4.ERR_INVALID_ARG
    assert L.dsv4_pool_rows(FAKE, FAKE, FAKE, 10, 4, 100, FAKE, None) == dsv4.ERR_UNSUPPORTED
    assert L.dsv4_read_status(None, None) == dsv4.ERR_INVALID_ARG


def test_decode_plan_on_host(dsv4):
    """The launch plan the decode calls take, computed on the host (148 SMs
    when no device can be queried): the batched CSA configuration (B = 32,
    top-512, window 128) takes 128-row tiles gathered two per CTA in three
    splits; the four-sequence decode step takes 32-row tiles; a window-only
    call plans the window tiles alone; D = 192 takes the CUDA-core path."""
    sms = dsv4.dsv4_decode_plan(_desc(dsv4), 64, 512)["sms"]
    if sms != 148:
        pytest.skip(f"plans below are worked out for 148 SMs, this device has {sms}")
    p = dsv4.dsv4_decode_plan(_desc(dsv4, batch=32, capacity=32768), 64, 512)
    assert (p["tensor_core"], p["tile_rows"], p["tiles_per_split"], p["splits"]) == (1, 128, 2, 3)
    p = dsv4.dsv4_decode_plan(_desc(dsv4, capacity=262144), 64, 512)
    assert (p["tensor_core"], p["tile_rows"], p["tiles_per_split"], p["splits"]) == (1, 32, 1, 20)
    p = dsv4.dsv4_decode_plan(_desc(dsv4, ratio=128, idx_dim=0, capacity=8192), 64, -1)
    assert (p["tile_rows"], p["tiles_per_split"], p["splits"]) == (128, 2, 33)
    p = dsv4.dsv4_decode_plan(_desc(dsv4, capacity=262144), 64, 0)
    assert (p["tile_rows"], p["splits"]) == (32, 4)                    # 128 window rows, no entries
    p = dsv4.dsv4_decode_plan(_desc(dsv4, d_nope=128, d_rope=64), 64, 512)
    assert p["tensor_core"] == 0
    p = dsv4.dsv4_decode_plan(_desc(dsv4), 128, 512)
    assert p["head_groups"] == 2
    with pytest.raises(dsv4.Dsv4Error):
        dsv4.dsv4_decode_plan(_desc(dsv4), 64, -2)


def test_projection_rejects_bad_arguments_on_host(dsv4):
    d = _desc(dsv4)
    L = dsv4.lib
    c = _cache(dsv4)

    def proj(desc, cache, T=4, d_model=512, hidden=FAKE, weight=FAKE, base=10000.0, x=FAKE, u=FAKE):
        return L.dsv4_project_streams(ctypes.byref(desc), ctypes.byref(cache), T, d_model, hidden, weight,
                                      ctypes.c_float(base), x, FAKE, u, FAKE, None)

    assert proj(d, c, T=-1) == dsv4.ERR_INVALID_ARG
    assert proj(d, c, d_model=0) == dsv4.ERR_INVALID_ARG
    assert proj(d, c, base=1.0) == dsv4.ERR_INVALID_ARG
    assert proj(d, c, d_model=100) == dsv4.ERR_UNSUPPORTED                   # not a multiple of 64
    assert proj(_desc(dsv4, separate_v=1), c) == dsv4.ERR_UNSUPPORTED        # shared K = V only
    assert proj(_desc(dsv4, d_nope=40), c) == dsv4.ERR_UNSUPPORTED           # d_nope not a multiple of 32
    assert proj(d, c, hidden=FAKE + 2) == dsv4.ERR_MISALIGNED
    assert proj(d, c, u=None) == dsv4.ERR_INVALID_ARG                        # indexer streams missing
    assert proj(d, _cache(dsv4, n_tokens=0)) == dsv4.ERR_INVALID_ARG
    assert proj(d, c, T=0, hidden=None, weight=None, x=None, u=None) == dsv4.OK   # nothing to do
