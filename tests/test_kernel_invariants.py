"""Index arithmetic the tensor-core attention kernel relies on, checked on the host.

These are properties of the kernel's own layouts (compressed_sparse_kv_05_b300/csrc/
attention_tc.cu), not of the method: the constants below restate that file's.
"""
import math

import pytest

K_WORKERS = 14 * 32          # worker warps 2-15
K_ROWS = 128                 # rows of a tile (MMA M)
K_ATOM_BYTES = K_ROWS * 128  # one 64-dim f16 swizzle atom of a chunk
K_ITEMS = math.ceil(K_ROWS * 16 / K_WORKERS)


@pytest.mark.parametrize("nch", range(1, 17))
def test_query_head_reciprocal_is_exact(nch):
    """Query staging: head = ((i >> 4) * ceil(2^16 / nch)) >> 16 equals i // (16 nch)
    for every 8-dim group index i of up to 128 heads (D = 128 nch)."""
    rcp = (65536 + nch - 1) // nch
    gpr = 16 * nch
    for i in range(128 * gpr):
        assert ((i >> 4) * rcp) >> 16 == i // gpr


@pytest.mark.parametrize("rc", range(16, K_ROWS + 1, 16))
def test_code_chunk_dequantisation_is_warp_local(rc):
    """A chunk of 128 code dims is dequantised in place with only a warp barrier
    between the read and write phases: every byte a warp writes is read (as a raw
    code) by no other warp. Item i = worker + it * workers is row i // 16, 8-dim
    group i % 16; raw codes of row j sit at [128 j, 128 j + 128); the f16 output of
    group g goes to atom g // 8, row j, granule (g % 8) ^ (j % 8)."""
    readers, writers = {}, {}
    for it in range(K_ITEMS):
        for w in range(K_WORKERS):
            i = w + it * K_WORKERS
            if i >= rc * 16:
                continue
            j, g = i >> 4, i & 15
            warp = w >> 5
            for byte in range(128 * j + 8 * g, 128 * j + 8 * g + 8):
                readers.setdefault(byte, set()).add(warp)
            base = (g >> 3) * K_ATOM_BYTES + j * 128 + (((g & 7) ^ (j & 7)) << 4)
            for byte in range(base, base + 16):
                writers.setdefault(byte, set()).add(warp)
    assert len(writers) == rc * 256   # every f16 byte of the rows written once
    for byte, ws in writers.items():
        assert len(ws) == 1
        assert readers.get(byte, set()) <= ws
