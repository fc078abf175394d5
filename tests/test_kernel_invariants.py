"""Index arithmetic the kernels rely on, checked on the host.

These are properties of the kernels' own layouts (compressed_sparse_kv_05_b300/csrc/
attention_tc.cu, and compress.cu's clustered pooling), not of the method: the
constants and shape rules below restate those files' (and kernels.h's).
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


# ----------------------------------------------------------------------------- clustered pooling


def _pool_shape(m, C):
    """kernels.h pool_shape: channel groups of 8, up to 512 threads a team."""
    cg = C // 8
    G = (m + 7) // 8
    gmax = 512 // cg if cg <= 512 else 1
    G = max(1, min(G, gmax))
    return cg, G, -(-m // G)


def _slice_cpt(G):
    return 2 if G <= 8 else (4 if G <= 16 else 8)


@pytest.mark.parametrize("D", range(64, 513, 64))
@pytest.mark.parametrize("two", [False, True])
def test_cluster_pooling_fits_and_covers(D, two):
    """For every ratio the clustered pooling takes (9..256) and every D it takes
    (multiples of 64 up to 512): the CTA has 64 to 256 threads;
    its shared memory (bias, z, x (, v), the combine buffer, four words, the
    pooled slice) fits the 200 KB the launch allows; pool_slice's threads cover
    every (channel, token group) of the 64-channel slice exactly once; the
    combine buffer's largest index is inside its G x 8 x (16 | 24) floats; the
    token groups tile [0, ratio); cp.async sources stay 16-byte aligned."""
    S = 3 if two else 2
    for m in range(9, 257):
        _, G, tpg = _pool_shape(m, D)
        cpt = _slice_cpt(G)
        threads = 64 * G // cpt
        assert 64 <= threads <= 256 and 64 * G % cpt == 0, (m, G)
        part = G * 8 * (24 if two else 16)
        smem = m * 64 * (4 + 2 * (3 if two else 2)) + part * 4 + 4 * 4 + 128 * 4
        assert smem <= 200 * 1024, (m, smem)
        seen = set()
        top = -1
        for t in range(threads):
            q, g = t % (64 // cpt), t // (64 // cpt)
            assert g < G
            for k in range(cpt):
                c = q * cpt + k
                assert (c, g) not in seen
                seen.add((c, g))
                top = max(top, (g * 64 + c) * S + S - 1)
        assert len(seen) == 64 * G
        assert top < part
        toks = [i for g in range(G) for i in range(g * tpg, min(g * tpg + tpg, m))]
        assert toks == list(range(m))
        assert (D * 2) % 16 == 0 and (64 * 2) % 16 == 0 and (D * 4) % 16 == 0

