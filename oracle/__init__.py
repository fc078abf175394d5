"""The oracle: a plain float64 CPU statement of CSA/HCA decode over the low-bit
compressed KV cache, written from the source pages (see ``method.py`` for the
citations and the readings taken).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code with
the CUDA library in ``compressed_sparse_kv_05_b300/`` and neither imports the
other; the seeded input generators in ``compressed_sparse_kv_05_b300/synth.py``
(random draws only, none of the method's arithmetic) serve both.

Every function here is pinned by a ``-m "not gpu"`` test against something other
than itself: format tables and a library conversion, closed forms, brute force
on tiny inputs, and the invariants listed in ``tests/test_oracle_*.py``.
"""
from .formats import (E2M1_MAX, E4M3_MAX, bf16_decode, bf16_encode, e2m1_decode,
                      e2m1_encode, e4m3_decode, e4m3_encode)
from .method import (attend, build_cache, csa_attend, dequant_fp4_rows,
                     dequant_kv_rows, hca_attend, index_scores, index_scores_causal,
                     lse_merge, multi_attend, pool_blocks, project_streams, quantize_fp4_rows,
                     quantize_kv_rows, query_positions, rope_rotate, topk_blocks, topk_boundary_gap,
                     window_tokens)
