"""Each pin must catch a plausible mistake: plant one in the oracle (CPU only,
via monkeypatch) and check that the corresponding pin fails."""
import numpy as np
import pytest

import oracle as O
import oracle.formats as F
import oracle.method as M
from tests import test_oracle_formats as TF
from tests import test_oracle_method as TM


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def _patch(monkeypatch, name, fn, *mods):
    for mod in (O,) + mods:
        monkeypatch.setattr(mod, name, fn)


def test_pooling_without_bias_is_caught(monkeypatch):
    orig = M.pool_blocks
    _patch(monkeypatch, "pool_blocks", lambda x, z, b, m: orig(x, z, np.zeros_like(b), m), M)
    _fails(TM.test_pool_ratio2_closed_form)


def test_pooling_unnormalised_weights_are_caught(monkeypatch):
    def bad(x, z, b, m):
        xd = F.bf16_decode(x)
        nb = xd.shape[0] // m
        lg = F.bf16_decode(z)[: nb * m].reshape(nb, m, -1) + b[None]
        return (np.exp(lg - lg.max(axis=1, keepdims=True)) * xd[: nb * m].reshape(nb, m, -1)).sum(1).astype(np.float32)
    _patch(monkeypatch, "pool_blocks", bad, M)
    _fails(TM.test_pool_zero_gates_is_mean)


def test_round_half_away_is_caught(monkeypatch):
    def bad_grid(a, mant_bits, emin):
        a = np.asarray(a, np.float64)
        _, ex = np.frexp(a)
        q = np.ldexp(1.0, np.maximum(ex - 1, emin) - mant_bits)
        return np.floor(a / q + 0.5) * q
    monkeypatch.setattr(F, "_round_to_grid", bad_grid)
    _fails(TF.test_e4m3_encode_midpoints_and_neighbours)
    _fails(TF.test_e2m1_tie_table)


def test_swapped_fp4_nibbles_are_caught(monkeypatch):
    orig = M.quantize_fp4_rows

    def bad(y):
        c, s = orig(y)
        return ((c >> 4) | (c << 4)).astype(np.uint8), s
    _patch(monkeypatch, "quantize_fp4_rows", bad, M)
    _fails(TM.test_fp4_quant_exact_on_representable_rows_and_nibble_order)


def test_missing_relu_is_caught(monkeypatch):
    def bad(kc, ks, q, w):
        Q = M.dequant_fp4_rows(*M.quantize_fp4_rows(F.bf16_decode(q).astype(np.float32)))
        return (M.dequant_fp4_rows(kc, ks) @ Q.T * w[None].astype(np.float64)).sum(1)
    _patch(monkeypatch, "index_scores", bad, M)
    _fails(TM.test_index_scores_single_head_is_relu_dot)


def test_transposed_indexer_operand_is_caught(monkeypatch):
    def bad(kc, ks, q, w):
        Q = M.dequant_fp4_rows(*M.quantize_fp4_rows(F.bf16_decode(q).astype(np.float32)))
        K = M.dequant_fp4_rows(kc, ks)
        K = K[:, ::-1]                       # dims reversed: a plausible layout slip
        return (np.maximum(K @ Q.T, 0) * w[None].astype(np.float64)).sum(1)
    _patch(monkeypatch, "index_scores", bad, M)
    _fails(TM.test_index_scores_exact_rational)


def test_topk_wrong_tie_rule_is_caught(monkeypatch):
    def bad(scores, k):
        s = np.asarray(scores, np.float64)
        order = np.lexsort((-np.arange(s.shape[0]), -s))
        sel = np.sort(order[: min(k, s.shape[0])]).astype(np.int32)
        return np.concatenate([sel, np.full(k - sel.shape[0], -1, np.int32)])
    _patch(monkeypatch, "topk_blocks", bad, M)
    for seed in range(6):
        try:
            TM.test_topk_matches_brute_force_with_ties(seed)
        except AssertionError:
            return
    pytest.fail("tie rule slip not caught")


def test_missing_softmax_scale_is_caught(monkeypatch):
    orig = M.attend
    _patch(monkeypatch, "attend", lambda q, K, V, s: orig(q, K, V, 1.0), M)
    _fails(TM.test_attend_matches_sdpa_fp64)


def test_window_one_token_short_is_caught(monkeypatch):
    monkeypatch.setattr(M, "window_tokens", lambda n, W: np.arange(max(0, n - W + 1), n))
    _fails(TM.test_csa_is_merge_of_window_and_selected_partials)


def test_scale_dropped_from_dequant_is_caught(monkeypatch):
    _patch(monkeypatch, "dequant_kv_rows",
           lambda nope, scale, rope: np.concatenate([F.e4m3_decode(nope), F.bf16_decode(rope)], axis=1), M)
    _fails(TM.test_csa_ratio1_all_selected_no_window_is_full_attention)


def test_dequant_row_slip_is_caught(monkeypatch):
    # each row takes its neighbour's scale (a row slip between the code and scale planes)
    _patch(monkeypatch, "dequant_kv_rows",
           lambda nope, scale, rope: np.concatenate([F.e4m3_decode(nope) * np.roll(np.asarray(scale, np.float64), 1)[:, None],
                                                     F.bf16_decode(rope)], axis=1), M)
    _fails(TM.test_dequant_kv_rows_against_library_decode)


def test_dequant_rope_block_dropped_is_caught(monkeypatch):
    _patch(monkeypatch, "dequant_kv_rows",
           lambda nope, scale, rope: np.concatenate([F.e4m3_decode(nope) * np.asarray(scale, np.float64)[:, None],
                                                     np.zeros(np.shape(rope))], axis=1), M)
    _fails(TM.test_dequant_kv_rows_against_library_decode)


def test_multi_token_window_one_token_long_is_caught(monkeypatch):
    # each query's window reaching one token further back than W
    orig = M.multi_attend

    def bad(q, sm, sel, n, ratio, W, *planes):
        return orig(q, sm, sel, n, ratio, W + 1, *planes[:3], np.concatenate([planes[3][:1], planes[3]]),
                    *planes[4:7], *([np.concatenate([planes[7][:1], planes[7]])] if len(planes) > 7 else []))
    _patch(monkeypatch, "multi_attend", bad, M)
    _fails(TM.test_multi_token_step_equals_single_token_decode_on_each_prefix, 90, 7)


def test_multi_token_selection_not_causal_is_caught(monkeypatch):
    # every query scoring all blocks of the sequence instead of those complete at its position
    def bad(codes, scales, q, w, n, ratio):
        return [M.index_scores(codes[: n // ratio], scales[: n // ratio], q[t], w[t]) for t in range(q.shape[0])]
    _patch(monkeypatch, "index_scores_causal", bad, M)
    # caught by the pin's comparison, or by the attention refusing a block not yet complete
    with pytest.raises((AssertionError, ValueError)):
        TM.test_multi_token_step_equals_single_token_decode_on_each_prefix(90, 7)


def test_rope_sin_sign_flipped_is_caught(monkeypatch):
    orig = M.rope_rotate
    _patch(monkeypatch, "rope_rotate", lambda x, pos, base: orig(x, -np.asarray(pos, np.float64), base), M)
    _fails(TM.test_rope_pairs_are_adjacent_dims_with_geometric_frequencies)


def test_rope_half_split_pairs_are_caught(monkeypatch):
    orig = M.rope_rotate

    def bad(x, pos, base):
        x = np.asarray(x, np.float64)
        d = x.shape[-1]
        perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])   # (i, i + d/2) pairs
        inv = np.argsort(perm)
        return orig(x[..., inv], pos, base)[..., perm]
    _patch(monkeypatch, "rope_rotate", bad, M)
    _fails(TM.test_rope_pairs_are_adjacent_dims_with_geometric_frequencies)


def test_rope_wrong_frequency_exponent_is_caught(monkeypatch):
    def bad(x, pos, base):
        x = np.asarray(x, np.float64)
        d = x.shape[-1]
        theta = float(base) ** (-np.arange(d // 2) / d)            # -i/d instead of -2i/d
        ang = np.asarray(pos, np.float64).reshape(-1, 1) * theta[None, :]
        out = np.empty_like(x)
        out[..., 0::2] = x[..., 0::2] * np.cos(ang) - x[..., 1::2] * np.sin(ang)
        out[..., 1::2] = x[..., 0::2] * np.sin(ang) + x[..., 1::2] * np.cos(ang)
        return out
    _patch(monkeypatch, "rope_rotate", bad, M)
    _fails(TM.test_rope_pairs_are_adjacent_dims_with_geometric_frequencies)


def test_projection_rope_on_leading_dims_is_caught(monkeypatch):
    orig = M.project_streams

    def bad(h_bits, w_bits, d_nope, d_rope, idx_dim, pos, base):
        h, w = O.bf16_decode(h_bits), O.bf16_decode(w_bits)
        D = d_nope + d_rope
        y = h @ w.T
        x = y[:, :D].copy()
        x[:, :d_rope] = M.rope_rotate(x[:, :d_rope], pos, base)   # the leading dims rotated
        u = y[:, 2 * D:2 * D + idx_dim].copy()
        return tuple(O.bf16_encode(a) for a in (x, y[:, D:2 * D], u, y[:, 2 * D + idx_dim:]))
    _patch(monkeypatch, "project_streams", bad, M)
    _fails(TM.test_project_streams_one_hot_hidden_rows_pick_weight_columns)


def test_projection_streams_swapped_is_caught(monkeypatch):
    orig = M.project_streams

    def bad(*a):
        x, z, u, zu = orig(*a)
        return x, z, zu, u
    _patch(monkeypatch, "project_streams", bad, M)
    _fails(TM.test_project_streams_small_integers_are_exact_dot_products)
