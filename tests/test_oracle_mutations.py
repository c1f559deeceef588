"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch them.

Each mutation replaces one oracle function with a subtly wrong variant; at least
one pin from ``test_oracle_pins`` must then fail.
"""
import numpy as np
import pytest

from oracle import hs2_oracle as O
import tests.test_oracle_pins as P


def _sel_no_lse(x, lse, n_far):  # dropped per-head normaliser
    return np.exp(x[:, :n_far]).sum(axis=0) if n_far > 0 else np.zeros(0)


def _sel_max_not_sum(x, lse, n_far):  # heads combined by max instead of sum
    return np.exp(x[:, :n_far] - lse[:, None]).max(axis=0) if n_far > 0 else np.zeros(0)


def _topk_upper_ties(score, k):  # ties to the higher position
    n = len(score)
    kk = min(int(k), n)
    order = np.lexsort((-np.arange(n), -np.asarray(score)))
    return np.sort(order[:kk])


def _far_off_by_one(t, w):
    return max(0, t - w + 1)


def _window_short(t, w):
    return np.arange(max(0, t - w + 1), t, dtype=np.int64)


def _full_attn_transposed(q, K, V, scale):  # softmax over the wrong axis
    x = (q @ K.T) * float(scale)
    m = x.max(axis=0, keepdims=True)
    p = np.exp(x - m)
    p /= p.sum(axis=0, keepdims=True)
    lse = np.log(np.exp(x).sum(axis=1))
    return x, lse, p @ V


def _sparse_two_softmaxes(q, K, V, scale, sink=None):  # window and far positions normalised apart
    half = max(1, K.shape[0] // 2)
    outs = []
    for sl in (slice(0, half), slice(half, None)):
        x = (q @ K[sl].T) * float(scale)
        if x.shape[1] == 0:
            continue
        p = np.exp(x - x.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        outs.append(p @ V[sl])
    return sum(outs) / len(outs)


_sparse_ref = O.sparse_attention


def _sparse_sink_ignored(q, K, V, scale, sink=None):  # sink bias dropped
    return _sparse_ref(q, K, V, scale)


def _sparse_sink_base2(q, K, V, scale, sink=None):  # sink added as 2^b instead of e^b
    return _sparse_ref(q, K, V, scale, None if sink is None else np.asarray(sink) * np.log(2.0))


def _gate_wrong_side(o, gate):  # o * (1 - sigmoid(g))
    return o if gate is None else o / (1.0 + np.exp(np.asarray(gate, np.float64)))


def _block_topk_mean(score, k, blk):  # block key = mean instead of max
    n = len(score)
    nb = (n + blk - 1) // blk
    kb = min(int(k) // blk, nb)
    if kb <= 0:
        return np.zeros(0, dtype=np.int64)
    keys = np.array([np.mean(score[b * blk:min(n, b * blk + blk)]) for b in range(nb)])
    blocks = np.sort(np.lexsort((np.arange(nb), -keys))[:kb])
    return np.concatenate([np.arange(b * blk, min(n, b * blk + blk)) for b in blocks]).astype(np.int64)


def _fp8_bias8(b):  # exponent bias 8 instead of 7
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e, m = (b >> 3) & 0xF, b & 0x7
    mag = np.where(e == 0, m * 2.0 ** -10, (1.0 + m / 8.0) * np.exp2(e - 8.0))
    return np.where((e == 15) & (m == 7), np.nan, sign * mag)


def _lightning_no_relu(q_idx, w_idx, K):
    return (np.asarray(w_idx)[:, None] * (q_idx @ K.T)).sum(axis=0)


def _block_max_past_t(I, t, blk):
    nb = (t + blk - 1) // blk
    padded = np.concatenate([I, np.full(nb * blk - len(I), 1e9)])
    return padded.reshape(nb, blk).max(axis=1)


def _gather_wrong_slot(pool, bt_row, g, positions, page, dtype):
    positions = np.asarray(positions, dtype=np.int64)
    pages = np.asarray(bt_row, dtype=np.int64)[positions // page]
    return O.to_f64(pool[pages, g, (positions + 1) % page, :], dtype)


def _append_past_current(kv, k_new, v_new=None):
    """Writes the new rows one position late (at t instead of t-1)."""
    import copy
    out = copy.copy(kv)
    out.k, out.v = np.array(kv.k, copy=True), np.array(kv.v, copy=True)
    for b in range(len(kv.seq_len)):
        pos = int(kv.seq_len[b])
        pg = int(kv.block_table[b][min(pos // kv.page, kv.block_table.shape[1] - 1)])
        out.k[pg, :, pos % kv.page, :] = k_new[b]
        out.v[pg, :, pos % kv.page, :] = v_new[b]
    return out


def _fp4_high_nibble_first(packed):
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = packed >> 4
    out[..., 1::2] = packed & 0xF
    return out


def _fp4_bias2(c):
    c = np.asarray(c, dtype=np.uint8).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    e, m = (c >> 1) & 0x3, c & 0x1
    return sign * np.where(e == 0, m * 0.25, (1.0 + m / 2.0) * np.exp2(e - 2.0))


def _sa_rows_variant(t_of, idx_row, gate_rows):
    """sa_prefill_rows with one of its three row bookkeeping choices swapped out."""
    def f(q, kv, rows, w, idx, cnt, scale, sink=None, gate=None):
        rows = np.asarray(rows, dtype=np.int64)
        qf = O.to_f64(q, O._qdtype(kv))
        _, Hq, d = qf.shape
        Hkv = kv.k.shape[1]
        G = Hq // Hkv
        o = np.zeros((len(rows), Hq, d))
        for r, i in enumerate(rows):
            t = t_of(int(i))
            j = idx_row(r, int(i))
            for g in range(Hkv):
                U = O._union(t, w, idx[j, g, :cnt[j, g]])
                K = O.gather_rows(kv.k, kv.block_table[0], g, U, kv.page, kv.dtype, O._scale(kv, "k"))
                V = O.gather_rows(kv.v, kv.block_table[0], g, U, kv.page, kv.dtype, O._scale(kv, "v"))
                hs = slice(g * G, (g + 1) * G)
                o[r, hs] = O.sparse_attention(qf[i, hs], K, V, scale, None if sink is None else np.asarray(sink)[hs])
        return O.output_gate(o, None if gate is None else O.to_f64(np.asarray(gate)[gate_rows(rows)], "f32"))
    return f


_sa_rows_t_is_i = _sa_rows_variant(lambda i: i, lambda r, i: i, lambda rows: rows)  # t = i, not i + 1
_sa_rows_t_is_i.__name__ = "_sa_rows_t_is_i"
_sa_rows_idx_by_sample = _sa_rows_variant(lambda i: i + 1, lambda r, i: r, lambda rows: rows)  # idx[r]
_sa_rows_idx_by_sample.__name__ = "_sa_rows_idx_by_sample"
_sa_rows_gate_by_sample = _sa_rows_variant(lambda i: i + 1, lambda r, i: i,
                                           lambda rows: np.arange(len(rows)))  # gate[r]
_sa_rows_gate_by_sample.__name__ = "_sa_rows_gate_by_sample"


def _bf16_as_f16(x, dtype):  # bf16 bit patterns read as IEEE half
    if dtype == "bf16":
        return np.ascontiguousarray(x, dtype=np.uint16).view(np.float16).astype(np.float64)
    return _to_f64_ref(x, dtype)


_to_f64_ref = O.to_f64


MUTATIONS = [
    ("selection_scores", _sel_no_lse),
    ("selection_scores", _sel_max_not_sum),
    ("topk_lower_index", _topk_upper_ties),
    ("far_count", _far_off_by_one),
    ("window", _window_short),
    ("full_attention", _full_attn_transposed),
    ("sparse_attention", _sparse_two_softmaxes),
    ("lightning_scores", _lightning_no_relu),
    ("block_max", _block_max_past_t),
    ("gather_rows", _gather_wrong_slot),
    ("sparse_attention", _sparse_sink_ignored),
    ("sparse_attention", _sparse_sink_base2),
    ("output_gate", _gate_wrong_side),
    ("block_topk", _block_topk_mean),
    ("fp8_e4m3_to_f64", _fp8_bias8),
    ("kv_append", _append_past_current),
    ("fp4_unpack", _fp4_high_nibble_first),
    ("fp4_e2m1_to_f64", _fp4_bias2),
    ("sa_prefill_rows", _sa_rows_t_is_i),
    ("sa_prefill_rows", _sa_rows_idx_by_sample),
    ("sa_prefill_rows", _sa_rows_gate_by_sample),
    ("to_f64", _bf16_as_f16),
]

PINS = [
    lambda: P.test_fa_prefill_matches_masked_dense(4, 2),
    P.test_fa_closed_forms,
    P.test_gather_rows_follows_block_table,
    P.test_window_and_far_range_match_one_based_statement,
    P.test_selection_scores_against_ratio_form,
    *[(lambda s=s: P.test_topk_is_best_subset_bruteforce(s)) for s in range(6)],
    P.test_selection_invariants_and_short_context,
    P.test_ties_go_to_lower_position,
    P.test_sa_equals_dense_when_k_covers_far_range,
    P.test_sa_window_zero_with_everything_selected_is_dense,
    P.test_sa_renormalisation_error_bound,
    P.test_lightning_score_special_cases,
    P.test_block_max_bruteforce_and_tail,
    P.test_reindex_over_all_blocks_is_flat_indexer,
    P.test_csa2_attention_over_whole_pool_is_dense_over_pool,
    P.test_sa_sink_limits_and_closed_form,
    P.test_output_gate_limits,
    P.test_sa_decode_sink_and_gate_reach_their_heads,
    P.test_block_topk_with_unit_blocks_is_token_topk,
    P.test_block_topk_bruteforce_and_invariants,
    P.test_block_decode_selection_respects_window_and_budget,
    P.test_fp8_e4m3_values_from_the_format,
    P.test_fp8_encoder_rounds_to_nearest_even,
    lambda: P.test_kv_append_writes_exactly_the_current_token_row("bf16"),
    P.test_fa_after_append_is_dense_over_sequence_ending_in_new_row,
    P.test_fp4_e2m1_values_from_the_format,
    P.test_fp4_unpack_channel_order,
    P.test_oracle_on_fp4_pool_equals_oracle_on_its_dequantised_values,
    *[(lambda sg=sg: P.test_sa_prefill_rows_dense_when_k_covers_far_range(sg)) for sg in (False, True)],
    *[(lambda sg=sg: P.test_sa_prefill_rows_partial_sets_bruteforce(sg)) for sg in (False, True)],
    P.test_sa_prefill_last_row_equals_decode,
    P.test_bf16_widening_known_bit_patterns,
]


@pytest.mark.parametrize("name,fn", MUTATIONS, ids=[f"{n}:{f.__name__}" for n, f in MUTATIONS])
def test_some_pin_catches_mutation(monkeypatch, name, fn):
    monkeypatch.setattr(O, name, fn)
    caught = 0
    for pin in PINS:
        try:
            pin()
        except Exception:  # noqa: BLE001 - any failure of a pin counts as a catch
            caught += 1
    assert caught > 0, f"no pin caught the mutation of {name}"
