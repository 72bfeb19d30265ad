"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each one.

Each mutant replaces one oracle function for the duration of one pin; the pin must
then fail.  This shows the pins in ``test_oracle_pins.py`` are strong enough to
reject the usual slips, not only that the oracle passes them.
"""

import numpy as np
import pytest

import oracle
from oracle import attention as A
from oracle import formats as F
import tests.test_oracle_pins as P
import tests.test_oracle_layouts as L
import tests.test_oracle_paged as PG
from oracle import paged as PGO
from oracle import passq as PQO
import tests.test_oracle_passq as PQ

_orig_attend = A.attend
_orig_merge = A.merge_lse
_orig_split = A.split_attention


def _attend_no_scale(q, k, v, scale, q_pos=None, kv_pos=None):
    return _orig_attend(q, k, v, 1.0, q_pos, kv_pos)


def _attend_causal_off_by_one(q, k, v, scale, q_pos=None, kv_pos=None):
    if q_pos is not None:
        q_pos = np.asarray(q_pos) - 1  # t < p instead of t <= p
    return _orig_attend(q, k, v, scale, q_pos, kv_pos)


def _attend_sign_flip(q, k, v, scale, q_pos=None, kv_pos=None):
    return _orig_attend(-np.asarray(q), k, v, scale, q_pos, kv_pos)


def _kv_head_interleaved(h, Hq, Hkv):
    return h % Hkv


def _merge_linear_weights(o_parts, lse_parts):
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    with np.errstate(all="ignore"):  # empty splits (lse = -inf) make this slip produce NaN
        w = lse_parts - lse_parts.min(axis=0) + 1.0  # weights not exponentiated
        o = (w[..., None] * np.asarray(o_parts)).sum(0) / w.sum(0)[..., None]
        return o, np.log(np.exp(lse_parts).sum(0))


def _merge_lse_without_max(o_parts, lse_parts):
    o, lse = _orig_merge(o_parts, lse_parts)
    m = np.asarray(lse_parts, dtype=np.float64).max(axis=0)
    return o, lse - np.where(np.isfinite(m), m, 0.0)  # dropped the "+ m" term


def _e4m3_bias8(codes):
    c = np.asarray(codes).astype(np.uint8)
    v = F.__dict__["_orig_e4m3"](c)
    return v / 2.0


def _split_ignores_seq_len(lo, hi, seq_len):
    return max(lo, 0), hi


_orig_gather = PGO.gather_pages


def _gather_row_and_block_swapped(pages, block_table, n_tokens):
    # token t taken from block table[b][t % L], row t // L (the two indices swapped)
    pages = np.asarray(pages)
    nb, Hkv, Lb, d = pages.shape
    table = np.asarray(block_table, dtype=np.int64)
    out = np.empty((table.shape[0], Hkv, n_tokens, d), dtype=pages.dtype)
    for b in range(table.shape[0]):
        for t in range(n_tokens):
            out[b, :, t] = pages[table[b, t % Lb] if t % Lb < table.shape[1] else 0, :, min(t // Lb, Lb - 1)]
    return out


def _gather_physical_order(pages, block_table, n_tokens):
    # block table ignored: physical blocks read in storage order
    pages = np.asarray(pages)
    table = np.asarray(block_table, dtype=np.int64)
    ident = np.arange(table.size).reshape(table.shape) % pages.shape[0]
    return _orig_gather(pages, ident, n_tokens)


def _visible_strict(q_pos, kv_pos):
    return np.asarray(kv_pos)[None, :] < np.asarray(q_pos)[:, None]  # t < p instead of t <= p


def _split_ignores_positions(q, k, v, seq_lens, split_bounds, causal_offset, scale, q_positions=None,
                             k_positions=None):
    return _orig_split(q, k, v, seq_lens, split_bounds, causal_offset, scale)  # storage index as position


def _split_swaps_positions(q, k, v, seq_lens, split_bounds, causal_offset, scale, q_positions=None,
                           k_positions=None):
    # each KV token's position taken from the wrong rank: the query chunk's layout repeated
    if q_positions is not None:
        S = np.asarray(k_positions).shape[1]
        reps = -(-S // np.asarray(q_positions).shape[1])
        k_positions = np.tile(np.asarray(q_positions), (1, reps))[:, :S]
    return _orig_split(q, k, v, seq_lens, split_bounds, causal_offset, scale, q_positions, k_positions)


_orig_rank_partial = PQO.rank_partial
_orig_gather_shards = PQO.gather_shards


def _rank_partial_without_batch_ids(q_block, batch_ids, k_local, v_local, lens_local, scale):
    # the block arrives without its batch ids: slot j reads the rank's entry of request j
    return _orig_rank_partial(q_block, list(range(len(batch_ids))), k_local, v_local, lens_local, scale)


def _return_to_computing_rank(arrived):
    # partials filed under the rank that computed them instead of the queries' owner
    N = len(arrived)
    received = [[None] * N for _ in range(N)]
    for k in range(N):
        for s in range(N):
            received[k][PQO.ring_source(k, s, N)] = arrived[k][s]
    return received


def _gather_shards_drops_last_rank(shards, shard_lens):
    lens = [list(r) for r in shard_lens]
    lens[-1] = [0] * len(lens[-1])
    return _orig_gather_shards(shards, lens)


MUTANTS = [
    ("attend without softmax scale", [(A, "attend", _attend_no_scale), (oracle, "attend", _attend_no_scale)],
     [P.test_golden_closed_forms]),
    ("causal mask off by one", [(A, "attend", _attend_causal_off_by_one)],
     [P.test_causal_offset_zero_is_dense_lower_triangle]),
    ("score sign flipped", [(A, "attend", _attend_sign_flip), (oracle, "attend", _attend_sign_flip)],
     [P.test_golden_closed_forms, P.test_two_tokens_is_a_logistic_blend]),
    ("interleaved GQA head map", [(A, "kv_head_of", _kv_head_interleaved)],
     [P.test_gqa_contiguous_groups]),
    ("merge weights not exponentiated", [(A, "merge_lse", _merge_linear_weights),
                                         (oracle, "merge_lse", _merge_linear_weights)],
     [P.test_merge_two_fragments_closed_form_and_empty_split, P.test_merged_fragments_merge_again]),
    ("merged lse drops the max", [(A, "merge_lse", _merge_lse_without_max),
                                  (oracle, "merge_lse", _merge_lse_without_max)],
     [P.test_merge_two_fragments_closed_form_and_empty_split, P.test_merged_fragments_merge_again]),
    ("e4m3 exponent bias 8", [(oracle, "e4m3_bits_to_f64", _e4m3_bias8)],
     [P.test_e4m3_all_codes_match_torch]),
    ("split not clipped to seq_len", [(A, "_visible_range", _split_ignores_seq_len)],
     [P.test_split_past_seq_len_is_empty_and_poison_is_never_read]),
    ("positional mask strict", [(A, "visible_mask", _visible_strict)],
     [L.test_every_zigzag_rank_processes_132_kv_positions, L.test_layout_attention_brute_force_tiny]),
    ("positions ignored", [(A, "split_attention", _split_ignores_positions)],
     [L.test_layout_attention_equals_original_order_attention]),
    ("KV positions from the wrong rank", [(A, "split_attention", _split_swaps_positions)],
     [L.test_layout_attention_equals_original_order_attention]),
    ("paged gather: row and block index swapped", [(PGO, "gather_pages", _gather_row_and_block_swapped),
                                                   (oracle, "gather_pages", _gather_row_and_block_swapped)],
     [PG.test_hand_worked_gather, PG.test_gather_inverts_the_generators_scatter_bf16]),
    ("paged gather ignores the block table", [(PGO, "gather_pages", _gather_physical_order),
                                              (oracle, "gather_pages", _gather_physical_order)],
     [PG.test_hand_worked_gather, PG.test_gather_inverts_the_generators_scatter_bf16]),
    ("pass-Q block travels without its batch ids", [(PQO, "rank_partial", _rank_partial_without_batch_ids)],
     [PQ.test_zero_query_is_the_mean_value_over_every_rank_and_log_count,
      PQ.test_one_token_per_request_returns_its_value_row]),
    ("pass-Q partials kept by the computing rank", [(PQO, "return_to_owners", _return_to_computing_rank)],
     [PQ.test_zero_query_is_the_mean_value_over_every_rank_and_log_count,
      PQ.test_one_token_per_request_returns_its_value_row]),
    ("shard gather drops the last rank", [(PQO, "gather_shards", _gather_shards_drops_last_rank),
                                          (oracle, "gather_shards", _gather_shards_drops_last_rank)],
     [PQ.test_hand_worked_gather]),
]


def _run_pin(fn):
    import inspect
    import json
    import os

    if fn is L.test_layout_attention_equals_original_order_attention:
        fn("zigzag", 32, 4)
        fn("striped", 24, 3)
    elif fn is P.test_golden_closed_forms:
        cases = json.load(open(os.path.join(P.GOLDEN, "closed_form_attention.json")))["cases"]
        for c in cases:
            fn(c)
    elif "seed" in inspect.signature(fn).parameters:
        fn(0)
    else:
        fn()


@pytest.mark.parametrize("name,patches,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, patches, pins, monkeypatch):
    F.__dict__.setdefault("_orig_e4m3", F.e4m3_bits_to_f64)
    for mod, attr, repl in patches:
        monkeypatch.setattr(mod, attr, repl)
    for pin in pins:
        with pytest.raises(AssertionError):
            _run_pin(pin)


def test_unmutated_pins_pass():
    for _, _, pins in MUTANTS:
        for pin in pins:
            _run_pin(pin)
