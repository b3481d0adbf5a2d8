"""Pin strength: plant one plausible mistake at a time in the oracle (on the
CPU, by monkeypatching) and check that at least one pin test fails.  The
oracle itself is never modified."""

import numpy as np
import pytest

import oracle.mla as O
from tests import test_oracle_decode as D
from tests import test_oracle_gather_prefill as G
from tests import test_oracle_rope as RP


def _fails(*pins):
    for pin in pins:
        try:
            pin()
        except AssertionError:
            return True
    return False


def test_causal_off_by_one(monkeypatch):
    orig = O.decode_range

    def bad(seq_len, q_len, i, causal, kv_start=None, kv_end=None):
        lo, hi = orig(seq_len, q_len, i, causal, kv_start, kv_end)
        return (lo, max(lo, hi - 1)) if causal else (lo, hi)
    monkeypatch.setattr(O, "decode_range", bad)
    assert _fails(D.test_paged_addressing_matches_contiguous,
                  D.test_causal_pair_reduces_to_single_token_decode)


def test_lse_without_max_term(monkeypatch):
    def bad(q_rows, keys, values, sm_scale):
        H = q_rows.shape[0]
        if keys.shape[0] == 0:
            return np.zeros((H, values.shape[1])), np.full(H, -np.inf)
        s = sm_scale * (q_rows @ keys.T)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        z = e.sum(axis=1, keepdims=True)
        return (e / z) @ values, np.log(z)[:, 0]          # forgot + m
    monkeypatch.setattr(O, "attend", bad)
    assert _fails(D.test_attend_brute_force, D.test_attend_golden_two_keys)


def test_scale_missing_in_scores(monkeypatch):
    orig = O.attend
    monkeypatch.setattr(O, "attend", lambda q, k, v, s: orig(q, k, v, 1.0))
    assert _fails(D.test_attend_brute_force, D.test_attend_golden_two_keys)


def test_merge_weight_sign(monkeypatch):
    def bad(parts_out, parts_lse):
        parts_lse = np.asarray(parts_lse, float)
        m = parts_lse.max(axis=0)
        w = np.exp(m[None] - parts_lse)                     # inverted
        z = w.sum(axis=0)
        return (np.asarray(parts_out) * w[..., None]).sum(0) / z[..., None], m + np.log(z)
    monkeypatch.setattr(O, "merge_states", bad)
    assert _fails(lambda: D.test_merge_of_shards_equals_unsplit("contiguous"))


def test_absorb_wrong_contraction(monkeypatch):
    def bad(q_nope, q_pe, w_uk_t):
        # contracts over the wrong weight axis pattern (per-head transpose)
        ql = np.einsum("thp,hpl->thl", q_nope[..., ::-1], w_uk_t)
        return np.concatenate([ql, q_pe], axis=-1)
    monkeypatch.setattr(O, "absorb_q", bad)
    assert _fails(D.test_absorb_brute_force, D.test_absorbed_mqa_equals_expanded_mha)


def test_v_up_transposed_weight(monkeypatch):
    monkeypatch.setattr(O, "v_up", lambda o, w: np.einsum("thl,hvl->thv", o, w[:, ::-1]))
    assert _fails(D.test_v_up_brute_force, D.test_absorbed_mqa_equals_expanded_mha)


def test_expand_swapped_halves(monkeypatch):
    orig = O.expand_kv

    def bad(kv_rows, w_kvb, H, heads=None):
        w = np.asarray(w_kvb).reshape(H, 256, 512)[:, ::-1].reshape(H * 256, 512)
        return orig(kv_rows, w, H, heads)
    monkeypatch.setattr(O, "expand_kv", bad)
    assert _fails(G.test_expand_brute_force, D.test_absorbed_mqa_equals_expanded_mha)


def test_reorg_ignores_interleave(monkeypatch):
    monkeypatch.setattr(O, "shard_local_index",
                        lambda t, W, I: (np.asarray(t) % W, np.asarray(t) // W))
    assert _fails(lambda: G.test_reorg_inverts_interleaved_sharding(4, 3),
                  G.test_shard_local_index_is_a_bijection)


def test_gather_ignores_seq_starts(monkeypatch):
    orig = O.gather_cache
    monkeypatch.setattr(O, "gather_cache",
                        lambda c, bt, cu, seq_starts=None: orig(c, bt, cu, None))
    assert _fails(G.test_gather_seq_starts_equals_slice_of_full_gather)


def test_prefill_causal_shift(monkeypatch):
    orig = O.prefill_attention

    def bad(q, k, v, cu_q, cu_k, causal, sm_scale, q_rows=None):
        if causal:   # aligns the mask top-left instead of bottom-right
            cu_k2 = np.asarray(cu_k).copy()
            return orig(q, k, v, cu_q, cu_k2, True, sm_scale * 1.01, q_rows)
        return orig(q, k, v, cu_q, cu_k, causal, sm_scale, q_rows)
    monkeypatch.setattr(O, "prefill_attention", bad)
    assert _fails(G.test_prefill_causal_brute_force,
                  lambda: G.test_chunked_prefill_equals_full_attention(2))


def test_rope_sin_sign_flipped(monkeypatch):
    """A rotation by -theta keeps norms and relative positions: only the
    hand-worked example catches it."""
    orig = O.rope
    monkeypatch.setattr(O, "rope", lambda x, p, base=10000.0, interleaved=True:
                        orig(x, -np.asarray(p), base, interleaved))
    assert _fails(lambda: RP.test_rope_matches_hand_worked_example(True, "interleaved"))


def test_rope_frequency_exponent_wrong(monkeypatch):
    monkeypatch.setattr(O, "rope_inv_freq", lambda dim=64, base=10000.0:
                        float(base) ** (-np.arange(dim // 2, dtype=np.float64) / dim))
    assert _fails(lambda: RP.test_rope_matches_hand_worked_example(True, "interleaved"))


def test_rope_pairs_wrong(monkeypatch):
    """Pairs taken as (i, i + d/2) where (2i, 2i + 1) is meant."""
    orig = O.rope
    monkeypatch.setattr(O, "rope", lambda x, p, base=10000.0, interleaved=True:
                        orig(x, p, base, not interleaved))
    assert _fails(lambda: RP.test_rope_matches_hand_worked_example(True, "interleaved"),
                  RP.test_rope_layouts_agree_under_the_pairing_permutation)


def test_cache_write_skips_no_padding(monkeypatch):
    orig = O.cache_write
    monkeypatch.setattr(O, "cache_write", lambda c, kv, kp, slots, dt="bf16", ks=1.0:
                        orig(c, kv, kp, np.abs(np.asarray(slots)), dt, ks))
    assert _fails(lambda: RP.test_cache_write_then_gather_returns_the_rows("bf16"))
