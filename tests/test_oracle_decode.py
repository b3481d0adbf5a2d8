"""Pins for the oracle's absorb / decode / merge / v_up definitions.

Each test checks the oracle against something other than itself: scalar
brute force with math.exp, closed forms, and the identities the pages fix
(absorbed MQA == expanded MHA; merged shards == unsplit attention)."""

import json
import math
import os

import numpy as np
import pytest

from oracle import mla

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(s):
    return np.random.Generator(np.random.PCG64(s))


def _brute_attend(q, K, Vv, scale):
    """Scalar loops, math.exp, no numpy reductions."""
    H, n = len(q), len(K)
    outs, lses = [], []
    for h in range(H):
        s = [scale * sum(float(q[h][d]) * float(K[j][d]) for d in range(len(q[h])))
             for j in range(n)]
        m = max(s)
        z = sum(math.exp(x - m) for x in s)
        lse = m + math.log(z)
        o = [sum(math.exp(s[j] - lse) * float(Vv[j][c]) for j in range(n))
             for c in range(len(Vv[0]))]
        outs.append(o)
        lses.append(lse)
    return np.array(outs), np.array(lses)


def test_attend_brute_force():
    g = _rng(1)
    q, K, Vv = g.standard_normal((3, 7)), g.standard_normal((5, 7)), g.standard_normal((5, 4))
    o, l = mla.attend(q, K, Vv, 0.37)
    ob, lb = _brute_attend(q, K, Vv, 0.37)
    assert np.allclose(o, ob, atol=1e-13, rtol=0)
    assert np.allclose(l, lb, atol=1e-13, rtol=0)


def test_attend_golden_two_keys():
    with open(os.path.join(GOLDEN, "decode_two_keys.json")) as f:
        g = json.load(f)
    q = np.array(g["q"], float)[None]
    K = np.array(g["keys"], float)
    Vv = np.array(g["values"], float)
    o, l = mla.attend(q, K, Vv, float(g["sm_scale"]))
    assert abs(l[0] - float(g["lse"])) < 1e-15
    assert np.allclose(o[0], np.array(g["out"], float), atol=1e-15, rtol=0)


def test_attend_single_key_and_empty():
    g = _rng(2)
    q, K, Vv = g.standard_normal((4, 9)), g.standard_normal((1, 9)), g.standard_normal((1, 3))
    o, l = mla.attend(q, K, Vv, 0.5)
    assert np.allclose(l, 0.5 * q @ K[0], atol=1e-14)
    assert np.allclose(o, np.broadcast_to(Vv[0], o.shape), atol=1e-15)
    o, l = mla.attend(q, K[:0], Vv[:0], 0.5)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_identical_keys_give_uniform_weights():
    g = _rng(3)
    n = 37
    q = g.standard_normal((5, 11))
    k = g.standard_normal(11)
    K = np.tile(k, (n, 1))
    Vv = g.standard_normal((n, 6))
    o, l = mla.attend(q, K, Vv, 0.3)
    assert np.allclose(o, np.broadcast_to(Vv.mean(0), o.shape), atol=1e-13)
    assert np.allclose(l, 0.3 * q @ k + math.log(n), atol=1e-13)


def test_output_is_convex_combination():
    g = _rng(4)
    q, K, Vv = g.standard_normal((8, 16)) * 3, g.standard_normal((50, 16)), g.standard_normal((50, 10))
    o, _ = mla.attend(q, K, Vv, 1.0)
    assert np.all(o <= Vv.max(0) + 1e-12) and np.all(o >= Vv.min(0) - 1e-12)


def _paged(g, seq_lens, H, q_len=1):
    pages = [(n + 63) // 64 for n in seq_lens]
    nb = sum(pages) + 2
    perm = g.permutation(nb)
    bt = np.full((len(seq_lens), max(pages)), -1, np.int64)
    o = 0
    for b, p in enumerate(pages):
        bt[b, :p] = perm[o:o + p]
        o += p
    cache = g.standard_normal((nb, 64, 576))
    q = g.standard_normal((len(seq_lens), q_len, H, 576)) * 0.1
    return q, cache, bt


def test_paged_addressing_matches_contiguous():
    g = _rng(5)
    seq = [1, 64, 65, 200]
    q, cache, bt = _paged(g, seq, 3)
    out, lse = mla.paged_decode(q, cache, bt, seq, 0.1)
    for b, n in enumerate(seq):
        rows = np.concatenate([cache[bt[b, p]] for p in range((n + 63) // 64)])[:n]
        o, l = mla.attend(q[b, 0], rows, rows[:, :512], 0.1)
        assert np.allclose(out[b, 0], o, atol=1e-14) and np.allclose(lse[b, 0], l, atol=1e-14)


def test_causal_pair_reduces_to_single_token_decode():
    g = _rng(6)
    seq = [2, 70, 129]
    q, cache, bt = _paged(g, seq, 2, q_len=2)
    out, lse = mla.paged_decode(q, cache, bt, seq, 0.2, causal=True)
    o1, l1 = mla.paged_decode(q[:, 1:2], cache, bt, seq, 0.2)
    o0, l0 = mla.paged_decode(q[:, 0:1], cache, bt, [n - 1 for n in seq], 0.2)
    assert np.allclose(out[:, 1], o1[:, 0], atol=1e-14) and np.allclose(lse[:, 1], l1[:, 0])
    assert np.allclose(out[:, 0], o0[:, 0], atol=1e-14) and np.allclose(lse[:, 0], l0[:, 0])


def test_seq_len_zero_and_empty_shard():
    g = _rng(7)
    q, cache, bt = _paged(g, [10], 2)
    out, lse = mla.paged_decode(q, cache, bt, [0], 0.2)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    out, lse = mla.paged_decode(q, cache, bt, [10], 0.2, kv_starts=[5], kv_ends=[5])
    assert np.all(out == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("kind", ["contiguous", "strided", "with_empty", "random"])
def test_merge_of_shards_equals_unsplit(kind):
    g = _rng(8)
    n, H = 300, 4
    q = g.standard_normal((H, 32))
    K, Vv = g.standard_normal((n, 32)), g.standard_normal((n, 12))
    full_o, full_l = mla.attend(q, K, Vv, 0.4)
    idx = np.arange(n)
    if kind == "contiguous":
        parts = np.array_split(idx, 5)
    elif kind == "strided":
        parts = [idx[s::4] for s in range(4)]
    elif kind == "with_empty":
        parts = [idx[:0], idx[:120], idx[120:120], idx[120:]]
    else:
        lab = g.integers(0, 6, n)
        parts = [idx[lab == s] for s in range(7)]          # part 6 is empty
    po, pl = zip(*[mla.attend(q, K[p], Vv[p], 0.4) for p in parts])
    o, l = mla.merge_states(np.stack(po), np.stack(pl))
    assert np.allclose(o, full_o, atol=1e-13) and np.allclose(l, full_l, atol=1e-13)


def test_merge_order_and_associativity():
    g = _rng(9)
    po = g.standard_normal((3, 5, 8))
    pl = g.standard_normal((3, 5)) * 4
    o, l = mla.merge_states(po, pl)
    o2, l2 = mla.merge_states(po[::-1], pl[::-1])
    oa, la = mla.merge_states(po[:2], pl[:2])
    o3, l3 = mla.merge_states(np.stack([oa, po[2]]), np.stack([la, pl[2]]))
    assert np.allclose(o, o2, atol=1e-14) and np.allclose(l, l2, atol=1e-14)
    assert np.allclose(o, o3, atol=1e-14) and np.allclose(l, l3, atol=1e-14)


def test_merge_all_empty_and_nan_in_empty_part():
    po = np.full((2, 3, 4), np.nan)
    pl = np.full((2, 3), -np.inf)
    o, l = mla.merge_states(po, pl)
    assert np.all(o == 0) and np.all(np.isneginf(l))
    po[1] = 2.0
    pl[1] = 0.5
    o, l = mla.merge_states(po, pl)
    assert np.all(o == 2.0) and np.all(l == 0.5)


def test_absorb_brute_force():
    g = _rng(10)
    T, H = 2, 3
    qn, qp = g.standard_normal((T, H, 128)), g.standard_normal((T, H, 64))
    w = g.standard_normal((H, 128, 512))
    got = mla.absorb_q(qn, qp, w)
    for t in range(T):
        for h in range(H):
            for l in (0, 17, 511):
                ref = sum(qn[t, h, p] * w[h, p, l] for p in range(128))
                assert abs(got[t, h, l] - ref) < 1e-11
            assert np.array_equal(got[t, h, 512:], qp[t, h])


def test_v_up_brute_force():
    g = _rng(11)
    o = g.standard_normal((2, 3, 512))
    w = g.standard_normal((3, 128, 512))
    got = mla.v_up(o, w)
    for t in range(2):
        for h in range(3):
            for v in (0, 64, 127):
                ref = sum(o[t, h, l] * w[h, v, l] for l in range(512))
                assert abs(got[t, h, v] - ref) < 1e-10


def test_absorbed_mqa_equals_expanded_mha():
    """MLA DCP prefill blog, §MLA Prefill vs Decode: decode (Q absorbed into
    the latent space, one 576-wide head) and prefill (kv_c expanded through
    W_UK/W_UV to N heads of width 192 / 128) compute the same attention."""
    g = _rng(12)
    H, n = 4, 90
    w_kvb = g.standard_normal((H * 256, 512)) * 0.05
    w_uk_t, w_uv = mla.absorbed_weights(w_kvb, H)
    kv = g.standard_normal((n, 576))
    q_nope, q_pe = g.standard_normal((1, H, 128)), g.standard_normal((1, H, 64))
    scale = 1 / math.sqrt(192)
    # absorbed path
    qa = mla.absorb_q(q_nope, q_pe, w_uk_t)
    o_lat, lse_a = mla.attend(qa[0], kv, kv[:, :512], scale)
    out_a = mla.v_up(o_lat[None], w_uv)[0]
    # expanded path
    K, Vv = mla.expand_kv(kv, w_kvb, H)
    for h in range(H):
        qh = np.concatenate([q_nope[0, h], q_pe[0, h]])
        o, l = mla.attend(qh[None], K[:, h], Vv[:, h], scale)
        assert np.allclose(o[0], out_a[h], atol=1e-12)
        assert abs(l[0] - lse_a[h]) < 1e-12


def test_concat_quant_divides_in_float32():
    from oracle import codecs
    q = np.array([[1.0, 3.0, -500.0, 1e-6]], np.float32)
    codes = mla.concat_quant_e4m3(q, 0.5)
    assert list(codes[0]) == [0x40, 0x4C, 0xFE, 0x00]    # 2, 6, sat, ~0
    x = (np.float32(0.1) / np.float32(0.3))
    assert codecs.e4m3_to_f64(mla.concat_quant_e4m3(np.array([0.1], np.float32), 0.3))[0] \
        == codecs.e4m3_to_f64(codecs.f32_to_e4m3(np.array([x])))[0]


def test_dims_match_pages_comm_table():
    """MLA DCP prefill blog, §核心思路：AllGather KV: 128 heads x 192 = 24576
    per-token Q elements against 512 + 64 = 576 latent KV elements."""
    assert 128 * (mla.P + mla.R) == 24576
    assert mla.L + mla.R == 576 == mla.D_QK
