"""Pins for the oracle's rotary embedding and cache write (the steps just
before the decode path).

The rotary embedding is checked against a hand-worked example written with
the math module only (tests/golden/rope_example.json), and against the
properties that define a rotary position embedding: position 0 is the
identity, every pair keeps its norm, rotations compose, and the dot product
of a rotated query and key depends only on their relative position.  The
rotate-half layout equals the interleaved one under the permutation of
dimensions that maps one pairing onto the other.  The cache write is
checked through the pinned gather and e4m3 codec."""

import json
import os

import numpy as np
import pytest

import synth
from oracle import codecs, mla

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(s):
    return np.random.Generator(np.random.PCG64(s))


@pytest.mark.parametrize("interleaved,key", [(True, "interleaved"), (False, "rotate_half")])
def test_rope_matches_hand_worked_example(interleaved, key):
    with open(os.path.join(GOLDEN, "rope_example.json")) as f:
        g = json.load(f)
    x = np.array(g["x"])
    for case in g["cases"]:
        got = mla.rope(x[None], [case["position"]], base=g["base"], interleaved=interleaved)[0]
        assert np.allclose(got, case[key], rtol=0, atol=1e-12), (case["position"], got)


@pytest.mark.parametrize("interleaved", [True, False])
def test_rope_position_zero_is_identity_and_norms_are_kept(interleaved):
    g = _rng(1)
    x = g.standard_normal((5, 3, 64))
    assert np.array_equal(mla.rope(x, [0] * 5, interleaved=interleaved), x)
    pos = g.integers(0, 40000, 5)
    y = mla.rope(x, pos, interleaved=interleaved)
    if interleaved:
        na, nb = x[..., 0::2] ** 2 + x[..., 1::2] ** 2, y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    else:
        na, nb = x[..., :32] ** 2 + x[..., 32:] ** 2, y[..., :32] ** 2 + y[..., 32:] ** 2
    assert np.allclose(na, nb, rtol=1e-12, atol=0)


@pytest.mark.parametrize("interleaved", [True, False])
def test_rope_composes_and_depends_on_relative_position_only(interleaved):
    g = _rng(2)
    q, k = g.standard_normal((4, 64)), g.standard_normal((4, 64))
    m, n = g.integers(0, 5000, 4), g.integers(0, 5000, 4)
    sft = g.integers(0, 5000, 4)
    # rope(rope(x, a), b) = rope(x, a + b)
    assert np.allclose(mla.rope(mla.rope(q, m, interleaved=interleaved), n, interleaved=interleaved),
                       mla.rope(q, m + n, interleaved=interleaved), rtol=0, atol=1e-9)
    # <rope(q, m), rope(k, n)> = <rope(q, m + s), rope(k, n + s)>
    d0 = np.sum(mla.rope(q, m, interleaved=interleaved) * mla.rope(k, n, interleaved=interleaved), -1)
    d1 = np.sum(mla.rope(q, m + sft, interleaved=interleaved) *
                mla.rope(k, n + sft, interleaved=interleaved), -1)
    assert np.allclose(d0, d1, rtol=0, atol=1e-9)


def test_rope_layouts_agree_under_the_pairing_permutation():
    g = _rng(3)
    x = g.standard_normal((6, 2, 64))
    pos = g.integers(0, 30000, 6)
    # interleaved dim 2i <-> rotate-half dim i, 2i+1 <-> i + 32
    perm = np.empty(64, np.int64)
    perm[0::2], perm[1::2] = np.arange(32), np.arange(32) + 32
    got = mla.rope(x[..., perm], pos, interleaved=True)
    want = mla.rope(x, pos, interleaved=False)[..., perm]
    assert np.allclose(got, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_cache_write_then_gather_returns_the_rows(kv_dtype):
    g = _rng(4)
    seq = np.array([70, 5, 130], np.int32)
    bt, nb = synth.paged_layout(g, seq)
    cache, ks = synth.fill_cache(g, bt, seq, nb, kv_dtype=kv_dtype)
    raw = cache.view(__import__("torch").int16).numpy().astype(np.uint16) if kv_dtype == "bf16" \
        else cache.view(__import__("torch").uint8).numpy()
    # the new tokens: the last position of each request, plus one padding row
    T = 4
    kv_c = codecs.f32_to_bf16(g.standard_normal((T, 512)).astype(np.float32))
    k_pe = codecs.f32_to_bf16(g.standard_normal((T, 64)).astype(np.float32))
    pos = np.array([69, 4, 129, 0])
    slots = np.array([bt[b, p // 64] * 64 + p % 64 for b, p in zip(range(3), pos[:3])] + [-1])
    out = mla.cache_write(raw, kv_c, k_pe, slots, kv_dtype, ks)
    rows = np.concatenate([kv_c, k_pe], axis=1)
    want = rows if kv_dtype == "bf16" else codecs.f32_to_e4m3(
        codecs.bf16_to_f64(rows).astype(np.float32) / np.float32(ks))
    cu = np.array([0, 1, 2, 3])
    got = mla.gather_cache(out, bt, cu, seq_starts=pos[:3])
    assert np.array_equal(got, want[:3])
    # only the three written rows changed (the padding slot wrote nothing)
    changed = np.argwhere(np.any(out != raw, axis=-1))
    assert len(changed) <= 3
    if kv_dtype == "e4m3":
        # stored codes decode to the value within half an e4m3 step
        dec = codecs.e4m3_to_f64(got) * ks
        val = codecs.bf16_to_f64(rows[:3])
        sat = np.abs(val) > 448 * ks
        ok = np.abs(dec - val) <= np.maximum(np.abs(val) * 2.0 ** -4, 2.0 ** -10 * ks) + 1e-12
        assert np.all(np.where(sat, np.abs(dec) == 448 * ks, ok))
