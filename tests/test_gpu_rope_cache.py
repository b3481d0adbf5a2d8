"""GPU parity of the step before the decode path: rotary embedding of the
query's rope slice and of k_pe, and the slot-mapping store of kv_c ‖ k_pe
into the paged cache (bf16 or e4m3), against the fp64 oracle.

The rotations are held to a bound derived from the kernel's arithmetic (the
angle and its sine / cosine in fp64, cos / sin rounded to fp32, one fused
fp32 rounding per output, one bf16 rounding):
    |gpu - ref| <= 2^-8 |ref| + 2^-20 * |(a, b)|
for an element of the pair (a, b).  The cache store is checked bit for bit,
over the whole cache, against the oracle's cache write fed the kernel's
own rotated k_pe (the e4m3 codes are taken in fp32, as the kernel does)."""

import numpy as np
import pytest
import torch

import synth
from oracle import codecs, mla as O
from tests._helpers import bits, check_attention, decode_terms, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_kv_uk_gb300 as mod
    return mod


def _i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()


def _pair_norm(x, interleaved):
    """|(a, b)| of the pair each element belongs to."""
    if interleaved:
        n = np.sqrt(x[..., 0::2] ** 2 + x[..., 1::2] ** 2)
        return np.repeat(n, 2, axis=-1)
    d = x.shape[-1] // 2
    n = np.sqrt(x[..., :d] ** 2 + x[..., d:] ** 2)
    return np.concatenate([n, n], axis=-1)


def _check_rot(got, x, pos, interleaved, label):
    ref = O.rope(x, pos, interleaved=interleaved)
    err = np.abs(f64(got) - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * _pair_norm(x, interleaved) + 1e-30
    print(f"{label}: max-abs {err.max():.3e} ({(err / bound).max():.3f} of its bound)")
    assert np.all(err <= bound)


def _setup(g, kv_dtype, T=40, H=128):
    seq = np.array([900, 64, 3, 2000], np.int32)
    bt, nb = synth.paged_layout(g, seq)
    cache, ks = synth.fill_cache(g, bt, seq, nb, kv_dtype=kv_dtype)
    q_pe = synth.as_bf16(g.standard_normal((T, H, 64)))
    k_pe = synth.as_bf16(g.standard_normal((T, 64)))
    kv_c = synth.as_bf16(g.standard_normal((T, 512)))
    pos = g.integers(0, 40000, T).astype(np.int32)
    pos[0] = 0
    # distinct physical rows anywhere in the pool, two padding slots
    slots = g.choice(nb * 64, T, replace=False).astype(np.int32)
    slots[3] = -1
    slots[T - 1] = -1
    return cache, ks, q_pe, k_pe, kv_c, pos, slots, nb


@pytest.mark.parametrize("layout", ["interleaved", "half"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_rope_and_cache_write(m, layout, kv_dtype):
    g = synth.generator(800 + (layout == "half") + 2 * (kv_dtype == "e4m3"))
    cache, ks, q_pe, k_pe, kv_c, pos, slots, nb = _setup(g, kv_dtype)
    inter = layout == "interleaved"
    before = bits(cache)
    d_q, d_k, d_c = q_pe.cuda(), k_pe.cuda(), cache.cuda()
    m.mla_get_device_error()
    m.mla_rope_cache_write(d_q, d_k, kv_c.cuda(), _i32(pos), _i32(slots), d_c,
                           layout=layout, k_scale=ks)
    assert m.mla_get_device_error() == 0
    _check_rot(d_q, f64(q_pe), pos, inter, f"q_pe {layout}")
    _check_rot(d_k, f64(k_pe), pos, inter, f"k_pe {layout}")
    want = O.cache_write(before.astype(np.uint16) if kv_dtype == "bf16" else before,
                         bits(kv_c).astype(np.uint16), bits(d_k).astype(np.uint16), slots,
                         kv_dtype, ks)
    got = bits(d_c)
    got = got.astype(np.uint16) if kv_dtype == "bf16" else got
    assert np.array_equal(got, want)


def test_out_of_range_slot_is_flagged_and_skipped(m):
    g = synth.generator(810)
    cache, ks, q_pe, k_pe, kv_c, pos, slots, nb = _setup(g, "bf16", T=6, H=4)
    slots[2] = nb * 64 + 5
    before = bits(cache)
    d_k, d_c = k_pe.cuda(), cache.cuda()
    m.mla_get_device_error()
    m.mla_rope_cache_write(None, d_k, kv_c.cuda(), _i32(pos), _i32(slots), d_c)
    assert m.mla_get_device_error() & 1
    ok = slots.copy()
    ok[2] = -1                                  # the bad token writes nothing
    want = O.cache_write(before.astype(np.uint16), bits(kv_c).astype(np.uint16),
                         bits(d_k).astype(np.uint16), ok, "bf16")
    assert np.array_equal(bits(d_c).astype(np.uint16), want)
    _check_rot(d_k, f64(k_pe), pos, True, "k_pe")


def test_new_tokens_written_then_decoded(m):
    """One decode step: each request's new token (at position seq_len - 1)
    is rotated and written by mla_rope_cache_write, the query is absorbed
    from q_nope and the rotated q_pe, and the decode reads the new rows;
    every stage against the oracle fed the GPU's own inputs."""
    g = synth.generator(820)
    B, H = 4, 128
    seq = np.array([1, 65, 700, 2049], np.int32)
    case = synth.decode_case("step", 821, B=B, H=H, seq_lens=seq, poison=True)
    q_nope = case.q_nope.cuda()
    q_pe = synth.as_bf16(g.standard_normal((B, H, 64)))
    k_pe = synth.as_bf16(g.standard_normal((B, 64)))
    kv_c = synth.as_bf16(g.standard_normal((B, 512)))
    pos = (seq - 1).astype(np.int32)
    slots = np.array([case.block_table[b, p // 64] * 64 + p % 64 for b, p in enumerate(pos)],
                     np.int32)
    cache = case.cache.cuda()
    before = bits(case.cache).astype(np.uint16)
    d_qp, d_kp = q_pe.cuda(), k_pe.cuda()
    m.mla_rope_cache_write(d_qp, d_kp, kv_c.cuda(), _i32(pos), _i32(slots), cache)
    _check_rot(d_qp, f64(q_pe), pos, True, "q_pe")
    want = O.cache_write(before, bits(kv_c).astype(np.uint16), bits(d_kp).astype(np.uint16),
                         slots)
    assert np.array_equal(bits(cache).astype(np.uint16), want)
    q = m.mla_absorb_q(q_nope, d_qp, case.w_uk_t.cuda()).view(B, 1, H, 576)
    out, lse = m.mla_decode_paged(q, cache, _i32(case.block_table), _i32(seq),
                                  sm_scale=case.sm_scale)
    assert m.mla_get_device_error() == 0
    q64, c64 = f64(q), f64(cache)
    ro, rl = O.paged_decode(q64, c64, case.block_table, seq, case.sm_scale)
    t = decode_terms(q64, c64, case.block_table, seq, case.sm_scale)
    check_attention(f64(out), lse.cpu().numpy(), ro, rl, t, out_tol=1e-2, lse_tol=1e-3,
                    label="decode after the cache write")
    # the rows the decode read at the new tokens' positions are the ones written
    assert np.array_equal(codecs.bf16_to_f64(want[slots // 64, slots % 64, :512]), f64(kv_c))
