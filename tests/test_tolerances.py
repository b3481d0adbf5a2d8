"""The scale-aware error bounds used by the GPU parity tests, checked on the
CPU: they must admit a result computed with exactly the roundings the
decode kernel performs (fp32 scores, bf16 P with an unrounded normaliser,
bf16 output), and must reject a plausible kernel mistake that the
spec max-abs tolerance (1e-2) lets through at the tiny config's
magnitudes.  The split path (bf16 partials of a job cut into spans, merged
in fp32) is emulated as well.  The mistakes are planted in a CPU emulation
built on the oracle's own definitions; no GPU result is involved."""

import math

import numpy as np
import pytest

import synth
from oracle import codecs, mla as O
from tests._helpers import bound_report, decode_terms, f64, merge_bounds

LOG2E = 1.0 / math.log(2.0)


def _bf16(x):
    """fp32 value -> its bf16 rounding (RNE), as float64."""
    return codecs.bf16_to_f64(codecs.f32_to_bf16(np.asarray(x, np.float32)))


def _emulate_decode(q, cache, block_table, seq_lens, sm_scale, *, drop_last_tile=False,
                    skip_scale=False):
    """The pair kernel's arithmetic on the CPU: fp32 scores, p = 2^(s*c - m)
    in fp32, P rounded to bf16 for the P.V product, normaliser l from the
    unrounded p, fp32 O / l rounded to bf16, lse = (m + log2 l) ln 2."""
    B, q_len, H, _ = q.shape
    out = np.zeros((B, q_len, H, 512))
    lse = np.full((B, q_len, H), -np.inf)
    for b in range(B):
        for i in range(q_len):
            lo, hi = O.decode_range(int(seq_lens[b]), q_len, i, True)
            if hi <= lo:
                continue
            blk, off = O.page_rows(block_table[b], np.arange(lo, hi))
            rows = cache[blk, off].astype(np.float32)
            s = q[b, i].astype(np.float32) @ rows.T
            c = np.float32(1.0 if skip_scale else sm_scale * LOG2E)
            x = (s * c).astype(np.float32)
            m = x.max(axis=1, keepdims=True)
            p = np.exp2(x - m).astype(np.float32)
            l = p.sum(axis=1, keepdims=True, dtype=np.float32)
            pt = _bf16(p).astype(np.float32)
            if drop_last_tile and hi - lo > 64:
                # requests of more than one tile lose their last tile's P.V
                last = ((hi - lo - 1) // 64) * 64
                pt[:, last:] = 0.0
            o = (pt @ rows[:, :512]).astype(np.float32) / l
            out[b, i] = _bf16(o)
            lse[b, i] = ((m[:, 0] + np.log2(l[:, 0])) * np.float32(math.log(2.0))).astype(np.float32)
    return out, lse


def _emulate_split_decode(q, cache, block_table, seq_lens, sm_scale, seg=64):
    """The split path: each request's key range cut into `seg`-token parts,
    each part computed as above and stored as a bf16 partial (O / l rounded
    to bf16, its lse in fp32), then the merge kernel's fp32 online fold
    (running max, rescaled sum and accumulator, parts in order) and one
    bf16 rounding of acc * (1 / z)."""
    B, q_len, H, _ = q.shape
    out = np.zeros((B, q_len, H, 512))
    lse = np.full((B, q_len, H), -np.inf)
    c = np.float32(sm_scale * LOG2E)
    ln2 = np.float32(math.log(2.0))
    for b in range(B):
        for i in range(q_len):
            lo, hi = O.decode_range(int(seq_lens[b]), q_len, i, True)
            if hi <= lo:
                continue
            m = np.full((H,), -np.inf, np.float32)
            z = np.zeros((H,), np.float32)
            acc = np.zeros((H, 512), np.float32)
            for a in range(lo, hi, seg):
                blk, off = O.page_rows(block_table[b], np.arange(a, min(hi, a + seg)))
                rows = cache[blk, off].astype(np.float32)
                x = ((q[b, i].astype(np.float32) @ rows.T) * c).astype(np.float32)
                ms = x.max(axis=1, keepdims=True)
                p = np.exp2(x - ms).astype(np.float32)
                ls = p.sum(axis=1, keepdims=True, dtype=np.float32)
                part = _bf16((_bf16(p).astype(np.float32) @ rows[:, :512]).astype(np.float32)
                             / ls).astype(np.float32)
                lse_s = ((ms[:, 0] + np.log2(ls[:, 0])) * ln2).astype(np.float32)
                mn = np.maximum(m, lse_s)
                sc = np.exp(m - mn).astype(np.float32)
                w = np.exp(lse_s - mn).astype(np.float32)
                z = (z * sc + w).astype(np.float32)
                acc = (acc * sc[:, None] + w[:, None] * part).astype(np.float32)
                m = mn
            out[b, i] = _bf16(acc * (np.float32(1.0) / z)[:, None])
            lse[b, i] = (m + np.log(z)).astype(np.float32)
    return out, lse


@pytest.fixture(scope="module")
def tiny():
    case = synth.tiny_decode(poison=False)
    q, cache = f64(case.q), f64(case.cache)
    ref_o, ref_l = O.paged_decode(q, cache, case.block_table, case.seq_lens, case.sm_scale)
    t = decode_terms(q, cache, case.block_table, case.seq_lens, case.sm_scale)
    return case, q, cache, ref_o, ref_l, t


def test_bounds_admit_the_kernel_roundings(tiny):
    case, q, cache, ref_o, ref_l, t = tiny
    o, l = _emulate_decode(q, cache, case.block_table, case.seq_lens, case.sm_scale)
    d_o, r_o, d_l, r_l, finite = bound_report(o, l, ref_o, ref_l, t)
    assert finite and r_o <= 0.6 and r_l <= 0.6, (r_o, r_l)


@pytest.mark.parametrize("seg", [64, 128])
def test_bounds_admit_the_split_path_with_bf16_partials(tiny, seg):
    """A job cut into spans stores each span's O / l in the output's type
    (bf16 here) and merges the parts in fp32: the rounding of the parts
    stays inside the same bounds."""
    case, q, cache, ref_o, ref_l, t = tiny
    o, l = _emulate_split_decode(q, cache, case.block_table, case.seq_lens, case.sm_scale, seg)
    d_o, r_o, d_l, r_l, finite = bound_report(o, l, ref_o, ref_l, t)
    assert finite and r_o <= 0.6 and r_l <= 0.6, (r_o, r_l)


def test_bounds_reject_a_dropped_pv_tile(tiny):
    """Dropping the last 64-token tile's P.V step of the 130-token request
    (keeping the normaliser) stays far inside the 1e-2 max-abs tolerance at
    the tiny decode's magnitudes; the scale-aware bound catches it."""
    case, q, cache, ref_o, ref_l, t = tiny
    o, l = _emulate_decode(q, cache, case.block_table, case.seq_lens, case.sm_scale,
                           drop_last_tile=True)
    d_o, r_o, _, _, _ = bound_report(o, l, ref_o, ref_l, t)
    assert d_o < 1e-2          # the plain max-abs check would pass it
    assert r_o > 1.0


def test_bounds_reject_a_missing_softmax_scale(tiny):
    case, q, cache, ref_o, ref_l, t = tiny
    o, l = _emulate_decode(q, cache, case.block_table, case.seq_lens, case.sm_scale,
                           skip_scale=True)
    _, r_o, _, r_l, _ = bound_report(o, l, ref_o, ref_l, t)
    assert r_o > 1.0 or r_l > 1.0


def test_merge_bounds_admit_fp32_merge_and_reject_swapped_weights():
    g = np.random.Generator(np.random.PCG64(7))
    S, T, H, D = 3, 2, 4, 64
    po = g.standard_normal((S, T, H, D)) * 0.05
    pl = g.standard_normal((S, T, H)) * 2
    ref_o, ref_l = O.merge_states(po, pl)
    bo, bl = merge_bounds(ref_o, ref_l, po, pl)
    # fp32 merge with a bf16 output
    m = pl.max(axis=0).astype(np.float32)
    w = np.exp((pl - m).astype(np.float32)).astype(np.float32)
    z = w.sum(axis=0, dtype=np.float32)
    o32 = (w[..., None] * po.astype(np.float32)).sum(axis=0, dtype=np.float32) / z[..., None]
    assert np.all(np.abs(_bf16(o32) - ref_o) <= bo)
    assert np.all(np.abs((m + np.log(z)).astype(np.float32) - ref_l) <= bl)
    # the weights of parts 0 and 1 exchanged
    w2 = w[[1, 0, 2]]
    o_bad = (w2[..., None] * po).sum(axis=0) / z[..., None]
    assert np.any(np.abs(_bf16(o_bad) - ref_o) > bo)
