"""GPU parity of the absorbed decode chain against the fp64 oracle:
absorb (+ e4m3 concat-quant, bit-exact), v_up, the split plan (validity)
and the paged decode with its on-device split merge."""

import math

import numpy as np
import pytest
import torch

import synth
from oracle import codecs, mla as O
from tests._helpers import (bits, check_attention, decode_terms, f64, gemm_tolerance, lse_close,
                            max_abs, merge_bounds)
from tests.plan_check import check_split_plan, job_ranges

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2      # bf16 decode output, max-abs (spec tolerance)
LSE_TOL = 1e-3      # bf16 decode LSE, max-abs


@pytest.fixture(scope="module")
def m():
    import mla_latent_kv_uk_gb300 as mod
    return mod


def _i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()


# ----------------------------------------------------------------- absorb
@pytest.mark.parametrize("T,H", [(1, 16), (32, 128), (37, 3), (300, 8)])
def test_absorb_bf16(m, T, H):
    g = synth.generator(400 + T)
    qn = synth.as_bf16(g.standard_normal((T, H, 128)))
    qp = synth.as_bf16(g.standard_normal((T, H, 64)))
    w = synth.as_bf16(g.standard_normal((H, 128, 512)) * 0.05)
    q = m.mla_absorb_q(qn.cuda(), qp.cuda(), w.cuda())
    ref = O.absorb_q(f64(qn), f64(qp), f64(w))
    abs_sum = np.concatenate([np.einsum("thp,hpl->thl", np.abs(f64(qn)), np.abs(f64(w))),
                              np.abs(f64(qp))], -1)
    err = np.abs(f64(q) - ref)
    assert np.all(err <= gemm_tolerance(ref, abs_sum)), float(err.max())
    assert np.array_equal(bits(q)[..., 512:], bits(qp))      # q_pe copied exactly


def test_absorb_fp32_and_e4m3_bit_exact(m):
    """The e4m3 encoder on the GPU must give the oracle's code for the very
    fp32 value it quantises: compare against the oracle's concat-quant of the
    kernel's own fp32 output (same accumulation order on both launches)."""
    g = synth.generator(410)
    T, H = 64, 128
    qn = synth.as_bf16(g.standard_normal((T, H, 128)))
    qp = synth.as_bf16(g.standard_normal((T, H, 64)))
    w = synth.as_bf16(g.standard_normal((H, 128, 512)) * 0.02)
    q32 = m.mla_absorb_q(qn.cuda(), qp.cuda(), w.cuda(), out_dtype=torch.float32)
    ref = O.absorb_q(f64(qn), f64(qp), f64(w))
    abs_sum = np.concatenate([np.einsum("thp,hpl->thl", np.abs(f64(qn)), np.abs(f64(w))),
                              np.abs(f64(qp))], -1)
    assert np.all(np.abs(f64(q32) - ref) <= abs_sum * 2.0 ** -20 + 1e-30)
    q_scale = float(np.float32(np.abs(f64(q32)).max() / 448.0))
    q8 = m.mla_absorb_q(qn.cuda(), qp.cuda(), w.cuda(), out_dtype=torch.float8_e4m3fn,
                        q_scale=q_scale)
    want = O.concat_quant_e4m3(q32.cpu().numpy(), q_scale)
    assert np.array_equal(bits(q8), want)


# ------------------------------------------------------------------ v_up
@pytest.mark.parametrize("T,H", [(1, 4), (32, 128), (256, 16), (300, 2)])
def test_v_up(m, T, H):
    g = synth.generator(420 + T)
    o = synth.as_bf16(g.standard_normal((T, H, 512)))
    w = synth.as_bf16(g.standard_normal((H, 128, 512)) * 0.02)
    out = m.mla_v_up(o.cuda(), w.cuda())
    ref = O.v_up(f64(o), f64(w))
    abs_sum = np.einsum("thl,hvl->thv", np.abs(f64(o)), np.abs(f64(w)))
    err = np.abs(f64(out) - ref)
    assert np.all(err <= gemm_tolerance(ref, abs_sum)), float(err.max())


# ------------------------------------------------------------------ plan
# The split plan is this library's schedule (the pages fix only that it is
# derived on the device from seq_lens and the true head count), so the GPU
# plan is checked for validity: every key tile of every job met by exactly
# one span, consistent prefixes, no more spans than CTA groups, none longer
# than C (tests/plan_check.py).
@pytest.mark.parametrize("split_tiles,n_groups,fp8", [(0, 76, False), (3, 5, False),
                                                     (0, 1, False), (1, 2, False),
                                                     (0, 76, True), (2, 3, True)])
def test_plan_is_valid(m, split_tiles, n_groups, fp8):
    g = synth.generator(430)
    B, q_len, H = 9, 2, 200
    seq = g.integers(0, 3000, B).astype(np.int32)
    seq[2] = 0
    starts = g.integers(0, 50, B).astype(np.int32)
    ends = (starts + g.integers(0, 2500, B)).astype(np.int32)
    plan = m.mla_decode_plan(_i32(seq), B, q_len, H, 64, kv_starts=_i32(starts),
                             kv_ends=_i32(ends), causal=True, split_tiles=split_tiles,
                             n_groups=n_groups,
                             kv_dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16
                             ).cpu().numpy()
    lo, hi = job_ranges(seq, q_len, H, True, starts, ends)
    check_split_plan(plan, lo, hi, n_groups, split_tiles)


@pytest.mark.parametrize("B,q_len,n_groups", [(200, 2, 76), (32, 1, 76), (1, 1, 76),
                                              (128, 2, 76)])
def test_plan_is_valid_many_jobs(m, B, q_len, n_groups):
    """Up to J = 400 jobs: the one-warp plan kernel (J <= 256) and the
    block-scan plan kernel beyond it; the DeepSeek-V3 decode and speculative decode shapes."""
    g = synth.generator(431 + B)
    H = 128
    seq = g.integers(0, 5000, B).astype(np.int32)
    plan = m.mla_decode_plan(_i32(seq), B, q_len, H, 80, causal=True,
                             n_groups=n_groups).cpu().numpy()
    lo, hi = job_ranges(seq, q_len, H, True)
    check_split_plan(plan, lo, hi, n_groups)


# ---------------------------------------------------------------- decode
# Every decode check applies the spec max-abs bounds (out 1e-2, LSE
# 1e-3; fp8 KV out 5e-2) and the scale-aware elementwise bounds derived from
# the kernel's roundings (tests/_helpers.py: bf16 output and P, e4m3 P on
# the fp8 path, fp32 score accumulation); the helper prints the achieved
# errors and their ratio to the bound.
def _oracle_decode(case, kv_starts=None, kv_ends=None, causal=None, pick=None):
    """(out, lse, error terms) of the oracle on the case's quantised inputs
    (dequantised exactly), optionally for a subset of requests."""
    q = f64(case.q) * case.q_scale
    cache = f64(case.cache) * case.k_scale
    bt, sl = case.block_table, case.seq_lens
    st, en = kv_starts, kv_ends
    if pick is not None:
        q, bt, sl = q[pick], bt[pick], sl[pick]
        st = None if st is None else np.asarray(st)[pick]
        en = None if en is None else np.asarray(en)[pick]
    c = case.causal if causal is None else causal
    ro, rl = O.paged_decode(q, cache, bt, sl, case.sm_scale, causal=c, kv_starts=st,
                            kv_ends=en)
    t = decode_terms(q, cache, bt, sl, case.sm_scale, causal=c, kv_starts=st, kv_ends=en,
                     fp8=case.kv_dtype == "e4m3")
    return ro, rl, t


def _run_decode(m, case, split_tiles=0, out_dtype=torch.bfloat16, kv_starts=None,
                kv_ends=None, causal=None):
    return m.mla_decode_paged(
        case.q.cuda(), case.cache.cuda(), _i32(case.block_table), _i32(case.seq_lens),
        sm_scale=case.sm_scale, q_scale=case.q_scale, k_scale=case.k_scale,
        kv_starts=None if kv_starts is None else _i32(kv_starts),
        kv_ends=None if kv_ends is None else _i32(kv_ends),
        causal=case.causal if causal is None else causal, split_tiles=split_tiles,
        out_dtype=out_dtype)


def _check(out, lse, ro, rl, t, out_tol=OUT_TOL, lse_tol=LSE_TOL, label="decode"):
    check_attention(f64(out).reshape(ro.shape), lse.cpu().numpy().reshape(rl.shape), ro, rl, t,
                    out_tol=out_tol, lse_tol=lse_tol, out_bf16=out.dtype == torch.bfloat16,
                    label=label)


def test_decode_tiny(m):
    case = synth.tiny_decode(poison=True)
    out, lse = _run_decode(m, case)
    _check(out, lse, *_oracle_decode(case), label="tiny decode")
    assert m.mla_get_device_error() == 0


@pytest.mark.parametrize("split_tiles", [0, 1, 3])
def test_decode_ragged_multi_tile(m, split_tiles):
    case = synth.decode_case("ragged", 440, B=4, H=128, seq_lens=[1, 33, 100, 1000],
                             poison=True)
    out, lse = _run_decode(m, case, split_tiles=split_tiles)
    _check(out, lse, *_oracle_decode(case))


def test_decode_fp32_out_and_head_groups(m):
    case = synth.decode_case("hg", 441, B=2, H=200, seq_lens=[77, 300], poison=True)
    out, lse = _run_decode(m, case, out_dtype=torch.float32, split_tiles=2)
    # an fp32 output drops only the final bf16 rounding; P is still bf16
    _check(out, lse, *_oracle_decode(case))


def test_decode_causal_pair(m):
    case = synth.decode_case("pair", 442, B=3, H=128, seq_lens=[2, 64, 513], q_len=2,
                             poison=True)
    out, lse = _run_decode(m, case, split_tiles=4)
    _check(out, lse, *_oracle_decode(case))


def test_decode_max_q_len(m):
    """The largest q_len the call takes (64 causal query tokens per request):
    token i of request b sees seq_len - 64 + i + 1 keys, so the first token
    of the short request sees a single key and its last token all 64."""
    case = synth.decode_case("qlen64", 443, B=2, H=128, seq_lens=[64, 700], q_len=64,
                             poison=True)
    out, lse = _run_decode(m, case)
    ro, rl, t = _oracle_decode(case)
    # a token that sees one or a few keys outputs (nearly) a raw value row,
    # |o| up to ~5, where the bf16 rounding of the output alone (half an
    # ulp, 2^-8 relative) exceeds 1e-2: the max-abs bound gets that
    # documented term; the elementwise bound is unchanged
    _check(out, lse, ro, rl, t, out_tol=OUT_TOL + 2.0 ** -8 * float(np.abs(ro).max()),
           label="q_len 64")
    assert m.mla_get_device_error() == 0


def test_decode_max_heads(m):
    """The largest head count the call takes (H = 4096: 32 head groups of
    128, each its own job), over a ragged pair of requests."""
    case = synth.decode_case("h4096", 444, B=2, H=4096, seq_lens=[300, 65], poison=True)
    out, lse = _run_decode(m, case)
    ro, rl, t = _oracle_decode(case)
    # 4.2M outputs reach |o| where the bf16 rounding of the output alone
    # exceeds 1e-2: the documented 2^-8 |o| term, elementwise bound unchanged
    _check(out, lse, ro, rl, t, out_tol=OUT_TOL + 2.0 ** -8 * float(np.abs(ro).max()),
           label="H 4096")
    assert m.mla_get_device_error() == 0


def test_decode_explicit_shards_then_merge(m):
    """Tiny decode shape: 2 shards per request via kv_starts/kv_ends, merged by
    mla_merge_states, equals the unsplit decode."""
    case = synth.tiny_decode(poison=True)
    B = case.B
    parts_o, parts_l = [], []
    for s in range(2):
        st = np.array([sh[s][0] for sh in case.shards], np.int32)
        en = np.array([sh[s][1] for sh in case.shards], np.int32)
        o, l = _run_decode(m, case, kv_starts=st, kv_ends=en, out_dtype=torch.float32)
        _check(o, l, *_oracle_decode(case, kv_starts=st, kv_ends=en), out_tol=1e-3,
               label=f"shard {s}")
        parts_o.append(o.reshape(B, case.H, 512))
        parts_l.append(l.reshape(B, case.H))
    mo, ml = m.mla_merge_states(torch.stack(parts_o), torch.stack(parts_l),
                                out_dtype=torch.bfloat16)
    # the merge on its own, against the oracle's merge of the GPU's own parts
    po = np.stack([f64(x) for x in parts_o])
    pl = np.stack([x.cpu().numpy().astype(np.float64) for x in parts_l])
    mro, mrl = O.merge_states(po, pl)
    bo, bl = merge_bounds(mro, mrl, po, pl)
    assert np.all(np.abs(f64(mo) - mro) <= bo)
    d, fin = lse_close(ml.cpu().numpy(), mrl, 1e-3)
    assert fin and np.all(np.where(np.isneginf(mrl), 0.0, np.abs(ml.cpu().numpy() - mrl)) <= bl)
    # and the whole split-and-merge against the unsplit oracle
    ro, rl, t = _oracle_decode(case)
    _check(mo, ml, ro.reshape(B, case.H, 512), rl.reshape(B, case.H),
           t.take((slice(None), 0)), label="merged shards")


def test_decode_empty_ranges(m):
    case = synth.decode_case("empty", 443, B=3, H=16, seq_lens=[0, 50, 50], poison=True)
    out, lse = _run_decode(m, case, kv_starts=[0, 20, 7], kv_ends=[0, 20, 9])
    _check(out, lse, *_oracle_decode(case, kv_starts=[0, 20, 7], kv_ends=[0, 20, 9]))
    assert np.all(np.isneginf(lse.cpu().numpy()[:2]))
    assert np.all(f64(out)[:2] == 0)


def test_decode_peaked_scores(m):
    """Large-magnitude queries make the softmax peaked and the running max
    jump between tiles (exercises the lazy rescale)."""
    case = synth.decode_case("peaked", 444, B=2, H=128, seq_lens=[700, 2000], q_std=4.0,
                             kv_std_c=0.5, kv_std_pe=0.5, poison=True)
    out, lse = _run_decode(m, case)
    ro, rl, t = _oracle_decode(case)
    # outputs reach |o| ~ 2, where the bf16 rounding of the output alone
    # (half an ulp, 2^-8 relative) exceeds 1e-2: the max-abs bound gets that
    # documented term; the elementwise bound is unchanged
    _check(out, lse, ro, rl, t, out_tol=OUT_TOL + 2.0 ** -8 * float(np.abs(ro).max()))


def test_chain_absorb_decode_vup_dsv3_sampled(m):
    """DeepSeek-V3 decode shape (B=32, H=128, ctx 4096) end to end; the
    oracle checks 4 requests in full (the GPU runs all 32)."""
    case = synth.dsv3_decode()
    q = m.mla_absorb_q(case.q_nope.cuda(), case.q_pe.cuda(), case.w_uk_t.cuda())
    q = q.view(case.B, 1, case.H, 576)
    out, lse = m.mla_decode_paged(q, case.cache.cuda(), _i32(case.block_table),
                                  _i32(case.seq_lens), sm_scale=case.sm_scale)
    y = m.mla_v_up(out.view(case.B, case.H, 512), case.w_uv.cuda())
    pick = [0, 7, 19, 31]
    qo = f64(q)[pick]
    cache = f64(case.cache)
    bt, sl = case.block_table[pick], case.seq_lens[pick]
    # stage by stage: the decode against the oracle fed the GPU's own query
    ro, rl = O.paged_decode(qo, cache, bt, sl, case.sm_scale)
    t = decode_terms(qo, cache, bt, sl, case.sm_scale)
    _check(out[pick], lse[pick], ro, rl, t, label="DeepSeek-V3 decode")
    ref_y = O.v_up(f64(out)[pick][:, 0], f64(case.w_uv))
    abs_sum = np.einsum("thl,hvl->thv", np.abs(f64(out)[pick][:, 0]), np.abs(f64(case.w_uv)))
    assert np.all(np.abs(f64(y)[pick] - ref_y) <= gemm_tolerance(ref_y, abs_sum))
    # end to end against the unrounded fp64 chain: the bf16 rounding of the
    # absorbed query moves the exact LSE by (rl - el), computed here in fp64;
    # beyond that shift the GPU stays within the 1e-3 LSE bound
    q_true = O.absorb_q(f64(case.q_nope)[pick], f64(case.q_pe)[pick], f64(case.w_uk_t))
    eo, el = O.paged_decode(q_true[:, None], cache, bt, sl, case.sm_scale)
    assert max_abs(f64(out)[pick], eo) <= OUT_TOL
    assert np.all(np.abs(lse.cpu().numpy()[pick] - el) <= LSE_TOL + np.abs(rl - el))


def test_decode_long_request_shards(m):
    """ctx 131072 as 8 explicit shards (one launch, B'=8 shard rows) merged
    on the GPU, against the unsplit oracle."""
    case = synth.long_request()
    S = 8
    q = case.q.cuda().expand(S, 1, case.H, 576).contiguous()
    bt = np.repeat(case.block_table, S, axis=0)
    seq = np.repeat(case.seq_lens, S)
    st = np.array([a for a, _ in case.shards[0]], np.int32)
    en = np.array([z for _, z in case.shards[0]], np.int32)
    o, l = m.mla_decode_paged(q, case.cache.cuda(), _i32(bt), _i32(seq),
                              sm_scale=case.sm_scale, kv_starts=_i32(st),
                              kv_ends=_i32(en), out_dtype=torch.float32)
    mo, ml = m.mla_merge_states(o.view(S, 1, case.H, 512), l.view(S, 1, case.H),
                                out_dtype=torch.bfloat16)
    ro, rl, t = _oracle_decode(case)
    _check(mo, ml, ro.reshape(1, case.H, 512), rl.reshape(1, case.H),
           t.take((slice(None), 0)), label="long request")


def test_decode_spec_sampled(m):
    """Spec decode shape (B=128, q_len 2, lognormal ctx): all requests run,
    12 are checked in full by the oracle."""
    case = synth.spec_decode()
    out, lse = _run_decode(m, case)
    pick = [0, 1, 5, 17, 33, 50, 64, 77, 90, 101, 120, 127]
    _check(out[pick], lse[pick], *_oracle_decode(case, pick=pick), label="speculative decode")


def test_decode_reruns_bit_identical(m):
    """Race check: the split-KV work assignment is fixed, so repeated runs
    must agree bit for bit.  The spec-decode shape (many jobs, spans that
    cross job boundaries, partial merges) exercises every hand-off of the
    paired-CTA kernel; a hand-off that is not ordered shows up as a rerun
    that differs (this is how a staging-buffer race was caught)."""
    case = synth.spec_decode()
    out0, lse0 = _run_decode(m, case)
    ob0, lb0 = bits(out0), bits(lse0)
    for _ in range(40):
        out, lse = _run_decode(m, case)
        assert np.array_equal(bits(out), ob0)
        assert np.array_equal(bits(lse), lb0)


def test_decode_many_short_jobs(m):
    """Many jobs (B = 150 requests x 2 query tokens) of short ragged lengths,
    empty ones included, so most spans hold several whole jobs and few are
    split: against the oracle."""
    g = synth.generator(470)
    B = 150
    seq = g.integers(0, 200, B).astype(np.int32)
    case = synth.decode_case("many_jobs", 471, B=B, H=16, seq_lens=seq, q_len=2, poison=True)
    out, lse = _run_decode(m, case)
    ro, rl, t = _oracle_decode(case)
    # contexts of a few tokens leave outputs near single value rows (|out|
    # up to ~4): the max-abs bound gets the bf16 half-ulp term of the output
    _check(out, lse, ro, rl, t, out_tol=OUT_TOL + 2.0 ** -8 * float(np.abs(ro).max()))
    assert m.mla_get_device_error() == 0


# ------------------------------------------------------------- fp8 decode
FP8_OUT_TOL, FP8_LSE_TOL = 5e-2, 1e-2


@pytest.mark.parametrize("split_tiles", [0, 2])
def test_decode_fp8_ragged(m, split_tiles):
    case = synth.decode_case("fp8_small", 450, B=3, H=128, seq_lens=[5, 100, 700],
                             kv_dtype="e4m3", q_dtype="e4m3", poison=True)
    out, lse = _run_decode(m, case, split_tiles=split_tiles)
    _check(out, lse, *_oracle_decode(case), out_tol=FP8_OUT_TOL, lse_tol=FP8_LSE_TOL,
           label="fp8 ragged")
    assert m.mla_get_device_error() == 0


def test_decode_fp8_causal_pair_head_groups(m):
    case = synth.decode_case("fp8_pair", 451, B=2, H=144, seq_lens=[70, 1000], q_len=2,
                             kv_dtype="e4m3", q_dtype="e4m3", poison=True)
    out, lse = _run_decode(m, case, out_dtype=torch.float32)
    _check(out, lse, *_oracle_decode(case), out_tol=FP8_OUT_TOL, lse_tol=FP8_LSE_TOL,
           label="fp8 pair")


def test_decode_fp8_sampled(m):
    """FP8 KV shape (B=64, ctx U[1024,16384], e4m3 cache and query with
    per-tensor scales): all requests run, 6 are checked in full."""
    case = synth.fp8_decode()
    out, lse = _run_decode(m, case)
    pick = [0, 9, 21, 40, 52, 63]
    _check(out[pick], lse[pick], *_oracle_decode(case, pick=pick), out_tol=FP8_OUT_TOL,
           lse_tol=FP8_LSE_TOL, label="fp8 decode")
