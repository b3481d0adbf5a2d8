"""GPU parity: paged gather / dequant / reorg (bit-exact) and the LSE merge
(within the decode tolerance) against the oracle."""

import math

import numpy as np
import pytest
import torch

import synth
from oracle import mla as O
from tests._helpers import bits, f64, lse_close, max_abs, merge_bounds

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_kv_uk_gb300 as mod
    return mod


def _dev(x):
    return torch.as_tensor(x).cuda()


def _i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_gather_bit_exact_with_seq_starts(m, kv_dtype):
    g = synth.generator(300)
    seq = np.array([1, 64, 130, 777, 5], np.int32)
    bt, nb = synth.paged_layout(g, seq)
    cache, ks = synth.fill_cache(g, bt, seq, nb, kv_dtype=kv_dtype, poison=True)
    starts = np.array([0, 13, 64, 100, 5], np.int32)
    cnt = np.minimum(seq - starts, [1, 40, 66, 600, 0]).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
    total = int(cu[-1]) + 3          # rows past cu[B] must stay untouched
    out = torch.full((total, 576), 7, dtype=cache.dtype, device="cuda") \
        if kv_dtype == "bf16" else torch.zeros((total, 576), dtype=cache.dtype, device="cuda")
    sentinel = bits(out)[-3:].copy()
    m.mla_gather_cache(_dev(cache), _i32(bt), _i32(seq), _i32(cu), total,
                       seq_starts=_i32(starts), k_scale=ks, out=out)
    ref = O.gather_cache(bits(cache), bt, cu, seq_starts=starts)
    got = bits(out)
    assert np.array_equal(got[:cu[-1]], ref)
    assert np.array_equal(got[cu[-1]:], sentinel)
    assert m.mla_get_device_error() == 0


def test_gather_dequant_bit_exact(m):
    g = synth.generator(301)
    seq = np.array([200, 64, 3], np.int32)
    bt, nb = synth.paged_layout(g, seq)
    cache, ks = synth.fill_cache(g, bt, seq, nb, kv_dtype="e4m3", poison=True)
    cu = np.concatenate([[0], np.cumsum(seq)]).astype(np.int32)
    out = m.mla_gather_cache(_dev(cache), _i32(bt), _i32(seq), _i32(cu), int(cu[-1]),
                             k_scale=ks, out_dtype=torch.bfloat16)
    codes = O.gather_cache(bits(cache), bt, cu)
    ref = O.dequant_e4m3_to_bf16(codes, ks)
    assert np.array_equal(bits(out).astype(np.uint16), ref)


def test_gather_flags_bad_ranges(m):
    g = synth.generator(302)
    seq = np.array([10], np.int32)
    bt, nb = synth.paged_layout(g, seq)
    cache, _ = synth.fill_cache(g, bt, seq, nb)
    m.mla_get_device_error()
    cu = np.array([0, 12], np.int32)      # asks for 2 rows past seq_len
    out = m.mla_gather_cache(_dev(cache), _i32(bt), _i32(seq), _i32(cu), 12)
    assert m.mla_get_device_error() & 4
    assert np.all(bits(out)[10:] == 0)
    bt_bad = bt.copy()
    bt_bad[0, 0] = nb + 5
    m.mla_gather_cache(_dev(cache), _i32(bt_bad), _i32(seq), _i32([0, 10]), 10)
    assert m.mla_get_device_error() & 1


@pytest.mark.parametrize("W,I,kv_dtype,out_dtype", [
    (4, 1, "bf16", "bf16"), (2, 3, "bf16", "bf16"), (4, 1, "e4m3", "e4m3"),
    (3, 2, "e4m3", "bf16"), (1, 1, "bf16", "bf16"),
    (16, 1, "bf16", "bf16"), (16, 5, "e4m3", "bf16")])   # the most shards the call takes
def test_reorg_bit_exact(m, W, I, kv_dtype, out_dtype):
    g = synth.generator(310 + W * 7 + I)
    ctx = np.array([1, 9, 64, 257, 1000], np.int32)
    bt, nb = synth.paged_layout(g, ctx)
    cache, ks = synth.fill_cache(g, bt, ctx, nb, kv_dtype=kv_dtype)
    shards = synth.shard_cache_interleaved(g, cache, bt, ctx, W, I)
    smb = max(s[1].shape[1] for s in shards)
    tables = []
    for _, sbt, _ in shards:
        t = np.full((len(ctx), smb), -1, np.int32)
        t[:, :sbt.shape[1]] = sbt
        tables.append(_i32(t))
    cu = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    p = (ctx // (I * W)) * I + np.minimum(ctx % (I * W), I)
    pcu = np.concatenate([[0], np.cumsum(p)]).astype(np.int32)
    odt = torch.bfloat16 if out_dtype == "bf16" else torch.float8_e4m3fn
    out, rm = m.mla_gather_cache_reorg([_dev(s[0]) for s in shards], tables, _i32(cu),
                                       int(cu[-1]), interleave=I, k_scale=ks,
                                       out_dtype=odt, padded_cu=_i32(pcu),
                                       rank_major_rows=W * int(pcu[-1]))
    ref_codes = O.gather_cache(bits(cache), bt, cu)
    np_shards = [(bits(s[0]), s[1], s[2]) for s in shards]
    buf, pp, off = O.rank_major_buffer(np_shards, ctx, W, I)
    assert np.array_equal(pp, p)
    if kv_dtype == out_dtype:
        assert np.array_equal(bits(out), ref_codes)
        assert np.array_equal(bits(rm), buf)
        assert np.array_equal(O.reorg(bits(rm), pp, off, ctx, W, I), ref_codes)
    else:
        assert np.array_equal(bits(out).astype(np.uint16), O.dequant_e4m3_to_bf16(ref_codes, ks))


@pytest.mark.parametrize("S,T,H,D,pdt,odt", [
    (2, 3, 16, 512, torch.float32, torch.bfloat16),
    (8, 1, 128, 512, torch.float32, torch.bfloat16),
    (3, 5, 7, 128, torch.bfloat16, torch.float32),
    (1, 2, 4, 64, torch.float32, torch.float32),
    # an odd number of 16-byte chunks per row (one chunk a thread), the
    # smallest row, and the warp-per-row form past eight parts up to the
    # largest part count the call takes
    (2, 3, 3, 24, torch.bfloat16, torch.bfloat16),
    (5, 2, 3, 8, torch.float32, torch.bfloat16),
    (12, 2, 5, 512, torch.bfloat16, torch.bfloat16),
    (256, 1, 2, 64, torch.float32, torch.float32)])
def test_merge_states(m, S, T, H, D, pdt, odt):
    g = synth.generator(320 + S)
    po = torch.from_numpy(g.standard_normal((S, T, H, D)).astype(np.float32)).to(pdt)
    pl = g.standard_normal((S, T, H)).astype(np.float32) * 3
    pl[0, 0, 0] = -np.inf                       # one empty part
    if S > 1:
        pl[:, 0, 1] = -np.inf                   # a fully empty row
        po[:, 0, 1] = float("nan")              # whose parts hold NaN
    out, lse = m.mla_merge_states(po.cuda(), torch.from_numpy(pl).cuda(), out_dtype=odt)
    ro, rl = O.merge_states(f64(po), pl.astype(np.float64))
    # output rounding plus the fp32 rescaling error (tests/_helpers.py)
    bo, bl = merge_bounds(ro, rl, f64(po), pl, out_bf16=odt == torch.bfloat16)
    err = np.abs(f64(out) - ro)
    print(f"merge S={S}: out max-abs {err.max():.3e} ({(err / bo).max():.3f} of its bound)")
    assert np.all(err <= bo)
    d, finite = lse_close(lse.cpu().numpy(), rl, 1e-3)
    assert finite and d <= 1e-3
    gl = lse.cpu().numpy()
    assert np.all(np.where(np.isneginf(rl), 0.0, np.abs(gl - rl)) <= bl)


def test_bounded_wait_timeout_is_reported_and_context_survives(m):
    """Failure detection without a fault: a device wait on a barrier that
    nothing completes gives up after ~1 ms of SM cycles and raises the
    timeout bit; the context stays usable (a decode right after is correct
    and raises nothing)."""
    m.mla_get_device_error()                     # start from a clear word
    m.mla_selftest_wait_timeout(2_000_000)
    assert m.mla_get_device_error() & 8
    case = synth.tiny_decode(poison=True)
    out, lse = m.mla_decode_paged(
        case.q.cuda(), case.cache.cuda(),
        torch.as_tensor(case.block_table, dtype=torch.int32).cuda(),
        torch.as_tensor(case.seq_lens, dtype=torch.int32).cuda(), sm_scale=case.sm_scale)
    ref_o, _ = O.paged_decode(f64(case.q), f64(case.cache), case.block_table, case.seq_lens,
                              case.sm_scale, causal=case.causal)
    assert max_abs(f64(out), ref_o) <= 1e-2
    assert m.mla_get_device_error() == 0
