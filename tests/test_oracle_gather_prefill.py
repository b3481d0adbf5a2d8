"""Pins for the oracle's gather / dequant / reorg, expand and prefill-attention
definitions, and for the split-plan validity checker."""

import math

import numpy as np
import pytest
import torch

from oracle import codecs, mla
import synth


def _rng(s):
    return np.random.Generator(np.random.PCG64(s))


def _paged_ints(g, seq_lens, width=576):
    bt, nb = synth.paged_layout(g, seq_lens)
    # distinct integer payload per (block, row, col) makes any misplacement visible
    cache = np.arange(nb * 64 * width, dtype=np.int64).reshape(nb, 64, width)
    return cache, bt


def test_gather_is_the_logical_sequence():
    g = _rng(20)
    seq = np.array([3, 64, 130, 1], np.int32)
    cache, bt = _paged_ints(g, seq)
    cu = np.concatenate([[0], np.cumsum(seq)])
    out = mla.gather_cache(cache, bt, cu)
    for b, n in enumerate(seq):
        for j in range(n):
            blk = bt[b, j // 64]
            assert np.array_equal(out[cu[b] + j], cache[blk, j % 64])


def test_gather_seq_starts_equals_slice_of_full_gather():
    """DCP + FP8 KV MLA decode digest, §实现拆解 4: the MLA gather with
    seq_starts.  A shifted gather is a slice of the unshifted one."""
    g = _rng(21)
    seq = np.array([100, 257, 64], np.int32)
    cache, bt = _paged_ints(g, seq)
    full = mla.gather_cache(cache, bt, np.concatenate([[0], np.cumsum(seq)]))
    starts = np.array([37, 64, 0])
    cnt = np.array([50, 193, 64])
    cu = np.concatenate([[0], np.cumsum(cnt)])
    part = mla.gather_cache(cache, bt, cu, seq_starts=starts)
    fcu = np.concatenate([[0], np.cumsum(seq)])
    for b in range(3):
        assert np.array_equal(part[cu[b]:cu[b + 1]],
                              full[fcu[b] + starts[b]:fcu[b] + starts[b] + cnt[b]])


def test_dequant_matches_torch_float8_cast():
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]
    for scale in (1.0, 0.0123, 3.7):
        ours = mla.dequant_e4m3_to_bf16(codes, scale)
        t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32)
        ref = (t * torch.tensor(scale, dtype=torch.float32)).to(torch.bfloat16)
        assert np.array_equal(ours, ref.view(torch.int16).numpy().astype(np.uint16))


@pytest.mark.parametrize("W,I", [(1, 1), (2, 1), (4, 1), (4, 3), (3, 2)])
def test_reorg_inverts_interleaved_sharding(W, I):
    """MLA DCP prefill blog, §与非 DCP 的流程对比: local gather on every rank,
    rank-major all-gather, reorg back to sequence order == plain gather."""
    g = _rng(30 + W * 10 + I)
    ctx = np.array([1, 9, 64, 200], np.int32)
    bt, nb = synth.paged_layout(g, ctx)
    cache = torch.arange(nb * 64 * 4, dtype=torch.int32).reshape(nb, 64, 4)
    shards = synth.shard_cache_interleaved(g, cache, bt, ctx, W, I)
    np_shards = [(sc.numpy(), sbt, sl) for sc, sbt, sl in shards]
    buf, p, off = mla.rank_major_buffer(np_shards, ctx, W, I)
    got = mla.reorg(buf, p, off, ctx, W, I)
    ref = mla.gather_cache(cache.numpy(), bt, np.concatenate([[0], np.cumsum(ctx)]))
    assert np.array_equal(got, ref)
    # the rank-major buffer holds each shard's run, padded with zero rows
    assert buf.shape[0] == W * int(p.sum())


def test_shard_local_index_is_a_bijection():
    for W, I in [(2, 1), (4, 1), (4, 5)]:
        t = np.arange(1000)
        k, j = mla.shard_local_index(t, W, I)
        pairs = set(zip(k.tolist(), j.tolist()))
        assert len(pairs) == 1000
        for kk in range(W):
            jj = np.sort(j[k == kk])
            assert np.array_equal(jj, np.arange(len(jj)))


# The split plan is the library's own schedule, not a definition from the
# pages, so it is checked for validity (tests/plan_check.py), not against a
# reference schedule.  These pins make sure the checker accepts a plan worked
# out by hand and rejects plausible corruptions of it.
#   jobs: [0,130) -> key tiles 0..2 (3 tiles); [10,10) empty; [0,64) -> 1 tile
#   units: 3 + 4 (switch cost), 0, 1 + 4  -> prefix 0, 7, 7, 12 (total 12)
#   auto, 3 groups: C = 4, spans [0,4) [4,8) [8,12); job 0's tiles sit at
#   units 4..6 (span 1 only), job 2's at unit 11 (span 2) -> segs 1, 0, 1
#   forced C = 2: spans of 2 units; job 0 at 4..6 meets spans 2 and 3,
#   job 2 at 11 meets span 5 -> segs 2, 0, 1
_LO, _HI = [0, 10, 0], [130, 10, 64]
_PLAN_AUTO3 = [12, 4, 3, 3, 0, 7, 7, 12, 0, 1, 1, 2, 0, 10, 0, 0, 130, 10, 64, 0]
_PLAN_FORCED2 = [12, 2, 3, 6, 0, 7, 7, 12, 0, 2, 2, 3, 0, 10, 0, 0, 130, 10, 64, 0]


def test_plan_checker_accepts_hand_worked_plans():
    from tests.plan_check import check_split_plan
    check_split_plan(_PLAN_AUTO3, _LO, _HI, n_groups=3)
    check_split_plan(_PLAN_FORCED2, _LO, _HI, n_groups=3, split_tiles=2)


@pytest.mark.parametrize("field,idx,value", [
    ("seg", 11, 3),         # one extra segment counted for job 2
    ("units", 1, 6),        # job 0 short of one tile (prefix 0, 6, 6, 11)
    ("chunk", 1, 3),        # C = 3 -> 4 spans for 3 groups
    ("hi", 16, 129),        # job 0's key range recorded wrong
    ("spans", 3, 2),        # span count inconsistent with C
])
def test_plan_checker_rejects_corrupted_plans(field, idx, value):
    from tests.plan_check import check_split_plan
    plan = list(_PLAN_AUTO3)
    if field == "units":
        plan[4:8] = [0, 6, 6, 11]
        plan[0] = 11
    elif field == "chunk":
        plan[1], plan[3] = 3, 4
    else:
        plan[idx] = value
    with pytest.raises(AssertionError):
        check_split_plan(plan, _LO, _HI, n_groups=3)


def test_job_ranges_follow_the_causal_definition():
    from tests.plan_check import job_ranges
    lo, hi = job_ranges([5, 0], 2, 200, True, kv_starts=[1, 0], kv_ends=[4, 9])
    # token-major: (token 0: request 0, request 1), (token 1: request 0,
    # request 1), two head groups each.  Request 0: token 0 sees keys < 4 ->
    # [1,4); token 1 < 5 -> [1, min(5,4)=4).  Request 1: empty.
    assert lo.tolist() == [1, 1, 0, 0, 1, 1, 0, 0]
    assert hi.tolist() == [4, 4, 0, 0, 4, 4, 0, 0]


def test_expand_brute_force():
    g = _rng(50)
    H = 2
    w = g.standard_normal((H * 256, 512))
    kv = g.standard_normal((3, 576))
    K, Vv = mla.expand_kv(kv, w, H)
    for n in range(3):
        for h in range(H):
            for c in (0, 127):
                assert abs(K[n, h, c] - sum(kv[n, l] * w[h * 256 + c, l] for l in range(512))) < 1e-10
                assert abs(Vv[n, h, c] - sum(kv[n, l] * w[h * 256 + 128 + c, l] for l in range(512))) < 1e-10
            assert np.array_equal(K[n, h, 128:], kv[n, 512:])


def test_prefill_causal_brute_force():
    g = _rng(51)
    H, d = 2, 6
    cu = np.array([0, 3, 7])
    q, k, v = g.standard_normal((7, H, d)), g.standard_normal((7, H, d)), g.standard_normal((7, H, 4))
    out, lse = mla.prefill_attention(q, k, v, cu, cu, True, 0.5)
    for b in range(2):
        for i in range(cu[b + 1] - cu[b]):
            t = cu[b] + i
            for h in range(H):
                s = [0.5 * float(q[t, h] @ k[cu[b] + j, h]) for j in range(i + 1)]
                m = max(s)
                z = sum(math.exp(x - m) for x in s)
                assert abs(lse[t, h] - (m + math.log(z))) < 1e-13
                o = sum(math.exp(s[j] - m) / z * v[cu[b] + j, h] for j in range(i + 1))
                assert np.allclose(out[t, h], o, atol=1e-13)


@pytest.mark.parametrize("n_chunks", [1, 2, 3])
def test_chunked_prefill_equals_full_attention(n_chunks):
    """MLA DCP prefill blog, §Chunked Prefill 与 LSE Merge: new-token causal
    attention, chunked context attention and N merges reproduce attention
    over [context ‖ new tokens] with the causal mask on the new part."""
    g = _rng(52 + n_chunks)
    H, d, dv = 3, 8, 5
    nq, nc = np.array([4, 6]), np.array([9, 5])
    cu_q = np.concatenate([[0], np.cumsum(nq)])
    cu_c = np.concatenate([[0], np.cumsum(nc)])
    q = g.standard_normal((nq.sum(), H, d))
    kn, vn = g.standard_normal((nq.sum(), H, d)), g.standard_normal((nq.sum(), H, dv))
    kc, vc = g.standard_normal((nc.sum(), H, d)), g.standard_normal((nc.sum(), H, dv))
    out, lse, merges = mla.chunked_prefill(q, kn, vn, kc, vc, cu_q, cu_c, 0.4, n_chunks)
    assert merges == n_chunks
    for b in range(2):
        K = np.concatenate([kc[cu_c[b]:cu_c[b + 1]], kn[cu_q[b]:cu_q[b + 1]]])
        Vv = np.concatenate([vc[cu_c[b]:cu_c[b + 1]], vn[cu_q[b]:cu_q[b + 1]]])
        for i in range(nq[b]):
            t = cu_q[b] + i
            lim = nc[b] + i + 1
            for h in range(H):
                o, l = mla.attend(q[t, h][None], K[:lim, h], Vv[:lim, h], 0.4)
                assert np.allclose(out[t, h], o[0], atol=1e-13)
                assert abs(lse[t, h] - l[0]) < 1e-13
