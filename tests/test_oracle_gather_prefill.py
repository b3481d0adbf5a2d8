"""Pins for the oracle's gather / dequant / reorg, split plan, expand and
prefill-attention definitions."""

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


@pytest.mark.parametrize("n_ctas", [1, 7, 152])
@pytest.mark.parametrize("job_cost", [0, 4])
def test_plan_covers_each_job_exactly_once(n_ctas, job_cost):
    g = _rng(40)
    lo = g.integers(0, 50, 30)
    hi = lo + g.integers(0, 3000, 30)
    hi[3] = lo[3]                     # an empty job
    plan = mla.decode_plan(lo, hi, n_ctas, job_cost=job_cost)
    C, tp = plan["chunk"], plan["tile_prefix"]
    assert C >= -(-plan["total"] // n_ctas)
    # brute force: walk every CTA's span and record which tiles of which job
    # it meets; every tile of every job must be met exactly once
    n = np.array([0 if hi[j] <= lo[j] else
                  len(set(range(lo[j] // 32, (hi[j] - 1) // 32 + 1))) for j in range(len(lo))])
    first = tp[:-1] + np.where(n > 0, job_cost, 0)
    segs = np.zeros(len(lo), np.int64)
    seen = [np.zeros(int(k), np.int64) for k in n]
    for p in range(-(-plan["total"] // C)):
        a, z = p * C, min((p + 1) * C, plan["total"])
        for j in range(len(lo)):
            u0, u1 = max(a, first[j]), min(z, tp[j + 1])
            if u0 < u1:
                segs[j] += 1
                seen[j][u0 - first[j]:u1 - first[j]] += 1
    assert all(np.all(s_ == 1) for s_ in seen)
    assert np.array_equal(np.diff(plan["seg_prefix"]), segs)
    assert -(-plan["total"] // C) <= n_ctas
    # units per job: its tiles of 32 that meet [lo, hi), plus the switch cost
    assert np.array_equal(np.diff(tp), np.where(n > 0, n + job_cost, 0))


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
