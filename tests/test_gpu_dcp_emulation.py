"""Single-GPU emulation of the decode-context-parallel arithmetic the pages
describe, built from the library's entry points:

* DCP decode (MLA DCP prefill blog, §DCP 在 Prefill 与 Decode 中的不同角色):
  every rank holds an interleaved shard of the KV cache, computes partial
  attention (out, lse) of the full query over its shard, and the partials
  are combined by LSE weighting.
* The query all-gather of the DCP + FP8 KV decode digest (§关键源码片段
  mla_attention.py): a fake group concatenates the per-rank queries along
  the head dimension and counts calls, as the digest's test does.
* Multi-chunk chunked prefill (MLA DCP prefill blog, §Chunked Prefill 与
  LSE Merge): N context chunks gathered with seq_starts, N-1 inter-chunk
  merges plus one final merge.
* q_len = 4 speculative decode with the causal mask inside the group.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import mla as O
from tests._helpers import (bits, check_attention, decode_terms, f64, gemm_tolerance, max_abs,
                            merge_bounds, prefill_terms)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_kv_uk_gb300 as mod
    return mod


def _i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()


class FakeDCPGroup:
    """Stands in for the DCP process group on one GPU: all_gather stacks the
    ranks' tensors along `dim` and records the call."""

    def __init__(self, world):
        self.world = world
        self.calls = 0
        self.shapes = []

    def all_gather(self, per_rank, dim):
        self.calls += 1
        self.shapes.append(tuple(per_rank[0].shape))
        return torch.cat(per_rank, dim=dim)


@pytest.mark.parametrize("W", [2, 4])
def test_dcp_decode_interleaved_shards_merge(m, W):
    g = synth.generator(600 + W)
    case = synth.decode_case("dcp", 601, B=3, H=128, seq_lens=[40, 513, 3000])
    shards = synth.shard_cache_interleaved(g, case.cache, case.block_table,
                                           case.seq_lens, W, interleave=1)
    # query heads are split over the ranks; the fake group all-gathers them
    grp = FakeDCPGroup(W)
    per_rank_q = list(case.q.cuda().chunk(W, dim=2))
    q_full = grp.all_gather(per_rank_q, dim=2)
    assert grp.calls == 1 and q_full.shape[2] == case.H
    parts_o, parts_l = [], []
    for cache_k, bt_k, lens_k in shards:
        o, l = m.mla_decode_paged(q_full, cache_k.cuda(), _i32(bt_k), _i32(lens_k),
                                  sm_scale=case.sm_scale, out_dtype=torch.float32)
        parts_o.append(o.view(case.B, case.H, 512))
        parts_l.append(l.view(case.B, case.H))
    mo, ml = m.mla_merge_states(torch.stack(parts_o), torch.stack(parts_l),
                                out_dtype=torch.bfloat16)
    q64, c64 = f64(case.q), f64(case.cache)
    ro, rl = O.paged_decode(q64, c64, case.block_table, case.seq_lens, case.sm_scale)
    t = decode_terms(q64, c64, case.block_table, case.seq_lens, case.sm_scale)
    check_attention(f64(mo), ml.cpu().numpy(), ro[:, 0], rl[:, 0], t.take((slice(None), 0)),
                    out_tol=1e-2, lse_tol=1e-3, label=f"DCP W={W}")


def test_spec_decode_q_len4(m):
    case = synth.decode_case("q4", 610, B=3, H=128, seq_lens=[4, 130, 2000], q_len=4,
                             poison=True)
    out, lse = m.mla_decode_paged(case.q.cuda(), case.cache.cuda(), _i32(case.block_table),
                                  _i32(case.seq_lens), sm_scale=case.sm_scale, causal=True)
    q64, c64 = f64(case.q), f64(case.cache)
    ro, rl = O.paged_decode(q64, c64, case.block_table, case.seq_lens, case.sm_scale, causal=True)
    t = decode_terms(q64, c64, case.block_table, case.seq_lens, case.sm_scale)
    check_attention(f64(out), lse.cpu().numpy(), ro, rl, t, out_tol=1e-2, lse_tol=1e-3,
                    label="q_len 4")


@pytest.mark.parametrize("n_chunks,kv_dtype", [(2, "bf16"), (3, "bf16"), (3, "e4m3")])
def test_multi_chunk_prefill(m, n_chunks, kv_dtype):
    """Context split into n chunks per request: each chunk is gathered with
    seq_starts (dequantising an e4m3 cache to bf16 on the way), expanded and
    attended (non-causal); the chunk results are merged pairwise (n-1
    merges), then merged with the causal new-token attention (1 merge).
    Stage by stage against the oracle fed the GPU's own inputs, then end to
    end against the unrounded chain."""
    g = synth.generator(620 + n_chunks)
    H = 8
    ctx = np.array([300, 1000], np.int32)
    new = np.array([64, 130], np.int32)
    bt, nb = synth.paged_layout(g, ctx)
    cache, ks = synth.fill_cache(g, bt, ctx, nb, kv_dtype=kv_dtype, poison=True)
    w = synth.as_bf16(g.standard_normal((H * 256, 512)) * 0.05)
    new_kv = synth.as_bf16(g.standard_normal((int(new.sum()), 576)))
    q = synth.as_bf16(g.standard_normal((int(new.sum()), H, 192)))
    scale = 1 / np.sqrt(192)
    cu_q = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    q64, w64 = f64(q), f64(w)
    wabs = np.abs(w64).reshape(H, 256, 512)

    def expand_ok(rows64, K, V):
        rk, rv = O.expand_kv(rows64, w64, H)
        absk = np.einsum("nl,hcl->nhc", np.abs(rows64[:, :512]), wabs)
        assert np.all(np.abs(f64(K)[..., :128] - rk[..., :128])
                      <= gemm_tolerance(rk[..., :128], absk[..., :128]))
        assert np.array_equal(f64(K)[..., 128:], rk[..., 128:])
        assert np.all(np.abs(f64(V) - rv) <= gemm_tolerance(rv, absk[..., 128:]))
        return rk, rv

    def attn_ok(o, l, K, V, cu_k, causal, label):
        ro, rl = O.prefill_attention(q64, f64(K), f64(V), cu_q, cu_k, causal, scale)
        t = prefill_terms(q64, f64(K), f64(V), cu_q, cu_k, causal, scale)
        # the first causal rows see one or two keys, so |o| reaches ~4, where
        # the bf16 rounding of the output alone (2^-8 relative) exceeds 1e-2:
        # the max-abs bound gets that documented term
        check_attention(f64(o), l.cpu().numpy(), ro, rl, t,
                        out_tol=1e-2 + 2.0 ** -8 * float(np.abs(ro).max()), lse_tol=1e-3,
                        label=label)

    def merge_ok(o, l, parts):
        po = np.stack([f64(x) for x, _ in parts])
        pl = np.stack([y.cpu().numpy().astype(np.float64) for _, y in parts])
        mo, ml = O.merge_states(po, pl)
        bo, bl = merge_bounds(mo, ml, po, pl)
        assert np.all(np.abs(f64(o) - mo) <= bo)
        assert np.all(np.abs(l.cpu().numpy() - ml) <= bl)

    kn, vn = m.mla_expand_kv(new_kv.cuda(), w.cuda(), H)
    Kn, Vn = expand_ok(f64(new_kv), kn, vn)
    o_new, l_new = m.mla_prefill_attn(q.cuda(), kn, vn, _i32(cu_q), _i32(cu_q),
                                      int(new.max()), causal=True, sm_scale=scale)
    attn_ok(o_new, l_new, kn, vn, cu_q, True, "new tokens")
    acc_o = acc_l = None
    merges = 0
    for c in range(n_chunks):
        a = ctx * c // n_chunks
        z = ctx * (c + 1) // n_chunks
        cnt = (z - a).astype(np.int32)
        cu_c = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
        rows = m.mla_gather_cache(cache.cuda(), _i32(bt), _i32(ctx), _i32(cu_c),
                                  int(cu_c[-1]), seq_starts=_i32(a), k_scale=ks,
                                  out_dtype=torch.bfloat16)
        codes = O.gather_cache(bits(cache), bt, cu_c, seq_starts=a)
        want = codes if kv_dtype == "bf16" else O.dequant_e4m3_to_bf16(codes, ks)
        assert np.array_equal(bits(rows).astype(np.uint16), want.astype(np.uint16))
        kc, vc = m.mla_expand_kv(rows, w.cuda(), H)
        expand_ok(f64(rows), kc, vc)
        o_c, l_c = m.mla_prefill_attn(q.cuda(), kc, vc, _i32(cu_q), _i32(cu_c),
                                      int(new.max()), causal=False, sm_scale=scale)
        attn_ok(o_c, l_c, kc, vc, cu_c, False, f"chunk {c}")
        if acc_o is None:
            acc_o, acc_l = o_c, l_c
        else:
            mo_, ml_ = m.mla_merge_states(torch.stack([acc_o, o_c]), torch.stack([acc_l, l_c]))
            merge_ok(mo_, ml_, [(acc_o, acc_l), (o_c, l_c)])
            acc_o, acc_l = mo_, ml_
            merges += 1
    out, lse = m.mla_merge_states(torch.stack([acc_o, o_new]), torch.stack([acc_l, l_new]))
    merge_ok(out, lse, [(acc_o, acc_l), (o_new, l_new)])
    merges += 1
    assert merges == n_chunks
    assert m.mla_get_device_error() == 0
    # end to end against the unrounded chain (dequantised values for e4m3)
    cu_ctx = np.concatenate([[0], np.cumsum(ctx)])
    ctx_rows = O.gather_cache(f64(cache) * ks, bt, cu_ctx)
    Kc, Vc = O.expand_kv(ctx_rows, w64, H)
    ro, rl, om = O.chunked_prefill(q64, Kn, Vn, Kc, Vc, cu_q, cu_ctx, scale, n_chunks=n_chunks)
    assert om == n_chunks
    assert max_abs(f64(out), ro) <= 1e-2
