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
from tests._helpers import f64, lse_close, max_abs

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
    ro, rl = O.paged_decode(f64(case.q), f64(case.cache), case.block_table, case.seq_lens,
                            case.sm_scale)
    assert max_abs(f64(mo), ro[:, 0]) <= 1e-2
    d, fin = lse_close(ml.cpu().numpy(), rl[:, 0], 1e-3)
    assert fin and d <= 1e-3


def test_spec_decode_q_len4(m):
    case = synth.decode_case("q4", 610, B=3, H=128, seq_lens=[4, 130, 2000], q_len=4,
                             poison=True)
    out, lse = m.mla_decode_paged(case.q.cuda(), case.cache.cuda(), _i32(case.block_table),
                                  _i32(case.seq_lens), sm_scale=case.sm_scale, causal=True)
    ro, rl = O.paged_decode(f64(case.q), f64(case.cache), case.block_table, case.seq_lens,
                            case.sm_scale, causal=True)
    assert max_abs(f64(out), ro) <= 1e-2
    d, fin = lse_close(lse.cpu().numpy(), rl, 1e-3)
    assert fin and d <= 1e-3


@pytest.mark.parametrize("n_chunks", [2, 3])
def test_multi_chunk_prefill(m, n_chunks):
    """Context split into n chunks per request: each chunk is gathered with
    seq_starts, expanded and attended (non-causal); the chunk results are
    merged pairwise (n-1 merges), then merged with the causal new-token
    attention (1 merge)."""
    g = synth.generator(620 + n_chunks)
    H = 8
    ctx = np.array([300, 1000], np.int32)
    new = np.array([64, 130], np.int32)
    bt, nb = synth.paged_layout(g, ctx)
    cache, _ = synth.fill_cache(g, bt, ctx, nb, poison=True)
    w = synth.as_bf16(g.standard_normal((H * 256, 512)) * 0.05)
    new_kv = synth.as_bf16(g.standard_normal((int(new.sum()), 576)))
    q = synth.as_bf16(g.standard_normal((int(new.sum()), H, 192)))
    scale = 1 / np.sqrt(192)
    cu_q = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    kn, vn = m.mla_expand_kv(new_kv.cuda(), w.cuda(), H)
    o_new, l_new = m.mla_prefill_attn(q.cuda(), kn, vn, _i32(cu_q), _i32(cu_q),
                                      int(new.max()), causal=True, sm_scale=scale)
    acc_o = acc_l = None
    merges = 0
    for c in range(n_chunks):
        a = ctx * c // n_chunks
        z = ctx * (c + 1) // n_chunks
        cnt = (z - a).astype(np.int32)
        cu_c = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
        rows = m.mla_gather_cache(cache.cuda(), _i32(bt), _i32(ctx), _i32(cu_c),
                                  int(cu_c[-1]), seq_starts=_i32(a))
        kc, vc = m.mla_expand_kv(rows, w.cuda(), H)
        o_c, l_c = m.mla_prefill_attn(q.cuda(), kc, vc, _i32(cu_q), _i32(cu_c),
                                      int(new.max()), causal=False, sm_scale=scale)
        if acc_o is None:
            acc_o, acc_l = o_c, l_c
        else:
            acc_o, acc_l = m.mla_merge_states(torch.stack([acc_o, o_c]),
                                              torch.stack([acc_l, l_c]))
            merges += 1
    out, lse = m.mla_merge_states(torch.stack([acc_o, o_new]), torch.stack([acc_l, l_new]))
    merges += 1
    assert merges == n_chunks
    cu_ctx = np.concatenate([[0], np.cumsum(ctx)])
    ctx_rows = O.gather_cache(f64(cache), bt, cu_ctx)
    Kc, Vc = O.expand_kv(ctx_rows, f64(w), H)
    Kn, Vn = O.expand_kv(f64(new_kv), f64(w), H)
    ro, rl, om = O.chunked_prefill(f64(q), Kn, Vn, Kc, Vc, cu_q, cu_ctx, scale,
                                   n_chunks=n_chunks)
    assert om == n_chunks
    assert max_abs(f64(out), ro) <= 1e-2
    d, fin = lse_close(lse.cpu().numpy(), rl, 2e-3)
    assert fin and d <= 2e-3
