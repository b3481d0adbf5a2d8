"""fp64 reference of every step of the absorbed-MLA decode path and of the
chunked-prefill context step (test infrastructure only).

All tensors are float64 numpy arrays unless stated; integer metadata is
int32/int64.  Notation: T query tokens, H heads, L = 512 latent rank,
R = 64 rope width, P = 128 per-head nope width, V = 128 per-head value
width, page size 64.

Each function restates one passage of the source pages (cited by page title
and section) as its plain definition.
"""

from __future__ import annotations

import math

import numpy as np

from . import codecs

BLOCK = 64
L, R, P, V = 512, 64, 128, 128
D_QK = L + R

NEG_INF = -math.inf


# --------------------------------------------------------------------------
# A1/A2: query absorption and concat(-quant)
# --------------------------------------------------------------------------

def absorb_q(q_nope, q_pe, w_uk_t):
    """ql[t,h,l] = sum_p q_nope[t,h,p] * W_UK_T[h,p,l]; q = ql ‖ q_pe.

    MLA DCP query replication digest, §实现拆解 5 (the decode branch runs the
    BMM against W_UK_T); MLA DCP prefill blog, §MLA Prefill vs Decode
    (decode absorbs Q into the latent space through an einsum, giving a
    576-wide single-latent-head query); DCP + FP8 KV MLA decode digest,
    §关键源码片段 mla_attention.py (nope and pe concatenated to (B, N, L+P)).
    Shapes: q_nope [T,H,P], q_pe [T,H,R], w_uk_t [H,P,L] -> [T,H,L+R]."""
    ql = np.einsum("thp,hpl->thl", q_nope, w_uk_t)
    return np.concatenate([ql, q_pe], axis=-1)


def concat_quant_e4m3(q_f32, q_scale):
    """e4m3 code of each query element divided by the per-tensor q scale.

    DCP + FP8 KV MLA decode digest, §关键源码片段 mla_attention.py
    (``_decode_concat_quant_fp8_op(mqa_ql_nope, mqa_q_pe, self._q_scale)``).
    Reading: x / q_scale in IEEE float32 (one correctly rounded division),
    then round-to-nearest-even with saturation to +-448.
    q_f32: float32 array (already concatenated, width 576) -> uint8 codes."""
    x = np.asarray(q_f32, dtype=np.float32) / np.float32(q_scale)
    return codecs.f32_to_e4m3(x)


# --------------------------------------------------------------------------
# A4: paged latent decode (forward_mqa)
# --------------------------------------------------------------------------

def page_rows(block_row, positions):
    """Physical cache rows (block, offset) of logical token positions."""
    positions = np.asarray(positions, dtype=np.int64)
    return block_row[positions // BLOCK].astype(np.int64), positions % BLOCK


def attend(q_rows, keys, values, sm_scale):
    """Plain softmax attention of H query rows over n keys.

    s_j = sm_scale * q·k_j;  lse = ln sum_j exp(s_j);  o = sum_j exp(s_j - lse) v_j.
    n == 0 gives o = 0, lse = -inf.  Computed stably as m + ln sum exp(s - m).
    q_rows [H, D], keys [n, D], values [n, Dv] -> (o [H, Dv], lse [H])."""
    H = q_rows.shape[0]
    n = keys.shape[0]
    if n == 0:
        return np.zeros((H, values.shape[1])), np.full(H, NEG_INF)
    s = sm_scale * (q_rows @ keys.T)               # [H, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(z))[:, 0]
    o = (e / z) @ values
    return o, lse


def decode_range(seq_len, q_len, i, causal, kv_start=None, kv_end=None):
    """Key range [lo, hi) seen by query token i of a request.

    Causal positions are absolute: query i of q_len sees keys
    < seq_len - q_len + i + 1 (the new tokens are already in the cache).
    kv_start/kv_end (an explicit shard) intersect that range."""
    hi = seq_len - q_len + i + 1 if causal else seq_len
    hi = min(hi, seq_len)
    lo = 0
    if kv_start is not None:
        lo = max(lo, int(kv_start))
    if kv_end is not None:
        hi = min(hi, int(kv_end))
    hi = max(hi, 0)
    lo = min(max(lo, 0), hi)
    return lo, hi


def paged_decode(q, cache, block_table, seq_lens, sm_scale, *, causal=True,
                 kv_starts=None, kv_ends=None):
    """Single-latent-head attention over a paged latent cache.

    DCP + FP8 KV MLA decode digest, §关键源码片段 mla_attention.py
    (``forward_mqa(mqa_q, kv_cache, attn_metadata)`` returns attn_out and
    lse); MLA DCP prefill blog, §MLA Prefill vs Decode (decode keeps KV in
    latent form, one head of width L+R = 576; the value is the L-wide latent
    part).  For request b, token i, head h:
        K_j = cache[slot(b,j)][0:576],  V_j = cache[slot(b,j)][0:512]
        slot(b,j) = block_table[b][j // 64] * 64 + j % 64
    q [B,q_len,H,576], cache [num_blocks,64,576] (dequantised values)
    -> out [B,q_len,H,512], lse [B,q_len,H] (natural log, scale included)."""
    B, q_len, H, _ = q.shape
    out = np.zeros((B, q_len, H, L))
    lse = np.full((B, q_len, H), NEG_INF)
    for b in range(B):
        for i in range(q_len):
            lo, hi = decode_range(int(seq_lens[b]), q_len, i, causal,
                                  None if kv_starts is None else kv_starts[b],
                                  None if kv_ends is None else kv_ends[b])
            blk, off = page_rows(block_table[b], np.arange(lo, hi))
            rows = cache[blk, off]                 # [n, 576]
            o, l = attend(q[b, i], rows, rows[:, :L], sm_scale)
            out[b, i], lse[b, i] = o, l
    return out, lse


# --------------------------------------------------------------------------
# A5/A10: LSE-rescaling merge (merge_attn_states)
# --------------------------------------------------------------------------

def merge_states(parts_out, parts_lse):
    """Merge S partial attention states over disjoint key sets.

    MLA DCP prefill blog, §Chunked Prefill 与 LSE Merge (merge_attn_states
    rescales each partial by its LSE; O(B×N×V) elementwise) and §DCP 在
    Prefill 与 Decode 中的不同角色 (decode combines per-rank partials by LSE
    weighting).  Per row: m = max_s lse_s, w_s = exp(lse_s - m),
    o = sum_s w_s o_s / sum_s w_s, lse = m + ln sum_s w_s.  Parts with
    lse = -inf get weight 0; if every part is -inf: o = 0, lse = -inf.
    parts_out [S, ..., D], parts_lse [S, ...] -> (out [..., D], lse [...])."""
    parts_out = np.asarray(parts_out, dtype=np.float64)
    parts_lse = np.asarray(parts_lse, dtype=np.float64)
    m = parts_lse.max(axis=0)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.where(np.isneginf(parts_lse), 0.0, np.exp(parts_lse - m_safe[None]))
    z = w.sum(axis=0)
    z_safe = np.where(empty, 1.0, z)
    contrib = np.where(w[..., None] > 0, parts_out, 0.0) * w[..., None]
    out = contrib.sum(axis=0) / z_safe[..., None]
    out = np.where(empty[..., None], 0.0, out)
    lse = np.where(empty, NEG_INF, m_safe + np.log(z_safe))
    return out, lse


# --------------------------------------------------------------------------
# A6: value up-projection
# --------------------------------------------------------------------------

def v_up(o_lat, w_uv):
    """out[t,h,v] = sum_l o_lat[t,h,l] * W_UV[h,v,l].

    MLA DCP prefill blog, §MLA Prefill vs Decode (W_UV decompresses the
    latent back to per-head values); MLA DCP query replication digest,
    §关键源码片段 mla.py (output_shape = (tokens, num_heads * v_head_dim)).
    o_lat [T,H,L], w_uv [H,V,L] -> [T,H,V]."""
    return np.einsum("thl,hvl->thv", o_lat, w_uv)


# --------------------------------------------------------------------------
# Before the path: rotary position embedding and the cache write
# --------------------------------------------------------------------------

def rope_inv_freq(dim=R, base=10000.0):
    """theta_i = base^(-2i/dim) for pair i < dim/2 (the rotary position
    embedding of RoFormer, Su et al. 2021, §3.2; the pages name the step,
    rotary_emb, but not its variant: this is the plain reading)."""
    i = np.arange(dim // 2, dtype=np.float64)
    return float(base) ** (-2.0 * i / dim)


def rope(x, positions, base=10000.0, interleaved=True):
    """Rotate the last axis of x (even width d) by each token's position.

    MLA DCP query replication digest, §关键源码片段 mla.py: rotary_emb is
    applied to the rope slice of the query (q[..., qk_nope_head_dim:]) and
    to k_pe before mla_attn.  Pair i of token t turns by angle
    positions[t] * theta_i:  (a, b) -> (a cos - b sin, a sin + b cos).
    interleaved: pair i = dims (2i, 2i+1) (RoFormer's layout);
    otherwise pair i = dims (i, i + d/2) (the rotate-half layout).
    x [T, ..., d] (fp64), positions [T] -> same shape."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(d, base)[None, :]
    shape = (ang.shape[0],) + (1,) * (x.ndim - 2) + (d // 2,)
    c, s = np.cos(ang).reshape(shape), np.sin(ang).reshape(shape)
    if interleaved:
        a, b = x[..., 0::2], x[..., 1::2]
    else:
        a, b = x[..., : d // 2], x[..., d // 2:]
    ra, rb = a * c - b * s, a * s + b * c
    out = np.empty_like(x)
    if interleaved:
        out[..., 0::2], out[..., 1::2] = ra, rb
    else:
        out[..., : d // 2], out[..., d // 2:] = ra, rb
    return out


def cache_write(cache, kv_c_bits, k_pe_bits, slot_mapping, kv_dtype="bf16", k_scale=1.0):
    """Store new tokens' latent rows kv_c ‖ k_pe into the paged cache.

    MLA DCP prefill blog, §Chunked Prefill 与 LSE Merge (the new tokens'
    KV is already in the cache when attention runs) and MLA DCP query
    replication digest, §关键源码片段 mla.py (kv_c_normed and the rotated
    k_pe are what the attention layer receives).  Token n goes to physical
    row slot_mapping[n] = block * 64 + offset; a negative slot is padding
    and writes nothing.  A bf16 cache stores the bits; an e4m3 cache stores
    e4m3(f32(value) / f32(k_scale)) (round to nearest even, saturating).
    cache: uint16 bf16 bits or uint8 e4m3 codes [num_blocks, 64, 576];
    kv_c_bits [T, 512], k_pe_bits [T, 64]: bf16 bits.  Returns a copy."""
    out = np.array(cache, copy=True)
    rows = np.concatenate([np.asarray(kv_c_bits, np.uint16),
                           np.asarray(k_pe_bits, np.uint16)], axis=1)
    if kv_dtype == "bf16":
        codes = rows
    else:
        vals = codecs.bf16_to_f64(rows).astype(np.float32) / np.float32(k_scale)
        codes = codecs.f32_to_e4m3(vals)
    for n, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        out[slot // BLOCK, slot % BLOCK] = codes[n]
    return out


# --------------------------------------------------------------------------
# A7: paged gather, dequantising gather, interleaved-shard reorg
# --------------------------------------------------------------------------

def gather_cache(cache, block_table, cu_out, seq_starts=None):
    """Gather each request's rows from the paged cache into a dense buffer.

    MLA DCP prefill blog, §与非 DCP 的流程对比 and §关于 cp_gather_cache 的命名澄清
    (cp_gather_cache is a gather without dequantisation);
    DCP + FP8 KV MLA decode digest, §实现拆解 3-4 (the MLA gather with
    seq_starts).  out[cu_out[b] + j] = cache[slot(b, seq_starts[b] + j)] for
    j < cu_out[b+1] - cu_out[b].  Works on any element type (bit copy)."""
    B = len(cu_out) - 1
    total = int(cu_out[-1])
    out = np.zeros((total,) + cache.shape[2:], dtype=cache.dtype)
    for b in range(B):
        n = int(cu_out[b + 1] - cu_out[b])
        s0 = 0 if seq_starts is None else int(seq_starts[b])
        blk, off = page_rows(block_table[b], np.arange(s0, s0 + n))
        out[int(cu_out[b]):int(cu_out[b]) + n] = cache[blk, off]
    return out


def dequant_e4m3_to_bf16(codes, k_scale):
    """bf16 bits of float32(e4m3 value) * float32(k_scale), RNE.

    DCP + FP8 KV MLA decode digest, §实现拆解 3 (gather_and_maybe_dequant_cache
    dequantises fp8 rows with the cache scale).  One float32 multiply and one
    round to bf16; both are exact-rule operations, so the result is unique."""
    v = codecs.e4m3_to_f64(codes).astype(np.float32)
    prod = v * np.float32(k_scale)
    return codecs.f32_to_bf16(prod)


def shard_local_index(t, W, interleave):
    """(shard k, local index j) of global token t under interleave I."""
    t = np.asarray(t, dtype=np.int64)
    return (t // interleave) % W, (t // (interleave * W)) * interleave + t % interleave


def rank_major_buffer(shards, ctx_lens, W, interleave):
    """The all-gathered buffer of per-shard local gathers, rank-major.

    MLA DCP prefill blog, §与非 DCP 的流程对比 steps 1-3: each rank gathers its
    local rows with padded per-request offsets, then all_gather(dim=0)
    stacks the ranks.  Reading: each request's local run on every shard is
    padded with zero rows to p_r = max_k n_{r,k}; shard k's block occupies
    rows [k*sum_r p_r, (k+1)*sum_r p_r).
    shards: W x (cache, block_table, local_lens).  Returns (buffer, p, off)."""
    B = len(ctx_lens)
    n = np.zeros((B, W), dtype=np.int64)
    for r in range(B):
        k, _ = shard_local_index(np.arange(int(ctx_lens[r])), W, interleave)
        for kk in range(W):
            n[r, kk] = int((k == kk).sum())
    p = n.max(axis=1)
    off = np.concatenate([[0], np.cumsum(p)])
    sum_p = int(off[-1])
    cache0 = shards[0][0]
    buf = np.zeros((W * sum_p,) + cache0.shape[2:], dtype=cache0.dtype)
    for kk, (sc, sbt, slens) in enumerate(shards):
        for r in range(B):
            cnt = int(n[r, kk])
            assert cnt == int(slens[r])
            blk, o = page_rows(sbt[r], np.arange(cnt))
            base = kk * sum_p + int(off[r])
            buf[base:base + cnt] = sc[blk, o]
    return buf, p, off


def reorg(buf, p, off, ctx_lens, W, interleave):
    """Rank-major all-gather buffer -> rows in original sequence order.

    MLA DCP prefill blog, §与非 DCP 的流程对比 step 4 (reorg_kvcache restores
    sequence order using the padded local lengths and every rank's local
    context lengths).  out[cu_r + t] = buf[k * sum_p + off_r + j] with
    (k, j) = shard_local_index(t)."""
    sum_p = int(off[-1])
    cu = np.concatenate([[0], np.cumsum(np.asarray(ctx_lens, dtype=np.int64))])
    out = np.zeros((int(cu[-1]),) + buf.shape[1:], dtype=buf.dtype)
    for r in range(len(ctx_lens)):
        t = np.arange(int(ctx_lens[r]))
        k, j = shard_local_index(t, W, interleave)
        out[int(cu[r]) + t] = buf[k * sum_p + int(off[r]) + j]
    return out


# --------------------------------------------------------------------------
# A8-A10: kv_b_proj expand, prefill attention, final merge
# --------------------------------------------------------------------------

def expand_kv(kv_rows, w_kvb, H, heads=None):
    """kv_b_proj: latent rows -> per-head K (nope ‖ rope) and V.

    MLA DCP prefill blog, §MLA Prefill vs Decode (prefill decompresses kv_c
    through W_UK/W_UV into N full heads; K head dim P+R = 192, V head 128)
    and §与非 DCP 的流程对比 step 5.  With W_kvb [H*256, L] (per head: rows
    [0,128) are W_UK, [128,256) are W_UV):
        K[n,h,0:128] = kv_c[n] · W_UK_h^T,  K[n,h,128:192] = k_pe[n],
        V[n,h,:]     = kv_c[n] · W_UV_h^T.
    ``heads`` restricts the expansion to a subset (sampled checks)."""
    heads = range(H) if heads is None else heads
    kv_c, k_pe = kv_rows[:, :L], kv_rows[:, L:]
    hs = list(heads)
    K = np.empty((kv_rows.shape[0], len(hs), P + R))
    Vv = np.empty((kv_rows.shape[0], len(hs), V))
    for idx, h in enumerate(hs):
        w = w_kvb[h * (P + V):(h + 1) * (P + V)]
        K[:, idx, :P] = kv_c @ w[:P].T
        K[:, idx, P:] = k_pe
        Vv[:, idx] = kv_c @ w[P:].T
    return K, Vv


def absorbed_weights(w_kvb, H):
    """W_UK_T [H,P,L] and W_UV [H,V,L] sliced from one kv_b_proj weight."""
    w = np.asarray(w_kvb).reshape(H, P + V, L)
    return w[:, :P, :].copy(), w[:, P:, :].copy()


def prefill_attention(q, k, v, cu_q, cu_k, causal, sm_scale, q_rows=None):
    """Multi-head attention of new tokens over keys, returning LSE.

    MLA DCP prefill blog, §Chunked Prefill 与 LSE Merge: step 1 is causal
    attention of the new tokens over themselves (return_softmax_lse), step 2
    the non-causal attention of the new tokens over the cached context.
    Causal alignment is bottom-right: query i of a request with nq queries
    and nk keys sees keys j <= i + nk - nq.
    q [Tq,H,192], k [Nk,H,192], v [Nk,H,Vd] -> out [Tq,H,Vd], lse [Tq,H].
    ``q_rows`` (optional) restricts the computation to those query rows;
    other rows are left as NaN."""
    Tq, H, _ = q.shape
    out = np.full((Tq, H, v.shape[2]), np.nan)
    lse = np.full((Tq, H), np.nan)
    rows = range(Tq) if q_rows is None else q_rows
    B = len(cu_q) - 1
    req = np.searchsorted(np.asarray(cu_q), np.arange(Tq), side="right") - 1
    for t in rows:
        b = int(req[t])
        nq = int(cu_q[b + 1] - cu_q[b])
        nk = int(cu_k[b + 1] - cu_k[b])
        i = t - int(cu_q[b])
        lim = min(nk, i + nk - nq + 1) if causal else nk
        lim = max(lim, 0)
        ks = slice(int(cu_k[b]), int(cu_k[b]) + lim)
        for h in range(H):
            o, l = attend(q[t, h][None], k[ks, h], v[ks, h], sm_scale)
            out[t, h], lse[t, h] = o[0], l[0]
    assert B >= 1
    return out, lse


def chunked_prefill(q, k_new, v_new, k_ctx, v_ctx, cu_q, cu_ctx, sm_scale,
                    n_chunks=1, q_rows=None):
    """forward_mha with cached context: causal new-token attention, chunked
    non-causal context attention with inter-chunk merges, final merge.

    MLA DCP prefill blog, §Chunked Prefill 与 LSE Merge: N context chunks
    need N-1 inter-chunk merges plus one final merge, N merges in all.
    Returns (out, lse, merges_done)."""
    out_new, lse_new = prefill_attention(q, k_new, v_new, cu_q, cu_q, True,
                                         sm_scale, q_rows)
    merges = 0
    B = len(cu_ctx) - 1
    ctx_out = ctx_lse = None
    for c in range(n_chunks):
        # chunk c of every request: an even split of its context
        lo = np.zeros(B + 1, dtype=np.int64)
        ks, vs = [], []
        for b in range(B):
            n = int(cu_ctx[b + 1] - cu_ctx[b])
            a, z = c * n // n_chunks, (c + 1) * n // n_chunks
            ks.append(k_ctx[int(cu_ctx[b]) + a:int(cu_ctx[b]) + z])
            vs.append(v_ctx[int(cu_ctx[b]) + a:int(cu_ctx[b]) + z])
            lo[b + 1] = lo[b] + (z - a)
        o_c, l_c = prefill_attention(q, np.concatenate(ks), np.concatenate(vs),
                                     cu_q, lo, False, sm_scale, q_rows)
        if ctx_out is None:
            ctx_out, ctx_lse = o_c, l_c
        else:
            ctx_out, ctx_lse = _merge_rows(ctx_out, ctx_lse, o_c, l_c, q_rows)
            merges += 1
    out, lse = _merge_rows(ctx_out, ctx_lse, out_new, lse_new, q_rows)
    merges += 1
    return out, lse, merges


def _merge_rows(o1, l1, o2, l2, q_rows):
    out = np.full_like(o1, np.nan)
    lse = np.full_like(l1, np.nan)
    rows = range(o1.shape[0]) if q_rows is None else q_rows
    for t in rows:
        o, l = merge_states(np.stack([o1[t], o2[t]]), np.stack([l1[t], l2[t]]))
        out[t], lse[t] = o, l
    return out, lse
