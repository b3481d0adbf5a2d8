"""Test helpers: bit-exact views of device/host tensors as fp64 for the oracle."""

import numpy as np
import torch

from oracle import codecs


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 value of every element of a bf16 / e4m3 / f32 tensor."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return codecs.bf16_to_f64(t.view(torch.int16).numpy())
    if t.dtype == torch.float8_e4m3fn:
        return codecs.e4m3_to_f64(t.view(torch.uint8).numpy())
    if t.dtype in (torch.float32, torch.float64):
        return t.numpy().astype(np.float64)
    raise TypeError(t.dtype)


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int32).numpy()


def max_abs(a, b, mask=None):
    d = np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))
    if mask is not None:
        d = d[mask]
    return float(d.max()) if d.size else 0.0


def gemm_tolerance(ref, abs_sum):
    """Bound for a bf16-output GEMM with fp32 accumulation: half a bf16 ulp of
    the result (2^-9 relative, 2^-8 used for margin) plus K-term fp32
    accumulation error (<= 2^-20 of the sum of |products| for K <= 512)."""
    return np.abs(ref) * 2.0 ** -8 + abs_sum * 2.0 ** -20 + 1e-30


def lse_close(gpu, ref, tol):
    g, r = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    both_inf = np.isneginf(g) & np.isneginf(r)
    d = np.where(both_inf, 0.0, np.abs(g - r))
    return float(np.nanmax(d)) if d.size else 0.0, bool(np.all(~np.isnan(d)))


# ----------------------------------------------------------------------
# Scale-aware error bounds for the attention outputs, derived from the
# arithmetic of the kernels (each term is a rounding the GPU performs that
# the fp64 oracle does not):
#   * the output is rounded to bf16 once: |bf16(x) - x| <= 2^-8 |x|
#     (unit roundoff of an 8-bit significand);
#   * P is rounded to bf16 before the P.V product while the normaliser l is
#     summed from the unrounded probabilities, so O moves by
#     sum_j w_j d_j V_j with |d_j| <= 2^-8: at most 2^-8 sum_j w_j |V_j|
#     (2^-7 is used: a factor 2 for the fp32 accumulation of the product
#     and second-order terms);
#   * the scores carry the fp32 accumulation error of the QK product,
#     |ds_j| <= 2^-14 sm_scale sum_i |q_i k_ji| (a generous bound on the
#     per-instruction roundings of the tensor-core accumulation), which moves
#     the LSE by at most max_j |ds_j| and the weights by
#     |dw_j| <= 2 max|ds| w_j;
#   * e4m3 P (fp8 path): |p~ - p| <= max(2^-4 p, 2^-10) (4-bit significand;
#     half the subnormal spacing 2^-9) with p relative to a running max that
#     is at or below the true one, so in weight units the error is at most
#     e_j = max(2^-4 w_j, 2^-10 / l*), l* = sum_j exp(s_j - s_max); whether
#     O is normalised by the rounded or the unrounded sum, the output moves
#     by at most (sum_j e_j |V_j| + E sum_j w_j |V_j|) / (1 - E), E = sum e_j.
# The LSE adds the fp32 rounding of m + log2(l) and of the merge:
# 2^-20 |lse| + 1e-5.
U_BF16 = 2.0 ** -8
U_E4M3 = 2.0 ** -4
E4M3_HALF_SUB = 2.0 ** -10


class AttnTerms:
    """abs_wv [..., Dv] = sum_j w_j |V_j|; smag [...] = sm_scale * max_j
    sum_i |q_i k_ji|; fp8_wv [..., Dv] the e4m3 P-rounding term (or None)."""

    def __init__(self, abs_wv, smag, fp8_wv=None):
        self.abs_wv, self.smag, self.fp8_wv = abs_wv, smag, fp8_wv

    def take(self, idx):
        return AttnTerms(self.abs_wv[idx], self.smag[idx],
                         None if self.fp8_wv is None else self.fp8_wv[idx])


def row_terms(q_rows, keys, values, sm_scale, fp8=False):
    """Error-analysis terms of softmax attention of H query rows (fp64)."""
    H, Dv = q_rows.shape[0], values.shape[1]
    if keys.shape[0] == 0:
        z = np.zeros((H, Dv))
        return z, np.zeros(H), (z.copy() if fp8 else None)
    s = sm_scale * (q_rows @ keys.T)
    smag = sm_scale * (np.abs(q_rows) @ np.abs(keys).T).max(axis=1)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    l = p.sum(axis=1, keepdims=True)
    w = p / l
    av = np.abs(values)
    abs_wv = w @ av
    fp8_wv = None
    if fp8:
        e = np.maximum(U_E4M3 * w, E4M3_HALF_SUB / l)
        E = e.sum(axis=1, keepdims=True)
        fp8_wv = np.where(E < 0.5, (e @ av + E * abs_wv) / np.maximum(1.0 - E, 0.5), np.inf)
    return abs_wv, smag, fp8_wv


def decode_terms(q, cache, block_table, seq_lens, sm_scale, causal=True, kv_starts=None,
                 kv_ends=None, fp8=False):
    """AttnTerms of the paged decode, over the same key ranges and rows as
    the oracle's paged_decode (q, cache: dequantised fp64 values)."""
    from oracle import mla as O
    B, q_len, H, _ = q.shape
    abs_wv = np.zeros((B, q_len, H, 512))
    smag = np.zeros((B, q_len, H))
    fp8_wv = np.zeros((B, q_len, H, 512)) if fp8 else None
    for b in range(B):
        for i in range(q_len):
            lo, hi = O.decode_range(int(seq_lens[b]), q_len, i, causal,
                                    None if kv_starts is None else kv_starts[b],
                                    None if kv_ends is None else kv_ends[b])
            blk, off = O.page_rows(block_table[b], np.arange(lo, hi))
            rows = cache[blk, off]
            a, s, f = row_terms(q[b, i], rows, rows[:, :512], sm_scale, fp8)
            abs_wv[b, i], smag[b, i] = a, s
            if fp8:
                fp8_wv[b, i] = f
    return AttnTerms(abs_wv, smag, fp8_wv)


def prefill_terms(q, k, v, cu_q, cu_k, causal, sm_scale, q_rows=None):
    """AttnTerms of the prefill attention (same ranges as the oracle's
    prefill_attention); rows not in q_rows are left at 0."""
    Tq, H, _ = q.shape
    abs_wv = np.zeros((Tq, H, v.shape[2]))
    smag = np.zeros((Tq, H))
    req = np.searchsorted(np.asarray(cu_q), np.arange(Tq), side="right") - 1
    for t in (range(Tq) if q_rows is None else q_rows):
        b = int(req[t])
        nq, nk = int(cu_q[b + 1] - cu_q[b]), int(cu_k[b + 1] - cu_k[b])
        i = t - int(cu_q[b])
        lim = max(min(nk, i + nk - nq + 1) if causal else nk, 0)
        ks = slice(int(cu_k[b]), int(cu_k[b]) + lim)
        for h in range(H):
            a, s, _ = row_terms(q[t, h][None], k[ks, h], v[ks, h], sm_scale)
            abs_wv[t, h], smag[t, h] = a[0], s[0]
    return AttnTerms(abs_wv, smag)


def attn_out_bound(ref, t, out_bf16=True):
    b = (2.0 ** -7 + 2.0 ** -13 * t.smag[..., None]) * t.abs_wv + 1e-7
    b = b + (U_BF16 if out_bf16 else 2.0 ** -20) * np.abs(ref)
    if t.fp8_wv is not None:
        b = b + 1.25 * t.fp8_wv
    return b


def attn_lse_bound(ref_l, t):
    r = np.where(np.isfinite(ref_l), np.abs(ref_l), 0.0)
    return 1e-5 + 2.0 ** -20 * r + 2.0 ** -14 * t.smag


def bound_report(out, lse, ref_o, ref_l, t, out_bf16=True):
    """(max-abs out error, max out error / bound, max-abs LSE error,
    max LSE error / bound, LSE finite where the oracle's is)."""
    o = np.asarray(out, np.float64)
    l = np.asarray(lse, np.float64)
    eo = np.abs(o - ref_o)
    ro = float((eo / attn_out_bound(ref_o, t, out_bf16)).max()) if eo.size else 0.0
    both_inf = np.isneginf(l) & np.isneginf(ref_l)
    el = np.where(both_inf, 0.0, np.abs(l - ref_l))
    finite = bool(np.all(~np.isnan(el)))
    rl = float(np.nanmax(el / attn_lse_bound(ref_l, t))) if el.size else 0.0
    return (float(eo.max()) if eo.size else 0.0, ro,
            float(np.nanmax(el)) if el.size else 0.0, rl, finite)


def check_attention(out, lse, ref_o, ref_l, t, *, out_tol, lse_tol, out_bf16=True, label=""):
    """North-star max-abs bounds plus the scale-aware elementwise bounds."""
    d_o, r_o, d_l, r_l, finite = bound_report(out, lse, ref_o, ref_l, t, out_bf16)
    print(f"{label}: out max-abs {d_o:.3e} ({r_o:.3f} of its bound), "
          f"lse max-abs {d_l:.3e} ({r_l:.3f} of its bound)")
    assert finite, "NaN in LSE"
    assert d_o <= out_tol, f"out max-abs {d_o}"
    assert d_l <= lse_tol, f"lse max-abs {d_l}"
    assert r_o <= 1.0, f"out error {r_o:.3f} x its scale-aware bound"
    assert r_l <= 1.0, f"lse error {r_l:.3f} x its scale-aware bound"


def merge_bounds(ref_o, ref_l, parts_o, parts_l, out_bf16=True):
    """Bounds for mla_merge_states: output rounding, and the fp32 rescaling
    (exp and sums) of S parts: 2^-18 sum_s w_s |o_s|."""
    po = np.asarray(parts_o, np.float64)
    pl = np.asarray(parts_l, np.float64)
    m = pl.max(axis=0)
    m_safe = np.where(np.isneginf(m), 0.0, m)
    w = np.where(np.isneginf(pl), 0.0, np.exp(pl - m_safe[None]))
    z = np.where(w.sum(axis=0) > 0, w.sum(axis=0), 1.0)
    wabs = (w[..., None] * np.where(w[..., None] > 0, np.abs(po), 0.0)).sum(axis=0) / z[..., None]
    bo = (U_BF16 if out_bf16 else 2.0 ** -20) * np.abs(ref_o) + 2.0 ** -18 * wabs + 1e-7
    S = po.shape[0]
    bl = 1e-6 + 2.0 ** -20 * (np.where(np.isfinite(ref_l), np.abs(ref_l), 0.0) + S)
    return bo, bl
