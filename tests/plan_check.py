"""Validity checker for the split-KV plan that mla_decode_plan / mla_decode_paged
write (test helper; not part of the oracle).

The pages fix only what the plan is derived from: the scheduler metadata of
the FlashMLA backend is built from seq_lens and the true query-head count
(DCP + FP8 KV MLA decode digest, §关键源码片段 flashmla.py).  How the key
tiles are cut into spans is this library's own schedule, so a plan is not
compared with a reference schedule: it is checked for validity.  Given the
per-job key ranges (from the causal definition the oracle states), a plan is
valid when, walking the spans the way the decode kernel consumes them,

* every job's key range is recorded exactly (job_lo / job_hi);
* the unit prefix starts at 0, never decreases, and gives an empty job no
  units and a non-empty job its key tiles plus one switch cost that is the
  same for every non-empty job;
* the spans [p*C, (p+1)*C) tile the flat unit space, none longer than C,
  and there are no more of them than CTA groups (auto split) or exactly
  ceil(total / split_tiles) of them (forced split);
* every key tile of every job is met by exactly one span;
* the segment prefix counts, per job, the spans that meet its tiles.

Plan layout (int32, documented with mla_decode_plan): [0] total units,
[1] C, [2] J, [3] spans, then unit_prefix[J+1], seg_prefix[J+1],
job_lo[J+1], job_hi[J+1].
"""

from __future__ import annotations

import numpy as np

from oracle import mla as O

TILE = 64   # key tokens per tile of the bf16 and e4m3 decode kernels


def job_ranges(seq_lens, q_len, H, causal, kv_starts=None, kv_ends=None):
    """Key range [lo, hi) of every job (query token i, request b, head group
    of 128: token-major, the documented plan order), from the oracle's
    causal-range definition."""
    HG = (H + 127) // 128
    lo, hi = [], []
    for i in range(q_len):
        for b in range(len(seq_lens)):
            a, z = O.decode_range(int(seq_lens[b]), q_len, i, causal,
                                  None if kv_starts is None else kv_starts[b],
                                  None if kv_ends is None else kv_ends[b])
            lo += [a] * HG
            hi += [z] * HG
    return np.asarray(lo, np.int64), np.asarray(hi, np.int64)


def split_plan_fields(plan, J):
    plan = np.asarray(plan, np.int64)
    off = 4
    tp = plan[off:off + J + 1]
    sp = plan[off + J + 1:off + 2 * (J + 1)]
    jl = plan[off + 2 * (J + 1):off + 3 * (J + 1)]
    jh = plan[off + 3 * (J + 1):off + 4 * (J + 1)]
    return dict(total=int(plan[0]), chunk=int(plan[1]), J=int(plan[2]),
                spans=int(plan[3]), unit_prefix=tp, seg_prefix=sp, job_lo=jl, job_hi=jh)


def check_split_plan(plan, lo, hi, n_groups, split_tiles=0, tile=TILE):
    """Raises AssertionError (with the reason) if ``plan`` is not a valid
    split of the jobs with key ranges [lo, hi)."""
    lo = np.asarray(lo, np.int64)
    hi = np.asarray(hi, np.int64)
    J = len(lo)
    f = split_plan_fields(plan, J)
    assert f["J"] == J, f"plan J {f['J']} != {J}"
    assert np.array_equal(f["job_lo"][:J], lo), "job_lo differs from the key ranges"
    assert np.array_equal(f["job_hi"][:J], hi), "job_hi differs from the key ranges"
    tp, sp, total, C = f["unit_prefix"], f["seg_prefix"], f["total"], f["chunk"]
    assert tp[0] == 0 and np.all(np.diff(tp) >= 0), "unit prefix not a prefix sum"
    assert tp[J] == total, "unit prefix does not end at the total"
    ntiles = np.where(hi > lo, (hi + tile - 1) // tile - lo // tile, 0)
    units = np.diff(tp)
    assert np.all((units == 0) == (ntiles == 0)), "an empty job has units or a job none"
    cost = units[ntiles > 0] - ntiles[ntiles > 0]
    assert cost.size == 0 or (np.all(cost == cost[0]) and cost[0] >= 0), \
        "switch cost differs between jobs"
    c0 = int(cost[0]) if cost.size else 0
    assert C >= 1, "span length C < 1"
    n_spans = -(-total // C) if total else 0
    assert f["spans"] == n_spans, "span count differs from ceil(total / C)"
    if split_tiles > 0:
        assert C == split_tiles, "forced span length ignored"
    else:
        assert n_spans <= n_groups, f"{n_spans} spans for {n_groups} CTA groups"
    # walk the spans, recording which tiles of which job each one meets
    first = tp[:-1] + np.where(ntiles > 0, c0, 0)
    seen = [np.zeros(int(n), np.int64) for n in ntiles]
    segs = np.zeros(J, np.int64)
    for p in range(n_spans):
        a, z = p * C, min((p + 1) * C, total)
        assert 0 < z - a <= C
        js = np.nonzero((first < z) & (tp[1:] > a) & (ntiles > 0))[0]
        for j in js:
            u0, u1 = max(a, first[j]), min(z, tp[j + 1])
            if u0 < u1:
                segs[j] += 1
                seen[j][u0 - first[j]:u1 - first[j]] += 1
    for j in range(J):
        assert np.all(seen[j] == 1), f"job {j}: a key tile met {seen[j].min()}..{seen[j].max()} times"
    assert sp[0] == 0 and np.array_equal(np.diff(sp), segs), "segment prefix inconsistent"
    return f
