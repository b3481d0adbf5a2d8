"""Benchmark of the absorbed MLA decode step on GB300.

One step = the whole absorbed decode chain on the DeepSeek-V3 decode shape
(B = 32 requests, 128 heads, 4096 context tokens each, bf16, 64-token pages
with shuffled physical blocks):
    mla_absorb_q (W_UK_T BMM + concat)  ->  mla_decode_paged (device split
    plan + tcgen05 paged decode + on-device merge)  ->  mla_v_up (W_UV).
Inputs are synthetic (seeded), resident in HBM when the timed region starts.
L2 is flushed (a 512 MiB write) before every timed step.  The timed step is
the three calls captured once into a CUDA graph and replayed; the eager
launch of the same calls is reported beside it (`step_eager_ms`), and the
end-to-end number (`e2e`) replays the same calls with the host copies
(pinned host buffer in, result out, moved by the library's staging copy)
captured into a graph of their own; the eager launch of that step and the
same step with copy-engine copies are reported beside it.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "MLA decode tokens/s and TFLOPS/HBM GB/s as % of GB300 roofline (1 GPU)"
WORKLOAD = "dsv3_decode_b32_h128_ctx4096_bf16"
B, H, CTX = 32, 128, 4096


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def algorithmic_counts(seq_lens, Bq, Hq):
    """Bytes / FLOPs the decode kernel must move / do (per launch)."""
    kv_tokens = int(np.sum(seq_lens))
    bytes_ = kv_tokens * 576 * 2 + Bq * Hq * 576 * 2 + Bq * Hq * 512 * 2 + Bq * Hq * 4
    flops = 2 * Hq * (576 + 512) * kv_tokens
    return bytes_, flops, kv_tokens


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        # samples go to a file read after the timed region: a reader thread
        # would take the GIL from the host thread while it enqueues a step
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.seek(0)
            self.lines = [ln.strip() for ln in self.out.read().splitlines()]
            self.out.close()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(values, world, device):
    """Per-rank timings -> the maximum over all ranks (replicas run
    independently; this reduction is measurement plumbing, not data path)."""
    if world <= 1:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank, world, ms_max):
    """Aggregate throughput: units all ranks processed / slowest rank's time."""
    return units_per_rank * world / (ms_max * 1e-3)


def make_inputs(device):
    import synth
    case = synth.dsv3_decode(B=B, ctx=CTX)
    d = dict(
        q_nope=case.q_nope.to(device), q_pe=case.q_pe.to(device),
        w_uk_t=case.w_uk_t.to(device), w_uv=case.w_uv.to(device),
        cache=case.cache.to(device),
        bt=torch.from_numpy(case.block_table).to(device),
        sl=torch.from_numpy(case.seq_lens).to(device),
    )
    return case, d


def run_ours(args, rank, world, device):
    import mla_latent_kv_uk_gb300 as m
    case, d = make_inputs(device)
    T = B
    ws = torch.empty(m.mla_decode_workspace_size(B, 1, H, d["bt"].shape[1] * 64),
                     dtype=torch.uint8, device=device)
    q = torch.empty((T, H, 576), dtype=torch.bfloat16, device=device)
    o_lat = torch.empty((B, 1, H, 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, 1, H), dtype=torch.float32, device=device)
    y = torch.empty((T, H, 128), dtype=torch.bfloat16, device=device)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def step(q_nope, q_pe, bt, sl):
        m.mla_absorb_q(q_nope, q_pe, d["w_uk_t"], out=q)
        m.mla_decode_paged(q.view(B, 1, H, 576), d["cache"], bt, sl,
                           sm_scale=case.sm_scale, out=o_lat, lse=lse, workspace=ws)
        m.mla_v_up(o_lat.view(T, H, 512), d["w_uv"], out=y)

    def timed(fn, k):
        """Per-step CUDA-event timing with an L2 flush before each step.  No
        event sits between the calls of a step: an event record between two
        kernels ends their programmatic-dependent-launch overlap."""
        tot = []
        for _ in range(k):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            tot.append(e0.elapsed_time(e1))
        return tot

    def device_step():
        step(d["q_nope"], d["q_pe"], d["bt"], d["sl"])

    def decode_call():
        m.mla_decode_paged(q.view(B, 1, H, 576), d["cache"], d["bt"], d["sl"],
                           sm_scale=case.sm_scale, out=o_lat, lse=lse, workspace=ws)

    def breakdown(k):
        """Per-call device times (ms) of the three entry points, each after an
        L2 flush (so each starts cold, as inside a real step)."""
        names = ("absorb", "decode", "v_up")
        calls = (
            lambda: m.mla_absorb_q(d["q_nope"], d["q_pe"], d["w_uk_t"], out=q),
            lambda: m.mla_decode_paged(q.view(B, 1, H, 576), d["cache"], d["bt"], d["sl"],
                                       sm_scale=case.sm_scale, out=o_lat, lse=lse, workspace=ws),
            lambda: m.mla_v_up(o_lat.view(T, H, 512), d["w_uv"], out=y))
        res = {}
        for nm, fn in zip(names, calls):
            ts = []
            for _ in range(k):
                flush.zero_()
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                fn()
                a1.record(stream)
                torch.cuda.synchronize()
                ts.append(a0.elapsed_time(a1))
            res[nm] = statistics.median(ts)
        return res

    # host-buffer (end-to-end) variant: the step's inputs (q_nope, q_pe,
    # block table, lengths) packed in one pinned host buffer and copied in
    # with one copy, the result (v_up output + LSE, packed likewise) read
    # back with one copy, all inside the timed region
    def packed(tensors):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += -(-t.numel() * t.element_size() // 256) * 256
        return offs, n

    ins = (d["q_nope"], d["q_pe"], d["bt"], d["sl"])
    in_offs, in_bytes = packed(ins)
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=device)

    def view(buf, off, like):
        nb = like.numel() * like.element_size()
        return buf[off:off + nb].view(like.dtype).view(like.shape)

    for t, o in zip(ins, in_offs):
        view(h_in, o, t).copy_(t.cpu())
    d_qn, d_qp, d_bt, d_sl = (view(d_in, o, t) for t, o in zip(ins, in_offs))
    outs = (y, lse)
    out_offs, out_bytes = packed(outs)
    d_out = torch.empty(out_bytes, dtype=torch.uint8, device=device)
    h_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    y_e, lse_e = (view(d_out, o, t) for t, o in zip(outs, out_offs))

    def e2e_calls():
        m.mla_absorb_q(d_qn, d_qp, d["w_uk_t"], out=q)
        m.mla_decode_paged(q.view(B, 1, H, 576), d["cache"], d_bt, d_sl,
                           sm_scale=case.sm_scale, out=o_lat, lse=lse_e, workspace=ws)
        m.mla_v_up(o_lat.view(T, H, 512), d["w_uv"], out=y_e)

    def e2e_step():
        # the library's staging copies: the SMs load the pinned input buffer
        # and store the result buffer over the host link
        m.mla_stage_copy(d_in, h_in)
        e2e_calls()
        m.mla_stage_copy(h_out, d_out)

    def e2e_step_copy_engine():
        d_in.copy_(h_in, non_blocking=True)
        e2e_calls()
        h_out.copy_(d_out, non_blocking=True)

    h2d, d2h = in_bytes, out_bytes   # the two copies' sizes (256-byte padded parts)

    for _ in range(args.warmup):
        device_step()
        e2e_step()
        e2e_step_copy_engine()
    torch.cuda.synchronize()
    # The timed step is the three calls captured once into a CUDA graph and
    # replayed (the kernels, their arguments and their programmatic-launch
    # edges are those of the eager calls; the host's launch work is gone).
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            device_step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        device_step()
    # the end-to-end step (host copy in, the three calls, host copy out)
    # captured the same way: the copies stay in every replayed step
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph):
        e2e_step()
    for _ in range(args.warmup):
        e2e_graph.replay()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        tot = timed(graph.replay, args.steps)
        # the same step with the three calls launched eagerly
        eager = timed(device_step, args.steps)
        # the decode call (plan + decode + merge) on its own, same flush, for
        # its roofline
        dec = timed(decode_call, args.steps)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e2e_tot = timed(e2e_graph.replay, args.steps)
    e2e_eager = timed(e2e_step, args.steps)
    e2e_ce = timed(e2e_step_copy_engine, args.steps)
    parts = breakdown(max(3, min(args.steps, 10)))
    err = m.mla_get_device_error()

    ms, ms_e2e, ms_dec, ms_e2e_eager, ms_e2e_ce = max_over_ranks(
        [statistics.mean(tot), statistics.mean(e2e_tot),
         statistics.mean(dec), statistics.mean(e2e_eager), statistics.mean(e2e_ce)],
        world, device)
    bytes_, flops, kv_tokens = algorithmic_counts(case.seq_lens, B, H)
    hbm, bf16, src = peaks()
    achieved = bytes_ / (ms_dec * 1e-3) / 1e9
    traffic, traffic_src = decode_traffic()
    res = {
        "metric": METRIC, "value": whole_job_rate(B, world, ms), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": WORKLOAD, "batch": B, "heads": H, "ctx": CTX,
                   "kv_tokens": kv_tokens, "page": 64, "l2": "flushed (512 MiB write) before every step",
                   "parallelism": "replicas" if world > 1 else "single"},
        "e2e": {"value": whole_job_rate(B, world, ms_e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "copies": "mla_stage_copy (pinned host buffer <-> device, SM loads/stores)",
                "launch": "CUDA graph of the copies and the three calls",
                "eager_value": whole_job_rate(B, world, ms_e2e_eager),
                "eager_ms_per_step": ms_e2e_eager,
                "copy_engine_ms_per_step": ms_e2e_ce},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "traffic_source": traffic_src, "algorithmic_bytes": bytes_,
                     "kernel": "mla_decode_paged (plan + decode + merge launches)",
                     "kernel_ms": ms_dec, "peak_source": src,
                     "tensor_tflops": flops / (ms_dec * 1e-3) / 1e12,
                     "tensor_frac_of_bf16_peak": flops / (ms_dec * 1e-3) / 1e12 / bf16},
        "step_eager_ms": max_over_ranks([statistics.mean(eager)], world, device)[0],
        "step_breakdown_ms": parts,
        "gpu_launches": 5 * args.steps,
        "clocks": clk.summary(),
        "device_error": err,
    }
    return res


# DRAM bytes (read + write) per launch of the decode kernel on this workload,
# from one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum), with
# the SHA-256 of the kernel sources it was taken on: when the sources differ
# the counters no longer describe the kernel and the line reports null.
DECODE_TRAFFIC = {"bytes": 159246592,
                  "sources_sha256": "bde1a38e1b58bedcace0ba38b6a3514b95a1759f11a165e7519b522c6a0dad2e",
                  "kernel": "decode_pair_kernel"}
DECODE_SOURCES = ("decode.cu", "sm100.cuh", "common.cuh", "merge_row.cuh")


def decode_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "mla_latent_kv_uk_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def decode_traffic():
    """(bytes per launch or None, where the figure comes from)."""
    if DECODE_TRAFFIC["bytes"] is None:
        return None, "no ncu capture of the current kernel"
    if DECODE_TRAFFIC["sources_sha256"] != decode_sources_sha256():
        return None, "kernel changed since the ncu capture"
    return DECODE_TRAFFIC["bytes"], ("ncu dram__bytes_read.sum + dram__bytes_write.sum, "
                                     f"{DECODE_TRAFFIC['kernel']}, one launch")


def _timed_call(fn, flush, stream, reps):
    """Median device time (ms) of fn() over reps calls, each after an L2
    flush, by CUDA events on the launching stream (fn's inputs resident)."""
    ts = []
    for _ in range(reps):
        flush.zero_()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        fn()
        a1.record(stream)
        torch.cuda.synchronize()
        ts.append(a0.elapsed_time(a1))
    return statistics.median(ts)


def _roof(ms, bytes_, flops, hbm, tensor_tf, tensor_name):
    """Achieved GB/s and TFLOP/s and the fraction of the binding roof
    (max of bytes / HBM and FLOPs / tensor peak)."""
    sec = ms * 1e-3
    t_hbm = bytes_ / (hbm * 1e9)
    t_ten = flops / (tensor_tf * 1e12) if flops else 0.0
    bound = "hbm" if t_hbm >= t_ten else "tensor"
    return {"ms": ms, "algorithmic_bytes": bytes_, "flops": flops,
            "gbs": bytes_ / sec / 1e9, "tflops": flops / sec / 1e12 if flops else 0.0,
            "bound": bound, "roof_ms": max(t_hbm, t_ten) * 1e3,
            "frac": max(t_hbm, t_ten) / sec, "tensor_peak": tensor_name}


def run_extras(device, flush, reps=10, only=None):
    """Every other workload of the path, timed on its own (each call after an
    L2 flush): the long single request, the fp8 KV cache, the speculative
    decode and its chunked-prefill context step, and the rotary embedding +
    cache write of one decode step.  Inputs are seeded and synthetic.
    `only` (long, fp8, spec, prefill or rope) runs just that one, e.g. for a
    profiler; `only` = gather or merge runs just that stage of the context
    step (a few hundred MB on the device instead of the whole step's GB)."""
    want = lambda name: only is None or only == name
    import mla_latent_kv_uk_gb300 as m
    import synth
    hbm, bf16, _ = peaks()
    fp8_tf = 2.0 * bf16            # nominal fp8 : bf16 dense ratio (4.5 : 2.25 PF/s)
    stream = torch.cuda.current_stream()
    i32 = lambda x: torch.as_tensor(np.asarray(x, dtype=np.int32), device=device)
    ex = {}

    # long single request: 131072 tokens as 8 explicit shards, merged
    if want("long"):
        c3 = synth.long_request()
        S = 8
        q3 = c3.q.to(device).expand(S, 1, 128, 576).contiguous()
        bt3, sl3 = i32(np.repeat(c3.block_table, S, axis=0)), i32(np.repeat(c3.seq_lens, S))
        st3 = i32([a for a, _ in c3.shards[0]])
        en3 = i32([z for _, z in c3.shards[0]])
        cache3 = c3.cache.to(device)
        ws3 = torch.empty(m.mla_decode_workspace_size(S, 1, 128, bt3.shape[1] * 64),
                          dtype=torch.uint8, device=device)
        o3 = torch.empty((S, 1, 128, 512), dtype=torch.float32, device=device)
        l3 = torch.empty((S, 1, 128), dtype=torch.float32, device=device)

        def long_req():
            m.mla_decode_paged(q3, cache3, bt3, sl3, sm_scale=c3.sm_scale, kv_starts=st3,
                               kv_ends=en3, out_dtype=torch.float32, out=o3, lse=l3, workspace=ws3)
            m.mla_merge_states(o3.view(S, 1, 128, 512), l3.view(S, 1, 128), out_dtype=torch.bfloat16)
        n3 = int(c3.seq_lens.sum())
        ex["long_b1_h128_ctx131072_8shards"] = dict(
            _roof(_timed_call(long_req, flush, stream, reps),
                  n3 * 1152 + 128 * 576 * 2 + 128 * 512 * 2 + 128 * 4, 278528 * n3, hbm, bf16,
                  "bf16 measured"), calls="decode (8 shard rows) + merge_states")
        del q3, cache3, ws3, o3, l3

    # fp8 KV cache: B = 64, ctx U[1024, 16384], e4m3 cache and query
    if want("fp8"):
        c4 = synth.fp8_decode()
        q4, cache4 = c4.q.to(device), c4.cache.to(device)
        bt4, sl4 = i32(c4.block_table), i32(c4.seq_lens)
        ws4 = torch.empty(m.mla_decode_workspace_size(c4.B, 1, 128, bt4.shape[1] * 64),
                          dtype=torch.uint8, device=device)
        o4 = torch.empty((c4.B, 1, 128, 512), dtype=torch.bfloat16, device=device)
        l4 = torch.empty((c4.B, 1, 128), dtype=torch.float32, device=device)
        n4 = int(c4.seq_lens.sum())
        ms4 = _timed_call(lambda: m.mla_decode_paged(
            q4, cache4, bt4, sl4, sm_scale=c4.sm_scale, q_scale=c4.q_scale, k_scale=c4.k_scale,
            out=o4, lse=l4, workspace=ws4), flush, stream, reps)
        ex["fp8_b64_h128_ctxU1k_16k"] = dict(
            _roof(ms4, n4 * 576 + c4.B * 128 * (576 + 512 * 2 + 4), 278528 * n4, hbm, fp8_tf,
                  "fp8 = 2 x bf16 measured (nominal ratio)"),
            tokens_per_s=c4.B / (ms4 * 1e-3), kv_tokens=n4)
        del q4, cache4, ws4, o4, l4

    # speculative decode: B = 128, q_len 2 (causal pair), lognormal contexts
    if want("spec"):
        c5 = synth.spec_decode()
        q5, cache5 = c5.q.to(device), c5.cache.to(device)
        bt5, sl5 = i32(c5.block_table), i32(c5.seq_lens)
        ws5 = torch.empty(m.mla_decode_workspace_size(c5.B, 2, 128, bt5.shape[1] * 64),
                          dtype=torch.uint8, device=device)
        o5 = torch.empty((c5.B, 2, 128, 512), dtype=torch.bfloat16, device=device)
        l5 = torch.empty((c5.B, 2, 128), dtype=torch.float32, device=device)
        n5 = int(c5.seq_lens.sum())
        keys5 = int(2 * c5.seq_lens.sum() - c5.B)        # token 0 sees seq-1 keys, token 1 seq
        ms5 = _timed_call(lambda: m.mla_decode_paged(q5, cache5, bt5, sl5, sm_scale=c5.sm_scale,
                                                     out=o5, lse=l5, workspace=ws5),
                          flush, stream, reps)
        ex["spec_b128_q2_h128_lognormal"] = dict(
            _roof(ms5, n5 * 1152 + c5.B * 2 * 128 * (576 * 2 + 512 * 2 + 4), 278528 * keys5,
                  hbm, bf16, "bf16 measured"),
            tokens_per_s=c5.B * 2 / (ms5 * 1e-3), kv_tokens=n5,
            note="the two query tokens of a request are separate jobs; the planner orders "
                 "jobs token-major so that their reads of a KV tile fall close together "
                 "and the later one hits L2")
        del q5, cache5, ws5, o5, l5

    # chunked-prefill context step: 4 x 8192 context rows on 4 interleaved
    # shards, 512 new tokens each, H = 128
    if want("prefill"):
        cp = synth.context_prefill()
        smb = max(s_[1].shape[1] for s_ in cp.shards)
        tables = []
        for _, sbt, _ in cp.shards:
            t_ = np.full((cp.B, smb), -1, np.int32)
            t_[:, :sbt.shape[1]] = sbt
            tables.append(i32(t_))
        caches = [s_[0].to(device) for s_ in cp.shards]
        cu_c = np.concatenate([[0], np.cumsum(cp.ctx_lens)]).astype(np.int32)
        cu_q = np.concatenate([[0], np.cumsum(cp.new_lens)]).astype(np.int32)
        dcu_c, dcu_q = i32(cu_c), i32(cu_q)
        Nc, Tq, Hp = int(cu_c[-1]), int(cu_q[-1]), cp.H
        rows = torch.empty((Nc, 576), dtype=torch.bfloat16, device=device)
        w = cp.w_kvb.to(device)
        kc = torch.empty((Nc, Hp, 192), dtype=torch.bfloat16, device=device)
        vc = torch.empty((Nc, Hp, 128), dtype=torch.bfloat16, device=device)
        new_kv = cp.new_kv.to(device)
        qp = cp.q.to(device)
        kn, vn = m.mla_expand_kv(new_kv, w, Hp)
        mq = int(cp.new_lens.max())
        oc = torch.empty((Tq, Hp, 128), dtype=torch.bfloat16, device=device)
        lc = torch.empty((Tq, Hp), dtype=torch.float32, device=device)
        on = torch.empty_like(oc)
        ln = torch.empty_like(lc)
        stages = {
            "gather_reorg": (lambda: m.mla_gather_cache_reorg(caches, tables, dcu_c, Nc, interleave=1,
                                                              out=rows),
                             2 * Nc * 1152, 0),
            "expand_context": (lambda: m.mla_expand_kv(rows, w, Hp, k_out=kc, v_out=vc),
                               Nc * 1152 + Hp * 256 * 512 * 2 + Nc * Hp * 320 * 2,
                               2 * Nc * 512 * Hp * 256),
            "prefill_context": (lambda: m.mla_prefill_attn(qp, kc, vc, dcu_q, dcu_c, mq, causal=False,
                                                           sm_scale=cp.sm_scale, out=oc, lse=lc),
                                Tq * Hp * 192 * 2 + Nc * Hp * 320 * 2 + Tq * Hp * (128 * 2 + 4),
                                2 * Hp * (192 + 128) * int(np.sum(cp.new_lens * cp.ctx_lens))),
            "prefill_new_causal": (lambda: m.mla_prefill_attn(qp, kn, vn, dcu_q, dcu_q, mq,
                                                              causal=True, sm_scale=cp.sm_scale,
                                                              out=on, lse=ln),
                                   Tq * Hp * (192 + 192 + 128) * 2 + Tq * Hp * (128 * 2 + 4),
                                   2 * Hp * (192 + 128) * int(np.sum(cp.new_lens * (cp.new_lens + 1) // 2))),
            "merge": (lambda: m.mla_merge_states(po, pl, out_dtype=torch.bfloat16, out=mo, out_lse=ml),
                      Tq * Hp * (3 * 128 * 2 + 3 * 4), 0),
        }
        po = torch.empty((2, Tq, Hp, 128), dtype=torch.bfloat16, device=device)
        pl = torch.empty((2, Tq, Hp), dtype=torch.float32, device=device)
        mo = torch.empty((Tq, Hp, 128), dtype=torch.bfloat16, device=device)
        ml = torch.empty((Tq, Hp), dtype=torch.float32, device=device)
        ex_p = {}
        for nm, (fn, b_, f_) in stages.items():
            if nm == "merge":   # the two states, stacked outside the timed region
                po[0].copy_(oc)
                po[1].copy_(on)
                pl[0].copy_(lc)
                pl[1].copy_(ln)
            fn()
            ex_p[nm] = _roof(_timed_call(fn, flush, stream, reps), b_, f_, hbm, bf16, "bf16 measured")
        ex["prefill_ctx_4x8192_w4_sq512_h128"] = ex_p
        del caches, rows, kc, vc, kn, vn, oc, on, po, pl, mo, ml

    # single stages of the context step, for a profiler: the gather + reorg
    # of the 4 x 8192 context rows, and the final merge of the two states
    # (synthetic states of the step's shape: 2048 new tokens x 128 heads)
    if only == "gather":
        cp = synth.context_prefill()
        smb = max(s_[1].shape[1] for s_ in cp.shards)
        tables = []
        for _, sbt, _ in cp.shards:
            t_ = np.full((cp.B, smb), -1, np.int32)
            t_[:, :sbt.shape[1]] = sbt
            tables.append(i32(t_))
        caches = [s_[0].to(device) for s_ in cp.shards]
        cu_c = np.concatenate([[0], np.cumsum(cp.ctx_lens)]).astype(np.int32)
        dcu_c, Nc = i32(cu_c), int(cu_c[-1])
        rows = torch.empty((Nc, 576), dtype=torch.bfloat16, device=device)
        fn = lambda: m.mla_gather_cache_reorg(caches, tables, dcu_c, Nc, interleave=1, out=rows)
        fn()
        ex["gather_reorg_ctx_4x8192_w4"] = _roof(_timed_call(fn, flush, stream, reps),
                                                 2 * Nc * 1152, 0, hbm, bf16, "bf16 measured")
    if only == "merge":
        cp = synth.context_prefill()
        Tq, Hp = int(np.sum(cp.new_lens)), cp.H
        g = torch.Generator(device="cpu").manual_seed(77)
        po = torch.randn((2, Tq, Hp, 128), generator=g).to(torch.bfloat16).to(device)
        pl = (torch.randn((2, Tq, Hp), generator=g) * 2.0 + 8.0).to(device)
        mo = torch.empty((Tq, Hp, 128), dtype=torch.bfloat16, device=device)
        ml = torch.empty((Tq, Hp), dtype=torch.float32, device=device)
        fn = lambda: m.mla_merge_states(po, pl, out_dtype=torch.bfloat16, out=mo, out_lse=ml)
        fn()
        ex["merge_ctx_2048q_h128"] = _roof(_timed_call(fn, flush, stream, reps),
                                           Tq * Hp * (3 * 128 * 2 + 3 * 4), 0, hbm, bf16,
                                           "bf16 measured")

    # rotary embedding + cache write of one decode step at the DeepSeek-V3
    # shape (32 new tokens, 128 query heads)
    if want("rope"):
        g = synth.generator(9001)
        T2 = 32
        qpe = synth.as_bf16(g.standard_normal((T2, 128, 64))).to(device)
        kpe = synth.as_bf16(g.standard_normal((T2, 64))).to(device)
        kvc = synth.as_bf16(g.standard_normal((T2, 512))).to(device)
        pos = i32(np.full(T2, 4095))
        cache_r = torch.zeros((2048, 64, 576), dtype=torch.bfloat16, device=device)
        slots = i32(np.arange(T2) * 64 + 63)
        ms_r = _timed_call(lambda: m.mla_rope_cache_write(qpe, kpe, kvc, pos, slots, cache_r),
                           flush, stream, reps)
        ex["rope_cache_write_b32_h128"] = _roof(ms_r, T2 * (128 * 64 * 2 * 2 + 64 * 2 * 2 + 512 * 2 + 1152),
                                                0, hbm, bf16, "-")
    return ex


def oracle_sample(n_req):
    """fp64 oracle on n_req requests of the workload; returns (seconds, tokens)."""
    import synth
    from oracle import codecs, mla as O
    case = synth.dsv3_decode(B=B, ctx=CTX)
    f = lambda t: codecs.bf16_to_f64(t.view(torch.int16).numpy())
    qn, qp = f(case.q_nope)[:n_req], f(case.q_pe)[:n_req]
    wk, wv = f(case.w_uk_t), f(case.w_uv)
    cache = f(case.cache)
    t0 = time.perf_counter()
    qa = O.absorb_q(qn, qp, wk)
    o, l = O.paged_decode(qa[:, None], cache, case.block_table[:n_req],
                          case.seq_lens[:n_req], case.sm_scale)
    O.v_up(o[:, 0], wv)
    return time.perf_counter() - t0, n_req


def run_reference(args, rank, world):
    n_req = 4
    times = []
    for _ in range(args.warmup):
        oracle_sample(n_req)
    for _ in range(args.steps):
        dt, n = oracle_sample(n_req)
        times.append(dt)
    sec = statistics.mean(times)
    v = n_req / sec
    cores = os.cpu_count()
    sample = f"{n_req} of {B} requests per step (absorb + decode + v_up in fp64)"
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "batch": B, "heads": H, "ctx": CTX},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads' timings (long request, fp8, spec decode, "
                         "prefill context step, rope + cache write)")
    ap.add_argument("--only-extra", choices=["long", "fp8", "spec", "prefill", "rope", "gather",
                                             "merge"],
                    help="time just that one of the other workloads and print its line "
                         "(for a profiler); no main bench")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if args.only_extra:
        if rank == 0:
            ex = run_extras(device, torch.empty(512 * 1024 * 1024, dtype=torch.uint8,
                                                device=device), only=args.only_extra)
            print(json.dumps({"extra": ex}), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    res = run_ours(args, rank, world, device)
    if rank == 0 and world == 1 and not args.no_extras:
        res["extra"] = run_extras(device, torch.empty(512 * 1024 * 1024, dtype=torch.uint8,
                                                      device=device))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, n = oracle_sample(2)
        res["cpu_baseline"] = {"value": n / dt, "unit": "tokens/s", "cores": os.cpu_count(),
                               "kind": "oracle",
                               "sample": "2 of 32 requests, absorb + decode + v_up in fp64"}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
