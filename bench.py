"""Benchmark of the absorbed MLA decode step on GB300.

One step = the whole absorbed decode chain on the DeepSeek-V3 decode shape
(B = 32 requests, 128 heads, 4096 context tokens each, bf16, 64-token pages
with shuffled physical blocks):
    mla_absorb_q (W_UK_T BMM + concat)  ->  mla_decode_paged (device split
    plan + tcgen05 paged decode + on-device merge)  ->  mla_v_up (W_UV).
Inputs are synthetic (seeded), resident in HBM when the timed region starts.
L2 is flushed (a 512 MiB write) before every timed step.

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
import threading
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
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

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
    case = synth.config2(B=B, ctx=CTX)
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

    def timed(fn, k, has_dec=True):
        """Per-step CUDA-event timing with an L2 flush before each step."""
        tot, dec = [], []
        for _ in range(k):
            flush.zero_()
            e0, e1, e2, e3 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
            e0.record(stream)
            fn(e1, e2)
            e3.record(stream)
            torch.cuda.synchronize()
            tot.append(e0.elapsed_time(e3))
            if has_dec:
                dec.append(e1.elapsed_time(e2))
        return tot, dec

    def device_step(e1, e2):
        m.mla_absorb_q(d["q_nope"], d["q_pe"], d["w_uk_t"], out=q)
        e1.record(stream)
        m.mla_decode_paged(q.view(B, 1, H, 576), d["cache"], d["bt"], d["sl"],
                           sm_scale=case.sm_scale, out=o_lat, lse=lse, workspace=ws)
        e2.record(stream)
        m.mla_v_up(o_lat.view(T, H, 512), d["w_uv"], out=y)

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

    # host-buffer (end-to-end) variant: inputs copied from pinned host memory
    # and the result read back every step, all inside the timed region
    h_qn = d["q_nope"].cpu().pin_memory()
    h_qp = d["q_pe"].cpu().pin_memory()
    h_bt = d["bt"].cpu().pin_memory()
    h_sl = d["sl"].cpu().pin_memory()
    h_y = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    d_qn, d_qp = torch.empty_like(d["q_nope"]), torch.empty_like(d["q_pe"])
    d_bt, d_sl = torch.empty_like(d["bt"]), torch.empty_like(d["sl"])

    def e2e_step(e1, e2):
        d_qn.copy_(h_qn, non_blocking=True)
        d_qp.copy_(h_qp, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        d_sl.copy_(h_sl, non_blocking=True)
        step(d_qn, d_qp, d_bt, d_sl)
        h_y.copy_(y, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    h2d = sum(t.numel() * t.element_size() for t in (h_qn, h_qp, h_bt, h_sl))
    d2h = h_y.numel() * h_y.element_size() + h_lse.numel() * h_lse.element_size()

    for _ in range(args.warmup):
        device_step(torch.cuda.Event(), torch.cuda.Event())
        e2e_step(None, None)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        tot, dec = timed(device_step, args.steps)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e2e_tot, _ = timed(e2e_step, args.steps, has_dec=False)
    parts = breakdown(max(3, min(args.steps, 10)))
    err = m.mla_get_device_error()

    ms, ms_e2e, ms_dec = max_over_ranks(
        [statistics.mean(tot), statistics.mean(e2e_tot),
         statistics.mean(dec) if dec else float("nan")], world, device)
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
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "traffic_source": traffic_src, "algorithmic_bytes": bytes_,
                     "kernel": "mla_decode_paged (plan + decode + merge launches)",
                     "kernel_ms": ms_dec, "peak_source": src,
                     "tensor_tflops": flops / (ms_dec * 1e-3) / 1e12,
                     "tensor_frac_of_bf16_peak": flops / (ms_dec * 1e-3) / 1e12 / bf16},
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
DECODE_TRAFFIC = {"bytes": None, "sources_sha256": None,
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


def oracle_sample(n_req):
    """fp64 oracle on n_req requests of the workload; returns (seconds, tokens)."""
    import synth
    from oracle import codecs, mla as O
    case = synth.config2(B=B, ctx=CTX)
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
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    res = run_ours(args, rank, world, device)
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
