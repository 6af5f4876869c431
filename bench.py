#!/usr/bin/env python
"""KDA forward-path benchmark on GB300.  Prints ONE JSON line (rank 0).

A step is one chunked prefill (``kda_chunk_fwd``) of the dense serving
workload B=2, T=4096, Hqk=Hv=16, D=128 (bf16 activations, fp32 initial state
read, fp32 final state written), inputs resident in HBM; L2 is flushed (a
256 MB write) before every timed step and the flush is outside the events.
The same line carries the decode / verify / varlen / long-context results
under ``extras``, the dominant kernel's roofline, the end-to-end number
through the public API with pinned host buffers, and the CPU oracle timed on
this host as a reported baseline.

Multi-GPU (torchrun): one replica per rank, no collective in the data path
("weak" scaling); a barrier brackets the timed region and the slowest rank's
time is used.

``--impl reference`` times the fp64 CPU oracle on the whole dense workload
per step on this host's cores (rank 0 only) and prints the same keys.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

D = 128
CHUNK = 64
WORKLOAD = dict(name="dense", B=2, T=4096, hqk=16, hv=16)
METRIC = "chunk_kda prefill tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--extras",
                    default="decode,verify,verify_conv,commit,decode_steps,decode_bf16,prefill_fp16,varlen,"
                            "checkpoint,prefill_conv,long",
                    help="comma list of extra workloads: decode, verify, verify_conv, commit, "
                         "decode_steps, decode_bf16, prefill_fp16, varlen, checkpoint, prefill_conv, long")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def workload_desc():
    w = WORKLOAD
    return (f"dense prefill B={w['B']} T={w['T']} Hqk={w['hqk']} Hv={w['hv']} D=128, bf16 "
            f"q/k/v/g/beta, fp32 initial state N(0,0.02), final state returned, "
            f"lower_bound=-5, A_log=log U[1,16], dt_bias N(0,0.1)")


def flop_per_token_head():
    return 6 * D * D + 10 * CHUNK * D


def prefill_bytes_per_token_head(hqk, hv):
    return 2 * 256 / (hv // hqk) + 512 + 2 + 256


# Sources each kernel is built from: a profiled DRAM traffic figure is only
# reported while these files are unchanged since the capture.
KERNEL_SOURCES = {
    "kda_prologue": ["kda_chunk.cu", "kda_common.cuh", "kda_tc.cuh", "kda_params.cuh", "kda_conv.cuh"],
    "kda_walk": ["kda_chunk.cu", "kda_common.cuh", "kda_tc.cuh", "kda_params.cuh", "kda_conv.cuh"],
    "kda_window": ["kda_window.cu", "kda_common.cuh", "kda_params.cuh", "kda_conv.cuh"],
}


def sources_sha256(kernel):
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "linear_attention_serving_fwd_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(kernel):
    """DRAM bytes per launch (read + write) from the committed ncu summary in
    profiles/, or None when the kernel's sources changed since the capture."""
    import re
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    try:
        text = open(path).read()
        block = re.search(r"```json\n(.*?)\n```", text, re.S).group(1)
        rec = json.loads(block).get(kernel)
    except Exception:
        return None
    if not rec or rec.get("sources_sha256") != sources_sha256(kernel):
        return None
    return int(rec["dram_bytes_per_launch"])


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = bus_id
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                rows.append(parts)
        os.unlink(self.file.name)
        if self.bus_id:
            mine = [r for r in rows if r[1].lower().endswith(self.bus_id.lower()[-12:])]
            rows = mine or rows
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        busy = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------
def make_flush(torch):
    buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def flush():
        buf.zero_()
    return flush


def time_device(torch, fn, steps, flush, barrier):
    """Sum of per-step CUDA-event durations of ``fn`` on the current stream
    (flush outside the events), bracketed by barrier + synchronize."""
    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    for i in range(steps):
        flush()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    return sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / 1e3  # seconds


def preroll(torch, fn, seconds=1.0):
    """Keep the GPU busy so the clock sampler sees the load."""
    t0 = time.time()
    while time.time() - t0 < seconds:
        for _ in range(5):
            fn()
        torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, barrier, reduce_max):
    import torch

    import linear_attention_serving_fwd_gb300 as kda
    from linear_attention_serving_fwd_gb300 import _native, workloads as W

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    dev = torch.device("cuda")
    pk = peaks()
    w = WORKLOAD
    x = W.dense_prefill(w["B"], w["T"], w["hqk"], w["hv"], seed=rank, device=dev)
    n = w["B"]
    T = x.t_total
    out = torch.empty((T, w["hv"], D), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((n, w["hv"], D, D), dtype=torch.float32, device=dev)
    ws = torch.empty(kda.chunk_workspace_bytes(n, T, w["hv"], 0), dtype=torch.uint8, device=dev)

    def step():
        kda.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, A_log=x.A_log, dt_bias=x.dt_bias,
                          scale=x.scale, lower_bound=x.lower_bound, n_seqs=n,
                          initial_state=x.initial_state, final_state=fin, out=out,
                          workspace=ws)

    flush = make_flush(torch)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        bus = None
    clocks = ClockSampler(str(bus) if bus else None)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    clocks.start()
    preroll(torch, step, 1.0)
    secs = time_device(torch, step, args.steps, flush, barrier)
    clk = clocks.stop()
    secs = reduce_max(secs)
    ms_per_step = secs / args.steps * 1e3
    tokens = n * w["T"] * world
    value = weak_scaling_value(n * w["T"], args.steps, world, secs)
    th = n * w["T"] * w["hv"]
    tflops = th * flop_per_token_head() * args.steps * world / secs / 1e12

    # dominant kernel, timed live with the library's event tracing (CUDA
    # events recorded by the library on its launch stream)
    _native.trace_enable(True)
    time_device(torch, step, args.steps, flush, barrier)
    tr = _native.trace_read()
    _native.trace_enable(False)
    launches = sum(c for _, c in tr.values())
    dom = max(tr, key=lambda k: tr[k][0])
    dom_ms = tr[dom][0] / tr[dom][1]
    # Algorithmic work per (token, v-head) by kernel.  The prologue streams the
    # step's inputs once (q, k per q/k head, v, g, beta): an HBM roofline.  The
    # walk carries the method's three 64 x 128 x 128 contractions (6 K V flop)
    # and writes o: a tensor roofline over a serial chain.
    r = w["hv"] // w["hqk"]
    in_bytes = 2 * 256 / r + 512 + 2
    kern = {
        "kda_prologue": {"bound": "hbm", "unit": "GB/s", "peak": pk["hbm"],
                         "work": th * in_bytes, "scale": 1e9,
                         "peak_source": f"{pk['src']} HBM copy bandwidth",
                         "per_unit": f"{in_bytes:.0f} B of q/k/v/g/beta per (token, v-head)"},
        "kda_walk": {"bound": "tensor", "unit": "TFLOP/s", "peak": pk["bf16"],
                     "work": th * 6 * D * D, "scale": 1e12,
                     "peak_source": f"{pk['src']} bf16 dense (burst)",
                     "per_unit": "6 K V flop per (token, v-head)"},
    }
    details = {}
    for name, kd in kern.items():
        if name not in tr:
            continue
        ms = tr[name][0] / tr[name][1]
        ach = kd["work"] / (ms / 1e3) / kd["scale"]
        details[name] = {"bound": kd["bound"], "achieved": round(ach, 3), "peak": kd["peak"],
                         "unit": kd["unit"], "frac": round(ach / kd["peak"], 4),
                         "per_launch_ms": round(ms, 4), "per_unit": kd["per_unit"]}
    d = details.get(dom)
    if d is None:  # a kernel without a model: report its time only
        d = {"bound": "tensor", "achieved": None, "peak": pk["bf16"], "unit": "TFLOP/s", "frac": None,
             "per_launch_ms": round(dom_ms, 4)}
    roofline = {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"],
                "unit": d["unit"], "frac": d["frac"],
                "traffic": profiled_traffic(dom) if dom in KERNEL_SOURCES else None,
                "peak_source": kern.get(dom, {}).get("peak_source"),
                "per_launch_ms": d["per_launch_ms"], "per_unit": d.get("per_unit"),
                "kernels": details,
                "kernels_ms_per_step": {k: round(v[0] / v[1], 4) for k, v in tr.items()}}

    # end to end through the public host-memory call: page-locked host
    # inputs, outputs and states; the library copies segments in, runs them
    # as chunked prefill and copies the outputs back, overlapped
    host = {name: getattr(x, name).cpu().pin_memory()
            for name in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state")}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    fin_h = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size() + fin_h.numel() * fin_h.element_size()
    ws_host = torch.empty(kda.chunk_fwd_host_workspace_bytes(
        host["q"], host["k"], host["v"], host["g"], host["beta"], A_log=host["A_log"],
        dt_bias=host["dt_bias"], n_seqs=n), dtype=torch.uint8, device=dev)

    def e2e_step():
        kda.kda_chunk_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"],
                               A_log=host["A_log"], dt_bias=host["dt_bias"], scale=x.scale,
                               lower_bound=x.lower_bound, n_seqs=n,
                               initial_state=host["initial_state"], final_state=fin_h, out=out_h,
                               workspace=ws_host)

    for _ in range(3):
        e2e_step()
    e2e_secs = reduce_max(time_device(torch, e2e_step, max(5, args.steps // 5), flush, barrier))
    e2e_value = tokens * max(5, args.steps // 5) / e2e_secs

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, random gate parameters, no weights)",
        "config": {"workload": workload_desc(), "global_batch": n * world, "seq_len": w["T"],
                   "parallelism": f"replicas x{world}", "l2": "flushed before each step (256 MB write)",
                   "groups": "auto"},
        "tflops": round(tflops, 3), "pct_bf16_peak": round(100 * tflops / pk["bf16"], 2),
        "hbm_gbs_algorithmic": round(th * prefill_bytes_per_token_head(w["hqk"], w["hv"])
                                     * args.steps * world / secs / 1e9, 1),
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x)
    if not args.no_extras:
        line["extras"] = extras(torch, kda, W, pk, args, flush, barrier, reduce_max, rank, world)
    return line


def extras(torch, kda, W, pk, args, flush, barrier, reduce_max, rank, world):
    from linear_attention_serving_fwd_gb300 import _native
    res = {}
    steps = max(5, min(args.steps, 20))
    sb = 4 * D * D

    def restoring(pool):
        """Before each timed run of a call that updates ``pool`` in place: put
        back its starting contents, then flush L2 (both outside the events)."""
        start = pool.clone()

        def fn():
            pool.copy_(start)
            flush()
        return fn
    # decode / verify on the 256-request batch, H=32, 512-slot pool
    want = set(args.extras.split(","))
    for window in (1, 4):
        if not ({"decode", "verify", "verify_conv", "commit"} & want):
            break
        y = W.workload("decode", window=window, seed=rank, device="cuda")
        pool = y.state_pool
        out = torch.empty((y.t_total, y.hv, D), dtype=torch.bfloat16, device="cuda")
        counter = torch.zeros(1, dtype=torch.int32, device="cuda")
        corr = torch.empty((y.n_seqs, y.hv, window, D), dtype=torch.float32, device="cuda")
        kg = torch.empty((y.n_seqs, y.hv, window, 2 * D), dtype=torch.bfloat16, device="cuda")
        for verify in (False, True):
            if verify and window == 1:
                continue
            if ("verify" if verify else "decode") not in want:
                continue

            def fn():
                if verify:
                    kda.kda_verify(y.q, y.k, y.v, y.g, y.beta, pool, y.cu_seqlens,
                                   y.state_indices, window, A_log=y.A_log, dt_bias=y.dt_bias,
                                   out=out, corr=corr, kg=kg, work_counter=counter)
                else:
                    kda.kda_decode(y.q, y.k, y.v, y.g, y.beta, pool, y.cu_seqlens,
                                   y.state_indices, window, A_log=y.A_log, dt_bias=y.dt_bias,
                                   out=out)
            for _ in range(3):
                fn()
            secs = reduce_max(time_device(torch, fn, steps, flush if verify else restoring(pool), barrier))
            items = y.n_seqs * y.hv
            t = secs / steps
            state_bytes = items * sb * (1 if verify else 2)
            act_bytes = y.t_total * y.hv * (2 * 256 + 256 + 2 + 256)  # q,k per v-head (GVA 1), v,g,o
            rec_bytes = (y.t_total * y.hv * (4 * D + 4 * D)) if verify else 0
            gbs = (state_bytes + act_bytes + rec_bytes) / t / 1e9
            key = f"{'verify' if verify else 'decode'}_q{window}"
            res[key] = {"tokens_per_s": round(y.t_total * world / t, 1),
                        "ms_per_step": round(t * 1e3, 4),
                        "state_gbs": round(state_bytes / t / 1e9, 1),
                        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"],
                                     "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4),
                                     "traffic": profiled_traffic("kda_window") if window == 1 and not verify
                                     else None,
                                     "peak_source": f"{pk['src']} HBM copy bandwidth"},
                        "workload": f"256 requests x window {window}, Hqk=Hv=32, 512-slot fp32 pool"}
        if "verify_conv" in want and window == 4:
            # verify on the raw projection bands: width-4 conv + SiLU after the
            # history at the accepted column, conv state rolled (bf16 taps)
            w, cst = W.conv_inputs(y.hqk, y.hv, pool.shape[0], window + 2, seed=rank, device="cuda")
            acc = torch.randint(1, window + 1, (y.n_seqs,), dtype=torch.int32, device="cuda")

            def fv():
                kda.kda_verify(y.q, y.k, y.v, y.g, y.beta, pool, y.cu_seqlens, y.state_indices, window,
                               A_log=y.A_log, dt_bias=y.dt_bias, out=out, corr=corr, kg=kg,
                               work_counter=counter, conv_weight=w, conv_state=cst,
                               num_accepted_tokens=acc)
            for _ in range(3):
                fv()
            secs = reduce_max(time_device(torch, fv, steps, flush, barrier))
            t = secs / steps
            items = y.n_seqs * y.hv
            nbytes = (items * sb + y.t_total * y.hv * (2 * 256 + 256 + 2 + 256)
                      + y.t_total * y.hv * (4 * D + 4 * D))
            gbs = nbytes / t / 1e9
            res["verify_conv_q4"] = {"tokens_per_s": round(y.t_total * world / t, 1),
                                     "ms_per_step": round(t * 1e3, 4),
                                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                                                  "peak": pk["hbm"], "unit": "GB/s",
                                                  "frac": round(gbs / pk["hbm"], 4), "traffic": None,
                                                  "peak_source": f"{pk['src']} HBM copy bandwidth"},
                                     "workload": "256 requests x window 4, Hqk=Hv=32, 512-slot fp32 pool, "
                                                 "width-4 conv + SiLU on raw q/k/v (bf16 taps), "
                                                 "6-position conv state, accepted U{1..4}"}
            del w, cst, acc
        if "commit" in want and window == 4:
            # rebuild every request's state after all 4 verified tokens from
            # verify's records, in place: 64 KB in + 64 KB out per item
            kda.kda_verify(y.q, y.k, y.v, y.g, y.beta, pool, y.cu_seqlens, y.state_indices, window,
                           A_log=y.A_log, dt_bias=y.dt_bias, out=out, corr=corr, kg=kg,
                           work_counter=counter)
            acc = torch.full((y.n_seqs,), window, dtype=torch.int32, device="cuda")

            def fc():
                kda.kda_commit(pool, y.state_indices, acc, corr, kg, window, A_log=y.A_log,
                               dt_bias=y.dt_bias, lower_bound=y.lower_bound)
            for _ in range(3):
                fc()
            secs = reduce_max(time_device(torch, fc, steps, restoring(pool), barrier))
            items = y.n_seqs * y.hv
            t = secs / steps
            nbytes = items * (2 * sb + window * (4 * D + 4 * D))
            gbs = nbytes / t / 1e9
            res["commit_q4"] = {"requests_per_s": round(y.n_seqs * world / t, 1),
                                "ms_per_step": round(t * 1e3, 4),
                                "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"],
                                             "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4),
                                             "traffic": None,
                                             "peak_source": f"{pk['src']} HBM copy bandwidth"},
                                "workload": "256 requests x 4 accepted tokens, Hv=32, 512-slot fp32 pool"}
        del y, pool
    if "decode_steps" in want:
        # speculative multi-token decode with a [request, step] slot table:
        # start from the accepted column's row, store the state after every
        # token into its own row (64 KB in + 4 x 64 KB out per item)
        window = 4
        y = W.decode_batch(256, window, 32, 32, slots=1280, seed=rank, device="cuda",
                           name="decode_steps_q4")
        table, acc = W.decode_slot_table(256, window, 1280, seed=rank, device="cuda")
        pool = y.state_pool
        out = torch.empty((y.t_total, y.hv, D), dtype=torch.bfloat16, device="cuda")

        def fs():
            kda.kda_decode_steps(y.q, y.k, y.v, y.g, y.beta, pool, y.cu_seqlens, table, window,
                                 num_accepted_tokens=acc, A_log=y.A_log, dt_bias=y.dt_bias, out=out)
        for _ in range(3):
            fs()
        secs = reduce_max(time_device(torch, fs, steps, restoring(pool), barrier))
        items = y.n_seqs * y.hv
        t = secs / steps
        nbytes = items * sb * (1 + window) + y.t_total * y.hv * (2 * 256 + 256 + 2 + 256)
        gbs = nbytes / t / 1e9
        res["decode_steps_q4"] = {"tokens_per_s": round(y.t_total * world / t, 1),
                                  "ms_per_step": round(t * 1e3, 4),
                                  "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"],
                                               "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4),
                                               "traffic": None,
                                               "peak_source": f"{pk['src']} HBM copy bandwidth"},
                                  "workload": "256 requests x 4 tokens, Hqk=Hv=32, 1280-row fp32 pool, "
                                              "slot table of 4 rows per request, accepted counts U{1..4}"}
        del y, pool, table, acc
        torch.cuda.empty_cache()
    if "decode_bf16" in want:
        # Q = 1 decode on a bf16 pool (rounded after the token): half the
        # state bytes of the fp32 pool
        y = W.decode_batch(256, 1, 32, 32, slots=512, seed=rank, device="cuda", state_dtype=torch.bfloat16,
                           name="decode_q1_bf16")
        out = torch.empty((y.t_total, y.hv, D), dtype=torch.bfloat16, device="cuda")

        def fb():
            kda.kda_decode(y.q, y.k, y.v, y.g, y.beta, y.state_pool, y.cu_seqlens, y.state_indices, 1,
                           A_log=y.A_log, dt_bias=y.dt_bias, out=out)
        for _ in range(3):
            fb()
        secs = reduce_max(time_device(torch, fb, steps, restoring(y.state_pool), barrier))
        t = secs / steps
        items = y.n_seqs * y.hv
        nbytes = items * (sb // 2) * 2 + y.t_total * y.hv * (2 * 256 + 256 + 2 + 256)
        gbs = nbytes / t / 1e9
        res["decode_q1_bf16_state"] = {"tokens_per_s": round(y.t_total * world / t, 1),
                                       "ms_per_step": round(t * 1e3, 4),
                                       "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"],
                                                    "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4),
                                                    "traffic": None,
                                                    "peak_source": f"{pk['src']} HBM copy bandwidth"},
                                       "workload": "256 requests x window 1, Hqk=Hv=32, 512-slot bf16 pool"}
        del y, out
    if "prefill_fp16" in want:
        # the headline prefill (B=2, T=4096, H=16) with fp16 activations and output
        z = W.dense_prefill(2, 4096, 16, 16, seed=rank, device="cuda", act_dtype=torch.float16)
        out = torch.empty((z.t_total, z.hv, D), dtype=torch.float16, device="cuda")
        fin = torch.empty((2, z.hv, D, D), dtype=torch.float32, device="cuda")
        ws = torch.empty(kda.chunk_workspace_bytes(2, z.t_total, z.hv, 0), dtype=torch.uint8, device="cuda")

        def ff():
            kda.kda_chunk_fwd(z.q, z.k, z.v, z.g, z.beta, A_log=z.A_log, dt_bias=z.dt_bias, n_seqs=2,
                              initial_state=z.initial_state, final_state=fin, out=out, workspace=ws)
        for _ in range(3):
            ff()
        secs = reduce_max(time_device(torch, ff, steps, flush, barrier))
        t = secs / steps
        res["prefill_fp16"] = {"tokens_per_s": round(z.t_total * world / t, 1), "ms_per_step": round(t * 1e3, 4),
                               "workload": "B=2 T=4096 Hqk=Hv=16, fp16 q/k/v/g/beta and output, fp32 states"}
        del z, out, fin, ws
    # varlen paged and long-context prefill
    for name in ("varlen", "checkpoint", "prefill_conv", "long"):
        if name not in want:
            continue
        z = W.workload("long" if name == "long" else "varlen", seed=rank, device="cuda")
        ck = {}
        q_in, k_in, v_in = z.q, z.k, z.v
        if name == "prefill_conv":
            # raw projection bands as strided views of one fused [T, C]
            # projection; width-4 conv + SiLU (bf16 taps) before the prologue
            T_, C_ = z.t_total, (2 * z.hqk + z.hv) * D
            qkv = torch.cat([z.q.reshape(T_, -1), z.k.reshape(T_, -1), z.v.reshape(T_, -1)], dim=1)
            a_, b_ = z.hqk * D, 2 * z.hqk * D
            q_in = qkv[:, :a_].view(T_, z.hqk, D)
            k_in = qkv[:, a_:b_].view(T_, z.hqk, D)
            v_in = qkv[:, b_:].view(T_, z.hv, D)
            w_, cst_ = W.conv_inputs(z.hqk, z.hv, z.state_pool.shape[0], 4, seed=rank, device="cuda")
            ck = dict(conv_weight=w_, conv_state=cst_, conv_state_indices=z.state_indices,
                      conv_has_initial_state=z.has_initial_state)
        if name == "checkpoint":
            # one snapshot per sequence at its last 64-aligned midpoint, into
            # pool rows no sequence of the batch uses (prefix caching)
            lens = (z.cu_seqlens[1:] - z.cu_seqlens[:-1]).to(torch.int64)
            used = set(z.state_indices.tolist())
            spare = [r for r in range(z.state_pool.shape[0]) if r not in used][:z.n_seqs]
            ck = dict(checkpoint_state=z.state_pool,
                      checkpoint_offsets=((lens // 2) // 64 * 64).to(torch.int32),
                      checkpoint_state_indices=torch.tensor(spare, dtype=torch.int32, device="cuda"))
        out = torch.empty((z.t_total, z.hv, D), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(kda.chunk_workspace_bytes(z.n_seqs, z.t_total, z.hv, 0),
                         dtype=torch.uint8, device="cuda")
        fin = None
        if z.state_pool is None:
            fin = torch.empty((z.n_seqs, z.hv, D, D), dtype=torch.float32, device="cuda")

        def fn():
            if z.state_pool is not None:
                kda.kda_chunk_fwd(q_in, k_in, v_in, z.g, z.beta, A_log=z.A_log, dt_bias=z.dt_bias,
                                  cu_seqlens=z.cu_seqlens, state_cache=z.state_pool,
                                  state_indices=z.state_indices,
                                  has_initial_state=z.has_initial_state, out=out, workspace=ws, **ck)
            else:
                kda.kda_chunk_fwd(z.q, z.k, z.v, z.g, z.beta, A_log=z.A_log, dt_bias=z.dt_bias,
                                  n_seqs=z.n_seqs, final_state=fin, out=out, workspace=ws)
        fn()
        torch.cuda.synchronize()
        s2 = 3 if name == "long" else steps
        secs = reduce_max(time_device(torch, fn, s2, flush, barrier))
        t = secs / s2
        th = z.t_total * z.hv
        tfl = th * flop_per_token_head() / t / 1e12
        res[name] = {"tokens_per_s": round(z.t_total * world / t, 1), "ms_per_step": round(t * 1e3, 3),
                     "tflops": round(tfl, 3), "pct_bf16_peak": round(100 * tfl / pk["bf16"], 2),
                     "workload": {"varlen": "8 seqs (U[64,8192] rescaled to 32768), Hqk=8 Hv=32, paged fp32 cache",
                                  "checkpoint": "varlen workload plus one snapshot per sequence at its "
                                                "64-aligned midpoint into a spare cache row",
                                  "prefill_conv": "varlen workload on raw q/k/v bands of a fused "
                                                  "projection: width-4 conv + SiLU (bf16 taps) in a "
                                                  "pass of its own into a conv scratch, conv state updated",
                                  "long": "B=1 T=131072 Hqk=Hv=32, zero initial state"}[name]}
        if name == "prefill_conv" and "varlen" in res:
            res[name]["overhead_vs_varlen"] = round(t * 1e3 / res["varlen"]["ms_per_step"] - 1, 4)
        if name == "checkpoint":
            res[name]["snapshot_bytes"] = int((ck["checkpoint_offsets"] > 0).sum().item()) * z.hv * 4 * D * D
            if "varlen" in res:
                res[name]["overhead_vs_varlen"] = round(t * 1e3 / res["varlen"]["ms_per_step"] - 1, 4)
        del z, out, ws
        torch.cuda.empty_cache()
    return res


def cpu_baseline(x, min_seconds=10.0, max_reps=200):
    """The fp64 oracle, as it stands, on the whole dense workload (every
    sequence and head), repeated until ``min_seconds`` of wall time."""
    import oracle
    q, k, v, g, b = (t.cpu() for t in (x.q, x.k, x.v, x.g, x.beta))
    A_log, dt = x.A_log.cpu(), x.dt_bias.cpu()
    h0 = x.initial_state.cpu() if x.initial_state is not None else None
    cu = x.cu_seqlens.cpu()
    threads = os.cpu_count() or 1
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.recurrence(q, k, v, g, b, cu, A_log=A_log, dt_bias=dt, lower_bound=x.lower_bound,
                          h0=h0, want_out=True, want_state=True, n_threads=threads)
        reps += 1
        dt_s = time.perf_counter() - t0
        if dt_s >= min_seconds or reps >= max_reps:
            break
    return {"value": round(x.t_total * reps / dt_s, 2), "unit": "tokens/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt_s, 3),
            "sample": f"the whole dense workload ({x.n_seqs} x {x.t_total // x.n_seqs} tokens, Hv={x.hv}) "
                      f"{reps} times (fp64 token recurrence, OpenMP over sequence, head and value block)"}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def run_reference(args):
    import torch  # noqa: F401

    import oracle
    from linear_attention_serving_fwd_gb300 import workloads as W
    w = WORKLOAD
    # one step = the whole dense workload (every sequence and head)
    x = W.dense_prefill(w["B"], w["T"], w["hqk"], w["hv"], seed=0)
    threads = os.cpu_count() or 1
    args_ = (x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens)
    kw = dict(A_log=x.A_log, dt_bias=x.dt_bias, lower_bound=x.lower_bound,
              h0=x.initial_state, n_threads=threads)
    for _ in range(max(1, args.warmup)):
        oracle.recurrence(*args_, **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.recurrence(*args_, **kw)
    secs = time.perf_counter() - t0
    value = x.t_total * args.steps / secs
    sample = (f"per step: the whole dense workload ({w['B']} x {w['T']} tokens, Hv={w['hv']}; fp64 token "
              f"recurrence, OpenMP, {threads} threads)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(), "global_batch": w["B"], "seq_len": w["T"],
                   "parallelism": "cpu oracle, rank 0"},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def collectives(world, backend="nccl"):
    """The job's (barrier, reduce_max) over its ``world`` ranks: the barrier
    that brackets the timed region and the slowest rank's seconds.  One rank:
    no-ops.  The process group (nccl on GPUs; gloo for the CPU tests) is
    created here if the launcher has not made one."""
    if world <= 1:
        return (lambda: None), (lambda s: s)
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend)
    dev = "cuda" if backend == "nccl" else "cpu"

    def barrier():
        dist.barrier()

    def reduce_max(s):
        t = torch.tensor([s], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return barrier, reduce_max


def weak_scaling_value(units_per_rank, steps, world, max_seconds):
    """Whole-job throughput of ``world`` replicas that each processed
    ``units_per_rank`` per step for ``steps`` steps, timed by the slowest."""
    return units_per_rank * world * steps / max_seconds


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    barrier, reduce_max = collectives(world, "nccl")
    line = run_ours(args, rank, world, barrier, reduce_max)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
