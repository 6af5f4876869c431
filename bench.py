#!/usr/bin/env python
"""KDA forward-path benchmark on GB300.  Prints ONE JSON line (rank 0).

A step is one chunked prefill (``kda_chunk_fwd``) of the long-context
workload B=1, T=131072, Hqk=Hv=32, D=128 (bf16 activations, zero initial
state, fp32 final state written; 2048 chunks of 64 per head), the largest
single-GPU prefill configuration, with inputs resident in HBM.  Its inputs
(4.3 GB) are larger than L2, so no flush runs between steps.  The same line
carries the dominant kernel's roofline (and the walk's), the end-to-end
number through the public host-memory call, the CPU oracle timed on this
host as a reported baseline, and under ``extras`` the dense and varlen
prefills (each with its own roofline; L2 flushed before every step), the
chunk-group counts on the long workload, and decode / verify / commit.

Multi-GPU (torchrun): one replica per rank, no collective in the data path
("weak" scaling); a barrier brackets the timed region and the slowest rank's
time is used.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload (two of the 32 heads over the whole sequence per step, scaled
to the workload's tokens) on this host's cores (rank 0 only) and prints the
same keys.
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
# --workload dense: the dense serving prefill as the headline (profiling aid;
# its inputs are about L2-sized, so L2 is flushed before every step)
WORKLOADS = {"long": dict(name="long", B=1, T=131072, hqk=32, hv=32),
             "dense": dict(name="dense", B=2, T=4096, hqk=16, hv=16)}
WORKLOAD = dict(WORKLOADS["long"])
METRIC = "chunk_kda prefill tokens/s"
REF_SAMPLE_HEADS = 2  # heads of the workload the reference arm's step runs


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--extras",
                    default="dense,varlen,groups,checkpoint,prefill_conv,prefill_fp16,commit,decode_steps,"
                            "decode_bf16,verify_conv,verify,decode",
                    help="comma list of extra workloads: dense, varlen, groups, checkpoint, prefill_conv, "
                         "prefill_fp16, commit, decode_steps, decode_bf16, verify_conv, verify, decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="long",
                    help="the headline workload: long (default, B=1 T=131072 H=32) or dense "
                         "(B=2 T=4096 H=16, h0 given)")
    args = ap.parse_args()
    WORKLOAD.clear()
    WORKLOAD.update(WORKLOADS[args.workload])
    return args


def workload_desc():
    w = WORKLOAD
    h0 = "zero initial state" if w["name"] == "long" else "initial state N(0,0.02)"
    kind = "long-context" if w["name"] == "long" else "dense"
    return (f"{kind} prefill B={w['B']} T={w['T']} Hqk={w['hqk']} Hv={w['hv']} D=128, bf16 "
            f"q/k/v/g/beta N(0,1), {h0}, final state returned, lower_bound=-5, "
            f"A_log=log U[1,16], dt_bias N(0,0.1)")


def config_dict(replicas):
    """The workload's config; both arms print this same dict."""
    w = WORKLOAD
    return {"workload": workload_desc(), "global_batch": w["B"] * replicas, "seq_len": w["T"],
            "heads": f"Hqk={w['hqk']} Hv={w['hv']}"}


def flop_per_token_head():
    return 6 * D * D + 10 * CHUNK * D


def prefill_bytes_per_token_head(hqk, hv):
    return 2 * 256 / (hv // hqk) + 512 + 2 + 256


# Sources each kernel is built from: a profiled DRAM traffic figure is only
# reported while these files are unchanged since the capture.
KERNEL_SOURCES = {
    "kda_prologue": ["kda_chunk.cu", "kda_common.cuh", "kda_tc.cuh", "kda_params.cuh", "kda_conv.cuh"],
    "kda_walk": ["kda_chunk.cu", "kda_common.cuh", "kda_tc.cuh", "kda_params.cuh", "kda_conv.cuh"],
    "kda_pipelined": ["kda_chunk.cu", "kda_common.cuh", "kda_tc.cuh", "kda_params.cuh", "kda_conv.cuh"],
    "kda_walk128": ["kda_chunk.cu", "kda_common.cuh", "kda_tc.cuh", "kda_params.cuh", "kda_conv.cuh"],
    "kda_window": ["kda_window.cu", "kda_common.cuh", "kda_params.cuh", "kda_conv.cuh"],
}


def sources_sha256(kernel):
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "linear_attention_serving_fwd_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch (read + write) of ``kernel`` on ``workload`` from
    the committed ncu summary in profiles/, or None when the kernel's sources
    changed since the capture."""
    import re
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    try:
        text = open(path).read()
        block = re.search(r"```json\n(.*?)\n```", text, re.S).group(1)
        rec = json.loads(block).get(f"{kernel}@{workload}")
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


def time_device(torch, fn, steps, flush, barrier, per_step=None):
    """Sum of per-step CUDA-event durations of ``fn`` on the current stream
    (flush outside the events), bracketed by barrier + synchronize; each
    step's milliseconds are appended to ``per_step`` when one is given."""
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
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    if per_step is not None:
        per_step.extend(ms)
    return sum(ms) / 1e3  # seconds


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
def prefill_kernels(torch, step, steps, flush, barrier, reduce_max, th, hqk, hv, pk, state_io=0):
    """Per-kernel live timing of a prefill step (the library's CUDA events on
    its launch stream) and each kernel's roofline: the prologue streams the
    step's inputs once (q, k per q/k head, v, g, beta) against HBM; the walk
    carries the three 64 x 128 x 128 contractions (6 K V flop) against the
    bf16 tensor peak; the pipelined kernel does the whole step, so it is held
    to the step's algorithmic HBM bytes: the inputs, the output (256 B per
    token-head) and ``state_io`` bytes of initial and final states."""
    from linear_attention_serving_fwd_gb300 import _native
    _native.trace_enable(True)
    time_device(torch, step, steps, flush, barrier)
    tr = _native.trace_read()
    _native.trace_enable(False)
    in_bytes = 2 * 256 / (hv // hqk) + 512 + 2
    model = {
        "kda_prologue": {"bound": "hbm", "unit": "GB/s", "peak": pk["hbm"], "work": th * in_bytes,
                         "scale": 1e9, "peak_source": f"{pk['src']} HBM copy bandwidth",
                         "per_unit": f"{in_bytes:.0f} B of q/k/v/g/beta per (token, v-head)"},
        "kda_walk": {"bound": "tensor", "unit": "TFLOP/s", "peak": pk["bf16"], "work": th * 6 * D * D,
                     "scale": 1e12, "peak_source": f"{pk['src']} bf16 dense (burst)",
                     "per_unit": "6 K V flop per (token, v-head)"},
        "kda_walk128": {"bound": "tensor", "unit": "TFLOP/s", "peak": pk["bf16"], "work": th * 6 * D * D,
                        "scale": 1e12, "peak_source": f"{pk['src']} bf16 dense (burst)",
                        "per_unit": "6 K V flop per (token, v-head)"},
        "kda_pipelined": {"bound": "hbm", "unit": "GB/s", "peak": pk["hbm"], "work": th * (in_bytes + 256) + state_io,
                          "scale": 1e9, "peak_source": f"{pk['src']} HBM copy bandwidth",
                          "per_unit": f"{in_bytes + 256:.0f} B of q/k/v/g/beta in and o out per (token, v-head), "
                                      f"plus {state_io} B of states in and out"},
    }
    kernels = {}
    for name, kd in model.items():
        if name not in tr:
            continue
        ms = reduce_max(tr[name][0] / tr[name][1])
        ach = kd["work"] / (ms / 1e3) / kd["scale"]
        kernels[name] = {"bound": kd["bound"], "achieved": round(ach, 3), "peak": kd["peak"],
                         "unit": kd["unit"], "frac": round(ach / kd["peak"], 4),
                         "per_launch_ms": round(ms, 4), "per_unit": kd["per_unit"],
                         "peak_source": kd["peak_source"]}
    launches = sum(c for _, c in tr.values()) // max(1, steps)
    ms_all = {k: round(v[0] / v[1], 4) for k, v in tr.items()}
    return kernels, launches, ms_all


def run_ours(args, rank, world, barrier, reduce_max):
    import torch

    import linear_attention_serving_fwd_gb300 as kda
    from linear_attention_serving_fwd_gb300 import workloads as W

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    dev = torch.device("cuda")
    pk = peaks()
    w = WORKLOAD
    x = W.workload(w["name"], seed=rank, device=dev)
    n, T = w["B"], x.t_total
    out = torch.empty((T, w["hv"], D), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((n, w["hv"], D, D), dtype=torch.float32, device=dev)
    ws = torch.empty(kda.chunk_workspace_bytes(n, T, w["hv"], 0), dtype=torch.uint8, device=dev)

    def step():
        kda.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, A_log=x.A_log, dt_bias=x.dt_bias,
                          scale=x.scale, lower_bound=x.lower_bound, n_seqs=n,
                          initial_state=x.initial_state, final_state=fin, out=out, workspace=ws)

    def no_flush():  # the long workload's inputs (4.3 GB) are larger than L2
        pass

    flush = make_flush(torch)
    step_flush = no_flush if w["name"] == "long" else flush
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
    secs = time_device(torch, step, args.steps, step_flush, barrier)
    clk = clocks.stop()
    secs = reduce_max(secs)
    ms_per_step = secs / args.steps * 1e3
    tokens = n * w["T"] * world
    value = weak_scaling_value(n * w["T"], args.steps, world, secs)
    th = n * w["T"] * w["hv"]
    tflops = th * flop_per_token_head() * args.steps * world / secs / 1e12

    state_io = n * w["hv"] * D * D * 4 * (2 if x.initial_state is not None else 1)
    kernels, launches, ms_all = prefill_kernels(torch, step, args.steps, step_flush, barrier, reduce_max,
                                                th, w["hqk"], w["hv"], pk, state_io)
    dom = max(ms_all, key=lambda k: ms_all[k])
    d = kernels.get(dom, {"bound": "tensor", "achieved": None, "peak": pk["bf16"], "unit": "TFLOP/s",
                          "frac": None, "per_launch_ms": ms_all.get(dom), "per_unit": None,
                          "peak_source": None})
    roofline = {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"],
                "unit": d["unit"], "frac": d["frac"],
                "traffic": profiled_traffic(dom, w["name"]) if dom in KERNEL_SOURCES else None,
                "peak_source": d["peak_source"], "per_launch_ms": d["per_launch_ms"],
                "per_unit": d["per_unit"], "kernels": kernels, "kernels_ms_per_step": ms_all}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, random gate parameters, no weights)",
        "config": config_dict(world),
        "parallelism": f"replicas x{world}",
        "l2": ("inputs (4.3 GB) larger than L2: no flush" if w["name"] == "long"
               else "flushed before each step (256 MB write)"),
        "groups": "auto: the pipelined launch (one walk CTA per (sequence, head) chain beside the prologue)",
        "tflops": round(tflops, 3), "pct_bf16_peak": round(100 * tflops / pk["bf16"], 2),
        "hbm_gbs_algorithmic": round(th * prefill_bytes_per_token_head(w["hqk"], w["hv"])
                                     * args.steps * world / secs / 1e9, 1),
        "roofline": roofline,
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }
    if not args.no_e2e:
        line["e2e"] = e2e(torch, kda, x, n, out, fin, args, barrier, reduce_max, tokens)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x)
    if not args.no_extras:
        line["extras"] = extras(torch, kda, W, pk, args, flush, barrier, reduce_max, rank, world, x)
        # the extras' headline figures once more, last on the line, where a
        # reader of only its tail still finds them
        summ = {}
        for k, v in line["extras"].items():
            if isinstance(v, dict) and "frac" in v:
                summ[k] = {"ms": v.get("ms"), "hbm_frac": v["frac"]}
            elif isinstance(v, dict) and "ms" in v:
                summ[k] = {"ms": v["ms"]}
            elif isinstance(v, dict):
                summ[k] = v
        line["extras_summary"] = summ
    return line


def e2e(torch, kda, x, n, out, fin, args, barrier, reduce_max, tokens):
    """End to end through the public host-memory call: page-locked host
    inputs, output and final state; the library copies segments in, runs them
    as chunked prefill and copies the outputs back, overlapped.  The figure is
    the mean over the timed steps; each step's milliseconds and their median
    come with it, since a step whose copies meet other traffic on a shared
    host link (one step of 110 ms among steps of 22 ms has been seen) moves
    the mean but not the median."""
    dev = out.device
    host = {name: getattr(x, name).cpu().pin_memory()
            for name in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state")
            if getattr(x, name) is not None}
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
                               lower_bound=x.lower_bound, n_seqs=n, initial_state=host.get("initial_state"),
                               final_state=fin_h, out=out_h, workspace=ws_host)

    for _ in range(2):
        e2e_step()
    k = max(3, args.steps // 2)
    per_step = []
    secs = reduce_max(time_device(torch, e2e_step, k, lambda: None, barrier, per_step))
    # the host link itself, for reading the figure: one plain copy of the
    # page-locked q buffer to the device, timed the same way
    qd = torch.empty(host["q"].shape, dtype=host["q"].dtype, device=dev)
    qd.copy_(host["q"], non_blocking=True)
    link_s = reduce_max(time_device(torch, lambda: qd.copy_(host["q"], non_blocking=True), 2, lambda: None,
                                    barrier)) / 2
    link = host["q"].numel() * host["q"].element_size() / link_s / 1e9
    del qd
    res = {"value": round(tokens * k / secs, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": round(secs / k * 1e3, 3),
           "step_ms": [round(t, 2) for t in per_step],
           "median_ms": round(sorted(per_step)[len(per_step) // 2], 3),
           "link_h2d_gbs": round(link, 1), "link_h2d_floor_ms": round(h2d / link / 1e6, 3),
           "call": "kda_chunk_fwd_host on page-locked host buffers"}
    del host, out_h, fin_h, ws_host
    torch.cuda.empty_cache()
    return res


def _hbm(gbs, pk):
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
            "frac": round(gbs / pk["hbm"], 4)}


def extras(torch, kda, W, pk, args, flush, barrier, reduce_max, rank, world, xl):
    res = {}
    steps = max(5, min(args.steps, 20))
    sb = 4 * D * D
    want = set(args.extras.split(","))

    def restoring(pool):
        """Before each timed run of a call that updates ``pool`` in place: put
        back its starting contents, then flush L2 (both outside the events)."""
        start = pool.clone()

        def fn():
            pool.copy_(start)
            flush()
        return fn

    # ---- the other prefill configurations, each with its kernels' rooflines
    for name in ("dense", "varlen", "checkpoint", "prefill_conv", "prefill_fp16"):
        if name not in want:
            continue
        wl = "dense" if name in ("dense", "prefill_fp16") else "varlen"
        z = (W.dense_prefill(2, 4096, 16, 16, seed=rank, device="cuda", act_dtype=torch.float16)
             if name == "prefill_fp16" else W.workload(wl, seed=rank, device="cuda"))
        ck = {}
        q_in, k_in, v_in = z.q, z.k, z.v
        if name == "prefill_conv":
            # raw projection bands as strided views of one fused [T, C]
            # projection; width-4 conv + SiLU (bf16 taps) before the prologue
            T_ = z.t_total
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
        out = torch.empty((z.t_total, z.hv, D), dtype=z.q.dtype, device="cuda")
        ws = torch.empty(kda.chunk_workspace_bytes(z.n_seqs, z.t_total, z.hv, 0), dtype=torch.uint8,
                         device="cuda")
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
                                  n_seqs=z.n_seqs, initial_state=z.initial_state, final_state=fin,
                                  out=out, workspace=ws)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        secs = reduce_max(time_device(torch, fn, steps, flush, barrier))
        t = secs / steps
        th = z.t_total * z.hv
        tfl = th * flop_per_token_head() / t / 1e12
        r = {"ms": round(t * 1e3, 4), "tokens_per_s": round(z.t_total * world / t, 1),
             "tflops": round(tfl, 3), "pct_bf16_peak": round(100 * tfl / pk["bf16"], 2),
             "workload": {"dense": "B=2 T=4096 Hqk=Hv=16, h0 N(0,0.02), final state; L2 flushed",
                          "varlen": "8 seqs U[64,8192] rescaled to 32768, Hqk=8 Hv=32, paged fp32 cache; "
                                    "L2 flushed",
                          "checkpoint": "varlen plus one snapshot per sequence at its 64-aligned midpoint",
                          "prefill_conv": "varlen on raw q/k/v bands: width-4 conv + SiLU (bf16 taps) "
                                          "in its own pass, conv state updated",
                          "prefill_fp16": "dense with fp16 q/k/v/g/beta and output"}[name]}
        if name in ("dense", "varlen"):
            sio = z.n_seqs * z.hv * D * D * 4 * 2  # initial and final states (or cache rows) in and out
            kern, _, _ = prefill_kernels(torch, fn, steps, flush, barrier, reduce_max, th, z.hqk, z.hv, pk, sio)
            r["roofline"] = {k: {"frac": v["frac"], "achieved": v["achieved"], "unit": v["unit"],
                                 "ms": v["per_launch_ms"],
                                 "traffic": profiled_traffic(k, name)} for k, v in kern.items()}
        if name in ("checkpoint", "prefill_conv") and "varlen" in res:
            r["overhead_vs_varlen"] = round(t * 1e3 / res["varlen"]["ms"] - 1, 4)
        res[name] = r
        del z, out, ws, fin, ck
        torch.cuda.empty_cache()

    # ---- the long workload's other launch forms: the pipelined launch (the
    # auto choice, -1), two launches with a serial walk (1), the group scan (4, 8)
    if "groups" in want:
        n, T, hv = 1, xl.t_total, xl.hv
        g = {}
        for G in (-1, 1, 4, 8):
            ws = torch.empty(kda.chunk_workspace_bytes(n, T, hv, G), dtype=torch.uint8, device="cuda")
            out = torch.empty((T, hv, D), dtype=torch.bfloat16, device="cuda")
            fin = torch.empty((n, hv, D, D), dtype=torch.float32, device="cuda")

            def fg():
                kda.kda_chunk_fwd(xl.q, xl.k, xl.v, xl.g, xl.beta, A_log=xl.A_log, dt_bias=xl.dt_bias,
                                  n_seqs=n, final_state=fin, out=out, workspace=ws, groups=G)
            for _ in range(2):
                fg()
            s2 = 5
            g["pipelined_ms" if G < 0 else f"G{G}_ms"] = round(reduce_max(time_device(torch, fg, s2, lambda: None, barrier)) / s2 * 1e3, 3)
            del ws, out, fin
            torch.cuda.empty_cache()
        res["groups_long"] = g

    # ---- speculative decode: commit and the slot-table decode
    if "commit" in want:
        y = W.workload("decode", window=4, seed=rank, device="cuda")
        pool = y.state_pool
        counter = torch.zeros(1, dtype=torch.int32, device="cuda")
        kda.kda_verify(y.q, y.k, y.v, y.g, y.beta, pool, y.cu_seqlens, y.state_indices, 4,
                       A_log=y.A_log, dt_bias=y.dt_bias, work_counter=counter)
        out, corr, kg = kda.kda_verify(y.q, y.k, y.v, y.g, y.beta, pool, y.cu_seqlens, y.state_indices, 4,
                                       A_log=y.A_log, dt_bias=y.dt_bias, work_counter=counter)
        acc = torch.full((y.n_seqs,), 4, dtype=torch.int32, device="cuda")

        def fc():
            kda.kda_commit(pool, y.state_indices, acc, corr, kg, 4, A_log=y.A_log,
                           dt_bias=y.dt_bias, lower_bound=y.lower_bound)
        for _ in range(3):
            fc()
        secs = reduce_max(time_device(torch, fc, steps, restoring(pool), barrier))
        t = secs / steps
        nbytes = y.n_seqs * y.hv * (2 * sb + 4 * (4 * D + 4 * D))
        res["commit_q4"] = {"ms": round(t * 1e3, 4), **_hbm(nbytes / t / 1e9, pk),
                            "workload": "256 requests x 4 accepted tokens, Hv=32, fp32 pool"}
        del y, pool, out, corr, kg
    if "decode_steps" in want:
        # a [request, step] slot table: start from the accepted column's row,
        # store the state after every token (64 KB in + 4 x 64 KB out per item)
        y = W.decode_batch(256, 4, 32, 32, slots=1280, seed=rank, device="cuda", name="decode_steps_q4")
        table, acc = W.decode_slot_table(256, 4, 1280, seed=rank, device="cuda")
        pool = y.state_pool
        out = torch.empty((y.t_total, y.hv, D), dtype=torch.bfloat16, device="cuda")

        def fs():
            kda.kda_decode_steps(y.q, y.k, y.v, y.g, y.beta, pool, y.cu_seqlens, table, 4,
                                 num_accepted_tokens=acc, A_log=y.A_log, dt_bias=y.dt_bias, out=out)
        for _ in range(3):
            fs()
        secs = reduce_max(time_device(torch, fs, steps, restoring(pool), barrier))
        t = secs / steps
        nbytes = y.n_seqs * y.hv * sb * 5 + y.t_total * y.hv * (2 * 256 + 256 + 2 + 256)
        res["decode_steps_q4"] = {"ms": round(t * 1e3, 4), "tokens_per_s": round(y.t_total * world / t, 1),
                                  **_hbm(nbytes / t / 1e9, pk),
                                  "workload": "256 requests x 4 tokens, H=32, slot table of 4 rows each"}
        del y, pool, table, acc, out
        torch.cuda.empty_cache()
    if "decode_bf16" in want:
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
        nbytes = y.n_seqs * y.hv * sb + y.t_total * y.hv * (2 * 256 + 256 + 2 + 256)
        res["decode_q1_bf16_state"] = {"ms": round(t * 1e3, 4), "tokens_per_s": round(y.t_total * world / t, 1),
                                       **_hbm(nbytes / t / 1e9, pk),
                                       "workload": "256 requests x 1 token, H=32, bf16 pool"}
        del y, out

    # ---- verify, then decode last (Q = 4, then Q = 1) on the serving batch:
    # 256 requests, Hqk=Hv=32, 512-slot fp32 pool
    for window in (4, 1):
        if not ({"decode", "verify", "verify_conv"} & want):
            break
        y = W.workload("decode", window=window, seed=rank, device="cuda")
        pool = y.state_pool
        out = torch.empty((y.t_total, y.hv, D), dtype=torch.bfloat16, device="cuda")
        counter = torch.zeros(1, dtype=torch.int32, device="cuda")
        corr = torch.empty((y.n_seqs, y.hv, window, D), dtype=torch.float32, device="cuda")
        kg = torch.empty((y.n_seqs, y.hv, window, 2 * D), dtype=torch.bfloat16, device="cuda")
        act = y.t_total * y.hv * (2 * 256 + 256 + 2 + 256)  # q, k per v-head (GVA 1), v, g, o
        rec = y.t_total * y.hv * (4 * D + 4 * D)           # verify's corr and kg records
        items = y.n_seqs * y.hv
        if window == 4 and "verify_conv" in want:
            wc, cst = W.conv_inputs(y.hqk, y.hv, pool.shape[0], window + 2, seed=rank, device="cuda")
            acc = torch.randint(1, window + 1, (y.n_seqs,), dtype=torch.int32, device="cuda")

            def fv():
                kda.kda_verify(y.q, y.k, y.v, y.g, y.beta, pool, y.cu_seqlens, y.state_indices, window,
                               A_log=y.A_log, dt_bias=y.dt_bias, out=out, corr=corr, kg=kg,
                               work_counter=counter, conv_weight=wc, conv_state=cst,
                               num_accepted_tokens=acc)
            for _ in range(3):
                fv()
            t = reduce_max(time_device(torch, fv, steps, flush, barrier)) / steps
            res["verify_conv_q4"] = {"ms": round(t * 1e3, 4), **_hbm((items * sb + act + rec) / t / 1e9, pk),
                                     "workload": "verify Q=4 on raw q/k/v: width-4 conv + SiLU, conv state"}
            del wc, cst, acc
        for verify in (True, False):
            if verify and (window == 1 or "verify" not in want):
                continue
            if not verify and "decode" not in want:
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
            t = reduce_max(time_device(torch, fn, steps, flush if verify else restoring(pool), barrier)) / steps
            state_bytes = items * sb * (1 if verify else 2)
            nbytes = state_bytes + act + (rec if verify else 0)
            key = f"{'verify' if verify else 'decode'}_q{window}"
            res[key] = {"ms": round(t * 1e3, 4), "tokens_per_s": round(y.t_total * world / t, 1),
                        "state_gbs": round(state_bytes / t / 1e9, 1), **_hbm(nbytes / t / 1e9, pk),
                        "traffic": profiled_traffic("kda_window", key) if not verify else None,
                        "workload": f"256 requests x {window}, H=32, 512-slot fp32 pool"}
        del y, pool
        torch.cuda.empty_cache()
    return res


def cpu_baseline(x, min_seconds=10.0):
    """The fp64 oracle, as it stands, on the whole long-context workload
    (every head over the whole sequence, eight heads per call), repeated
    until ``min_seconds`` of wall time have passed."""
    import oracle
    threads = os.cpu_count() or 1
    hv, T = x.hv, x.t_total
    slabs = [(h, min(hv, h + 8)) for h in range(0, hv, 8)]
    cpu = {name: getattr(x, name).cpu() for name in ("q", "k", "v", "g", "beta", "A_log", "dt_bias")}
    cu = x.cu_seqlens.cpu()
    s0 = None if x.initial_state is None else x.initial_state.cpu()
    reps, elapsed = 0, 0.0
    while elapsed < min_seconds:
        for h0, h1 in slabs:
            q, k, v, g, b = (cpu[nm][:, h0:h1] for nm in ("q", "k", "v", "g", "beta"))
            t0 = time.perf_counter()
            oracle.recurrence(q, k, v, g, b, cu, A_log=cpu["A_log"][h0:h1], dt_bias=cpu["dt_bias"][h0:h1],
                              lower_bound=x.lower_bound, h0=None if s0 is None else s0[:, h0:h1],
                              want_out=True, want_state=True, n_threads=threads)
            elapsed += time.perf_counter() - t0
        reps += 1
    return {"value": round(T * reps / elapsed, 2), "unit": "tokens/s", "cores": threads,
            "kind": "oracle", "seconds": round(elapsed, 3),
            "sample": f"the whole {x.name} workload ({T} tokens, Hv={hv}), {reps} time(s), eight "
                      f"heads per oracle call (fp64 token recurrence, OpenMP over head and value block)"}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def run_reference(args):
    import torch  # noqa: F401

    import oracle
    from linear_attention_serving_fwd_gb300 import workloads as W
    w = WORKLOAD
    x = W.workload(w["name"], seed=0)
    threads = os.cpu_count() or 1
    hs = REF_SAMPLE_HEADS
    # one step = heads 0 .. hs-1 of the workload over the whole sequence;
    # its tokens/s is scaled to the workload's (all Hv heads)
    args_ = tuple(t[:, :hs].contiguous() for t in (x.q, x.k, x.v, x.g, x.beta)) + (x.cu_seqlens,)
    kw = dict(A_log=x.A_log[:hs].contiguous(), dt_bias=x.dt_bias[:hs].contiguous(),
              lower_bound=x.lower_bound, n_threads=threads)
    del x
    for _ in range(max(1, args.warmup)):
        oracle.recurrence(*args_, **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.recurrence(*args_, **kw)
    secs = time.perf_counter() - t0
    value = w["T"] * w["B"] * (hs / w["hv"]) * args.steps / secs
    sample = (f"per step: heads 0..{hs - 1} of the {w['hv']} over the whole sequence ({w['T']} tokens), "
              f"value scaled by {hs}/{w['hv']} to the workload's tokens/s; fp64 token recurrence, OpenMP, "
              f"{threads} threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(args.gpus),
        "parallelism": "cpu oracle, rank 0",
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
