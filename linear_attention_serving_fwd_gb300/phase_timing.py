"""Per-phase cycles of the chunk prologue, from a measurement build.

    python -m linear_attention_serving_fwd_gb300.phase_timing [--workload dense|long] [--steps N] [--groups G]

builds the library with ``-DKDA_PHASE_TIMING`` into ``_build/phase_timing/``
(the regular library is untouched), runs the prefill of the chosen workload
``steps`` times and prints, per phase of a (chunk, head) item, the mean SM
cycles between the barriers that close it (thread 0's clock64, summed over
CTAs and items, divided by the items).  The stamps add a few instructions per
phase; the totals come within a few percent of an uninstrumented item.
When the call takes the pipelined launch, the walk CTAs' counters follow:
the chain's waits and work and the loader's waits, per chunk step.
Needs a GPU.
"""
from __future__ import annotations

import argparse
import ctypes
import json

PHASES = (
    "tile wait (next item's q/k/v/g tiles)",
    "gate, gate cumsum, v record, row norms",
    "(offsets, references and norms: now inside the next phase)",
    "offsets, references, norms; X / Y operands (tf32)",
    "A_kk / A_qk product (N = 160) with the Kg / qg / kg build; next tiles issued",
    "TMEM read, A carve",
    "inverse: diagonal 16 x 16 blocks (forward substitution)",
    "inverse: 16-row pairs (two products)",
    "inverse: 32-row halves (two products)",
    "T^T and the identity block",
    "A_qk T + R products, -A_qk T and R to shared memory",
    "qg' + P + o_intra products, records staged and bulk-stored",
)


WALK = (
    "chain: next record and S16 buffer",
    "chain: P S (and R v) product",
    "chain: state update, S16 write",
    "chain: barrier and next issue",
    "loader: ready-flag waits",
    "loader: buffer waits",
)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=["dense", "long"], default="dense")
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--groups", type=int, default=0, help="as kda_chunk_fwd: 0 auto, 1 two launches, -1 pipelined")
    args = ap.parse_args(argv)

    from . import _native
    _native.select_variant("phase_timing")
    import torch

    import linear_attention_serving_fwd_gb300 as kda
    from . import workloads as W

    lib = _native.lib()
    for fn in (lib.kda_phase_cycles, lib.kda_walk_cycles):
        fn.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int32, ctypes.c_int32]
        fn.restype = ctypes.c_int
    n = len(PHASES)
    buf = (ctypes.c_ulonglong * (n + 1))()
    nw = len(WALK)
    wbuf = (ctypes.c_ulonglong * (nw + 1))()

    x = W.workload(args.workload, device="cuda")
    fin = torch.empty((x.n_seqs, x.hv, 128, 128), dtype=torch.float32, device="cuda")
    out = torch.empty((x.t_total, x.hv, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(kda.chunk_workspace_bytes(x.n_seqs, x.t_total, x.hv, 0), dtype=torch.uint8,
                     device="cuda")

    def step():
        kda.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, A_log=x.A_log, dt_bias=x.dt_bias, n_seqs=x.n_seqs,
                          initial_state=x.initial_state, final_state=fin, out=out, workspace=ws,
                          groups=args.groups)
    for _ in range(3):
        step()
    assert lib.kda_phase_cycles(buf, n, 1) == 0
    assert lib.kda_walk_cycles(wbuf, nw, 1) == 0
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(args.steps):
        step()
    ev1.record()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / args.steps
    assert lib.kda_phase_cycles(buf, n, 1) == 0
    assert lib.kda_walk_cycles(wbuf, nw, 1) == 0
    assert kda.kda_device_status(clear=True) == 0
    items = buf[n]
    rows = [(name, buf[i] / items) for i, name in enumerate(PHASES)]
    total = sum(c for _, c in rows)
    print(f"# prologue phases, {args.workload} workload, groups {args.groups}, {items // args.steps} items per "
          f"step, {args.steps} steps of {ms:.3f} ms: mean SM cycles per item")
    for name, c in rows:
        print(f"{c:9.0f}  {100 * c / total:5.1f} %  {name}")
    print(f"{total:9.0f}  100.0 %  total")
    rec = {"workload": args.workload, "groups": args.groups, "ms_per_step": round(ms, 4), "items": items, "cycles_per_item": round(total, 1),
           "phases": {name: round(c, 1) for name, c in rows}}
    steps_w = wbuf[nw]
    if steps_w:  # the pipelined launch ran: its walk's counters per chunk step
        print(f"# pipelined walk, {steps_w // args.steps} chunk steps per step: mean SM cycles per chunk step")
        for i, name in enumerate(WALK):
            print(f"{wbuf[i] / steps_w:9.0f}  {name}")
        rec["walk"] = {name: round(wbuf[i] / steps_w, 1) for i, name in enumerate(WALK)}
    if steps_w:  # per-CTA spans of the last launch: wall time and the SM clock it implies
        lib.kda_cta_spans.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int32]
        lib.kda_cta_spans.restype = ctypes.c_int
        nc = 152
        sp = (ctypes.c_ulonglong * (4 * nc))()
        assert lib.kda_cta_spans(sp, nc) == 0
        walk_ctas = x.n_seqs * x.hv
        t0 = min(sp[4 * i] for i in range(nc) if sp[4 * i])
        spans = {}
        for role, ids in (("walk", range(walk_ctas)), ("prologue", range(walk_ctas, nc))):
            ids = [i for i in ids if sp[4 * i]]
            st = [(sp[4 * i] - t0) / 1e3 for i in ids]
            en = [(sp[4 * i + 1] - t0) / 1e3 for i in ids]
            mhz = [sp[4 * i + 2] / max(1, sp[4 * i + 1] - sp[4 * i]) * 1e3 for i in ids]
            if st:
                print(f"# {role} CTAs ({len(st)}): start {min(st):.1f}..{max(st):.1f} us, end {min(en):.1f}.."
                      f"{max(en):.1f} us, SM clock {min(mhz):.0f}..{max(mhz):.0f} MHz")
                spans[role] = sorted((round(e, 1), int(sp[4 * i + 3])) for e, i in zip(en, ids))
        rec["cta_end_us_and_sm"] = spans
    print(json.dumps(rec))


if __name__ == "__main__":
    main()
