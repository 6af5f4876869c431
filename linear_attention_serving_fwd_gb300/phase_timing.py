"""Per-phase cycles of the chunk prologue, from a measurement build.

    python -m linear_attention_serving_fwd_gb300.phase_timing [--workload dense|long] [--steps N]

builds the library with ``-DKDA_PHASE_TIMING`` into ``_build/phase_timing/``
(the regular library is untouched), runs the prefill of the chosen workload
``steps`` times and prints, per phase of a (chunk, head) item, the mean SM
cycles between the barriers that close it (thread 0's clock64, summed over
CTAs and items, divided by the items).  The stamps add a few instructions per
phase; the totals come within a few percent of an uninstrumented item.
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


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=["dense", "long"], default="dense")
    ap.add_argument("--steps", type=int, default=20)
    args = ap.parse_args(argv)

    from . import _native
    _native.select_variant("phase_timing")
    import torch

    import linear_attention_serving_fwd_gb300 as kda
    from . import workloads as W

    lib = _native.lib()
    lib.kda_phase_cycles.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int32, ctypes.c_int32]
    lib.kda_phase_cycles.restype = ctypes.c_int
    n = len(PHASES)
    buf = (ctypes.c_ulonglong * (n + 1))()

    x = W.workload(args.workload, device="cuda")
    fin = torch.empty((x.n_seqs, x.hv, 128, 128), dtype=torch.float32, device="cuda")
    out = torch.empty((x.t_total, x.hv, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(kda.chunk_workspace_bytes(x.n_seqs, x.t_total, x.hv, 0), dtype=torch.uint8,
                     device="cuda")

    def step():
        kda.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, A_log=x.A_log, dt_bias=x.dt_bias, n_seqs=x.n_seqs,
                          initial_state=x.initial_state, final_state=fin, out=out, workspace=ws)
    for _ in range(3):
        step()
    assert lib.kda_phase_cycles(buf, n, 1) == 0
    for _ in range(args.steps):
        step()
    assert lib.kda_phase_cycles(buf, n, 1) == 0
    assert kda.kda_device_status(clear=True) == 0
    items = buf[n]
    rows = [(name, buf[i] / items) for i, name in enumerate(PHASES)]
    total = sum(c for _, c in rows)
    print(f"# prologue phases, {args.workload} workload, {items // args.steps} items per step, "
          f"{args.steps} steps: mean SM cycles per item")
    for name, c in rows:
        print(f"{c:9.0f}  {100 * c / total:5.1f} %  {name}")
    print(f"{total:9.0f}  100.0 %  total")
    print(json.dumps({"workload": args.workload, "items": items, "cycles_per_item": round(total, 1),
                      "phases": {name: round(c, 1) for name, c in rows}}))


if __name__ == "__main__":
    main()
