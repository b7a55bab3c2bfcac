"""KV-cache staleness study on the GPU (Polestar, App. C.2 and §3, Fig. 3).

Runs one synthetic trajectory on three library contexts that share the weights:

* ``polestar``: the method (block-entry forward, sparse layer-wise refresh on
  the tau_upd trigger);
* ``none``: the same block entries but no refresh inside a block (tau_upd set
  out of reach), i.e. block-wise cache reuse;
* ``reference``: ``polestar_full_forward`` at every step, the no-cache decoding
  that recomputes every position (the "fully recomputed" K/V of App. C.2).

After every step the staleness E_i(t, l) of the two caches against the
reference is computed on the device (``polestar_cache_staleness``) and averaged
over the local window (and over all positions).  The wall time of a Polestar
step (calibrate + commit) and of a full-sequence forward are taken with CUDA
events, and so is the staleness kernel itself (algorithmic bytes: both caches
read once, E written).

  python -m drift_aware_kv_gb300.staleness --workload llada8b_p512_g256_b1 --steps 20
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from drift_aware_kv_gb300 import polestar as P  # noqa: E402
from drift_aware_kv_gb300 import synth  # noqa: E402


def _events():
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def run(name: str, steps: int, kernel_iters: int = 10, progress: bool = False, **overrides) -> dict:
    """overrides: workload fields to change (e.g. topk, the refresh budget k);
    progress: print each step's record to stderr as it completes."""
    w = synth.WORKLOADS[name].replace(n_steps=None, **overrides)
    dt = synth.torch_dtype(w)
    W = synth.make_weights(w, "cuda")
    ctx = {"polestar": P.Polestar(w, W), "none": P.Polestar(w.replace(tau_upd=10 ** 6), W),
           "reference": P.Polestar(w, W)}
    tr = synth.Trajectory(w)
    E = {k: torch.empty(w.n_layers, w.batch, w.seq_len, device="cuda") for k in ("polestar", "none")}
    rows = []
    t_step, t_full = [], []
    stream = torch.cuda.current_stream()
    for _ in range(steps):
        st = tr.next_step()
        if st is None:
            break
        x0 = st["x0"].to(dt).cuda()
        lg = st["logits"].cuda()
        mk = st["masked"].to(torch.uint8).cuda()
        cm = torch.empty(w.batch, 2 * w.block, dtype=torch.uint8, device="cuda")
        fired = 0
        for k in ("polestar", "none"):
            e0, e1 = _events()
            e0.record(stream)
            out = ctx[k].calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])
            ctx[k].commit(lg, mk, cm)
            e1.record(stream)
            torch.cuda.synchronize()
            if k == "polestar":
                fired = sum(int(out.fire[s]) for s in range(w.batch)) if not st["block_entry"] else 0
                if not st["block_entry"]:
                    t_step.append(e0.elapsed_time(e1))
        e0, e1 = _events()
        e0.record(stream)
        ctx["reference"].full_forward(x0)
        e1.record(stream)
        for k in ("polestar", "none"):
            ctx[k].staleness(ctx["reference"], E[k])
        torch.cuda.synchronize()
        t_full.append(e0.elapsed_time(e1))
        win = synth.window_positions(w, st["block_index"])
        rec = dict(t=st["t"], block=st["block_index"], entry=bool(st["block_entry"]), refreshed=fired)
        for k in ("polestar", "none"):
            ew = E[k][:, :, win].mean(dim=(1, 2))  # per layer, over sequences and window rows
            rec[k] = dict(window_mean=float(ew.mean()), window_per_layer=[round(float(v), 6) for v in ew],
                          all_mean=float(E[k].mean()))
        rows.append(rec)
        if progress:
            print(json.dumps({"t": rec["t"], "block": rec["block"], "entry": rec["entry"],
                              "polestar": round(rec["polestar"]["window_mean"], 6),
                              "none": round(rec["none"]["window_mean"], 6)}), file=sys.stderr, flush=True)
    # the staleness kernel alone (cache pair already resident)
    e0, e1 = _events()
    e0.record(stream)
    for _ in range(kernel_iters):
        ctx["polestar"].staleness(ctx["reference"], E["polestar"])
    e1.record(stream)
    torch.cuda.synchronize()
    k_ms = e0.elapsed_time(e1) / kernel_iters
    nrow = w.n_layers * w.batch * w.seq_len
    esz = 2 if w.dtype == "bf16" else 4
    k_bytes = nrow * (4 * w.n_kv_heads * w.head_dim * esz + 4)
    within = [r for r in rows if not r["entry"]]
    summary = dict(
        workload=name, topk=w.topk, K=w.K, steps=len(rows), within_block_steps=len(within),
        window_staleness={k: sum(r[k]["window_mean"] for r in within) / max(1, len(within))
                          for k in ("polestar", "none")},
        all_positions_staleness={k: sum(r[k]["all_mean"] for r in within) / max(1, len(within))
                                 for k in ("polestar", "none")},
        polestar_within_step_ms=sum(t_step) / max(1, len(t_step)),
        full_forward_ms=sum(t_full) / max(1, len(t_full)),
        staleness_kernel=dict(ms=k_ms, bytes=k_bytes, gbs=k_bytes / (k_ms * 1e-3) / 1e9),
        per_step=rows,
    )
    for c in ctx.values():
        c.close()
    return summary


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llada8b_p512_g256_b1", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--json", default=None, help="also write the summary to this file")
    ap.add_argument("--topk", type=int, default=None, help="refresh budget k (clusters refreshed per layer)")
    ap.add_argument("--progress", action="store_true", help="print every step's staleness to stderr")
    a = ap.parse_args()
    from drift_aware_kv_gb300.build import build
    build()
    s = run(a.workload, a.steps, progress=a.progress, **({"topk": a.topk} if a.topk is not None else {}))
    brief = {k: v for k, v in s.items() if k != "per_step"}
    print(json.dumps(brief))
    if a.json:
        with open(a.json, "w") as f:
            json.dump(s, f, indent=1)


if __name__ == "__main__":
    main()
