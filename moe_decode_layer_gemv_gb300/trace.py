"""Phase timing of the persistent decode kernel from its device timestamps.

trace_stack() runs one stack forward with the trace buffer set and returns,
per layer, the duration of each phase (median and max over CTAs, in us):
  route   layer start -> routing done (logits, top-k, grouping)
  poll    layer start -> every logit word of the layer complete (the wait
          for the other CTAs' router contributions; there is no
          end-of-layer barrier)
  gate    routing done -> this CTA's gate/up pairs done
  mid     wait in the barrier after the gate/up pass
  down    down rows done (weights mostly already in shared memory)
  tail    combine, residual, next router partial sums
  end     the CTA-wide barrier closing the layer
and the layer's wall time (first start to last layer exit).
"""
from __future__ import annotations

import statistics

import torch

EVENTS = ("start", "routed", "gate_done", "mid_exit", "down_done", "work_done", "end_exit")


def trace_stack(api, x, stack, top_k, sms=None, flags=0):
    dev = x.device
    G = sms or torch.cuda.get_device_properties(dev).multi_processor_count
    L = stack.L
    words = (L + 1) * G * 48
    buf = torch.zeros(words, dtype=torch.int64, device=dev)
    xx = x.clone()
    api.set_trace_buffer(buf)
    try:
        api.stack_forward_(xx, stack, top_k, flags=flags)
        torch.cuda.synchronize()
    finally:
        api.set_trace_buffer(None)
    t = buf.view(L + 1, G, 24, 2)[..., 0].cpu().to(torch.float64) / 1000.0  # us
    cyc = buf.view(L + 1, G, 24, 2)[..., 1].cpu().to(torch.float64)
    out = []
    for l in range(1, L + 1):
        ev = t[l]
        d = lambda a, b: (ev[:, b] - ev[:, a]).tolist()
        row = {}
        for name, a, b in (("route", 0, 1), ("gate", 1, 2), ("mid", 2, 3), ("down", 3, 4),
                           ("tail", 4, 5), ("end", 5, 6), ("poll", 0, 14), ("topk", 0, 7), ("xload", 0, 8), ("group", 7, 9),
                           ("handoff", 9, 1), ("combine", 4, 10), ("cpwait", 10, 11), ("partial", 11, 5),
                           ("gate1st", 1, 12), ("issued", 1, 18), ("land0", 1, 19), ("gate_land", 1, 16), ("all_land", 1, 17)):
            v = d(a, b)
            row[name] = (statistics.median(v), max(v))
        row["wall"] = float(ev[:, 6].max() - ev[:, 0].min()) if l < L else float(ev[:, 5].max() - ev[:, 0].min())
        c = cyc[l]
        row["route_cycles"] = statistics.median((c[:, 1] - c[:, 0]).tolist())
        # SM-clock intervals (same SM, any warps): exact where globaltimer is coarse
        for name, a, b in (("cy_land", 1, 16), ("cy_after_land", 16, 2), ("cy_lead_wait", 1, 12),
                           ("cy_lead_compute", 12, 2), ("cy_mid", 2, 3), ("cy_down", 3, 4),
                           ("cy_combine", 4, 10), ("cy_partial", 11, 5), ("cy_end", 5, 6), ("cy_poll", 0, 14),
                           ("cy_topk", 0, 7),
                           ("cy_group", 7, 9), ("cy_xload", 0, 8), ("cy_route", 0, 1)):
            v = (c[:, b] - c[:, a]).tolist()
            row[name] = (statistics.median(v), max(v))
        out.append(row)
    init = t[0]
    return {"layers": out, "init_wall": float(init[:, 1].max() - init[:, 0].min())}


def format_detail(res) -> str:
    names = ("poll", "topk", "xload", "group", "handoff", "combine", "partial", "issued", "gate_land", "all_land")
    lines = ["layer  " + "  ".join(f"{n:>11s}" for n in names) + "  route_cycles"]
    for l, r in enumerate(res["layers"]):
        lines.append(f"{l:5d}  " + "  ".join(f"{r[n][0]:5.2f}/{r[n][1]:5.2f}" for n in names)
                     + f"  {r['route_cycles']:.0f}")
    return "\n".join(lines)


def format_cycles(res) -> str:
    names = ("cy_poll", "cy_topk", "cy_group", "cy_xload", "cy_route", "cy_land", "cy_after_land", "cy_lead_wait", "cy_lead_compute", "cy_mid", "cy_down",
             "cy_combine", "cy_partial", "cy_end")
    lines = ["layer " + " ".join(f"{n[3:]:>15s}" for n in names) + "   (SM cycles, median/max)"]
    for l, r in enumerate(res["layers"]):
        lines.append(f"{l:5d} " + " ".join(f"{r[n][0]:7.0f}/{r[n][1]:7.0f}" for n in names))
    return "\n".join(lines)


def format_trace(res) -> str:
    lines = ["layer  wall   route(med/max)  gate(med/max)   mid(med/max)   down(med/max)  tail(med/max)  end(med/max)"]
    for l, r in enumerate(res["layers"]):
        cells = "  ".join(f"{r[n][0]:5.2f}/{r[n][1]:5.2f}" for n in ("route", "gate", "mid", "down", "tail", "end"))
        lines.append(f"{l:5d} {r['wall']:6.2f}  {cells}")
    return "\n".join(lines)
