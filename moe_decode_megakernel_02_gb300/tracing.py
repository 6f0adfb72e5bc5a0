"""Summaries of the per-CTA stage trace of a decode step.

`Model.trace()` (the C call `mk_trace_read`, with MK_TRACE=1 set when the
model was loaded) returns, per CTA, records of (code, n, t_wait, t_ready,
t_end): code = stage << 16 | layer, n = the stage's items on that CTA, and
three device `%globaltimer` times in ns (the CTA began waiting for the
stage's inputs, they were ready, its items were done). Records with bit 31
of `code` set are item-level detail (MK_TRACE=2 or 3) and are left out here.

A stage's span in a layer runs from the first CTA whose inputs were ready
to the last CTA done; a layer's time is the step between the latest ends of
consecutive layers. Host-side arithmetic on the records only.
"""
from __future__ import annotations

import numpy as np

# stage codes in the order the kernel numbers its completion counters
STAGES = ("A", "QB", "APP", "QLAT", "ATTN", "COMB", "UV", "O", "ROUTER", "SHGU", "CARRY", "SHDOWN", "FFN",
          "INIT", "LM", "AMAX")
ROUTE_WAIT = 0x40  # routing: wait for the logits, then top-k (recorded by every FFN CTA)


def stage_name(code: int) -> str:
    s = (int(code) >> 16) & 0x7FFF
    if s == ROUTE_WAIT:
        return "ROUTE"
    return STAGES[s] if s < len(STAGES) else str(s)


def stage_spans(per_cta):
    """{(layer, stage name): dict(ctas, items, ready_min, ready_max, end_max, span, busy_median)} in us,
    times relative to the earliest record of the step."""
    recs = [r for t in per_cta for r in t if not (int(r["code"]) & 0x80000000)]
    if not recs:
        return {}
    t0 = min(int(r["t_wait"]) for r in recs)
    groups = {}
    for r in recs:
        code = int(r["code"])
        key = (code & 0xFFFF, stage_name(code))
        groups.setdefault(key, []).append(((int(r["t_ready"]) - t0) / 1e3, (int(r["t_end"]) - t0) / 1e3,
                                           int(r["n"])))
    out = {}
    for key, v in groups.items():
        ready = np.array([x[0] for x in v])
        end = np.array([x[1] for x in v])
        out[key] = dict(ctas=len(v), items=int(sum(x[2] for x in v)), ready_min=float(ready.min()),
                        ready_max=float(ready.max()), end_max=float(end.max()),
                        span=float(end.max() - ready.min()), busy_median=float(np.median(end - ready)))
    return out


def layer_times(spans, n_layers):
    """Time per layer (us): differences of the latest stage end of consecutive layers."""
    ends = {}
    for (layer, _), s in spans.items():
        if layer < n_layers:
            ends[layer] = max(ends.get(layer, -np.inf), s["end_max"])
    lays = [ends[l] for l in range(n_layers) if l in ends]
    return np.diff(np.array(lays)) if len(lays) > 1 else np.array([])


def summary(per_cta, n_layers):
    """Mean span per stage over the interior layers (the first and last are
    skipped: the step's start and the LM head distort them) and the mean time
    per layer, both in us."""
    spans = stage_spans(per_cta)
    agg = {}
    for (layer, name), s in spans.items():
        if 1 <= layer < n_layers - 1:
            agg.setdefault(name, []).append(s["span"])
    per_layer = layer_times(spans, n_layers)
    return {"stage_span_us": {k: float(np.mean(v)) for k, v in agg.items()},
            "layer_us": float(per_layer.mean()) if len(per_layer) else None}
