"""Stage-trace summaries (moe_decode_megakernel_02_gb300.tracing) on hand-built records (CPU)."""
import numpy as np

from moe_decode_megakernel_02_gb300 import tracing

DT = np.dtype([("code", "<u4"), ("n", "<u4"), ("t_wait", "<i8"), ("t_ready", "<i8"), ("t_end", "<i8")])


def rec(stage, layer, n, tw, tr, te, item=False):
    code = (stage << 16) | layer | (0x80000000 if item else 0)
    return (code, n, tw, tr, te)


def test_spans_and_layer_times():
    A, QB, FFN = 0, 1, 12
    base = 1_000_000
    cta0 = np.array([rec(A, 0, 2, base, base + 1000, base + 4000), rec(QB, 0, 1, base + 4000, base + 5000, base + 6000),
                     rec(FFN, 0, 3, base + 6000, base + 6000, base + 20000),
                     rec(A, 1, 1, base + 20000, base + 21000, base + 23000),
                     rec(FFN, 1, 3, base + 23000, base + 23000, base + 40000),
                     rec(A, 1, 7, 0, 0, 0, item=True)], dtype=DT)
    cta1 = np.array([rec(A, 0, 1, base, base + 2000, base + 3000), rec(FFN, 0, 2, base + 3000, base + 3000, base + 25000),
                     rec(A, 1, 2, base + 25000, base + 26000, base + 30000),
                     rec(FFN, 1, 2, base + 30000, base + 30000, base + 45000),
                     rec(tracing.ROUTE_WAIT, 1, 0, base + 30000, base + 31000, base + 31000)], dtype=DT)
    sp = tracing.stage_spans([cta0, cta1])
    a0 = sp[(0, "A")]
    assert a0["ctas"] == 2 and a0["items"] == 3
    assert a0["ready_min"] == 1.0 and a0["ready_max"] == 2.0 and a0["end_max"] == 4.0
    assert a0["span"] == 3.0 and a0["busy_median"] == 2.0
    assert sp[(1, "A")]["items"] == 3  # the item-level record is left out
    assert sp[(1, "ROUTE")]["ctas"] == 1
    # latest ends: layer 0 at 25 us, layer 1 at 45 us
    assert np.allclose(tracing.layer_times(sp, 2), [20.0])
    s = tracing.summary([cta0, cta1], 3)
    assert s["layer_us"] == 20.0
    assert s["stage_span_us"]["FFN"] == 45.0 - 23.0


def test_empty_trace():
    assert tracing.stage_spans([np.zeros(0, dtype=DT)]) == {}
    assert tracing.summary([np.zeros(0, dtype=DT)], 4) == {"stage_span_us": {}, "layer_us": None}
