"""Decoding of the per-unit trace (reducescatter_tcgen05_tmem_gb300/trace.py) on a
hand-built buffer: no GPU, no compiled library."""
import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _trace_module():
    # the package __init__ loads the compiled library; the decoder does not need it
    spec = importlib.util.spec_from_file_location(
        "flux_trace", os.path.join(ROOT, "reducescatter_tcgen05_tmem_gb300", "trace.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _buffer(grid, per, items):
    """items: {(cta, i): (unit, rank, k0, [7 stamps])}"""
    w = np.zeros(8 + grid * per * 8, dtype=np.uint64)
    w[0], w[1] = grid, per
    for (b, i), (unit, rank, k0, st) in items.items():
        base = 8 + (b * per + i) * 8
        w[base] = (unit + 1) | (rank << 32) | (k0 << 40)
        w[base + 1:base + 8] = st
    return w.view(np.int64)


def test_records_decode_tags_and_stamps():
    ft = _trace_module()
    buf = _buffer(2, 3, {(0, 0): (5, 3, 17, [10, 20, 30, 40, 50, 60, 70]),
                         (1, 1): (0, 7, 0, [1, 2, 3, 4, 5, 6, 7])})
    t = ft.records(buf)
    assert t["grid"] == 2 and t["per_cta"] == 3
    assert t["unit"][0, 0] == 5 and t["rank"][0, 0] == 3 and t["k0"][0, 0] == 17
    assert t["unit"][1, 1] == 0 and t["rank"][1, 1] == 7
    assert t["unit"][0, 1] == -1  # empty record
    assert t["mma_first"][0, 0] == 40 and t["epi_end"][1, 1] == 7


def test_summary_shares_of_a_known_timeline():
    ft = _trace_module()
    # one MMA CTA, two units: acc free at 0 / 150, first operands at 10 / 160,
    # last commit at 100 / 250; epilogue full / done 110-130 and 260-300
    ns = 1000
    items = {
        (0, 0): (0, 0, 0, [0, 90 * ns, 0, 10 * ns, 100 * ns, 110 * ns, 130 * ns]),
        (0, 1): (1, 0, 0, [95 * ns, 240 * ns, 150 * ns, 160 * ns, 250 * ns, 260 * ns, 300 * ns]),
    }
    s = ft.summary(ft.records(_buffer(1, 2, items)))
    assert s["span_us"] == 300.0
    assert s["units_per_cta"] == 2
    assert abs(s["kloop_share"] - 180 / 300) < 1e-4        # 90 + 90 (shares rounded to 4 places)
    assert abs(s["acc_wait_share"] - 50 / 300) < 1e-4      # 0 + (150 - 100)
    assert abs(s["operand_wait_share"] - 20 / 300) < 1e-4  # 10 + 10
    assert abs(s["idle_after_last_share"] - 50 / 300) < 1e-4
    assert s["unit_kloop_us"] == 90.0 and s["unit_epilogue_us"] == 30.0
    assert ft.summary(ft.records(_buffer(1, 2, {}))) is None
