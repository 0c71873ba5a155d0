"""Host-side logic of bench.py and of the seeded packed workload (no GPU)."""
from __future__ import annotations

import importlib.util
import os

from gated_delta_rule_gdr_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_varlen_lengths_seeded_and_in_range():
    a, b = I.varlen_lengths(I.VARLEN), I.varlen_lengths(I.VARLEN)
    assert a == b and len(a) == I.VARLEN.B
    assert all(16 <= n <= I.VARLEN.T for n in a)
    assert len(set(a)) > I.VARLEN.B // 2          # a spread of lengths, not one value


def test_varlen_counts_match_dense_counts_for_equal_lengths():
    bench = _bench()
    w = I.PREFILL
    by_d, fl_d = bench.prefill_algorithmic(w)
    by_v, fl_v = bench.varlen_algorithmic(w, [w.T] * w.B)
    assert (by_d, fl_d) == (by_v, fl_v)


def test_workload_choices_cover_the_packed_workload():
    bench = _bench()
    assert bench.WORKLOAD_ARG["varlen"] is I.VARLEN
    assert bench.WORKLOAD_ARG["prefill"] is I.PREFILL
