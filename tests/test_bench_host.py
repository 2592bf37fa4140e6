"""Host parts of bench.py on CPU: the oracle's CPU-baseline record."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_cpu_baseline_record_has_all_cores_and_single_thread_legs():
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_decode_inputs(w)
    step = bench.OracleStep(w, max(w.budgets), inp)
    threads = step.cores()
    rec = bench.cpu_baseline(step, budget_s=0.2, max_calls=4, single_s=0.1)
    assert rec["kind"] == "oracle" and rec["unit"] == "us" and rec["value"] > 0
    assert rec["cores"] == threads
    assert rec["single_thread"]["cores"] == 1 and rec["single_thread"]["value"] > 0
    assert step.cores() == threads          # the thread count is restored afterwards
    assert isinstance(rec["cpu_model"], str) and rec["cpu_model"]
