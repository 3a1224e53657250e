"""Failure detection on the GPU without a fault: a launch whose K/V load is
dropped on purpose (test hook) must end on its own, report FA_ERR_TIMEOUT
through fa_status(), and leave the CUDA context usable (a following normal
launch still matches the oracle). Runs in a child process so the test
process's own context is never involved."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np, torch
from exact_attention_16_gb300 import api
from exact_attention_16_gb300.workloads import Workload, draw_inputs
from parity import compare
import oracle

w = Workload("fault", 1, 512, 512, 2, 2, 128, "bf16", True, 1.0, 1.0, 5)
api.fa_debug_set_schedule(int(sys.argv[2]))   # 0 row-tile pairs, 1 key-split items
q, k, v = draw_inputs(w)
qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
out = {}
api.fa_debug_set_fault(2, 100)          # every CTA drops its third K/V load
try:
    t0 = time.perf_counter()
    api.fa_fwd(qd, kd, vd, causal=True)
    out["status_fault"] = api.fa_status()
    out["fault_seconds"] = time.perf_counter() - t0
finally:
    api.fa_debug_set_fault(-1)
o, lse = api.fa_fwd(qd, kd, vd, causal=True)
out["status_after"] = api.fa_status()
o_ref, l_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.scale, True)
out["stats_after"] = compare(o.float().cpu().numpy().transpose(0, 2, 1, 3), lse.cpu().numpy(),
                             o_ref.transpose(0, 2, 1, 3), l_ref)
print("RESULT " + json.dumps(out))
"""


@pytest.mark.parametrize("schedule", [0, 1], ids=["pairs", "keysplit"])
def test_dropped_load_times_out_and_context_survives(schedule):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    proc = subprocess.run([sys.executable, "-c", CHILD, ROOT, str(schedule)], capture_output=True, text=True,
                          timeout=300)
    line = [ln for ln in proc.stdout.splitlines() if ln.startswith("RESULT ")]
    assert proc.returncode == 0 and line, proc.stdout[-2000:] + proc.stderr[-2000:]
    res = json.loads(line[0][len("RESULT "):])
    assert res["status_fault"] == 4, res          # FA_ERR_TIMEOUT
    assert res["fault_seconds"] < 30, res
    assert res["status_after"] == 0, res
