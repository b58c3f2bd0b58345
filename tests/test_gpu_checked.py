"""The checked build (libqevict_check.so, compiled with -DQEVICT_CHECK): every index the kernels read from
device data (table entries, slots, task records, counts) is tested before the access it guards; an
index outside its buffer sets bit 8 of the device status word and the access is skipped.  It stands in
for a memory checker.  Each test runs in a child process with QEVICT_LIB=check, so that process loads
the checked library instead of libqevict.so.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ENV = dict(os.environ, QEVICT_LIB="check")


def _child(code, timeout=600):
    return subprocess.run([sys.executable, "-c", code], env=ENV, capture_output=True, text=True, timeout=timeout,
                          cwd=ROOT)


def test_parity_cases_on_the_checked_build(lib):
    """The small-shape lockstep cases (ragged prompts, GQA 1 to 8, batch 2, INT4, the rankers, pre-RoPE
    keys, two-tier and quantized-only budgets, a cache decoded until full) pass on the checked build,
    and every run ends with the device status word clear (the lockstep reads it through the counters)."""
    r = _child("from recoverable_quantized_kv_gb300 import binding; print(binding.LIB_PATH)")
    assert r.returncode == 0 and r.stdout.strip().endswith("libqevict_check.so"), r.stderr
    sel = ("tiny_workload or edge_shapes or int4_w64 or rankers or rope_domain or scores_absorbed or two_tier "
           "or minimal_prompt or slot_exhaustion")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_parity.py"), "-m", "gpu",
                        "-x", "-q", "-k", sel], env=ENV, capture_output=True, text=True, timeout=1800, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_an_index_past_its_buffer_is_reported(lib):
    """A Quantized-table entry naming the window one past the last is caught by the score flush of the
    checked build: qevict_check returns QEVICT_EDEVICE and the status word holds bit 8 alone.  (The planted index stays
    inside the arena, so even an unchecked read of it would not leave the allocation.)"""
    code = r'''
import torch
from recoverable_quantized_kv_gb300 import binding, synth
from oracle import qevict_oracle as O
wl = synth.workload("tiny_4k", prompt_len=1200, steps=16, n_plant=2)
c = binding.Cache(binding.make_config(wl))
p = synth.prompt_inputs(wl, 0, 0)
s0 = torch.rand(1, O.prompt_windows(O.Config.from_obj(wl)), device="cuda")
c.prefill_route(0, p["k"][None].cuda(), p["v"][None].cuda(), s0=s0)
q = torch.zeros(1, wl.h_q, 128, dtype=torch.bfloat16, device="cuda")
kv = torch.zeros(1, wl.h_kv, 128, dtype=torch.bfloat16, device="cuda")
c.decode_step(0, q, kv, kv, torch.empty_like(q))
c.check()
N = c.bud.n_windows
assert c.bud.k_q > 0
assert c.status_word() == 0
c.region("qtab", 0, 8).view(torch.int32)[0] = N
c.flush_scores()
try:
    c.check()
    raise SystemExit("not reported")
except binding.QEvictError as e:
    assert e.status == binding.EDEVICE, e.status
assert c.status_word() == 8, c.status_word()
print("reported")
'''
    r = _child(code)
    assert r.returncode == 0 and "reported" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
