"""CPU checks of the C-ABI library: it builds, loads, exports every declared entry point, and its
host-side budget arithmetic agrees with the oracle (no compute call needs a GPU here)."""
import os
import re

import numpy as np
import pytest

import layout as LY
from oracle import qevict_oracle as O
from recoverable_quantized_kv_gb300 import binding, build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cpu_lib():
    build.build()
    return binding.load()


def test_exports_every_declared_symbol(cpu_lib):
    header = open(os.path.join(ROOT, "include", "qevict.h")).read()
    declared = set(re.findall(r"\b(qevict_\w+)\s*\(", header))
    assert declared == set(binding.exported_symbols())
    for name in declared:
        assert hasattr(cpu_lib, name), name


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_budget_matches_oracle(cpu_lib, name):
    wl = synth.workload(name)
    b = binding.budget(binding.make_config(wl))
    ob = O.budget(O.Config.from_obj(wl))
    assert (b.full_bytes, b.b_total, b.b_sink, b.b_local, b.b_hist, b.payload, b.m_f, b.m_q, b.k_f, b.k_q) == \
        (ob.full_bytes, ob.b_total, ob.b_sink, ob.b_local, ob.b_hist, ob.payload, ob.m_f, ob.m_q, ob.k_f, ob.k_q)


def test_budget_sweep_matches_oracle(cpu_lib):
    """The 131K sweep (budget 10/20/40%, q 0.5/0.7/0.9) in both formats, INT2/W=32 and INT4/W=64."""
    base = synth.workload("long_131k")
    for fmt in (dict(window=32, bits=2), dict(window=64, bits=4)):
        for bn in (10, 20, 40):
            for qn in (50, 70, 90):
                wl = base.replace(budget_num=bn, q_num=qn, **fmt)
                b = binding.budget(binding.make_config(wl))
                ob = O.budget(O.Config.from_obj(wl))
                assert (b.payload, b.m_f, b.m_q, b.k_f, b.k_q, b.n_windows) == \
                    (ob.payload, ob.m_f, ob.m_q, ob.k_f, ob.k_q, O.Config.from_obj(wl).n_windows_cap())


def test_int4_payload_and_capacities(cpu_lib):
    """INT4/W=64 record of the 131K shape: 2*8*64*128*4/8 code bytes + 8*128*4 key and 8*64*4 value
    parameter bytes = 71680 per window (8960 per KV head); at 20% and q = 0.7: K_f = 95, K_q = 1036."""
    wl = synth.workload("long_131k", window=64, bits=4)
    b = binding.budget(binding.make_config(wl))
    assert b.payload == 71680 and b.payload // wl.h_kv == 8960
    assert (b.k_f, b.k_q) == (95, 1036)


def test_rejections(cpu_lib):
    wl = synth.workload("tiny_4k")
    for over, status in [(dict(budget_num=1, budget_den=1000), binding.EBUDGET), (dict(d_head=64), binding.EINVAL),
                         (dict(h_q=6, h_kv=4), binding.EINVAL), (dict(n_sink=17), binding.EINVAL),
                         (dict(prompt_len=4), binding.EINVAL), (dict(q_num=101), binding.EINVAL)]:
        with pytest.raises(binding.QEvictError) as e:
            binding.budget(binding.make_config(wl, **over))
        assert e.value.status == status, over


def test_documented_layouts_are_bijections():
    for W, bits in ((32, 2), (64, 4)):
        for is_v in (False, True):
            idx = LY.fn_index(W, is_v)
            assert np.array_equal(np.sort(idx.ravel()), np.arange(W * 128))
            byte, shift = LY.code_position(W, bits, is_v)
            key = byte * 8 + shift
            assert len(np.unique(key)) == W * 128 and byte.max() < W * 128 * bits // 8
            assert np.all(shift % bits == 0)


def test_router_capacity(cpu_lib):
    """A unit holds at most 8192 windows (the router sorts them in one CTA): max_len one token past that
    capacity is rejected, at it accepted."""
    wl = synth.workload("tiny_4k")
    cap = wl.n_sink + 8192 * wl.window
    assert binding.budget(binding.make_config(wl, max_len=cap)).n_windows == 8192
    with pytest.raises(binding.QEvictError) as e:
        binding.budget(binding.make_config(wl, max_len=cap + 1))
    assert e.value.status == binding.EINVAL


def test_budget_fraction_does_not_overflow(cpu_lib):
    """full_bytes * budget_num passes 2^63 for a wide, long unit and a huge fraction: the budget clamps
    at the largest int64 instead of wrapping to a negative (EBUDGET) value."""
    wl = synth.workload("tiny_4k", h_q=1024, h_kv=1024, prompt_len=1 << 18, budget_num=(1 << 31) - 1,
                        budget_den=1)
    b = binding.budget(binding.make_config(wl, max_len=1 << 18))
    assert b.full_bytes == 4 * 1024 * 128 * (1 << 18)
    assert b.b_total == (1 << 63) - 1 and b.k_f > 0 and b.k_q > 0


def _golden_budget_rows():
    path = os.path.join(ROOT, "tests", "golden", "budget_capacities.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    cols = ["name", "h_kv", "window", "bits", "n_sink", "n_recent", "prompt_len", "budget_num", "budget_den",
            "c_tok", "full", "b_total", "b_sink", "b_local", "b_hist", "payload", "m_q", "m_f", "k_f", "k_q"]
    return [dict(zip(cols, [r[0]] + [int(x) for x in r[1:]])) for r in rows]


@pytest.mark.parametrize("row", _golden_budget_rows(), ids=lambda r: r["name"])
def test_budget_against_hand_worked_capacities(cpu_lib, row):
    """The oracle's and the library's budgets equal the capacities worked by hand from QEvict §4.3
    Eq. (3) and App. B.4 Eq. (7)-(8) (tests/golden/budget_capacities.txt)."""
    wl = synth.workload("tiny_4k", h_q=4 * row["h_kv"], h_kv=row["h_kv"], window=row["window"], bits=row["bits"],
                        n_sink=row["n_sink"], n_recent=row["n_recent"], prompt_len=row["prompt_len"],
                        budget_num=row["budget_num"], budget_den=row["budget_den"], q_num=70, q_den=100)
    ob = O.budget(O.Config.from_obj(wl))
    b = binding.budget(binding.make_config(wl))
    want = (row["full"], row["b_total"], row["b_sink"], row["b_local"], row["b_hist"], row["payload"], row["m_q"],
            row["m_f"], row["k_f"], row["k_q"])
    for got in (ob, b):
        assert (got.full_bytes, got.b_total, got.b_sink, got.b_local, got.b_hist, got.payload, got.m_q, got.m_f,
                got.k_f, got.k_q) == want


def test_binding_fails_loudly_without_the_library(monkeypatch):
    """No CPU fallback: without the built library every entry point's loader raises."""
    monkeypatch.setattr(binding, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libqevict.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        binding.load()
    with pytest.raises(RuntimeError, match="missing"):
        binding.budget(binding.make_config(synth.workload("tiny_4k")))
