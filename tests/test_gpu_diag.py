"""GPU parity of the routing diagnostics (QEvict App. I Eq. (13)-(19), App. K) through the C ABI.

A policy cache runs in lockstep with the oracle (tests/gpu_lockstep.py) and a FullKV cache (every
window Full) decodes the same inputs on both sides.  The GPU diagnostics are compared with the
diagnostics oracle over the oracle's trace of the same run: event, term and episode counts and the
lagged transition counts exactly; FMM within the masses' tolerance; churn, QSA, R_Q and the tier
shares (computed from identical scores) to rounding.
"""
import numpy as np
import pytest
import torch

from diag_driver import fullkv_config
from gpu_lockstep import Lockstep
from oracle import qevict_diag as QD
from oracle import qevict_oracle as O
from recoverable_quantized_kv_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from recoverable_quantized_kv_gb300 import build
    build.build()
    return binding.load()


def _run(wl, steps, churn=None, horizon=32, lir_m=3, oracle_prefill_scores=True):
    ls = Lockstep(wl, churn=churn, oracle_prefill_scores=oracle_prefill_scores)
    ls.prefill()
    fwl = fullkv_config(wl)
    rc = binding.Cache(binding.make_config(fwl))
    ocfg_f = O.Config.from_obj(fwl)
    full = {key: O.Unit(ocfg_f) for key in ls.units}
    if getattr(wl, "rope_base", 0.0) > 0:
        table = synth.rope_table(wl.max_len, wl.rope_base)
        rc.set_rope_table(torch.from_numpy(table).cuda())
        for u in full.values():
            u.set_rope_table(table)
    B, L = wl.batch, wl.n_layers
    for l in range(L):
        ins = [synth.prompt_inputs(wl, b, l) for b in range(B)]
        k = torch.stack([x["k"] for x in ins]).cuda()
        v = torch.stack([x["v"] for x in ins]).cuda()
        rc.prefill_route(l, k, v, s0=ls.s0[l])
        s0h = ls.s0[l].cpu().numpy()
        for b in range(B):
            full[(l, b)].prefill_route(ins[b]["k"].float().numpy(), ins[b]["v"].float().numpy(), s0h[b])
    diag = binding.Diagnostics(ls.cache, rc, horizon=horizon, lir_m=lir_m)
    ls.route_hook = diag.route
    k_f = ls.bud.k_f
    traces = {key: QD.Trace(wl.n_sink, wl.window, k_f) for key in ls.units}
    N = ls.N

    def rc_scores(l, b):
        return rc.region("score", l * B + b, 4 * wl.h_kv * N).view(torch.float32).view(wl.h_kv, N)[0].cpu().numpy()

    for key in ls.units:
        traces[key].add_event(ls.units[key].T, ls.units[key].n_route, ls.units[key].z.copy(), ls.units[key].S.copy(),
                              full[key].S.copy())
    for s in range(steps):
        for l in range(L):   # the FullKV step first: the policy's routing event reads its masses
            q = torch.stack([ls.dec[(l, b)]["q"][s] for b in range(B)]).cuda()
            k = torch.stack([ls.dec[(l, b)]["k"][s] for b in range(B)]).cuda()
            v = torch.stack([ls.dec[(l, b)]["v"][s] for b in range(B)]).cuda()
            out = torch.empty(B, wl.h_q, 128, dtype=torch.bfloat16, device="cuda")
            rc.decode_step(l, q, k, v, out)
            for b in range(B):
                d = ls.dec[(l, b)]
                _, masses, sink = full[(l, b)].decode_step(d["q"][s].float().numpy(), d["k"][s].float().numpy(),
                                                           d["v"][s].float().numpy())
                traces[(l, b)].add_step(full[(l, b)].T, masses, sink)
        ls.decode(1)
        if ls.step % wl.omega == 0:
            torch.cuda.synchronize()
            for (l, b), u in ls.units.items():
                rv = rc_scores(l, b).astype(np.float64)
                full[(l, b)].route(scores=rv)
                traces[(l, b)].add_event(u.T, u.n_route, u.z.copy(), u.S.copy(), full[(l, b)].S.copy())
    got = diag.report()
    want = QD.report(list(traces.values()), H=horizon, m=lir_m)
    return got, want


def _compare(got, want):
    for key in ("events", "fmm_terms", "churn_terms", "qsa_terms", "lir_eligible", "lir_rescued",
                "lir_fullkv_eligible", "lir_fullkv_rescued"):
        assert got[key] == want[key], (key, got[key], want[key])
    assert np.array_equal(got["lag"], want["lag"]), (got["lag"], want["lag"])
    assert abs(got["fmm"] - want["fmm"]) <= 1e-3 * max(want["fmm"], 1e-3), (got["fmm"], want["fmm"])
    for key in ("churn", "qsa", "r_q"):
        assert abs(got[key] - want[key]) <= 1e-9 + 1e-6 * abs(want[key]), (key, got[key], want[key])
    assert np.allclose(got["tier_mass"], want["tier_mass"], rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("variant", [dict(), dict(no_promotion=1), dict(batch=2, h_q=8, h_kv=2),
                                     dict(window=64, bits=4, prompt_len=3000), dict(rope_base=10000.0),
                                     dict(n_layers=2, batch=2)])
def test_diagnostics_match_the_oracle(lib, variant):
    wl = synth.workload("tiny_4k", prompt_len=1500, steps=64, n_plant=4, kappa=6.0, budget_num=35, q_num=40)
    wl = wl.replace(**variant)
    got, want = _run(wl, 64, churn=5)
    _compare(got, want)
    assert got["fmm_terms"] > 0 and got["lir_eligible"] > 0
    if variant.get("no_promotion"):
        assert got["lir_rescued"] == 0


def test_diagnostics_without_forced_scores(lib):
    """The policy routes on its own attention: planted windows drift every 16 steps."""
    wl = synth.workload("tiny_4k", prompt_len=2000, steps=64, n_plant=6, kappa=6.0, budget_num=30, q_num=50)
    got, want = _run(wl, 64, horizon=16, lir_m=1)
    _compare(got, want)
    assert got["qsa_terms"] > 0 and 0 < got["qsa"] <= 1.0 + 1e-12


def test_diagnostics_at_32k(lib):
    """One layer of the Llama-3-8B-shaped 32K workload (about 1000 windows, 32 query heads), forced churn:
    five routing events, two of them with a complete FMM horizon."""
    wl = synth.workload("llama8b_32k", n_layers=1, steps=40)
    got, want = _run(wl, 40, churn=3, oracle_prefill_scores=False)
    _compare(got, want)
    assert got["events"] == 6 and got["fmm_terms"] == 2 * wl.h_q and got["lir_eligible"] >= 0


def test_diagnostics_argument_rules(lib):
    wl = synth.workload("tiny_4k", prompt_len=600, steps=16, n_plant=2, budget_num=60)
    pc = binding.Cache(binding.make_config(wl))
    fc = binding.Cache(binding.make_config(fullkv_config(wl)))
    with pytest.raises(binding.QEvictError) as e:     # not prefilled yet
        binding.Diagnostics(pc, fc)
    assert e.value.status == binding.ESCHEDULE
    p = synth.prompt_inputs(wl, 0, 0)
    s0 = torch.rand(1, O.prompt_windows(O.Config.from_obj(wl)), device="cuda")
    for c in (pc, fc):
        c.prefill_route(0, p["k"][None].cuda(), p["v"][None].cuda(), s0=s0)
    with pytest.raises(binding.QEvictError) as e:     # the FullKV cache can evict
        binding.Diagnostics(fc, pc)
    assert e.value.status == binding.EINVAL
    with pytest.raises(binding.QEvictError) as e:     # horizon not a multiple of omega
        binding.Diagnostics(pc, fc, horizon=12)
    assert e.value.status == binding.EINVAL
    d = binding.Diagnostics(pc, fc)
    with pytest.raises(binding.QEvictError) as e:     # no routing event due yet
        d.route()
    assert e.value.status == binding.ESCHEDULE
    r = d.report()
    assert r["events"] == 1 and r["fmm_terms"] == 0
