"""Oracle-side driver of the routing diagnostics: a policy unit and a FullKV unit (every window Full)
decode the same inputs; the FullKV step masses and the per-event tiers and scores form the trace."""
import numpy as np

from oracle import qevict_diag as QD
from oracle import qevict_oracle as O


def fullkv_config(wl):
    """The workload with a budget that keeps every window Full (K_f >= the window count)."""
    return wl.replace(budget_num=1000, q_num=0)


def event(tr, pol, full, s_rank=None):
    tr.add_event(pol.T, pol.n_route, pol.z.copy(), pol.S.copy(), full.S.copy(), s_rank)


def run_oracle(wl, steps, prompt, dec, scores=None):
    """prompt: dict of q, k, v numpy arrays; dec: dict of per-step q, k, v.  Returns the trace.
    scores(step) -> optional forced scores for both units' routing (cumulative ranker)."""
    cfg = O.Config.from_obj(wl)
    fcfg = O.Config.from_obj(fullkv_config(wl))
    pol, full = O.Unit(cfg), O.Unit(fcfg)
    assert O.budget(fcfg).k_f >= fcfg.n_windows_cap()
    s0 = O.prefill_scores(prompt["q"], prompt["k"], cfg)
    pol.prefill_route(prompt["k"], prompt["v"], s0)
    full.prefill_route(prompt["k"], prompt["v"], s0)
    tr = QD.Trace(cfg.n_sink, cfg.window, O.budget(cfg).k_f)
    event(tr, pol, full)
    for s in range(steps):
        pol.decode_step(dec["q"][s], dec["k"][s], dec["v"][s])
        _, masses, sink = full.decode_step(dec["q"][s], dec["k"][s], dec["v"][s])
        tr.add_step(full.T, masses, sink)
        if (s + 1) % cfg.omega == 0:
            forced = scores(s + 1) if scores is not None else None
            pol.route(forced)
            full.route()
            event(tr, pol, full)
    return tr
