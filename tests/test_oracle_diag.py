"""Pins of the diagnostics oracle (QEvict App. I Eq. (13)-(19), App. K).

Checks:
- Global LIR and the lagged transition counts on hand-made selection histories;
- selection churn, QSA, R_Q and the tier-mass shares on hand-made events;
- Future Missed Mass on a hand-made trace, including the horizon and "existed at r" rules;
- whole runs: a policy that keeps every window (FullKV against itself) misses nothing, agrees with
  itself exactly and evicts no mass; under no-promotion no inactive episode is ever rescued (the
  pages note this zero holds by construction); the shares sum to one and FMM lies in [0, 1].
"""
import numpy as np
import pytest

from diag_driver import fullkv_config, run_oracle
from oracle import qevict_diag as QD
from oracle import qevict_oracle as O
from recoverable_quantized_kv_gb300 import synth

F, Q, E, L = O.FULL, O.QUANT, O.EVICTED, O.LOCAL


def _X(*cols):
    return np.array(cols).T


@pytest.mark.parametrize("seq,m,want", [
    ([1, 0, 0, 0, 1], 3, (1, 1)),        # left, inactive 3 events, returns
    ([1, 0, 0, 1], 3, (0, 0)),           # too short to be eligible
    ([1, 0, 0, 0, 0], 3, (1, 0)),        # eligible, never returns
    ([0, 0, 0, 0, 1], 3, (0, 0)),        # never selected before: nothing to re-enter
    ([1, 0, 0, 0, 1, 0, 0, 0], 3, (2, 1)),
    ([1, 0, 1, 0, 0, 1], 1, (2, 2)),
])
def test_global_lir_episodes(seq, m, want):
    X = _X(seq)
    assert QD.global_lir(X, np.array([0]), m) == want


def test_lir_starts_at_the_first_routed_event():
    X = _X([0, 0, 1, 0, 0, 0, 1], [1, 0, 0, 0, 1, 1, 1])
    # window 0 is routed from event 2 on: one episode (events 3-5), rescued at 6
    # window 1 from event 0: one episode (events 1-3), rescued at 4
    assert QD.global_lir(X, np.array([2, 0]), 3) == (2, 2)
    assert QD.global_lir(X, np.array([-1, 0]), 3) == (1, 1)


def test_lagged_transition_counts():
    X = _X([1, 1, 0, 0, 1])
    n = QD.lagged_counts(X, np.array([0]), max_lag=2)
    # Delta 1: (1,1) (1,0) (0,0) (0,1); Delta 2: (1,0) (1,0) (0,1)
    assert n[0].tolist() == [[1, 1], [1, 1]]
    assert n[1].tolist() == [[0, 1], [2, 0]]


def _trace(events, n_sink=4, window=32, k_f=1):
    tr = QD.Trace(n_sink, window, k_f)
    for T, n_route, tiers, sp, sf in events:
        tr.add_event(T, n_route, np.array(tiers), np.array(sp, float), np.array(sf, float))
    return tr


def test_churn_qsa_and_tier_mass():
    ev0 = (100, 3, [F, Q, E, L], [1, 1, 1, 1], [1, 1, 1, 1])
    ev1 = (108, 4, [F, E, E, Q], [3, 1, 1, 2], [6, 2, 1, 4])
    tr = _trace([ev0, ev1])
    # retained {0, 1} then {0, 3}: Jaccard distance 1 - 1/3
    assert QD.churn_terms(tr) == pytest.approx([2 / 3])
    qsa, rq = QD.qsa_terms(tr)     # event 1: the Quantized window 3 alone, scores 2 and 4
    assert qsa == pytest.approx([1.0]) and rq == pytest.approx([0.5])
    # windows 0-3 start at 4, 36, 68, 100 < 108: all exist; shares of 6, 4, (2 + 1), 0 over 13
    assert QD.tier_mass(tr, tr.events[1]) == pytest.approx([6 / 13, 4 / 13, 3 / 13, 0.0])
    two = _trace([ev0, (108, 4, [Q, Q, E, L], [3, 4, 0, 0], [6, 8, 1, 1])])
    qsa, rq = QD.qsa_terms(two)    # proportional vectors: cosine 1, ratio 1/2
    assert qsa == pytest.approx([1.0]) and rq == pytest.approx([0.5])
    orth = _trace([ev0, (108, 4, [Q, Q, E, L], [1, 0, 0, 0], [0, 1, 1, 1])])
    assert QD.qsa_terms(orth)[0] == pytest.approx([0.0])


def test_future_missed_mass_by_hand():
    # one head, windows 0..2 (starts 4, 36, 68); event at T = 68: window 2 did not exist yet
    tr = _trace([(68, 2, [E, F, L], [0, 0, 0], [0, 0, 0])])
    H = 2
    tr.add_step(68, [[0.7, 0.1, 0.0]], [0.2])     # the step that ended at the event: in the past
    tr.add_step(69, [[0.2, 0.3, 0.1]], [0.4])     # tau = r + 1
    tr.add_step(70, [[0.1, 0.5, 0.2]], [0.2])     # tau = r + 2 = r + H
    tr.add_step(71, [[0.9, 0.0, 0.0]], [0.1])     # beyond the horizon
    # numerator: window 0 at both steps; denominator: sinks + windows 0, 1 at both steps
    assert QD.fmm_terms(tr, H) == pytest.approx([(0.2 + 0.1) / (0.4 + 0.5 + 0.2 + 0.6)])
    short = _trace([(68, 2, [E, F, L], [0, 0, 0], [0, 0, 0])])
    short.add_step(69, [[0.2, 0.3, 0.1]], [0.4])
    assert QD.fmm_terms(short, H) == []           # horizon not reached: not eligible


def test_fullkv_selection_episodes():
    """The FullKV selection takes the top K_f routed windows by FullKV score (descending, ties to the
    older window): window 0 ranks first, drops below window 1 for three events, and returns."""
    sc = [[5, 1, 0], [1, 5, 0], [1, 5, 0], [1, 5, 0], [5, 1, 0]]
    tr = _trace([(100 + 8 * r, 3, [F, Q, Q], [0, 0, 0], row) for r, row in enumerate(sc)], k_f=1)
    X, first = QD.selections(tr, fullkv_topk=True)
    assert X[:, 0].tolist() == [1, 0, 0, 0, 1] and X[:, 1].tolist() == [0, 1, 1, 1, 0]
    assert QD.global_lir(X, first, 3) == (1, 1)
    tie = _trace([(100, 3, [F, Q, Q], [0, 0, 0], [2, 2, 2])], k_f=2)
    assert QD.selections(tie, fullkv_topk=True)[0][0].tolist() == [1, 1, 0]


def _inputs(wl):
    p = synth.prompt_inputs(wl, 0, 0)
    d = synth.decode_inputs(wl, 0, 0)
    prompt = {k: p[k].float().numpy() for k in ("q", "k", "v")}
    dec = {k: d[k].float().numpy() for k in ("q", "k", "v")}
    return prompt, dec


def test_fullkv_against_itself():
    wl = synth.workload("tiny_4k", prompt_len=900, steps=48, n_plant=4)
    prompt, dec = _inputs(wl)
    tr = run_oracle(fullkv_config(wl), 48, prompt, dec)
    r = QD.report([tr])
    assert r["fmm_terms"] > 0 and r["fmm"] == 0.0
    assert r["tier_mass"][1] == 0.0 and r["tier_mass"][2] == 0.0
    assert r["qsa_terms"] == 0                    # nothing is Quantized


@pytest.mark.parametrize("no_promotion", [0, 1])
def test_policy_runs(no_promotion):
    wl = synth.workload("tiny_4k", prompt_len=1500, steps=64, n_plant=4, kappa=6.0, no_promotion=no_promotion,
                        budget_num=35, q_num=40)
    prompt, dec = _inputs(wl)
    rng = np.random.default_rng(5)
    n = O.Config.from_obj(wl).n_windows_cap()
    tr = run_oracle(wl, 64, prompt, dec, scores=lambda s: rng.random(n) * 10)   # forced churn
    r = QD.report([tr])
    assert 0.0 < r["fmm"] < 1.0 and r["fmm_terms"] == (64 // 8 + 1 - 32 // 8) * wl.h_q
    assert r["tier_mass"].sum() == pytest.approx(1.0)
    assert 0.0 < r["churn"] < 1.0 and r["qsa_terms"] == 64 // 8
    assert r["lir_eligible"] > 0
    if no_promotion:
        assert r["lir_rescued"] == 0
    else:
        assert r["lir_rescued"] > 0
    lag = r["lag"]
    assert lag.sum() > 0 and np.all(lag[0].sum(axis=1) > 0)
