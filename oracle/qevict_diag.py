"""CPU oracle for QEvict's routing diagnostics.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU legs may import this module.  The product
path never calls it and it shares no code with the CUDA sources.

Definitions, from "QEvict: Recoverable Quantized KV Eviction for Attention-Drift-Robust Long-Context
Decoding" (arXiv 2608.05326), App. I and App. K:

  * Future Missed Mass (FMM), App. I.2 Eq. (13), horizon H = 32 decode steps
  * Selection Churn, App. I.2 Eq. (14)
  * tier attention-mass shares mu(z), App. I.3 Eq. (15)
  * Quantized-Score Agreement (QSA) and the mass ratio R_Q, App. I.3 Eq. (16)-(17), App. K
  * Global LIR(m), App. I.4 Eq. (18), m = 3
  * lagged transition probabilities P_ab(Delta), App. I.4 Eq. (19)

Inputs are a trace of two runs fed the same queries, keys and values: the evaluated policy and a
FullKV run whose every window stays Full.  Per decode step the trace holds the FullKV attention of
every query head on every window and on the sinks; per routing event the policy's tiers and the
window scores of both runs.  Everything is float64 and follows the equations term by term.

Readings (the pages define the diagnostics on token positions of model traces):
  * States are windows.  The evicted set E_r of Eq. (13) is the windows the policy holds Evicted
    after routing event r; "states that existed at r" are the sinks and every window whose first
    position is below T_r (the token count at r).  The FullKV attention of such a window at a later
    step includes its tokens appended after r (at most one window, inside the protected recent
    region, never evicted).
  * FMM averages over the (event, head) pairs whose full horizon was decoded (T_r + H reached).
  * Churn compares the historical sets retained (Full or Quantized) at consecutive events, sinks
    and the recent region excluded (Eq. (14)); all windows hold W tokens, so the Jaccard distance
    of the token sets equals that of the window sets.
  * QSA and R_Q use the cumulative window scores S (QEvict §4.2 Eq. (1)) of both runs over the
    windows Quantized after routing event r, for r >= 1 (at the prefill event both runs hold the same
    prompt scores).
  * mu(z) is taken at each event over the windows that exist then (Local = not yet routed).
  * An inactive episode of Eq. (18) starts when a window leaves the selected set (X goes 1 -> 0): a
    window that was never selected cannot re-enter.  The FullKV selection (the pages' "oracle") is the top K_f of the
    routed windows by FullKV score (descending, ties to the older window).
  * P_ab(Delta) counts every pair of events (r, r + Delta) at which the window was already routed.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

from oracle.qevict_oracle import EVICTED, FULL, LOCAL, QUANT


@dataclasses.dataclass
class StepRec:
    T: int                 # tokens cached after the step; its query sits at position T - 1
    masses: np.ndarray     # [H_q][n_windows] FullKV attention on each window
    sink: np.ndarray       # [H_q] FullKV attention on the sinks


@dataclasses.dataclass
class EventRec:
    T: int                 # tokens cached at the routing event
    n_route: int           # windows routed so far (ids below it left the recent region)
    tiers: np.ndarray      # [n_windows] policy tier after routing (LOCAL for unrouted ids)
    s_policy: np.ndarray   # [n_windows] the policy's window scores after routing
    s_full: np.ndarray     # [n_windows] the FullKV run's window scores after routing
    s_rank: np.ndarray     # [n_windows] scores the FullKV selection ranks (normally s_full)


class Trace:
    def __init__(self, n_sink: int, window: int, k_f: int):
        self.n_sink, self.window, self.k_f = n_sink, window, k_f
        self.steps: List[StepRec] = []
        self.events: List[EventRec] = []

    def add_step(self, T: int, masses: np.ndarray, sink: np.ndarray) -> None:
        self.steps.append(StepRec(int(T), np.asarray(masses, np.float64).copy(), np.asarray(sink, np.float64).copy()))

    def add_event(self, T: int, n_route: int, tiers, s_policy, s_full, s_rank=None) -> None:
        tiers = np.asarray(tiers).astype(np.int64).copy()
        tiers[n_route:] = LOCAL
        s_full = np.asarray(s_full, np.float64).copy()
        self.events.append(EventRec(int(T), int(n_route), tiers, np.asarray(s_policy, np.float64).copy(), s_full,
                                    s_full if s_rank is None else np.asarray(s_rank, np.float64).copy()))

    def existed(self, T: int, n: int) -> np.ndarray:
        """Windows whose first position n_s + wW lies below T."""
        return self.n_sink + np.arange(n) * self.window < T


def fmm_terms(tr: Trace, H: int = 32) -> List[float]:
    """Eq. (13) for every (event, head) with a complete horizon:
    sum over the steps tau in (r, r + H] of the FullKV attention on E_r, over the same sum on every
    state that existed at r."""
    out = []
    for ev in tr.events:
        fut = [s for s in tr.steps if ev.T < s.T <= ev.T + H]
        if not any(s.T == ev.T + H for s in fut):
            continue
        n = len(ev.tiers)
        evicted = ev.tiers == EVICTED
        existed = tr.existed(ev.T, n)
        for h in range(fut[0].masses.shape[0]):
            num = sum(float(s.masses[h, :n][evicted].sum()) for s in fut)
            den = sum(float(s.sink[h]) + float(s.masses[h, :n][existed].sum()) for s in fut)
            out.append(num / den)
    return out


def churn_terms(tr: Trace) -> List[float]:
    """Eq. (14) between consecutive events: 1 - |R_r and R_r+1| / |R_r or R_r+1|."""
    out = []
    for a, b in zip(tr.events, tr.events[1:]):
        ra = np.isin(a.tiers, (FULL, QUANT))
        rb = np.isin(b.tiers, (FULL, QUANT))
        union = int(np.sum(ra | rb))
        if union:
            out.append(1.0 - int(np.sum(ra & rb)) / union)
    return out


def qsa_terms(tr: Trace):
    """Eq. (16) and Eq. (17) at each event r >= 1 whose Quantized tier is not empty."""
    qsa, rq = [], []
    for ev in tr.events[1:]:
        q = ev.tiers == QUANT
        if not q.any():
            continue
        sq, sf = ev.s_policy[q], ev.s_full[q]
        qsa.append(float(np.dot(sq, sf) / (np.linalg.norm(sq) * np.linalg.norm(sf))))
        rq.append(float(sq.sum() / sf.sum()))
    return qsa, rq


def tier_mass(tr: Trace, ev: EventRec) -> np.ndarray:
    """Eq. (15) at one event: shares of the FullKV scores per policy tier (Full, Quantized, Evicted,
    Local) over the windows that exist."""
    ex = tr.existed(ev.T, len(ev.tiers))
    tot = ev.s_full[ex].sum()
    return np.array([ev.s_full[ex & (ev.tiers == z)].sum() / tot for z in (FULL, QUANT, EVICTED, LOCAL)])


def selections(tr: Trace, fullkv_topk: bool):
    """X[r][w] of App. I.4: 1 if window w is in the selected full-precision set at event r; and the
    first event at which each window was routed (-1 if never)."""
    n = len(tr.events[0].tiers)
    X = np.zeros((len(tr.events), n), np.int64)
    first = np.full(n, -1)
    for r, ev in enumerate(tr.events):
        routed = np.arange(n) < ev.n_route
        first[(first < 0) & routed] = r
        if fullkv_topk:
            ids = sorted(np.flatnonzero(routed).tolist(), key=lambda w: (-ev.s_rank[w], w))
            X[r, ids[:tr.k_f]] = 1
        else:
            X[r] = (ev.tiers == FULL) & routed
    return X, first


def global_lir(X: np.ndarray, first: np.ndarray, m: int = 3):
    """Eq. (18): (eligible inactive episodes, those that later re-enter).  An episode is a maximal run
    of X = 0 after the window was selected; it is eligible after m inactive events and rescued when
    the window is selected again before the trace ends."""
    eligible = rescued = 0
    for w in range(X.shape[1]):
        if first[w] < 0:
            continue
        seq = X[first[w]:, w]
        i, seen = 0, False
        while i < len(seq):
            if seq[i]:
                seen = True
                i += 1
                continue
            j = i
            while j < len(seq) and not seq[j]:
                j += 1
            if seen and j - i >= m:
                eligible += 1
                rescued += 1 if j < len(seq) else 0
            i = j
    return eligible, rescued


def lagged_counts(X: np.ndarray, first: np.ndarray, max_lag: int = 8) -> np.ndarray:
    """Eq. (19) counts: n[Delta - 1][a][b] = #{(w, r): routed at r, X[r][w] = a, X[r + Delta][w] = b}."""
    n = np.zeros((max_lag, 2, 2), np.int64)
    R = X.shape[0]
    for w in range(X.shape[1]):
        if first[w] < 0:
            continue
        for d in range(1, max_lag + 1):
            for r in range(first[w], R - d):
                n[d - 1, X[r, w], X[r + d, w]] += 1
    return n


def report(traces: List[Trace], H: int = 32, m: int = 3, max_lag: int = 8) -> dict:
    """All diagnostics over the (layer, sequence) traces of a run, each mean taken over its terms."""
    fmm, churn, qsa, rq, mus = [], [], [], [], []
    lir = np.zeros(2, np.int64)
    lir_o = np.zeros(2, np.int64)
    lag = np.zeros((max_lag, 2, 2), np.int64)
    for tr in traces:
        fmm += fmm_terms(tr, H)
        churn += churn_terms(tr)
        a, b = qsa_terms(tr)
        qsa += a
        rq += b
        mus.append(tier_mass(tr, tr.events[-1]))
        X, first = selections(tr, fullkv_topk=False)
        lir += global_lir(X, first, m)
        lag += lagged_counts(X, first, max_lag)
        Xo, fo = selections(tr, fullkv_topk=True)
        lir_o += global_lir(Xo, fo, m)

    def mean(v):
        return float(np.mean(v)) if v else 0.0
    return {"events": len(traces[0].events), "fmm": mean(fmm), "fmm_terms": len(fmm), "churn": mean(churn),
            "churn_terms": len(churn), "qsa": mean(qsa), "r_q": mean(rq), "qsa_terms": len(qsa),
            "tier_mass": np.mean(mus, axis=0), "lir_eligible": int(lir[0]), "lir_rescued": int(lir[1]),
            "lir_fullkv_eligible": int(lir_o[0]), "lir_fullkv_rescued": int(lir_o[1]), "lag": lag}
