"""Pins of the oracle's budget, candidate pool, TopK routing and migration bookkeeping.

QEvict §4.1 (budget constraint), §4.3 Eq. (3)-(6), App. A Algorithm 1, App. B.4 Eq. (7)-(8).
Checks: brute-force enumeration of all tier assignments on tiny pools, the
byte budget measured on the oracle's own stored arrays, and the invariants the
pages state (budget never exceeded, sinks and recent tokens never routed,
evicted windows never return, F/Q/E partition the history, codes written once).
"""
import itertools

import numpy as np
import pytest

from oracle import qevict_oracle as O

TINY = dict(h_q=4, h_kv=2, d_head=8, n_sink=2, n_recent=4, window=4, bits=2, omega=2)


def _bf16(rng, shape, scale=1.0):
    return O.bf16_round((rng.standard_normal(shape) * scale).astype(np.float32))


# ----------------------------------------------------------------------------- budget

@pytest.mark.parametrize("name", ["tiny_4k", "llama8b_32k", "batched_32k", "long_131k", "drift_16k"])
def test_capacities_are_the_largest_that_fit(name):
    from recoverable_quantized_kv_gb300 import synth
    cfg = O.Config.from_obj(synth.workload(name))
    b = O.budget(cfg)
    # floor optimality of Eq. (3) in exact rationals: K*M <= share < (K+1)*M
    share_f = (cfg.q_den - cfg.q_num) * b.b_hist
    share_q = cfg.q_num * b.b_hist
    assert b.k_f * b.m_f * cfg.q_den <= share_f < (b.k_f + 1) * b.m_f * cfg.q_den
    assert b.k_q * b.m_q * cfg.q_den <= share_q < (b.k_q + 1) * b.m_q * cfg.q_den
    # all windows of both tiers fit in the total budget together with the protected regions
    assert b.b_sink + b.b_local + b.k_f * b.m_f + b.k_q * b.m_q <= b.b_total
    assert b.b_total <= b.full_bytes


@pytest.mark.parametrize("bits,window", [(2, 32), (4, 64), (2, 4)])
def test_window_costs_match_the_stored_arrays(bits, window):
    """M_q / M_f count exactly the bytes of the arrays the oracle stores for one window."""
    cfg = O.Config(h_q=8, h_kv=2, d_head=128, window=window, bits=bits, prompt_len=8192, max_len=8200)
    b = O.budget(cfg)
    rng = np.random.default_rng(0)
    K = _bf16(rng, (window, cfg.h_kv, cfg.d_head))
    led = O.quantize_window(K, K, bits)
    code_bytes = (led.codes_k.size + led.codes_v.size) * bits // 8
    param_bytes = led.s_k.nbytes + led.m_k.nbytes + led.s_v.nbytes + led.m_v.nbytes
    assert led.s_k.dtype == np.float16 and led.s_v.dtype == np.float16
    assert code_bytes + param_bytes == b.payload
    positions, q_record, f_record = window * 4, 16, 8
    assert b.m_q == b.payload + positions + q_record
    bf16_window = 2 * K.size * 2                       # K and V of the window in bf16
    assert b.m_f == bf16_window + positions + f_record + b.payload
    # full KV of one layer and sequence: K and V, bf16, every prompt token (Eq. (7))
    assert b.full_bytes == cfg.prompt_len * 2 * cfg.h_kv * cfg.d_head * 2


def test_budget_below_protected_regions_is_rejected():
    cfg = O.Config(h_q=8, h_kv=2, prompt_len=64, max_len=80, b_total=100)
    with pytest.raises(ValueError):
        O.budget(cfg)


def test_aging_rule_brute_force():
    """A window ages once every one of its tokens lies before the last n_recent positions."""
    cfg = O.Config(**TINY, prompt_len=10, max_len=200)
    for T in range(0, 120):
        recent_lo = T - cfg.n_recent
        aged = [j for j in range(60) if all(p < recent_lo for p in range(cfg.n_sink + j * cfg.window,
                                                                           cfg.n_sink + (j + 1) * cfg.window))]
        assert O.n_hist(T, cfg) == len(aged) and aged == list(range(len(aged)))


# ----------------------------------------------------------------------------- TopK

def _fresh_unit(n_windows, k_f, k_q, seed=0, **policy):
    """A unit whose prompt holds exactly n_windows historical windows, with capacities forced."""
    P = TINY["n_sink"] + TINY["n_recent"] + n_windows * TINY["window"]
    cfg = O.Config(**TINY, prompt_len=P, max_len=P + 64, b_total=10 ** 9, **policy)
    u = O.Unit(cfg)
    u.bud = O.Budget(0, 10 ** 9, 0, 0, 10 ** 9, 0, 1, 1, k_f, k_q)
    rng = np.random.default_rng(seed)
    k = _bf16(rng, (P, cfg.h_kv, cfg.d_head))
    return u, k


def _pad(u, S):
    """Scores for the historical windows, zeros for the prompt windows still in the recent region."""
    return np.concatenate([S, np.zeros(O.prompt_windows(u.cfg) - len(S))])


def _brute_force(S, k_f, k_q):
    n = len(S)
    nf = min(k_f, n)
    nq = min(k_q, n - nf)
    best, best_key = None, None
    for assign in itertools.product((O.FULL, O.QUANT, O.EVICTED), repeat=n):
        if assign.count(O.FULL) != nf or assign.count(O.QUANT) != nq:
            continue
        key = (sum(S[i] for i in range(n) if assign[i] == O.FULL),
               sum(S[i] for i in range(n) if assign[i] != O.EVICTED))
        if best_key is None or key > best_key:
            best, best_key = assign, key
    return list(best)


@pytest.mark.parametrize("n,k_f,k_q,seed", [(n, kf, kq, s) for n in (1, 3, 5, 8) for kf in (0, 1, 2, 9)
                                            for kq in (0, 2, 3) for s in (0, 1)])
def test_routing_equals_brute_force(n, k_f, k_q, seed):
    u, k = _fresh_unit(n, k_f, k_q, seed)
    S = np.random.default_rng(100 + seed).permutation(n).astype(np.float64) + 0.5   # distinct scores
    u.prefill_route(k, k, _pad(u, S))
    assert u.z[:n].tolist() == _brute_force(list(S), k_f, k_q)


def test_ties_prefer_the_older_window():
    u, k = _fresh_unit(6, 2, 2)
    u.prefill_route(k, k, _pad(u, np.ones(6)))
    assert u.z[:6].tolist() == [O.FULL, O.FULL, O.QUANT, O.QUANT, O.EVICTED, O.EVICTED]


# ----------------------------------------------------------------------------- long runs: invariants

def _drive(cfg, steps, seed, churn=True, check=None):
    rng = np.random.default_rng(seed)
    u = O.Unit(cfg)
    P = cfg.prompt_len
    k = _bf16(rng, (P, cfg.h_kv, cfg.d_head))
    v = _bf16(rng, (P, cfg.h_kv, cfg.d_head))
    s0 = rng.random(O.prompt_windows(cfg))
    u.prefill_route(k, v, s0)
    if check:
        check(u)
    for s in range(1, steps + 1):
        q = _bf16(rng, (cfg.h_q, cfg.d_head), 2.0)
        u.decode_step(q, _bf16(rng, (cfg.h_kv, cfg.d_head)), _bf16(rng, (cfg.h_kv, cfg.d_head)))
        if s % cfg.omega == 0:
            scores = rng.random(len(u.S)) * 10 if churn else None     # forced churn: promotions and demotions
            u.route(scores)
            if check:
                check(u)
    return u


def _small_cfg(**kw):
    base = dict(TINY, prompt_len=64, max_len=64 + 200, budget_num=60, budget_den=100, d_head=16)
    base.update(kw)
    return O.Config(**base)


@pytest.mark.parametrize("q_num", [0, 30, 70, 100])
def test_invariants_after_every_event(q_num):
    cfg = _small_cfg(q_num=q_num)
    bud = O.budget(cfg)
    state = {"evicted": set()}

    def check(u):
        n = u.n_route
        assert u.stored_bytes() <= bud.b_total                                   # budget never exceeded
        assert np.all(u.z[n:] == O.LOCAL)                                        # recent tokens never routed
        assert set(np.unique(u.z[:n]).tolist()) <= {O.FULL, O.QUANT, O.EVICTED}  # F/Q/E partition the history
        ev = set(np.flatnonzero(u.z[:n] == O.EVICTED).tolist())
        assert state["evicted"] <= ev                                            # evicted never return
        state["evicted"] = ev
        fw = np.flatnonzero(u.z == O.FULL)
        qw = np.flatnonzero(u.z == O.QUANT)
        assert len(fw) <= bud.k_f and len(qw) <= bud.k_q
        assert sorted(u.f_slot) == fw.tolist()
        assert len(set(u.f_slot.values())) == len(fw) and all(0 <= s < bud.k_f for s in u.f_slot.values())
        slots = [led.slot for led in u.ledger.values()]
        assert len(set(slots)) == len(slots) and all(0 <= s < bud.k_f + bud.k_q for s in slots)
        for w in qw:
            assert u.ledger[w].status == O.ACTIVE
        for w, led in u.ledger.items():
            assert u.z[w] in (O.FULL, O.QUANT)
            assert (led.status == O.DORMANT) == (u.z[w] == O.FULL)
        # deterministic slots: retained windows keep theirs; newcomers (ascending id) take the lowest free ones
        prev_f, prev_l = state.get("f", {}), state.get("l", {})
        cur_l = {w: led.slot for w, led in u.ledger.items()}
        for cur, prev, pool in ((dict(u.f_slot), prev_f, bud.k_f), (cur_l, prev_l, bud.k_f + bud.k_q)):
            kept = {w: sl for w, sl in cur.items() if w in prev}
            assert all(prev[w] == sl for w, sl in kept.items())
            newcomers = sorted(w for w in cur if w not in prev)
            free = sorted(set(range(pool)) - set(kept.values()))
            assert [cur[w] for w in newcomers] == free[:len(newcomers)]
        state["f"], state["l"] = dict(u.f_slot), cur_l
        lo = cfg.n_sink + n * cfg.window                                         # local region size after an event
        assert all(p >= lo for p in u.local) and len(u.local) == u.T - lo
        assert cfg.n_recent <= len(u.local) <= cfg.n_recent + cfg.window - 1
        assert u.sink_k.shape[0] == cfg.n_sink                                   # sinks kept, never in a table

    u = _drive(cfg, 120, seed=q_num, check=check)
    if q_num == 0:
        assert bud.k_q == 0 and not np.any(u.z == O.QUANT)                      # two-tier window eviction
    if q_num == 100:
        assert bud.k_f == 0 and not np.any(u.z == O.FULL)                       # pure quantised retention
    if 0 < q_num < 100:
        c = dict(zip(O.COUNTER_NAMES, u.counters.tolist()))
        assert c["promotions"] > 0 and c["demotions"] > 0 and c["evictions"] > 0 and c["reactivations"] > 0


def test_codes_are_written_once():
    """Across many promote/demote cycles a window's codes and parameters never change (QEvict §4.3)."""
    cfg = _small_cfg(q_num=70)
    first = {}

    def check(u):
        for w, led in u.ledger.items():
            snap = (led.codes_k.tobytes(), led.s_k.tobytes(), led.m_k.tobytes(),
                    led.codes_v.tobytes(), led.s_v.tobytes(), led.m_v.tobytes())
            assert first.setdefault(w, snap) == snap

    u = _drive(cfg, 160, seed=3, check=check)
    assert u.counters[O.COUNTER_NAMES.index("reactivations")] >= 10


def test_promoted_window_holds_the_dequantised_copy():
    """Promotion rebuilds the low-bit approximation, not the original (QEvict App. K, §4.3)."""
    cfg = _small_cfg(q_num=70)
    rng = np.random.default_rng(5)
    u = _drive(cfg, 40, seed=5, churn=True)
    for w, led in u.ledger.items():
        if led.status == O.DORMANT:
            K, V = u.full[w]
            Kh, Vh = led.dequantize()
            assert np.array_equal(K, Kh) and np.array_equal(V, Vh)
    del rng


def _golden_events(name="routing_events.txt"):
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)
    rows = []
    for ln in open(path):
        if ln.strip() and not ln.startswith("#"):
            f = [p.split() for p in ln.split("|")]
            rows.append(dict(event=int(f[0][0]), T=int(f[1][0]), scores=[float(x) for x in f[2]], tier=f[3],
                             fslot=f[4], lslot=f[5], ledger=f[6], counters=[int(x) for x in f[7]]))
    return rows


@pytest.mark.parametrize("fixture,policy", [("routing_events.txt", {}),
                                            ("routing_no_promotion.txt", {"no_promotion": 1})])
def test_routing_events_worked_by_hand(fixture, policy):
    """Tiers, F slots, ledger slots and statuses, and transition counters of three routing events worked
    by hand (tests/golden/; QEvict §4.3 Eq. (4)-(6), App. A Algorithm 1, and App. K's policy without
    promotion, where a Quantized window that out-scores a Full one stays Quantized)."""
    rows = _golden_events(fixture)
    u, k = _fresh_unit(6, 2, 2, seed=3, **policy)
    P = u.cfg.prompt_len
    assert P == 30 and O.prompt_windows(u.cfg) == 7
    rng = np.random.default_rng(4)
    tier_of = {O.FULL: "F", O.QUANT: "Q", O.EVICTED: "E", O.LOCAL: "L"}
    for row in rows:
        if row["event"] == 0:
            before = u.counters.copy()
            u.prefill_route(k, _bf16(rng, k.shape), np.array(row["scores"]))
        else:
            for _ in range(u.cfg.omega):
                u.decode_step(_bf16(rng, (u.cfg.h_q, u.cfg.d_head)), _bf16(rng, (u.cfg.h_kv, u.cfg.d_head)),
                              _bf16(rng, (u.cfg.h_kv, u.cfg.d_head)))
            before = u.counters.copy()
            scores = np.zeros(len(u.S))
            scores[:7] = row["scores"]
            u.route(scores)
        assert u.T == row["T"]
        assert [tier_of[int(z)] for z in u.z[:7]] == row["tier"]
        assert [str(u.f_slot[w]) if w in u.f_slot else "-" for w in range(7)] == row["fslot"]
        assert [str(u.ledger[w].slot) if w in u.ledger else "-" for w in range(7)] == row["lslot"]
        st = {O.ACTIVE: "a", O.DORMANT: "d"}
        assert [st[u.ledger[w].status] if w in u.ledger else "-" for w in range(7)] == row["ledger"]
        assert (u.counters - before).tolist() == row["counters"]
