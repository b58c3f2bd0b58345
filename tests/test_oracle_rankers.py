"""Pins of the oracle's alternative window rankers (QEvict App. J Eq. (20)-(24)) and of the
no-promotion policy (QEvict App. K).

Checks:
- decayed attention with lambda = 1 and the p-norm with p = 1 reduce to cumulative attention (the
  default ranking of §4.2 Eq. (1)), on whole runs;
- the decayed value follows its geometric series for a constant per-event attention;
- the p-norm value is the sum of the event attentions raised to p;
- key-norm ranking keeps the windows with the smallest keys;
- under no-promotion a quantized window never returns to the full tier, the full tier holds the
  best-ranked eligible windows, and the quantized tier the best of the rest.
"""
import numpy as np
import pytest

from oracle import qevict_oracle as O
from test_oracle_routing import _bf16, _small_cfg


def _run(cfg, steps, seed):
    """A random run without forced scores: tiers follow the attention the unit itself measures."""
    rng = np.random.default_rng(seed)
    u = O.Unit(cfg)
    P = cfg.prompt_len
    k = _bf16(rng, (P, cfg.h_kv, cfg.d_head))
    v = _bf16(rng, (P, cfg.h_kv, cfg.d_head))
    u.prefill_route(k, v, rng.random(O.prompt_windows(cfg)))
    history = [u.z.copy()]
    for s in range(1, steps + 1):
        q = _bf16(rng, (cfg.h_q, cfg.d_head), 3.0)
        u.decode_step(q, _bf16(rng, (cfg.h_kv, cfg.d_head)), _bf16(rng, (cfg.h_kv, cfg.d_head)))
        if s % cfg.omega == 0:
            u.route()
            history.append(u.z.copy())
    return u, history


@pytest.mark.parametrize("variant", [dict(ranker=1, decay=1.0), dict(ranker=2, pnorm=1.0)])
def test_unit_parameters_reduce_to_cumulative_attention(variant):
    base, hb = _run(_small_cfg(q_num=70), 96, seed=11)
    other, ho = _run(_small_cfg(q_num=70, **variant), 96, seed=11)
    assert all(np.array_equal(a, b) for a, b in zip(hb, ho))
    assert np.array_equal(base.counters, other.counters)
    n = base.n_route
    assert np.allclose(other.R[:n], base.S[:n], rtol=1e-12, atol=0.0)


def test_decayed_value_is_the_geometric_series():
    """Eq. (22) with the same u at every event: R_n = u (1 - lam^(n+1)) / (1 - lam)."""
    lam, u_ev = 0.9, 0.25
    cfg = _small_cfg(q_num=70, ranker=1, decay=lam)
    u = O.Unit(cfg)
    ncap = len(u.R)
    for n in range(6):
        u.U[:] = u_ev
        u.rank_values(list(range(ncap)), [])
        assert np.allclose(u.R, u_ev * (1 - lam ** (n + 1)) / (1 - lam), rtol=1e-14)
        assert np.all(u.U == 0.0)


def test_pnorm_value_is_the_sum_of_powers():
    """Eq. (23): ranking by (sum_r u_r^p)^(1/p) is ranking by sum_r u_r^p; p = 3 by default."""
    cfg = _small_cfg(q_num=70, ranker=2)
    assert cfg.pnorm == 3.0
    u = O.Unit(cfg)
    events = [np.array([0.6, 0.1, 0.2]), np.array([0.0, 0.6, 0.2]), np.array([0.0, 0.1, 0.2])]
    for ev in events:
        u.U[:3] = ev
        u.rank_values([0, 1, 2], [])
    expect = sum(e ** 3 for e in events)
    assert np.allclose(u.R[:3], expect, rtol=1e-14)
    # the p-norm prefers a single strong event over the same total spread out (peak sensitivity)
    assert u.R[0] > u.R[2] and abs(sum(e[0] for e in events) - sum(e[2] for e in events)) < 1e-12


def test_key_norm_ranking_keeps_the_smallest_keys():
    """Eq. (24): windows are ranked by -mean ||k||, so the smallest-key windows take the full tier,
    the next the quantized tier, the largest are evicted."""
    cfg = _small_cfg(q_num=50, ranker=3, budget_num=60)
    bud = O.budget(cfg)
    rng = np.random.default_rng(2)
    P = cfg.prompt_len
    nw = O.n_hist(P, cfg)
    scale = rng.permutation(nw) + 1.0                     # a distinct key scale for every window
    k = _bf16(rng, (P, cfg.h_kv, cfg.d_head))
    for w in range(nw):
        lo = cfg.n_sink + w * cfg.window
        k[lo:lo + cfg.window] = O.bf16_round(k[lo:lo + cfg.window] * np.float32(scale[w] / 8))
    u = O.Unit(cfg)
    u.prefill_route(k, k, rng.random(O.prompt_windows(cfg)))
    norms = [u.R[w] for w in range(nw)]
    want = sorted(range(nw), key=lambda w: (norms[w], w))
    assert sorted(np.flatnonzero(u.z[:nw] == O.FULL).tolist()) == sorted(want[:bud.k_f])
    assert sorted(np.flatnonzero(u.z[:nw] == O.QUANT).tolist()) == sorted(want[bud.k_f:bud.k_f + bud.k_q])
    # the window's value is the mean over its tokens of the key's norm across all KV heads
    w = want[0]
    lo = cfg.n_sink + w * cfg.window
    ref = np.mean([np.linalg.norm(k[p].astype(np.float64)) for p in range(lo, lo + cfg.window)])
    assert abs(u.R[w] - ref) < 1e-9 * ref


@pytest.mark.parametrize("q_num", [30, 70])
def test_no_promotion_invariants(q_num):
    cfg = _small_cfg(q_num=q_num, no_promotion=1)
    bud = O.budget(cfg)
    rng = np.random.default_rng(q_num)
    u = O.Unit(cfg)
    P = cfg.prompt_len
    k = _bf16(rng, (P, cfg.h_kv, cfg.d_head))
    u.prefill_route(k, k, rng.random(O.prompt_windows(cfg)))
    for s in range(1, 161):
        q = _bf16(rng, (cfg.h_q, cfg.d_head), 3.0)
        u.decode_step(q, _bf16(rng, (cfg.h_kv, cfg.d_head)), _bf16(rng, (cfg.h_kv, cfg.d_head)))
        if s % cfg.omega == 0:
            before = u.z.copy()
            scores = rng.random(len(u.S)) * 10         # forced churn
            u.route(scores)
            # candidates: the windows that were full or quantized, and the windows aged at this event
            cand = [w for w in range(u.n_route) if before[w] in (O.FULL, O.QUANT) or before[w] == O.LOCAL]
            rank = sorted(cand, key=lambda w: (-scores[w], w))
            fw = [w for w in cand if u.z[w] == O.FULL]
            qw = [w for w in cand if u.z[w] == O.QUANT]
            assert not any(before[w] == O.QUANT for w in fw)                   # never Q -> F
            eligible = [w for w in rank if before[w] != O.QUANT]
            assert sorted(fw) == sorted(eligible[:bud.k_f])                    # F: best eligible
            rest = [w for w in rank if w not in fw]
            assert sorted(qw) == sorted(rest[:bud.k_q])                        # Q: best of the rest
    c = dict(zip(O.COUNTER_NAMES, u.counters.tolist()))
    assert c["promotions"] == 0 and c["reactivations"] == 0 and c["demotions"] > 0 and c["evictions"] > 0
