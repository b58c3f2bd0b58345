"""Pins of the oracle's attention, window masses and prefill scores.

QEvict §4.1 (attention over the accessible set), §4.2 Eq. (1) and its last
paragraph (prompt attention initialises the scores).  Checks: the all-Full
special case against torch's scaled_dot_product_attention, uniform attention
(zero queries) against closed forms, probability conservation, and a
pure-Python brute force of the prefill scores on a tiny prompt.
"""
import math

import numpy as np
import pytest
import torch

from oracle import qevict_oracle as O


def _bf16(rng, shape, scale=1.0):
    return O.bf16_round((rng.standard_normal(shape) * scale).astype(np.float32))


def _cfg(**kw):
    base = dict(h_q=4, h_kv=2, d_head=16, n_sink=2, n_recent=4, window=4, bits=2, omega=2,
                prompt_len=66, max_len=66 + 40)
    base.update(kw)
    return O.Config(**base)


def _sdpa(q, K, V, h_kv):
    """Dense attention of one query per head over all tokens, by torch (float64, CPU)."""
    h_q = q.shape[0]
    G = h_q // h_kv
    qt = torch.from_numpy(np.asarray(q, np.float64))[:, None, :]                   # [H_q][1][d]
    Kt = torch.from_numpy(np.asarray(K, np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
    Vt = torch.from_numpy(np.asarray(V, np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
    return torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt)[:, 0, :].numpy()


def test_all_full_equals_dense_attention():
    """Budget >= full cache with K_f >= every window: QEvict reduces to dense attention."""
    cfg = _cfg(q_num=0, b_total=10 ** 9)
    rng = np.random.default_rng(0)
    P = cfg.prompt_len
    k, v = _bf16(rng, (P, cfg.h_kv, cfg.d_head)), _bf16(rng, (P, cfg.h_kv, cfg.d_head))
    u = O.Unit(cfg)
    assert u.bud.k_f >= cfg.n_windows_cap()
    u.prefill_route(k, v, rng.random(O.prompt_windows(cfg)))
    allk, allv = [k], [v]
    for s in range(1, 33):
        q = _bf16(rng, (cfg.h_q, cfg.d_head), 3.0)
        kn, vn = _bf16(rng, (cfg.h_kv, cfg.d_head)), _bf16(rng, (cfg.h_kv, cfg.d_head))
        allk.append(kn[None])
        allv.append(vn[None])
        o, masses, sink = u.decode_step(q, kn, vn)
        ref = _sdpa(q, np.concatenate(allk), np.concatenate(allv), cfg.h_kv)
        assert np.max(np.abs(o - ref)) < 1e-12
        if s % cfg.omega == 0:
            u.route()
    assert not np.any(u.z == O.EVICTED) and not np.any(u.z == O.QUANT)


def test_mass_is_conserved_every_step():
    cfg = _cfg(budget_num=30)
    rng = np.random.default_rng(1)
    P = cfg.prompt_len
    u = O.Unit(cfg)
    u.prefill_route(_bf16(rng, (P, 2, 16)), _bf16(rng, (P, 2, 16)), rng.random(O.prompt_windows(cfg)))
    for s in range(1, 25):
        S_before = u.S.copy()
        o, masses, sink = u.decode_step(_bf16(rng, (4, 16), 2.0), _bf16(rng, (2, 16)), _bf16(rng, (2, 16)))
        assert np.allclose(masses.sum(axis=1) + sink, 1.0, atol=1e-12)
        assert np.allclose(u.S - S_before, masses.sum(axis=0) / cfg.h_q, atol=1e-15)
        assert np.isclose((u.S - S_before).sum() + sink.sum() / cfg.h_q, 1.0, atol=1e-12)
        if s % cfg.omega == 0:
            u.route()


def test_zero_query_is_uniform_over_the_accessible_set():
    """q = 0: every accessible token gets 1/N; the output is the mean of the accessible values and a
    window's mass is its accessible token count over N (this pins the token -> window attribution)."""
    cfg = _cfg(budget_num=30)
    rng = np.random.default_rng(2)
    P = cfg.prompt_len
    u = O.Unit(cfg)
    u.prefill_route(_bf16(rng, (P, 2, 16)), _bf16(rng, (P, 2, 16)), rng.random(O.prompt_windows(cfg)))
    for s in range(1, 12):
        kn, vn = _bf16(rng, (2, 16)), _bf16(rng, (2, 16))
        o, masses, sink = u.decode_step(np.zeros((4, 16), np.float32), kn, vn)
        K, V, wid = u.accessible()
        N = len(wid)
        for h in range(4):
            assert np.allclose(o[h], V[:, h // 2, :].astype(np.float64).mean(axis=0), atol=1e-12)
        counts = {}
        for p in range(cfg.n_sink):
            counts[-1] = counts.get(-1, 0) + 1
        for w in range(u.n_route):
            if u.z[w] in (O.FULL, O.QUANT):
                counts[w] = cfg.window
        for p in range(cfg.n_sink + u.n_route * cfg.window, u.T):
            w = (p - cfg.n_sink) // cfg.window
            counts[w] = counts.get(w, 0) + 1
        assert sum(counts.values()) == N
        for w in range(len(u.S)):
            assert np.allclose(masses[:, w], counts.get(w, 0) / N, atol=1e-14)
        assert np.allclose(sink, counts[-1] / N)
        if s % cfg.omega == 0:
            u.route()


def test_prefill_scores_uniform_closed_form():
    """q = 0: a_tau(i) = 1/(tau+1), so column i collects H_P - H_i (harmonic numbers)."""
    cfg = _cfg(prompt_len=50, max_len=60)
    P = cfg.prompt_len
    q = np.zeros((P, 4, 16), np.float32)
    k = _bf16(np.random.default_rng(3), (P, 2, 16))
    S0 = O.prefill_scores(q, k, cfg, row_block=7)
    H = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, P + 1))])     # H[n] = sum_{m<=n} 1/m
    col = H[P] - H[np.arange(P)]
    n_win = math.ceil((P - cfg.n_sink) / cfg.window)
    ref = [col[cfg.n_sink + j * 4: min(P, cfg.n_sink + j * 4 + 4)].sum() for j in range(n_win)]
    assert np.allclose(S0, ref, rtol=1e-13)
    assert np.isclose(S0.sum() + col[:cfg.n_sink].sum(), P)


def test_prefill_scores_brute_force():
    cfg = O.Config(h_q=2, h_kv=1, d_head=3, n_sink=1, n_recent=2, window=3, prompt_len=11, max_len=12)
    rng = np.random.default_rng(4)
    P = cfg.prompt_len
    q = _bf16(rng, (P, 2, 3), 2.0)
    k = _bf16(rng, (P, 1, 3), 2.0)
    col = [0.0] * P
    for h in range(2):
        for tau in range(P):
            logits = [sum(float(q[tau, h, c]) * float(k[i, 0, c]) for c in range(3)) / math.sqrt(3)
                      for i in range(tau + 1)]
            mx = max(logits)
            e = [math.exp(x - mx) for x in logits]
            z = sum(e)
            for i in range(tau + 1):
                col[i] += e[i] / z
    ref = [sum(col[1 + 3 * j: min(P, 4 + 3 * j)]) / 2 for j in range(4)]
    assert np.allclose(O.prefill_scores(q, k, cfg, row_block=4), ref, rtol=1e-12)


def test_promotion_leaves_attention_unchanged():
    """A window's tokens read the same values whether it is Quantized (dequantised on the fly) or
    promoted to Full, so promotion does not change attention (QEvict §4.3, App. K)."""
    cfg = _cfg(budget_num=60)
    rng = np.random.default_rng(6)
    P = cfg.prompt_len
    u = O.Unit(cfg)
    u.prefill_route(_bf16(rng, (P, 2, 16)), _bf16(rng, (P, 2, 16)), rng.random(O.prompt_windows(cfg)))
    qw = [w for w in range(u.n_route) if u.z[w] == O.QUANT]
    assert qw
    w = qw[0]
    K0, V0, wid0 = u.accessible()
    S = u.S.copy()
    S[w] = 1e6
    u.route(S)
    assert u.z[w] == O.FULL and u.ledger[w].status == O.DORMANT
    K1, V1, wid1 = u.accessible()
    assert np.array_equal(K0[wid0 == w], K1[wid1 == w]) and np.array_equal(V0[wid0 == w], V1[wid1 == w])
