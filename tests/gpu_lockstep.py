"""Lockstep driver: runs the CUDA path (through the C ABI) and the CPU oracle on the same seeded
inputs and compares them step by step.

Tolerances (reading of the stated bar): attention outputs max-abs <= 2e-2 (bf16 outputs); window
masses and scores relative <= 1e-3 wherever the value is at least 2^-100 of the largest in the same
row, else absolute <= 2^-100 of that largest.  The floor only covers values that fp32 cannot carry:
the kernels' exponentials flush results below 2^-126 of their running maximum to zero, so a window
whose every probability lies that far below the maximum reads as 0.  Tier states, slots, tables,
INT2 codes, fp16 parameters and bf16 window data bit-exact, with the router of the oracle fed the
scores the GPU ranked ("identical scores").
"""
import numpy as np
import torch

import layout as LY
from oracle import qevict_oracle as O
from recoverable_quantized_kv_gb300 import binding, synth

OUT_TOL = 2e-2
REL_TOL = 1e-3
FLOOR = 2.0 ** -100     # of the row's largest value: below it, values are compared in absolute terms


def close_rel(gpu, ref, what, rel=REL_TOL, floor_frac=FLOOR):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return
    floor = max(floor_frac * np.abs(ref).max(), np.finfo(np.float64).tiny)
    big = np.abs(ref) >= floor
    err_big = np.abs(gpu - ref)[big] / np.abs(ref)[big]
    err_small = np.abs(gpu - ref)[~big]
    assert err_big.size == 0 or err_big.max() <= rel, f"{what}: max rel err {err_big.max():.3e}"
    assert err_small.size == 0 or err_small.max() <= floor, f"{what}: small-value abs err {err_small.max():.3e}"


class Lockstep:
    def __init__(self, wl, check_state=True, oracle_prefill_scores=True, layers=None, per_step=True, state_seqs=None,
                 churn=None):
        """per_step: flush the scores after every decode step and check that step's window masses;
        otherwise scores absorb the steps' masses only inside route(), checked after routing.
        churn: a seed; before every routing event the scores are replaced by seeded random values
        (cumulative ranker only), so that windows move between the tiers in both directions."""
        self.wl = wl
        self.cfg = binding.make_config(wl)
        self.cache = binding.Cache(self.cfg)
        self.ocfg = O.Config.from_obj(wl)
        self.bud = binding.budget(self.cfg)
        self.lay = self.cache.layout
        self.B, self.L = wl.batch, wl.n_layers
        self.W = wl.window
        self.N = self.bud.n_windows
        self.check_state = check_state
        self.layers = list(range(self.L)) if layers is None else layers
        self.units = {(l, b): O.Unit(self.ocfg) for l in range(self.L) for b in range(self.B)}
        self.dec = {(l, b): synth.decode_inputs(wl, b, l) for l in range(self.L) for b in range(self.B)}
        self.step = 0
        self.oracle_prefill_scores = oracle_prefill_scores
        self.max_out_err = 0.0
        self.per_step = per_step
        # sequences whose full tier state / tables / window data are compared (outputs, masses, scores
        # and counters are compared for every sequence)
        self.state_seqs = list(range(self.B)) if state_seqs is None else state_seqs
        self.churn = churn
        self.route_hook = None   # replaces the cache's own routing call (e.g. a diagnostics route)
        self.s0 = {}             # per layer: the prompt scores the prefill routed on
        # pre-RoPE Quantized keys: both sides get the same (cos, sin) table, a model input
        if getattr(wl, "rope_base", 0.0) > 0:
            table = synth.rope_table(wl.max_len, wl.rope_base)
            for u in self.units.values():
                u.set_rope_table(table)
            self.cache.set_rope_table(torch.from_numpy(table).cuda())

    # ---- views of one unit's state
    def _u(self, l, b):
        return l * self.B + b

    def scores(self, l, b):
        raw = self.cache.region("score", self._u(l, b), 4 * self.wl.h_kv * self.N).view(torch.float32)
        return raw.view(self.wl.h_kv, self.N).cpu().numpy()

    def meta(self, l, b):
        return self.cache.region("meta", self._u(l, b), 64).view(torch.int32).cpu().numpy()

    def prefill(self):
        wl = self.wl
        npw = O.prompt_windows(self.ocfg)
        for l in range(self.L):
            ins = [synth.prompt_inputs(wl, b, l) for b in range(self.B)]
            q = torch.stack([x["q"] for x in ins]).cuda()
            k = torch.stack([x["k"] for x in ins]).cuda()
            v = torch.stack([x["v"] for x in ins]).cuda()
            s0 = torch.empty(self.B, npw, dtype=torch.float32, device="cuda")
            self.cache.prefill_scores(q, k, s0)
            s0h = s0.cpu().numpy()
            for b in range(self.B):
                if self.oracle_prefill_scores:
                    ref = O.prefill_scores(ins[b]["q"].float().numpy(), ins[b]["k"].float().numpy(), self.ocfg)
                    close_rel(s0h[b], ref, f"prefill scores layer {l} seq {b}")
                    # conservation: windows + sinks collect exactly one unit of mass per prompt query
                    assert abs(s0h[b].sum() + self._sink_share(ins[b]) - wl.prompt_len) < 1e-3 * wl.prompt_len
                else:   # at full size: every query's mass lands on windows or sinks, sinks take a little
                    assert 0 < wl.prompt_len - s0h[b].sum() < 0.01 * wl.prompt_len
            self.cache.prefill_route(l, k, v, s0=s0)
            self.s0[l] = s0.clone()
            for b in range(self.B):
                self.units[(l, b)].prefill_route(ins[b]["k"].float().numpy(), ins[b]["v"].float().numpy(), s0h[b])
            del q, k, v
        torch.cuda.synchronize()
        if self.check_state:
            for l in self.layers:
                for b in self.state_seqs:
                    self.compare_state(l, b)

    def _sink_share(self, ins):
        """Prompt attention mass on the sink tokens, (1/H_q) sum_h sum_tau a_tau^h(sinks), fp64 exact on the sinks."""
        q = ins["q"].double()
        k = ins["k"].double()
        P, Hq, d = q.shape
        G = Hq // k.shape[1]
        tot = 0.0
        ns = self.wl.n_sink
        for h in range(Hq):
            kg = k[:, h // G, :]
            # row log-sum-exp over the causal prefix, chunked
            for r0 in range(0, P, 4096):
                r1 = min(P, r0 + 4096)
                lg = (q[r0:r1, h, :] @ kg[:r1].T) / np.sqrt(d)
                mask = torch.arange(r1)[None, :] > torch.arange(r0, r1)[:, None]
                lg[mask] = -float("inf")
                lse = torch.logsumexp(lg, dim=1)
                tot += torch.exp(lg[:, :ns] - lse[:, None]).sum().item()
        return tot / Hq

    def compare_state(self, l, b):
        u = self.units[(l, b)]
        wl, W, N = self.wl, self.W, self.N
        unit = self._u(l, b)
        meta = self.meta(l, b)
        assert meta[0] == u.T and meta[1] == u.n_route, (meta[:4], u.T, u.n_route)
        st = self.cache.region("state", unit, N).cpu().numpy()
        assert np.array_equal(st & 3, u.z[:N].astype(np.uint8)), "tier states differ"
        assert np.array_equal((st >> 2) & 3, u.ledger_status()[:N].astype(np.uint8)), "ledger status differs"
        fs = self.cache.region("fslot", unit, 4 * N).view(torch.int32).cpu().numpy()
        ls = self.cache.region("lslot", unit, 4 * N).view(torch.int32).cpu().numpy()
        exp_fs = np.full(N, -1, np.int32)
        for w, s in u.f_slot.items():
            exp_fs[w] = s
        exp_ls = np.full(N, -1, np.int32)
        for w, led in u.ledger.items():
            exp_ls[w] = led.slot
        assert np.array_equal(fs, exp_fs), "F slots differ"
        assert np.array_equal(ls, exp_ls), "ledger slots differ"
        ft, qt = u.f_table(), u.q_table()
        assert meta[2] == len(ft) and meta[3] == len(qt)
        if ft:
            g_ft = self.cache.region("ftab", unit, 8 * len(ft)).view(torch.int32).view(-1, 2).cpu().numpy()
            assert np.array_equal(g_ft, np.array(ft, np.int32)), "F table differs"
        if qt:
            g_qt = self.cache.region("qtab", unit, 8 * len(qt)).view(torch.int32).view(-1, 2).cpu().numpy()
            assert np.array_equal(g_qt, np.array(qt, np.int32)), "Q table differs"
        H = wl.h_kv
        blk_bytes = 2 * W * 128 * 2
        fpool = self.cache.region("fpool", unit, max(1, min(self.bud.k_f, N)) * H * blk_bytes).view(torch.int16)
        fpool = fpool.cpu().numpy().view(np.uint16)
        for w, (Kw, Vw) in u.full.items():
            s = u.f_slot[w]
            for g in range(H):
                base = ((s * H + g) * 2) * W * 128
                kb = LY.unpack_block(fpool[base:base + W * 128], W, False)
                vb = LY.unpack_block(fpool[base + W * 128:base + 2 * W * 128], W, True)
                assert np.array_equal(kb, Kw[:, g, :]) and np.array_equal(vb, Vw[:, g, :]), f"F data of window {w}"
        qb = self.lay.qblock
        nled = max(1, min(self.bud.k_f + self.bud.k_q, N))
        ledger = self.cache.region("ledger", unit, nled * H * qb).cpu().numpy()
        for w, led in u.ledger.items():
            for g in range(H):
                off = (led.slot * H + g) * qb
                ck, cv, ks, km, vs, vm = LY.parse_ledger_block(ledger[off:off + qb], W, wl.bits)
                assert np.array_equal(ck, led.codes_k[g]) and np.array_equal(cv, led.codes_v[g]), f"codes of {w}"
                assert np.array_equal(ks.view(np.uint16), led.s_k[g].view(np.uint16)), f"key scales of {w}"
                assert np.array_equal(km.view(np.uint16), led.m_k[g].view(np.uint16)), f"key offsets of {w}"
                assert np.array_equal(vs.view(np.uint16), led.s_v[g].view(np.uint16)), f"value scales of {w}"
                assert np.array_equal(vm.view(np.uint16), led.m_v[g].view(np.uint16)), f"value offsets of {w}"

    def decode(self, n_steps):
        wl = self.wl
        H = wl.h_kv
        for _ in range(n_steps):
            s = self.step
            for l in range(self.L):
                q = torch.stack([self.dec[(l, b)]["q"][s] for b in range(self.B)]).cuda()
                k = torch.stack([self.dec[(l, b)]["k"][s] for b in range(self.B)]).cuda()
                v = torch.stack([self.dec[(l, b)]["v"][s] for b in range(self.B)]).cuda()
                out = torch.empty(self.B, wl.h_q, 128, dtype=torch.bfloat16, device="cuda")
                saved = {}
                if self.per_step:
                    for b in range(self.B):   # zero the score partials so this step's masses can be read alone
                        reg = self.cache.region("score", self._u(l, b), 4 * H * self.N)
                        saved[b] = reg.clone()
                        reg.zero_()
                self.cache.decode_step(l, q, k, v, out)
                if self.per_step:
                    self.cache.flush_scores()   # scores absorb this step's masses
                torch.cuda.synchronize()
                for b in range(self.B):
                    u = self.units[(l, b)]
                    o_ref, masses, sink = u.decode_step(self.dec[(l, b)]["q"][s].float().numpy(),
                                                        self.dec[(l, b)]["k"][s].float().numpy(),
                                                        self.dec[(l, b)]["v"][s].float().numpy())
                    if l in self.layers:
                        o = out[b].float().cpu().numpy()
                        err = np.abs(o - o_ref).max()
                        self.max_out_err = max(self.max_out_err, float(err))
                        assert err <= OUT_TOL, f"step {s + 1} layer {l} seq {b}: output max-abs err {err:.3e}"
                    if not self.per_step:
                        continue
                    reg = self.cache.region("score", self._u(l, b), 4 * H * self.N)
                    delta = reg.view(torch.float32).view(H, self.N).clone()
                    base = saved[b].view(torch.float32).view(H, self.N)
                    reg.view(torch.float32).view(H, self.N).copy_(base + delta)   # what the kernel adds
                    if l in self.layers:
                        gm = delta.sum(dim=0).cpu().numpy().astype(np.float64)
                        close_rel(gm[:len(u.S)], masses.sum(axis=0)[:self.N] / wl.h_q,
                                  f"step {s + 1} layer {l} seq {b} window masses")
                        assert abs(gm.sum() + sink.sum() / wl.h_q - 1.0) < 1e-4
            self.step += 1
            if self.step % wl.omega == 0:
                self.route()

    def route(self):
        ranker = getattr(self.wl, "ranker", 0)
        # before routing: the sum of the KV-head partials is the oracle's cumulative S (ranker 0), or
        # the attention since the previous event (the other rankers, QEvict App. J Eq. (20))
        if self.per_step:
            for l in self.layers:
                for b in range(self.B):
                    sg = self.scores(l, b).astype(np.float32)
                    tot = sg[0].copy()
                    for g in range(1, sg.shape[0]):
                        tot = (tot + sg[g]).astype(np.float32)
                    u = self.units[(l, b)]
                    ref = u.S if ranker == 0 else u.U
                    close_rel(tot, ref[:self.N], f"scores before event {self.step} layer {l} seq {b}")
        if self.churn is not None:
            assert ranker == 0
            rng = np.random.default_rng([self.churn, self.step])
            H = self.wl.h_kv
            for l in range(self.L):
                for b in range(self.B):
                    forced = torch.zeros(H, self.N, dtype=torch.float32)
                    forced[0] = torch.from_numpy((rng.random(self.N) * 10).astype(np.float32))
                    self.cache.region("score", self._u(l, b), 4 * H * self.N).view(torch.float32).copy_(
                        forced.view(-1).cuda())
        (self.route_hook or self.cache.route)()   # absorbs the pending steps' masses, then ranks
        torch.cuda.synchronize()
        for l in range(self.L):
            for b in range(self.B):
                u = self.units[(l, b)]
                if ranker == 0:
                    rv = self.scores(l, b)[0]
                    if not self.per_step and l in self.layers:
                        close_rel(rv, u.S[:self.N], f"scores at event {self.step} layer {l} seq {b}")
                    u.route(scores=rv.astype(np.float64))
                else:
                    rv = self.cache.region("agg", self._u(l, b), 4 * self.N).view(torch.float32).cpu().numpy()
                    what = f"rank values at event {self.step} layer {l} seq {b}"
                    hook = (lambda R, rv=rv, what=what: close_rel(rv, R[:self.N], what)) if l in self.layers else None
                    u.route(scores=rv.astype(np.float64), rank_hook=hook)
        if self.check_state:
            for l in self.layers:
                for b in self.state_seqs:
                    self.compare_state(l, b)

    def counters(self):
        got = self.cache.counters()
        want = np.zeros(7, np.int64)
        for u in self.units.values():
            want += u.counters
        return got, dict(zip(binding.COUNTER_NAMES, want.tolist()))
