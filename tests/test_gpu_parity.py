"""GPU parity: the CUDA path through the C ABI against the CPU oracle (QEvict §4.1-§4.3, App. A).

Every test here is marked gpu and runs in lockstep (tests/gpu_lockstep.py): outputs within
2e-2 max-abs, window masses and scores within 1e-3 relative, tier states / slots / tables /
INT2 codes / fp16 parameters / bf16 window data bit-exact given identical scores.
"""
import numpy as np
import pytest
import torch

from gpu_lockstep import close_rel, Lockstep, OUT_TOL
from oracle import qevict_oracle as O
from recoverable_quantized_kv_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def _run(wl, steps, **kw):
    ls = Lockstep(wl, **kw)
    ls.prefill()
    ls.decode(steps)
    got, want = ls.counters()
    assert got == want, (got, want)
    return ls


def test_tiny_workload_full_run(lib):
    """The tiny workload end to end: 4096-token prefill, 64 decode steps, 8 routing events."""
    ls = _run(synth.workload("tiny_4k"), 64)
    c = ls.cache.counters()
    assert c["evictions"] > 0 and c["first_quant"] > 0


@pytest.mark.parametrize("shape", [
    dict(h_q=8, h_kv=2, prompt_len=1000, n_sink=5, batch=2),        # ragged prompt, odd sink, batch 2
    dict(h_q=8, h_kv=8, prompt_len=777, n_sink=1),                  # G = 1
    dict(h_q=16, h_kv=2, prompt_len=1500, n_sink=16, n_recent=64),  # G = 8, 16 sinks
    dict(h_q=4, h_kv=2, prompt_len=600, n_sink=3, omega=4, budget_num=40),
])
def test_edge_shapes(lib, shape):
    base = synth.workload("tiny_4k", steps=24, n_plant=4, kappa=6.0)
    _run(base.replace(**shape), 24)


def test_scores_absorbed_only_at_routing(lib):
    """Window masses of Omega decode steps absorbed by the router's own flush, no flush in between,
    reach the oracle's per-step cumulative scores (QEvict §4.2 Eq. (1))."""
    base = synth.workload("tiny_4k", prompt_len=1500, steps=32, n_plant=4)
    _run(base, 32, per_step=False)
    _run(base.replace(h_q=16, h_kv=2, batch=2, omega=5), 20, per_step=False)


@pytest.mark.parametrize("shape", [
    dict(h_q=8, h_kv=2, prompt_len=1500, n_sink=4, batch=2),          # G = 4, batch 2
    dict(h_q=8, h_kv=8, prompt_len=1111, n_sink=7, budget_num=40),     # G = 1, ragged prompt
    dict(h_q=16, h_kv=2, prompt_len=2000, n_sink=16, omega=5),         # G = 8, 16 sinks
])
def test_int4_w64_shapes(lib, shape):
    """The INT4 / 64-token-window format (QEvict §5 INT4 setting): 4-bit codes with fp16 scale and
    offset, three-chunk ledger records, windows decoded as two 32-token halves."""
    base = synth.workload("tiny_4k", window=64, bits=4, steps=24, n_plant=4, kappa=6.0)
    _run(base.replace(**shape), 24)


@pytest.mark.parametrize("policy", [dict(ranker=1), dict(ranker=2), dict(ranker=3), dict(no_promotion=1),
                                    dict(ranker=1, no_promotion=1), dict(ranker=3, window=64, bits=4)])
def test_alternative_rankers_and_no_promotion(lib, policy):
    """QEvict App. J rankers (decayed attention, p-norm, key norm) and App. K's no-promotion policy:
    rank values, tiers, codes and counters in lockstep with the oracle."""
    base = synth.workload("tiny_4k", prompt_len=1500, steps=24, n_plant=4, kappa=6.0, key_lognormal_sigma=0.5)
    ls = _run(base.replace(**policy), 24)
    if policy.get("no_promotion"):
        assert ls.cache.counters()["promotions"] == 0


@pytest.mark.parametrize("fmt", [dict(), dict(window=64, bits=4, prompt_len=3000), dict(h_q=16, h_kv=2, n_sink=16, batch=2, n_recent=64)])
def test_rope_domain_keys(lib, fmt):
    """QEvict §4.3 "Cache Execution": the keys carry RoPE; Quantized keys are stored before it and
    rotated back to their positions after dequantisation, in attention and on promotion.  Codes,
    parameters and promoted bf16 windows bit-exact, outputs and masses within tolerance; forced score
    churn moves windows both ways."""
    base = synth.workload("tiny_4k", prompt_len=1500, steps=32, n_plant=4, kappa=6.0, rope_base=10000.0)
    ls = _run(base.replace(**fmt), 32, churn=7)
    c = ls.cache.counters()
    assert c["promotions"] > 0 and c["demotions"] > 0 and c["first_quant"] > 0


def test_rope_table_rules(lib):
    """The RoPE table is required before the first prefill of a rope cache, and refused for a cache
    without RoPE, with too few rows, or after a prefill."""
    wl = synth.workload("tiny_4k", prompt_len=600, steps=16, n_plant=2, budget_num=60, rope_base=10000.0)
    table = torch.from_numpy(synth.rope_table(wl.max_len, wl.rope_base)).cuda()
    p = synth.prompt_inputs(wl, 0, 0)
    s0 = torch.rand(1, O.prompt_windows(O.Config.from_obj(wl)), device="cuda")
    plain = binding.Cache(binding.make_config(wl, rope=0))
    with pytest.raises(binding.QEvictError) as e:
        plain.set_rope_table(table)
    assert e.value.status == binding.EINVAL
    c = binding.Cache(binding.make_config(wl))
    with pytest.raises(binding.QEvictError) as e:
        c.set_rope_table(table[:wl.max_len - 1].contiguous())
    assert e.value.status == binding.EINVAL
    with pytest.raises(binding.QEvictError) as e:
        c.prefill_route(0, p["k"][None].cuda(), p["v"][None].cuda(), s0=s0)
    assert e.value.status == binding.ESCHEDULE
    c.set_rope_table(table)
    c.prefill_route(0, p["k"][None].cuda(), p["v"][None].cuda(), s0=s0)
    with pytest.raises(binding.QEvictError) as e:
        c.set_rope_table(table)
    assert e.value.status == binding.ESCHEDULE
    c.check()


def test_prefill_scores_at_32k(lib):
    """The tensor-core prefill passes over a full 32K prompt: one KV head with its group of four query
    heads (the group shape of the Llama-3-8B layout, planted windows included) against the oracle's
    fp64 causal attention, window by window."""
    wl = synth.workload("llama8b_32k", n_layers=1, h_q=4, h_kv=1)
    cache = binding.Cache(binding.make_config(wl))
    ins = synth.prompt_inputs(wl, 0, 0)
    npw = O.prompt_windows(O.Config.from_obj(wl))
    s0 = torch.empty(1, npw, dtype=torch.float32, device="cuda")
    cache.prefill_scores(ins["q"][None].cuda(), ins["k"][None].cuda(), s0)
    ref = O.prefill_scores(ins["q"].float().numpy(), ins["k"].float().numpy(), O.Config.from_obj(wl))
    close_rel(s0.cpu().numpy()[0], ref, "32K prefill window scores")


def test_minimal_prompt_until_the_cache_is_full(lib):
    """A prompt of n_sink + 1 tokens (no historical window at prefill) decoded until T = max_len: every
    window the cache ever routes ages out of the recent region during decode, and one more step is
    refused."""
    wl = synth.workload("tiny_4k", prompt_len=5, steps=240, n_plant=0, budget_num=4000)
    ls = _run(wl, 240)
    assert ls.bud.k_q > 0 and ls.cache.counters()["aged_quant"] > 0
    q = torch.zeros(1, wl.h_q, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(1, wl.h_kv, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.QEvictError) as e:
        ls.cache.decode_step(0, q, kv, kv, torch.empty_like(q))
    assert e.value.status == binding.ESCHEDULE


def test_two_tier_and_quantized_only(lib):
    """q = 0: Full/Evicted only (two-tier window eviction); q = 1: K_f = 0 (quantised retention)."""
    base = synth.workload("tiny_4k", prompt_len=1200, steps=16, n_plant=4)
    ls = _run(base.replace(q_num=0), 16)
    assert ls.bud.k_q == 0
    ls = _run(base.replace(q_num=100), 16)
    assert ls.bud.k_f == 0


def test_budget_above_full_is_dense_attention(lib):
    """B_total >= the full cache with K_f >= every window: the step is dense softmax attention (torch SDPA)."""
    wl = synth.workload("tiny_4k", prompt_len=700, steps=16, q_num=0, budget_num=400, n_plant=2)
    ls = Lockstep(wl)
    ls.prefill()
    pk = synth.prompt_inputs(wl, 0, 0)
    K = [pk["k"].float()]
    V = [pk["v"].float()]
    dec = synth.decode_inputs(wl, 0, 0)
    for s in range(16):
        K.append(dec["k"][s:s + 1].float())
        V.append(dec["v"][s:s + 1].float())
        q = dec["q"][s:s + 1].cuda()
        out = torch.empty(1, wl.h_q, 128, dtype=torch.bfloat16, device="cuda")
        ls.cache.decode_step(0, q, dec["k"][s:s + 1].cuda(), dec["v"][s:s + 1].cuda(), out)
        Kt = torch.cat(K).cuda().permute(1, 0, 2).repeat_interleave(wl.h_q // wl.h_kv, 0)
        Vt = torch.cat(V).cuda().permute(1, 0, 2).repeat_interleave(wl.h_q // wl.h_kv, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(q[0].float()[:, None, :], Kt, Vt)[:, 0, :]
        assert (out[0].float() - ref).abs().max().item() <= OUT_TOL
        if (s + 1) % wl.omega == 0:
            ls.cache.route()
    torch.cuda.synchronize()
    st = ls.cache.region("state", 0, ls.N).cpu().numpy() & 3
    assert not np.any(st == O.EVICTED) and not np.any(st == O.QUANT)


def test_router_at_window_capacity(lib):
    """The largest unit the router sorts in one CTA: 8192 windows (a 262K-token context at W = 32).
    Prefill routing over every prompt window and one routing event, in lockstep with the oracle: the
    tier states, slots, tables and ledgers of all 8192 windows, every output and every window mass."""
    wl = synth.workload("tiny_4k", prompt_len=262148 - 8, steps=8, n_plant=8, kappa=6.0, budget_num=20)
    assert binding.budget(binding.make_config(wl)).n_windows == 8192
    ls = _run(wl, 8, oracle_prefill_scores=False)
    assert ls.max_out_err <= OUT_TOL


def test_full_size_llama_shape(lib):
    """The 32K Llama-3-8B-shaped workload in the bench's launch configuration (batch 1, 8 KV heads),
    two layers, 16 steps and 2 routing events, every output and window compared."""
    wl = synth.workload("llama8b_32k", n_layers=2, steps=16)
    ls = _run(wl, 16, oracle_prefill_scores=False)
    assert ls.max_out_err <= OUT_TOL


@pytest.mark.parametrize("name,over,steps,state_seqs", [
    # 16 sequences of the 32K shape: 128 (sequence, KV head) units, 2 splits each
    ("batched_32k", dict(n_layers=1, steps=8), 8, "ends"),
    # 131K prompt, lognormal per-window key scales (INT2, 20%, q = 0.7): outputs, masses and the
    # transition counters of every unit every step; the full state (4091 windows: tiers, slots,
    # tables, every ledger record and Full window) of the first sequence after prefill and routing
    ("long_131k", dict(n_layers=1, batch=2, steps=8), 8, [0]),
    # random-walk queries, 12.5% budget, 256 recent tokens, batch 8: three routing events
    ("drift_16k", dict(n_layers=1, steps=24), 24, "ends"),
    # the 131K point in the INT4 / 64-token-window format
    ("long_131k", dict(n_layers=1, batch=1, steps=8, window=64, bits=4), 8, None),
    # pre-RoPE Quantized keys at positions up to 131K (RoPE base 500000)
    ("long_131k", dict(n_layers=1, batch=1, steps=8, rope_base=500000.0), 8, None),
    # the corners of the budget x q sweep at 131K: 10% with q = 0.9 (the most Quantized-heavy point,
    # full state checked) and 40% with q = 0.5 (the most Full-heavy)
    ("long_131k", dict(n_layers=1, batch=1, steps=8, budget_num=10, q_num=90), 8, [0]),
    ("long_131k", dict(n_layers=1, batch=1, steps=8, budget_num=40, q_num=50), 8, None),
])
def test_full_size_workloads(lib, name, over, steps, state_seqs):
    """The other workloads at their full per-layer shapes (one layer each), in lockstep: outputs,
    window masses, scores and counters of every sequence; the full state of the listed sequences
    ("ends": the first, middle and last)."""
    wl = synth.workload(name, **over)
    if state_seqs == "ends":
        state_seqs = sorted({0, wl.batch // 2, wl.batch - 1})
    ls = _run(wl, steps, oracle_prefill_scores=False, check_state=state_seqs is not None,
              state_seqs=state_seqs or [])
    assert ls.max_out_err <= OUT_TOL


@pytest.mark.parametrize("name,over,steps", [
    # the bench's launch configuration: batch 1, 8 KV heads, 19 splits per head on 152 SMs
    ("llama8b_32k", dict(n_layers=2, steps=16), 16),
    # 16 sequences: 128 (sequence, KV head) units
    ("batched_32k", dict(n_layers=1, steps=8), 8),
])
def test_full_size_deferred_score_flush(lib, name, over, steps):
    """The production score path at full size (QEvict §4.2 Eq. (1), read as an update that the
    router absorbs): every decode step records its window masses in its own step slot, and only the
    routing event's flush adds them to the scores, step by step.  At every routing event the scores
    of every window of every unit equal the oracle's per-step cumulative scores; outputs are compared
    every step and the full state after each event."""
    wl = synth.workload(name, **over)
    ls = _run(wl, steps, oracle_prefill_scores=False, per_step=False, state_seqs=sorted({0, wl.batch - 1}))
    assert ls.max_out_err <= OUT_TOL


def test_status_codes(lib):
    wl = synth.workload("tiny_4k", prompt_len=600, steps=16, n_plant=2, budget_num=60)
    cfg = binding.make_config(wl)
    small = binding.make_config(wl, budget_num=1, budget_den=1000)
    with pytest.raises(binding.QEvictError) as e:
        binding.budget(small)
    assert e.value.status == binding.EBUDGET
    with pytest.raises(binding.QEvictError) as e:
        binding.Cache(cfg, arena=torch.empty(1024, dtype=torch.uint8, device="cuda"))
    assert e.value.status == binding.ENOMEM
    with pytest.raises(binding.QEvictError) as e:
        binding.budget(binding.make_config(wl, d_head=64))
    assert e.value.status == binding.EINVAL
    c = binding.Cache(cfg)
    q = torch.zeros(1, wl.h_q, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(1, wl.h_kv, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(binding.QEvictError) as e:     # decode before prefill
        c.decode_step(0, q, kv, kv, out)
    assert e.value.status == binding.ESCHEDULE
    # q one bf16 element off a 4-byte boundary: refused on the host, nothing is launched
    qbuf = torch.zeros(1 + wl.h_q * 128, dtype=torch.bfloat16, device="cuda")
    q_odd = qbuf[1:].view(1, wl.h_q, 128)
    assert q_odd.data_ptr() % 4 == 2
    with pytest.raises(binding.QEvictError) as e:
        c.decode_step(0, q_odd, kv, kv, out)
    assert e.value.status == binding.EINVAL
    p = synth.prompt_inputs(wl, 0, 0)
    s0 = torch.rand(1, O.prompt_windows(O.Config.from_obj(wl)), device="cuda")
    c.prefill_route(0, p["k"][None].cuda(), p["v"][None].cuda(), s0=s0)
    with pytest.raises(binding.QEvictError) as e:     # prefill twice
        c.prefill_route(0, p["k"][None].cuda(), p["v"][None].cuda(), s0=s0)
    assert e.value.status == binding.ESCHEDULE
    with pytest.raises(binding.QEvictError) as e:     # route off the Omega cadence
        c.route()
    assert e.value.status == binding.ESCHEDULE
    for _ in range(wl.omega):
        c.decode_step(0, q, kv, kv, out)
    with pytest.raises(binding.QEvictError) as e:     # a routing event is due
        c.decode_step(0, q, kv, kv, out)
    assert e.value.status == binding.ESCHEDULE
    c.route()
    c.decode_step(0, q, kv, kv, out)
    c.check()


def test_slot_exhaustion_guard(lib):
    """Failure detection of the router's slot allocation (QEvict App. A Algorithm 1): with a host-set
    cap that hides free slots, a routing event whose newcomers need more F or ledger slots than it sees
    records the failure (qevict_check returns QEVICT_EDEVICE) and leaves every tier, slot, table and
    ledger record as it was; the pending masses are still absorbed.  No GPU fault is involved."""
    wl = synth.workload("tiny_4k", prompt_len=1200, steps=24, n_plant=4)
    ls = Lockstep(wl)
    ls.prefill()
    ls.decode(3 * wl.omega - 1)   # the event after step 24 is the first one with a newly aged window
    one = ls.dec[(0, 0)]
    s = ls.step
    out = torch.empty(1, wl.h_q, 128, dtype=torch.bfloat16, device="cuda")
    ls.cache.decode_step(0, one["q"][s][None].cuda(), one["k"][s][None].cuda(), one["v"][s][None].cuda(), out)
    torch.cuda.synchronize()
    u, N = 0, ls.N
    regions = {"state": N, "fslot": 4 * N, "lslot": 4 * N, "ftab": 8 * max(1, min(ls.bud.k_f, N)),
               "qtab": 8 * max(1, min(ls.bud.k_q, N)), "ledger": ls.lay.stride_ledger, "fpool": ls.lay.stride_fpool}
    before = {k: ls.cache.region(k, u, n).clone() for k, n in regions.items()}
    meta_before = ls.meta(0, 0).copy()
    # a window ages out of the recent region at this event; ranked first, it enters F and needs an F
    # slot, which the cap hides
    aged = int(meta_before[1])
    assert O.n_hist(int(meta_before[0]), ls.ocfg) > aged
    ls.cache.region("score", u, 4 * wl.h_kv * N).view(torch.float32)[aged] = 1e6
    ls.cache.debug_cap_free_slots(0)
    ls.cache.route()
    with pytest.raises(binding.QEvictError) as e:
        ls.cache.check()
    assert e.value.status == binding.EDEVICE
    assert ls.cache.status_word() == 2                           # the slot bit alone
    for k, t in before.items():
        assert torch.equal(ls.cache.region(k, u, regions[k]), t), k
    m = ls.meta(0, 0)
    assert m[1] == meta_before[1] and m[2] == meta_before[2] and m[3] == meta_before[3]   # windows routed, |F|, |Q|
    ls.cache.debug_cap_free_slots(-1)
    with pytest.raises(binding.QEvictError):
        ls.cache.debug_cap_free_slots(-2)


def test_wait_timeout_is_reported_and_recoverable(lib):
    """Failure detection without a GPU fault: a bounded wait that runs out (an mbarrier phase that
    nothing completes) records a timeout in the device status word and returns.  qevict_check and
    qevict_read_counters then report QEVICT_EDEVICE, the rest of the cache is untouched, and
    importing a state exported before the timeout resumes the run in lockstep with the oracle."""
    wl = synth.workload("tiny_4k", prompt_len=1200, steps=24, n_plant=4)
    ls = Lockstep(wl)
    ls.prefill()
    ls.decode(8)
    snap = ls.cache.export_state()
    ls.cache.selftest_wait()
    for call in (ls.cache.check, ls.cache.counters):
        with pytest.raises(binding.QEvictError) as e:
            call()
        assert e.value.status == binding.EDEVICE
    assert ls.cache.status_word() == 1                           # the timeout bit alone
    after = ls.cache.export_state()
    diff = np.flatnonzero(snap != after)
    # one byte changed: the low byte of the status word, 0 -> the timeout bit
    assert diff.size == 1 and int(snap[diff[0]]) == 0 and int(after[diff[0]]) == 1, diff
    ls.cache.import_state(snap)
    ls.cache.check()
    ls.decode(16)                                               # two more routing events
    got, want = ls.counters()
    assert got == want, (got, want)


@pytest.mark.parametrize("rope_base", [0.0, 10000.0])
def test_tuple_views_and_checkpoint(lib, rope_base):
    """qevict_get_tuple points at each unit's regions; an exported cache imported into a fresh arena
    resumes the run: the same next steps and routing event as the original cache (with pre-RoPE keys,
    the RoPE table travels inside the arena)."""
    wl = synth.workload("tiny_4k", prompt_len=1200, steps=32, n_plant=4, batch=2, rope_base=rope_base)
    ls = Lockstep(wl)
    ls.prefill()
    ls.decode(10)                      # one routing event, then two steps with pending masses
    cache, lay = ls.cache, ls.cache.layout
    base = cache.arena.data_ptr()
    for layer in range(wl.n_layers):
        for b in range(wl.batch):
            t = cache.tuple(layer, b)
            u = layer * wl.batch + b
            for name, region in (("sink", "sink"), ("ring", "ring"), ("fpool", "fpool"), ("ledger", "ledger"),
                                 ("score", "score"), ("state", "state"), ("f_slot", "fslot"), ("l_slot", "lslot"),
                                 ("f_table", "ftab"), ("q_table", "qtab"), ("meta", "meta")):
                assert getattr(t, name) == base + getattr(lay, f"off_{region}") + u * getattr(lay, f"stride_{region}")
    snap = cache.export_state()
    twin = binding.Cache(ls.cfg)
    twin.import_state(snap)
    assert np.array_equal(twin.export_state(), snap)
    with pytest.raises(binding.QEvictError):   # a different configuration is refused
        other = binding.Cache(binding.make_config(wl.replace(omega=4)))
        other.import_state(snap)
    # both caches take the same six steps (a routing event after the sixth)
    outs = {}
    for name, c in (("orig", cache), ("twin", twin)):
        res = []
        for s in range(10, 16):
            for layer in range(wl.n_layers):
                d = [ls.dec[(layer, b)] for b in range(wl.batch)]
                q = torch.stack([x["q"][s] for x in d]).cuda()
                k = torch.stack([x["k"][s] for x in d]).cuda()
                v = torch.stack([x["v"][s] for x in d]).cuda()
                out = torch.empty(wl.batch, wl.h_q, 128, dtype=torch.bfloat16, device="cuda")
                c.decode_step(layer, q, k, v, out)
                res.append(out.float().cpu())
        c.route()
        torch.cuda.synchronize()
        outs[name] = torch.stack(res)
    assert (outs["orig"] - outs["twin"]).abs().max().item() <= 1e-2
    for region in ("state", "fslot", "lslot", "ftab", "qtab", "meta"):
        n = getattr(lay, f"stride_{region}")
        for u in range(wl.n_layers * wl.batch):
            assert torch.equal(cache.region(region, u, n), twin.region(region, u, n)), region
