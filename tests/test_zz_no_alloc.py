"""The allocation-free prefill-scoring entry point (qevict_prefill_scores_noalloc).

Callers that cannot allocate device memory (a framework owning every byte through its pool, a
plugin given only its inputs and outputs) use this entry point; its scratch is a fixed array in the
library image.  Its window scores must match the oracle's prompt attention (QEvict §4.2) and be
identical to those of the cache-based qevict_prefill_scores (the same kernels), on consecutive calls
that reuse the same scratch, including a call that fills the scratch exactly.  This file is collected
last so that a stop-at-first-failure run has already run every other test.
"""
import numpy as np
import pytest
import torch

from gpu_lockstep import close_rel
from oracle import qevict_oracle as O
from recoverable_quantized_kv_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def _prompt(wl, layer):
    ins = [synth.prompt_inputs(wl, b, layer) for b in range(wl.batch)]
    return ins, torch.stack([x["q"] for x in ins]).cuda(), torch.stack([x["k"] for x in ins]).cuda()


def _noalloc(wl, q, k, out):
    binding.prefill_scores_noalloc(wl.batch, wl.prompt_len, wl.h_q, wl.h_kv, wl.n_sink, wl.window, q, k, out)


def test_noalloc_scores_match_the_oracle_on_consecutive_calls(lib):
    wl = synth.workload("tiny_4k", batch=2, prompt_len=3000, n_sink=5, n_plant=4)
    cfg = O.Config.from_obj(wl)
    npw = O.prompt_windows(cfg)
    cache = binding.Cache(binding.make_config(wl))
    for layer in (0, 1):                      # two calls in a row, different inputs, one shared scratch
        ins, q, k = _prompt(wl, layer)
        ref = torch.empty(wl.batch, npw, dtype=torch.float32, device="cuda")
        got = torch.full((wl.batch, npw), float("nan"), dtype=torch.float32, device="cuda")
        cache.prefill_scores(q, k, ref)
        _noalloc(wl, q, k, got)
        torch.cuda.synchronize()
        binding.prefill_scores_noalloc_status()            # no device failure recorded
        assert torch.equal(got, ref), f"call {layer + 1}: differs from qevict_prefill_scores"
        for b in range(wl.batch):
            want = O.prefill_scores(ins[b]["q"].float().numpy(), ins[b]["k"].float().numpy(), cfg)
            close_rel(got[b].cpu().numpy(), want, f"call {layer + 1} seq {b} against the oracle")


def test_noalloc_call_that_fills_the_scratch(lib):
    """2 * batch * h_q * prompt_len == QEVICT_NOALLOC_SCRATCH_FLOATS: one 32K prompt with 32 query heads
    (the Llama-3-8B layer), so the end of the column-sum region is written and read.  Identical to the
    cache entry point; every prompt query's mass lands on the windows or the sinks."""
    wl = synth.workload("llama8b_32k", n_layers=1)
    assert 2 * wl.batch * wl.h_q * wl.prompt_len == 2 * 1024 * 1024
    _, q, k = _prompt(wl, 0)
    npw = O.prompt_windows(O.Config.from_obj(wl))
    ref = torch.empty(1, npw, dtype=torch.float32, device="cuda")
    got = torch.full((1, npw), float("nan"), dtype=torch.float32, device="cuda")
    binding.Cache(binding.make_config(wl)).prefill_scores(q, k, ref)
    _noalloc(wl, q, k, got)
    torch.cuda.synchronize()
    binding.prefill_scores_noalloc_status()
    assert torch.equal(got, ref)
    total = got.double().sum().item()
    assert 0 < wl.prompt_len - total < 0.01 * wl.prompt_len


def test_noalloc_rejects_bad_requests(lib):
    q = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(binding.QEvictError) as e:          # 2 * 1 * 32 * 40000 floats > 2 Mi
        binding.prefill_scores_noalloc(1, 40000, 32, 8, 4, 32, q, q, out)
    assert e.value.status == binding.ENOMEM
    with pytest.raises(binding.QEvictError) as e:          # s0_out off its 4-byte boundary
        binding.prefill_scores_noalloc(1, 64, 4, 1, 4, 32, q, q, out.view(torch.uint8)[1:])
    assert e.value.status == binding.EINVAL
