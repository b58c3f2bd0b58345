"""The allocation-free prefill-scoring entry point (qevict_prefill_scores_noalloc).

Callers that cannot allocate device memory (a framework owning every byte through its pool, a
plugin given only its inputs and outputs) use this entry point; its scratch is a fixed array in the
library image.  It must return what the cache-based qevict_prefill_scores returns, on consecutive
calls that reuse the same scratch.  This file is collected last so that a stop-at-first-failure run
has already run every other test.
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
    return torch.stack([x["q"] for x in ins]).cuda(), torch.stack([x["k"] for x in ins]).cuda()


def test_noalloc_scores_match_the_cache_entry_point_on_consecutive_calls(lib):
    wl = synth.workload("tiny_4k", batch=2, prompt_len=3000, n_sink=5, n_plant=4)
    npw = O.prompt_windows(O.Config.from_obj(wl))
    cache = binding.Cache(binding.make_config(wl))
    for layer in (0, 1):                      # two calls in a row, different inputs, one shared scratch
        q, k = _prompt(wl, layer)
        ref = torch.empty(wl.batch, npw, dtype=torch.float32, device="cuda")
        got = torch.full((wl.batch, npw), float("nan"), dtype=torch.float32, device="cuda")
        cache.prefill_scores(q, k, ref)
        binding.prefill_scores_noalloc(wl.batch, wl.prompt_len, wl.h_q, wl.h_kv, wl.n_sink, wl.window, q, k, got)
        torch.cuda.synchronize()
        close_rel(got.cpu().numpy(), ref.cpu().numpy(), f"call {layer + 1}")
        assert np.isfinite(got.cpu().numpy()).all()


def test_noalloc_rejects_requests_above_its_scratch(lib):
    q = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    with pytest.raises(binding.QEvictError) as e:          # 2 * 1 * 32 * 40000 floats > 2 Mi
        binding.prefill_scores_noalloc(1, 40000, 32, 8, 4, 32, q, q, out)
    assert e.value.status == binding.ENOMEM
