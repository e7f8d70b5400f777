"""GPU parity at the full sizes of the serving workloads, in the launch
configuration the benchmark times (one fused kvi_retrieve_and_inject call
over all requests).

At these sizes the oracle checks everything: every request's selected ids
(bit-exact), scores and placements; every injected token's rows -- all
layers and heads, K within the rotation tolerance and V bit-exact -- element
by element (the oracle's check_rows over chunks read back from the device,
on all host cores); and, for the whole pool, that exactly the rows the
oracle's placement maps tokens to were written in every layer and every
other row kept its canary.

Workloads ("InferScale: GPU-Native KV Injection for Personalized LLM
Serving" serving setting, synthetic stand-ins for its LoCoMo stores):
Llama-3-8B KV geometry with 10k facts (k = 5..50); 64 concurrent requests
over their own 5k-fact stores (k = 5..50); Mistral-7B geometry with 50k
facts of 8-128 tokens placed at random bases up to 32k (theta 1e6);
Llama-3-70B geometry, 256 requests, pool of about 150 GB.
"""
import gc

import numpy as np
import pytest
import torch

from tests import kvi_check as kc
from tests import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    kc.ensure_built()


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _run_and_check(b, k, label):
    f = kc.Fused(b, k)
    f()
    ids, scores, pos, status = f.results()
    assert status == 0, f"device status {status}"
    orc = kc.oracle_select(b, k)
    kc.check_selection(ids, scores, pos, orc)
    place = kc.placements_from_oracle(orc)
    n_tok, n_el, _ = kc.check_pool_exhaustive(b, place, label=label)
    assert n_tok == sum(T for (_s, _sel, _p, T) in orc)
    kc.check_canaries_by_row(b, place)
    return n_el


def test_llama3_8b_10k_k_sweep():
    b = synth.build_workload(synth.WORKLOADS["llama3_8b_10k"])
    try:
        for k in (5, 10, 20, 50):
            synth.fill_canary(b.pool)
            _run_and_check(b, k, f"llama3_8b_10k k={k}")
    finally:
        del b
        _free()


def test_concurrent_64x5k_k_sweep():
    b = synth.build_workload(synth.WORKLOADS["concurrent_64x5k"])
    try:
        for k in (5, 10, 20, 50):
            synth.fill_canary(b.pool)
            _run_and_check(b, k, f"concurrent_64x5k k={k}")
    finally:
        del b
        _free()


def test_mistral_long_placement_50k():
    b = synth.build_workload(synth.WORKLOADS["mistral_long_50k"])
    try:
        assert int(b.start_pos[0]) < 32768
        _run_and_check(b, 50, "mistral_long_50k k=50")
    finally:
        del b
        _free()


def test_llama3_70b_capacity_256_requests():
    w = synth.WORKLOADS["llama3_70b_capacity"]
    b = synth.build_workload(w, with_pool=False)
    try:
        # block tables sized to each request's injected tokens, as an engine
        # allocates them once it knows how many memory tokens it will receive
        orc = kc.oracle_select(b)
        synth.attach_pool(b, tokens_needed=[T for (_s, _sel, _p, T) in orc])
        assert b.pool.numel() * 2 > 140e9
        _run_and_check(b, 50, "llama3_70b_capacity k=50")
    finally:
        del b
        _free()
