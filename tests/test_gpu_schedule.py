"""Steps planned by the host block manager, run through the C ABI and
checked against the oracle at every step.

The schedule is Figure 3 of "vLLM engine anatomy" ("V1: unified
scheduling": R1..R4 with prompts of 40, 20, 16 and 4 tokens, prompt chunks of
at most 16 tokens, prefill chunks and decodes in the same step), followed by
a request that hits R1's cached prefix blocks ("01. vLLM", prefix caching)
and a fork whose shared partial block is copied before the write
("PagedAttention", copy-on-write).  Each step runs pa_copy_blocks, then
pa_reshape_and_cache of the step's new tokens, then pa_attention; the
oracle runs the same three operations on its own copy of the caches.  The
K and V of a token are a seeded function of (token id, position), as a
token's K/V are fixed by its prefix: a prefix hit then reads the same values
a recomputation would write.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_82_gb300 as pa
from paged_kv_cache_82_gb300.block_manager import KVCacheManager, Scheduler
from paged_kv_cache_82_gb300.metadata import build_step_metadata
from tests._gpu_step import assert_close, cache_bits, oracle_cache_bits

pytestmark = pytest.mark.gpu

HQ, HKV, D, NB = 32, 8, 128, 64


def _kv_rows(tokens, positions, which):
    out = np.empty((len(tokens), HKV, D), dtype=np.float32)
    for i, (t, p) in enumerate(zip(tokens, positions)):
        out[i] = np.random.default_rng([82100, which, int(t), int(p)]
                                       ).standard_normal((HKV, D))
    return torch.from_numpy(out).to(torch.bfloat16)


def _tokens(seed, n):
    return np.random.default_rng(seed).integers(0, 32000, size=n).tolist()


def test_block_manager_schedule_through_the_kernels():
    kv = KVCacheManager(NB)
    sched = Scheduler(kv, token_budget=2048, long_prefill_threshold=16)
    arrivals = {1: ("R1", _tokens(1, 40), 4), 2: ("R2", _tokens(2, 20), 3),
                3: ("R3", _tokens(3, 16), 4), 4: ("R4", _tokens(4, 4), 9)}
    # step 8: R5 shares R1's first 32 tokens (two full cached blocks)
    arrivals[8] = ("R5", _tokens(1, 40)[:32] + _tokens(5, 30), 3)
    shape = (NB, HKV, 16, D)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16)
    vc = torch.full(shape, float("nan"), dtype=torch.bfloat16)
    kg, vg = kc.cuda(), vc.cuda()
    ko = oracle._as_np(kc)[0].copy()
    vo = oracle._as_np(vc)[0].copy()
    rng = np.random.default_rng(82101)
    seen_kinds = set()
    for step in range(1, 15):
        if step in arrivals:
            sched.add_request(*arrivals[step])
        if step == 10:
            # parallel sampling: R4 gets a sibling that shares its blocks and
            # has sampled a different token
            child = sched.fork("R4", "R4b")
            child.token_ids[-1] = 31999
        plan = sched.schedule()
        if not plan.requests:
            continue
        md = build_step_metadata(plan.requests)
        key = _kv_rows(plan.new_token_ids, plan.new_positions, 0)
        value = _kv_rows(plan.new_token_ids, plan.new_positions, 1)
        T = len(plan.new_token_ids)
        q = torch.from_numpy(rng.standard_normal((T, HQ, D)).astype(
            np.float32)).to(torch.bfloat16)
        slots = torch.from_numpy(md["slot_mapping"])
        # GPU: copies, writes, attention
        if plan.copy_pairs:
            pa.pa_copy_blocks(kg, vg, torch.tensor(plan.copy_pairs).cuda())
            seen_kinds.add("cow")
        pa.pa_reshape_and_cache(key.cuda(), value.cuda(), kg, vg, slots.cuda())
        out = pa.pa_attention(
            q.cuda(), kg, vg, torch.from_numpy(md["block_tables"]).cuda(),
            torch.from_numpy(md["seq_lens"]).cuda(),
            torch.from_numpy(md["query_start_loc"]).cuda(),
            md["max_query_len"], md["max_seq_len"], D ** -0.5)
        assert pa.pa_get_device_error() == 0, f"step {step}"
        # oracle: the same operations on its own caches
        if plan.copy_pairs:
            oracle.copy_blocks(ko, vo, np.asarray(plan.copy_pairs),
                               cache_dtype="bf16")
        oracle.reshape_and_cache(key, value, ko, vo, md["slot_mapping"],
                                 cache_dtype="bf16")
        ref = oracle.paged_attention(q, ko, vo, md["block_tables"],
                                     md["seq_lens"], md["query_start_loc"],
                                     scale=D ** -0.5, cache_dtype="bf16")
        assert np.array_equal(cache_bits(kg), oracle_cache_bits(ko)), step
        assert np.array_equal(cache_bits(vg), oracle_cache_bits(vo)), step
        assert_close(out, ref, md, "bf16", "bf16")
        if any(r.num_new > 1 for r in plan.requests):
            seen_kinds.add("prefill")
        if any(r.num_new == 1 for r in plan.requests):
            seen_kinds.add("decode")
        if any(r.request_id == "R5" and r.num_computed == 32
               for r in plan.requests):
            seen_kinds.add("prefix_hit")
        sched.update(plan, {r: int(rng.integers(0, 32000))
                            for r in plan.scheduled})
    assert seen_kinds == {"cow", "prefill", "decode", "prefix_hit"}
