"""CPU checks of the host block manager and step planner against what the
pages fix: the Figure 3 schedule ("vLLM engine anatomy", "V1: unified
scheduling"), the Figure 2 layout, the 2,000-token prefix = 125 blocks ("01.
vLLM", prefix caching), the hash-chain rules (full blocks only, parent in the
hash, salt in the first block only, lookup stops at the first miss), the LRU
free queue (head out, tail in, O(1) removal from the middle), reference
counts, preemption by recompute, and copy-on-write of a shared block.
"""
import json
import os

import numpy as np
import pytest

from paged_kv_cache_82_gb300.block_manager import (BLOCK_SIZE, BlockPool,
                                                   FreeBlockQueue, KVBlock,
                                                   KVCacheManager, Scheduler,
                                                   hash_block)
from paged_kv_cache_82_gb300.metadata import build_step_metadata

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tokens(seed, n):
    return np.random.default_rng(seed).integers(0, 32000, size=n).tolist()


def run_figure3(sched_kwargs=None):
    """Requests R1..R4 of Figure 3 (prompts of 40, 20, 16 and 4 tokens)
    arrive one per step; prompt chunks are capped at 16 tokens.  Output
    lengths 4, 3, 4 and 5 end R1 and R3 after step 6, R2 after step 5."""
    kv = KVCacheManager(64)
    sched = Scheduler(kv, token_budget=2048, long_prefill_threshold=16,
                      **(sched_kwargs or {}))
    prompts = {"R1": 40, "R2": 20, "R3": 16, "R4": 4}
    outs = {"R1": 4, "R2": 3, "R3": 4, "R4": 5}
    rng = np.random.default_rng(5)
    steps = []
    for step in range(1, 9):
        rid = f"R{step}"
        if rid in prompts:
            sched.add_request(rid, _tokens(step, prompts[rid]), outs[rid])
        plan = sched.schedule()
        steps.append(plan)
        sched.update(plan, {r: int(rng.integers(0, 32000))
                            for r in plan.scheduled})
    return steps, sched


def test_figure3_schedule():
    steps, sched = run_figure3()
    got = [plan.scheduled for plan in steps]
    assert got[:7] == [
        {"R1": 16},
        {"R1": 16, "R2": 16},
        {"R1": 8, "R2": 4, "R3": 16},
        {"R1": 1, "R2": 1, "R3": 1, "R4": 4},      # three decodes + a prefill
        {"R1": 1, "R2": 1, "R3": 1, "R4": 1},
        {"R1": 1, "R3": 1, "R4": 1},               # R2 has left
        {"R4": 1},                                 # R1, R3 have left
    ]
    # prompt chunks cover tokens 0-15, 16-31, 32-39 (R1) and 0-15, 16-19 (R2)
    r1 = [r for p in steps[:3] for r in p.requests if r.request_id == "R1"]
    assert [(r.num_computed, r.num_new) for r in r1] == [(0, 16), (16, 16),
                                                         (32, 8)]
    assert [s.request_id for s in sched.finished] == ["R2", "R1", "R3",
                                                      "R4"]
    # every block went back to the pool
    assert sched.kv.pool.num_free == 64


def test_figure2_layout_and_next_slots():
    # A with 40 tokens and B with 20 on a fresh pool: blocks [0,1,2] and
    # [3,4]; their next tokens land in slots 40 and 68
    g = json.load(open(os.path.join(GOLDEN, "fig2_layout.json")))
    kv = KVCacheManager(12)
    sched = Scheduler(kv, token_budget=4096)
    sched.add_request("A", _tokens(1, 40), 2)
    sched.add_request("B", _tokens(2, 20), 2)
    plan = sched.schedule()
    tables = {r.request_id: r.block_ids for r in plan.requests}
    assert tables == {k: g["sequences"][k]["block_table"] for k in "AB"}
    free = [b.block_id for b in kv.pool.free_queue]
    assert free == g["free_blocks"]
    sched.update(plan, {"A": 7, "B": 9})
    plan = sched.schedule()
    md = build_step_metadata(plan.requests)
    assert md["slot_mapping"].tolist() == [g["next_token_slot"]["A"],
                                           g["next_token_slot"]["B"]]


def test_shared_prefix_of_2000_tokens_hits_125_blocks():
    kv = KVCacheManager(1024)
    sched = Scheduler(kv, token_budget=8192)
    prefix = _tokens(10, 2000)
    sched.add_request("first", prefix + _tokens(11, 37), 1)
    plan = sched.schedule()
    sched.update(plan, {"first": 1})
    sched.add_request("second", prefix + _tokens(12, 500), 1)
    plan = sched.schedule()
    second = plan.requests[-1]
    assert second.num_computed == 2000 == 125 * BLOCK_SIZE
    assert second.num_new == 500
    first_blocks = sched.finished[0].blocks  # freed, but kept as cache
    assert first_blocks == []
    # the hit blocks are exactly the first request's prefix blocks
    assert second.block_ids[:125] == plan_first_blocks(kv, prefix)


def plan_first_blocks(kv, prefix):
    hashes, parent = [], None
    for k in range(len(prefix) // 16):
        parent = hash_block(parent, prefix[16 * k:16 * (k + 1)])
        hashes.append(parent)
    return [kv.pool.lookup(h).block_id for h in hashes]


def test_only_full_blocks_are_cached_and_the_last_token_runs():
    kv = KVCacheManager(64)
    sched = Scheduler(kv, token_budget=4096)
    p = _tokens(20, 40)                      # 2 full blocks + 8 tokens
    sched.add_request("a", p, 1)
    sched.update(sched.schedule(), {"a": 1})
    assert len(kv.pool.cached) == 2          # the partial tail is not cached
    # the same 40-token prompt again: 2 blocks hit, the tail recomputed
    sched.add_request("b", p, 1)
    plan = sched.schedule()
    assert (plan.requests[0].num_computed, plan.requests[0].num_new) == (32, 8)
    sched.update(plan, {"b": 1})
    # a 32-token prompt fully cached still computes its last block
    sched.add_request("c", p[:32], 1)
    plan = sched.schedule()
    assert (plan.requests[0].num_computed, plan.requests[0].num_new) == (16, 16)


def test_hash_chain_parent_and_salt():
    a, b = _tokens(30, 16), _tokens(31, 16)
    h_a = hash_block(None, a)
    assert hash_block(None, a) == h_a                       # deterministic
    assert hash_block(h_a, b) != hash_block(None, b)        # parent counts
    assert hash_block(hash_block(None, b), b) != hash_block(h_a, b)
    assert hash_block(None, a, (("salt", "x"),)) != h_a     # extra keys count
    kv = KVCacheManager(64)
    sched = Scheduler(kv, token_budget=4096)
    p = _tokens(32, 48)
    sched.add_request("t1", p + [1], 1, cache_salt="tenant-1")
    sched.update(sched.schedule(), {"t1": 1})
    # another tenant with the same text: no hit anywhere in the chain
    sched.add_request("t2", p + [1], 1, cache_salt="tenant-2")
    plan = sched.schedule()
    assert plan.requests[0].num_computed == 0
    sched.update(plan, {"t2": 1})
    # same tenant: all three full blocks hit
    sched.add_request("t1b", p + [2], 1, cache_salt="tenant-1")
    plan = sched.schedule()
    assert plan.requests[0].num_computed == 48


def test_lookup_stops_at_the_first_miss():
    kv = KVCacheManager(64)
    sched = Scheduler(kv, token_budget=4096)
    p = _tokens(40, 64)
    sched.add_request("a", p + [0], 1)
    sched.update(sched.schedule(), {"a": 1})
    q = list(p)
    q[20] += 1                # block 1 differs: blocks 2, 3 cannot hit
    sched.add_request("b", q + [0], 1)
    plan = sched.schedule()
    assert plan.requests[0].num_computed == 16


def test_free_queue_is_lru_with_o1_removal():
    blocks = [KVBlock(i) for i in range(6)]
    q = FreeBlockQueue(blocks)
    assert [b.block_id for b in q] == [0, 1, 2, 3, 4, 5]
    q.remove(blocks[3])                       # from the middle
    assert [b.block_id for b in q] == [0, 1, 2, 4, 5] and len(q) == 5
    assert q.popleft().block_id == 0           # head out
    q.append(blocks[3])                        # tail in
    assert [b.block_id for b in q] == [1, 2, 4, 5, 3]
    with pytest.raises(RuntimeError):
        q.append(blocks[3])                    # already free
    with pytest.raises(RuntimeError):
        q.remove(blocks[0])                    # not in the queue


def test_refcounts_and_eviction_order():
    pool = BlockPool(4)
    a, b = pool.allocate(), pool.allocate()
    assert (a.block_id, b.block_id, pool.num_free) == (0, 1, 2)
    pool.register(a, b"ha")
    pool.touch(a)
    assert a.ref_cnt == 2
    pool.release(a)
    pool.release(a)                            # ref 0: back at the tail
    assert [x.block_id for x in pool.free_queue] == [2, 3, 0]
    assert pool.lookup(b"ha") is a             # still cached while free
    pool.touch(a)                              # a hit takes it out of the queue
    assert [x.block_id for x in pool.free_queue] == [2, 3]
    pool.release(a)
    pool.release(b)
    # allocation takes the least recently released first: 2, 3, then 0, 1
    got = [pool.allocate().block_id for _ in range(4)]
    assert got == [2, 3, 0, 1]
    assert pool.lookup(b"ha") is None          # reallocated: cache entry gone
    with pytest.raises(RuntimeError):
        pool.allocate()


def test_request_blocks_are_released_tail_first():
    kv = KVCacheManager(8)
    sched = Scheduler(kv, token_budget=4096)
    sched.add_request("a", _tokens(50, 40), 1)
    plan = sched.schedule()
    sched.update(plan, {"a": 1})               # finishes, releases [0, 1, 2]
    assert [b.block_id for b in kv.pool.free_queue][-3:] == [2, 1, 0]


def test_preemption_recomputes_and_hits_its_own_blocks():
    # 6 blocks; two requests fit, the third decode block does not
    kv = KVCacheManager(6)
    sched = Scheduler(kv, token_budget=4096)
    pa_ = _tokens(60, 47)
    pb_ = _tokens(61, 47)
    sched.add_request("a", pa_, 10)
    sched.add_request("b", pb_, 10)
    plan = sched.schedule()
    assert plan.scheduled == {"a": 47, "b": 47}      # 3 blocks each
    b_blocks = plan.requests[1].block_ids
    sched.update(plan, {"a": 1, "b": 2})
    plan = sched.schedule()      # a's 48th token fits its block; b too
    assert plan.scheduled == {"a": 1, "b": 1}
    sched.update(plan, {"a": 3, "b": 4})
    # 49th tokens need a 4th block each: none free, the last joined (b) goes
    plan = sched.schedule()
    assert plan.preempted == ["b"]
    assert plan.scheduled == {"a": 1}
    assert sched.waiting[0].request_id == "b" and sched.waiting[0].num_computed == 0
    sched.update(plan, {"a": 5})
    # b released its blocks tail first, so a's fourth block is b's third
    # (the least recently released); b's first two full blocks stay cached
    a = sched.running[0]
    assert a.blocks[3].block_id == b_blocks[2]
    while sched.running:
        plan = sched.schedule()
        sched.update(plan, {r: 0 for r in plan.scheduled})
    # b comes back: its 49 tokens, 2 blocks of them hit, the rest recomputed
    plan = sched.schedule()
    assert plan.scheduled == {"b": 49 - 32}
    assert plan.requests[0].num_computed == 32
    assert plan.requests[0].block_ids[:2] == b_blocks[:2]


def test_fork_shares_blocks_and_copies_on_write():
    kv = KVCacheManager(16)
    sched = Scheduler(kv, token_budget=4096)
    sched.add_request("p", _tokens(70, 20), 5)      # block 0 full, block 1 partial
    plan = sched.schedule()
    sched.update(plan, {"p": 11})                   # pending token 21 (pos 20)
    child = sched.fork("p", "c")
    child.token_ids[-1] = 12                        # its own sampled token
    parent = sched.running[0]
    assert [b.ref_cnt for b in parent.blocks] == [2, 2]
    plan = sched.schedule()
    # the parent writes first into the shared partial block: it gets a copy
    assert plan.copy_pairs == [(1, 2)]
    tables = {r.request_id: r.block_ids for r in plan.requests}
    assert tables == {"p": [0, 2], "c": [0, 1]}
    assert [b.ref_cnt for b in parent.blocks] == [2, 1]
    assert [b.ref_cnt for b in child.blocks] == [2, 1]
    md = build_step_metadata(plan.requests)
    assert md["slot_mapping"].tolist() == [2 * 16 + 4, 1 * 16 + 4]


def test_planned_steps_are_valid_attention_metadata():
    """Every planned step respects the budget, the per-request bounds
    (0 < S_i <= pending) and gives the metadata builder consistent tables."""
    rng = np.random.default_rng(7)
    kv = KVCacheManager(200)
    sched = Scheduler(kv, token_budget=256, long_prefill_threshold=64)
    shared = _tokens(80, 96)
    for step in range(60):
        if step % 3 == 0 and step < 40:
            p = (shared if rng.random() < 0.5 else []) + _tokens(
                100 + step, int(rng.integers(1, 120)))
            sched.add_request(f"q{step}", p, int(rng.integers(1, 12)))
        plan = sched.schedule()
        assert sum(plan.scheduled.values()) <= 256
        for r in plan.requests:
            assert r.num_new > 0
            L = r.num_computed + r.num_new
            assert len(r.block_ids) == -(-L // 16)
        ids = [b for r in plan.requests for b in r.block_ids]
        assert all(0 <= b < 200 for b in ids)
        if plan.requests:
            md = build_step_metadata(plan.requests)
            assert len(md["slot_mapping"]) == sum(plan.scheduled.values())
            # no two new tokens share a slot
            assert len(set(md["slot_mapping"].tolist())) == len(
                md["slot_mapping"])
        sched.update(plan, {r: int(rng.integers(0, 32000))
                            for r in plan.scheduled})
    while sched.running or sched.waiting:
        plan = sched.schedule()
        sched.update(plan, {r: 0 for r in plan.scheduled})
    assert kv.pool.num_free == 200
    assert all(b.ref_cnt == 0 for b in kv.pool.blocks)


def test_block_id_rows_follow_the_blocks():
    """Each request's block-id list (the step's block-table row) stays equal
    to its blocks' ids through admissions with prefix hits, chunked
    prompts, copy-on-write of forked requests, preemption and release."""
    import random
    rnd = random.Random(7)
    head = [rnd.randrange(1000) for _ in range(40)]
    sched = Scheduler(KVCacheManager(64), token_budget=96, max_num_seqs=8,
                      long_prefill_threshold=24)
    for i in range(12):
        tail = [rnd.randrange(1000) for _ in range(rnd.randrange(1, 30))]
        sched.add_request(f"r{i}", head + tail, rnd.randrange(1, 20))
    forked = False
    for _ in range(400):
        if not (sched.waiting or sched.running):
            break
        plan = sched.schedule()
        md = build_step_metadata(plan.requests)
        md2 = build_step_metadata(plan.requests, block_tables=plan.block_tables)
        for k in ("block_tables", "slot_mapping", "seq_lens", "query_start_loc"):
            assert np.array_equal(md[k], md2[k]), k
        for req in plan.requests:
            seq = next(s for s in sched.running if s.request_id == req.request_id)
            assert req.block_ids == [b.block_id for b in seq.blocks]
        sched.update(plan, {rid: rnd.randrange(1000) for rid in plan.scheduled})
        if not forked and sched.running and sched.running[0].num_computed > 20:
            sched.fork(sched.running[0].request_id, "child", 5)
            forked = True
        for seq in sched.running:
            assert seq.block_ids == [b.block_id for b in seq.blocks]
            assert list(seq.ids[:len(seq.blocks)]) == seq.block_ids
    assert not sched.waiting and not sched.running
