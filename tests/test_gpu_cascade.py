"""Shared-prefix (cascade) steps through pa_attention_cascade.

Requests that share a cached prompt prefix share its full blocks ("01.
vLLM", prefix caching); cascade attention ("01. vLLM", the attention-backend
paragraph) reads that prefix once for every query and merges its part of
the attention with each request's own part by the split-K merge rule ("vLLM
engine anatomy", "Boundaries: FlashAttention").  The result must be the
attention the oracle computes over each request's whole row (the oracle has
no cascade), within the same bar as every other step, and the hint must
change nothing where it is not used.
"""
import numpy as np
import pytest
import torch

import workloads
import paged_kv_cache_82_gb300 as pa
from paged_kv_cache_82_gb300.metadata import build_step_metadata
from tests._gpu_step import assert_close, cache_bits, gpu_step, oracle_cache_bits
from tests.test_gpu_parity import _oracle_full, _sampled_check

pytestmark = pytest.mark.gpu


def _step(prefix_blocks, private, q_lens, Hq=32, Hkv=8, cache_dtype="bf16",
          dtype="bf16", seed=82300, D=128):
    fp8 = cache_dtype == "e4m3"
    return workloads.shared_prefix_step(
        "cascade", seed, prefix_blocks=prefix_blocks, private=private,
        q_lens=q_lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        dtype=dtype, cache_dtype=cache_dtype,
        k_scale=0.02 if fp8 else 1.0, v_scale=0.03 if fp8 else 1.0)


def _check(wl, n):
    out, kc, vc, md, flags = gpu_step(wl, cascade_blocks=n)
    assert flags == 0, f"device error flags 0x{flags:x}"
    ref, kco, vco, _ = _oracle_full(wl)
    assert np.array_equal(cache_bits(kc), oracle_cache_bits(kco).reshape(
        cache_bits(kc).shape))
    assert np.array_equal(cache_bits(vc), oracle_cache_bits(vco).reshape(
        cache_bits(vc).shape))
    assert_close(out, ref, md, wl.cache_dtype, wl.q_dtype)
    return out, md


# private contexts: none (the request's keys after the prefix are its new
# tokens only), short, a full block, ragged, long (cut by several range
# boundaries of the decode kernel's plan)
PRIVATE = [0, 3, 16, 17, 200, 1000, 2500, 61]


@pytest.mark.parametrize("prefix_blocks", [1, 3, 8, 9, 17])
def test_decode_step_with_shared_prefix(prefix_blocks):
    wl = _step(prefix_blocks, PRIVATE, [1] * len(PRIVATE))
    _check(wl, prefix_blocks)


@pytest.mark.parametrize("Hq,Hkv,cache_dtype,q_len", [
    (32, 8, "bf16", 2),     # G = 4: two query tokens (8 rows per KV head)
    (64, 8, "f16", 1),      # G = 8
    (16, 4, "e4m3", 1),     # FP8 cache, bf16 q
    (32, 8, "e4m3", 2),
])
def test_group_sizes_and_types(Hq, Hkv, cache_dtype, q_len):
    dtype = "f16" if cache_dtype == "f16" else "bf16"
    wl = _step(5, PRIVATE, [q_len] * len(PRIVATE), Hq=Hq, Hkv=Hkv,
               cache_dtype=cache_dtype, dtype=dtype)
    _check(wl, 5)


@pytest.mark.parametrize("cache_dtype", ["bf16", "e4m3"])
def test_mixed_step_with_shared_prefix(cache_dtype):
    # decodes and two chunked prefills behind the same prefix: the prefill
    # tiles see every key of their rows, the decodes take the cascade
    private = PRIVATE + [40, 300]
    q_lens = [1] * len(PRIVATE) + [150, 77]
    wl = _step(7, private, q_lens, cache_dtype=cache_dtype)
    _check(wl, 7)


# A long prefix is split into key ranges of at least 32 blocks, each with a
# tile and a partial row of its own, merged in range order: ranges of
# unequal length, several token tiles per range, FP8 pages, G = 8, and a
# prefix far longer than the requests' own contexts (many ranges).
@pytest.mark.parametrize("prefix_blocks,n_req,cache_dtype,Hq", [
    (100, 8, "bf16", 32),     # 4 ranges of 25 blocks
    (77, 40, "bf16", 32),     # 3 ranges (25, 26, 26 blocks), two token tiles
    (1000, 3, "bf16", 32),    # 19 ranges of 52 or 53 blocks
    (300, 5, "e4m3", 32),
    (70, 9, "f16", 64),       # G = 8: tiles of 16 tokens
])
def test_long_prefix_in_key_ranges(prefix_blocks, n_req, cache_dtype, Hq):
    dtype = "f16" if cache_dtype == "f16" else "bf16"
    private = [PRIVATE[i % len(PRIVATE)] for i in range(n_req)]
    wl = _step(prefix_blocks, private, [1] * n_req, Hq=Hq, cache_dtype=cache_dtype,
               dtype=dtype, seed=82310 + prefix_blocks)
    _check(wl, prefix_blocks)


def test_long_prefix_mixed_step():
    # a chunked prefill (its own tiles, whole rows) beside decodes whose
    # 90-block prefix runs in key ranges
    private = PRIVATE + [40]
    q_lens = [1] * len(PRIVATE) + [200]
    wl = _step(90, private, q_lens, seed=82320)
    _check(wl, 90)


def test_prefill_requests_first_and_decodes_after():
    # the prefix tiles take the tokens up to the last decode-class request's
    # (rows of prefill requests among them are computed and not used)
    wl = _step(4, [100, 5, 900, 33], [130, 1, 1, 2])
    _check(wl, 4)


def test_zero_prefix_blocks_is_the_plain_step():
    wl = _step(3, PRIVATE, [1] * len(PRIVATE))
    a, _, _, _, fa = gpu_step(wl, cascade_blocks=0)
    b, _, _, _, fb = gpu_step(wl)
    assert fa == fb == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("Hq,Hkv,D", [(12, 6, 128), (32, 8, 64)])
def test_hint_unused_without_a_cascade_path(Hq, Hkv, D):
    # KV heads not a multiple of 4, or head_dim 64: the plain step runs
    wl = _step(3, PRIVATE, [1] * len(PRIVATE), Hq=Hq, Hkv=Hkv, D=D)
    a, _, _, md, fa = gpu_step(wl, cascade_blocks=3)
    b, _, _, _, fb = gpu_step(wl)
    assert fa == fb == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ref, _, _, _ = _oracle_full(wl)
    assert_close(a, ref, md, wl.cache_dtype, wl.q_dtype)


def _raw_call(wl, md, n, block_tables):
    dev = "cuda"
    kc, vc = wl.k_cache.to(dev), wl.v_cache.to(dev)
    pa.pa_reshape_and_cache(wl.key.to(dev), wl.value.to(dev), kc, vc,
                            torch.from_numpy(md["slot_mapping"]).to(dev))
    out = pa.pa_attention_cascade(
        wl.q.to(dev), kc, vc, torch.from_numpy(block_tables).to(dev),
        torch.from_numpy(md["seq_lens"]).to(dev),
        torch.from_numpy(md["query_start_loc"]).to(dev), md["max_query_len"],
        md["max_seq_len"], wl.scale, n)
    return pa.pa_get_device_error()


def test_prefix_block_mismatch_is_flagged():
    wl = _step(4, PRIVATE, [1] * len(PRIVATE))
    md = build_step_metadata(wl.requests, wl.block_size)
    bt = md["block_tables"].copy()
    bt[3, 2] = bt[3, 5]  # another valid block of the same request
    assert _raw_call(wl, md, 4, bt) & pa.PA_DEV_ERR_METADATA
    assert _raw_call(wl, md, 4, md["block_tables"]) == 0


def test_prefix_reaching_the_queries_is_flagged():
    # request 0 has no private context: with one block more than the shared
    # prefix claimed, its first query would lie inside the claimed prefix
    wl = _step(4, [0, 300, 40], [1, 1, 1])
    md = build_step_metadata(wl.requests, wl.block_size)
    assert _raw_call(wl, md, 5, md["block_tables"]) & pa.PA_DEV_ERR_METADATA
    assert pa.pa_get_device_error() == 0


def test_argument_checks():
    wl = _step(2, [5, 6], [1, 1])
    md = build_step_metadata(wl.requests, wl.block_size)
    for bad in (-1, md["block_tables"].shape[1] + 1):
        with pytest.raises(pa.PaError):
            _raw_call(wl, md, bad, md["block_tables"])


def test_mixed_step_full_size_sampled():
    """The 120-decode mixed step after a 2000-token shared prefix (125
    blocks), with the prefix as a cascade: sampled rows against the oracle."""
    wl = workloads.config4()
    _sampled_check(wl, 48, 41, cascade_blocks=len(wl.shared_blocks))


def test_shared_prefix_decode_full_size_sampled():
    """The bench's shared-prefix decode step: 32 decodes behind a 1024-block
    (16,384-token) prefix, run as a cascade in key ranges (as many as keep
    the prefix tiles within one per SM): sampled rows against the oracle."""
    wl = workloads.shared_prefix_decode()
    from paged_kv_cache_82_gb300.metadata import cascade_prefix_blocks
    n = cascade_prefix_blocks(wl.requests, wl.num_q_heads // wl.num_kv_heads)
    assert n == len(wl.shared_blocks) == 1024
    _sampled_check(wl, 32, 43, cascade_blocks=n)
