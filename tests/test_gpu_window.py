"""Sliding-window attention and speculative-verify query shapes on the GPU,
against the oracle.

"01. vLLM", section "KV cache management and prefix caching" (the hybrid KV
cache manager paragraph): layers with sliding-window attention, whose blocks
outside the window can be released; a window of W keys lets the query at
position p see keys p - W + 1 .. p.  Same page, scheduler section: a request
verifying k draft tokens runs 1 + k query tokens in one step.

Every kernel path takes the window: the head-group decode kernel, the
one-head kernel (narrow and 16-row), the tensor-core prefill tiles (each
tile starts at its first row's first page inside the window), the FP8
prefill tiles on the warp-level MMA and the generic kernel (fp32, head_dim
64).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_82_gb300 as pa
from paged_kv_cache_82_gb300.metadata import build_step_metadata
from tests._gpu_step import assert_close, gpu_step
from tests.test_gpu_parity import _check_step, _custom

pytestmark = pytest.mark.gpu

RAGGED = [(L, 1) for L in (1, 15, 16, 17, 31, 33, 100, 257, 700, 4000)]

CASES = {
    # decode steps, KV heads a multiple of 4: head-group kernel
    "hg_bf16_w1": (RAGGED, 32, 8, 128, "bf16", None, 1),
    "hg_bf16_w16": (RAGGED, 32, 8, 128, "bf16", None, 16),
    "hg_bf16_w17": (RAGGED, 32, 8, 128, "bf16", None, 17),
    "hg_bf16_w100": (RAGGED, 32, 8, 128, "bf16", None, 100),
    "hg_fp8_w300": (RAGGED, 64, 8, 128, "bf16", "e4m3", 300),
    # one-head kernel: 8-row (narrow) and 12-row (16-row path) requests
    "onehead_f16_g2": (RAGGED, 12, 6, 128, "f16", None, 50),
    "onehead_bf16_16rows": ([(300, 4), (40, 3), (1000, 2)], 24, 6, 128,
                            "bf16", None, 33),
    # spec-verify shapes and prefill tiles on the tensor cores
    "tc_spec_verify": ([(300, 4), (41, 8), (1000, 1), (77, 2)], 64, 8, 128,
                       "bf16", None, 40),
    "tc_prefill_w256": ([(3000, 1000), (200, 1), (900, 900)], 32, 8, 128,
                        "bf16", None, 256),
    "tc_prefill_w7": ([(700, 300), (64, 1)], 32, 8, 128, "bf16", None, 7),
    "tc_prefill_f16_w129": ([(1500, 600)], 8, 8, 128, "f16", None, 129),
    # FP8 cache with prefill tiles: planner + warp-level MMA tiles
    "fp8_prefill_w300": ([(2000, 1), (900, 100)], 32, 8, 128, "bf16", "e4m3",
                         300),
    # generic kernel
    "generic_d64_bf16": ([(100, 1), (50, 9)], 8, 2, 64, "bf16", None, 20),
    "generic_f32": ([(100, 1), (50, 9), (70, 3)], 8, 2, 64, "f32", None, 33),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_sliding_window(name):
    seq_q, Hq, Hkv, D, dtype, cdt, window = CASES[name]
    wl = _custom(seq_q, Hq, Hkv, D=D, dtype=dtype, cache_dtype=cdt,
                 write_new=True)
    wl.sliding_window = window
    _check_step(wl)


@pytest.mark.parametrize("window", [0, 4000, 10 ** 6])
def test_window_that_cuts_nothing_is_pa_attention_bitwise(window):
    seq_q = [(4000, 1), (300, 3), (1200, 200)]
    wl = _custom(seq_q, 32, 8, write_new=True)
    a, *_ = gpu_step(wl)
    wl.sliding_window = window
    b, _, _, md, flags = gpu_step(wl)
    assert flags == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_blocks_outside_the_window_are_never_read():
    """Blocks wholly before each request's first visible key may already be
    released: NaN contents and table entries past the pool change nothing
    and raise no device flag."""
    seq_q = [(3000, 1), (2000, 300), (500, 4), (40, 1)]
    window = 200
    wl = _custom(seq_q, 32, 8)
    wl.sliding_window = window
    a, *_ , md, flags = gpu_step(wl)
    assert flags == 0
    bt = md["block_tables"].copy()
    kc, vc = wl.k_cache.clone(), wl.v_cache.clone()
    for r, req in enumerate(wl.requests):
        first = max(0, req.num_computed - window + 1)
        for k in range(first // 16):
            kc[bt[r, k]] = float("nan")
            vc[bt[r, k]] = float("nan")
            bt[r, k] = wl.num_blocks + 1000
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa
    b = pa.pa_attention_window(
        wl.q.cuda(), kc.cuda(), vc.cuda(), dev(bt), dev(md["seq_lens"]),
        dev(md["query_start_loc"]), md["max_query_len"], md["max_seq_len"],
        wl.scale, window)
    assert pa.pa_get_device_error() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_window_sampled_at_full_size():
    """The Llama-3.1-8B decode batch (64 requests, contexts of 512 to 4096)
    through a 1024-key window: sampled rows against the oracle's row
    function."""
    import workloads
    wl = workloads.config2()
    wl.sliding_window = 1024
    out, kc, vc, md, flags = gpu_step(wl)
    assert flags == 0
    g = out.float().cpu().double().numpy()
    rng = np.random.default_rng(9)
    for r in rng.choice(len(wl.requests), size=12, replace=False):
        h = int(rng.integers(0, 32))
        row = oracle.paged_attention_row(
            wl.q, wl.k_cache, wl.v_cache, md["block_tables"], md["seq_lens"],
            md["query_start_loc"], int(r), 0, h, scale=wl.scale, window=1024)
        assert float(np.abs(g[md["query_start_loc"][r], h] - row).max()) <= 2e-3


@pytest.mark.parametrize("k", [3, 7])
def test_spec_verify_one_plus_k_at_group_8(k):
    """Verification of k draft tokens: 1 + k query tokens per request at
    8 query heads per KV head, i.e. 32 and 64 rows: past the head-group
    decode kernel's 8 rows and the one-head kernel's 16, onto the
    tensor-core tiles, next to plain decodes."""
    rng = np.random.default_rng(k)
    seq_q = [(int(L), 1 + k) for L in rng.integers(1 + k, 3000, size=20)]
    seq_q += [(int(L), 1) for L in rng.integers(1, 3000, size=20)]
    _check_step(_custom(seq_q, 64, 8, write_new=True))
