"""Lower-bit KV caches on the GPU ("01. vLLM", KV cache options table:
--kv-cache-dtype nvfp4 and int4_per_token_head), against the oracle.

Writes (pa_reshape_and_cache quantising each (token, KV head)) and block
copies must be bit-exact; attention reads the same codes as the oracle and
meets the 16-bit bar.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_82_gb300 as pa
import workloads
from tests._gpu_step import gpu_step, half_ulp
from tests.test_gpu_parity import _check_step

pytestmark = pytest.mark.gpu

FMTS = ["int4", "nvfp4"]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("src,D", [("bf16", 128), ("f16", 128), ("f32", 64),
                                   ("bf16", 64)])
def test_4bit_writes_bit_exact(fmt, src, D):
    rng = np.random.default_rng([FMTS.index(fmt), len(src), D])
    T, Hkv, NB = 70, 3, 9
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16,
           "f32": torch.float32}[src]
    # token rows with a stride (a slice of a wider buffer), values spanning
    # several orders of magnitude, an all-zero row, a padding token
    wide = torch.from_numpy((rng.standard_normal((T, Hkv * D + 32)) *
                             rng.uniform(0.01, 50, (T, 1))).astype(np.float32))
    wide[5] = 0.0
    key = wide[:, :Hkv * D].to(tdt).view(T, Hkv, D)
    wide2 = torch.from_numpy((rng.standard_normal((T, Hkv * D + 32)) * 3.0
                              ).astype(np.float32))
    value = wide2[:, :Hkv * D].to(tdt).view(T, Hkv, D)
    slots = rng.permutation(NB * 16)[:T].astype(np.int64)
    slots[7] = -1
    pb = workloads.page_bytes_4bit(fmt, D)
    init = rng.integers(0, 256, size=(NB, Hkv, pb), dtype=np.uint8)
    g = (0.37, 0.011)
    kc = torch.from_numpy(init.copy()).cuda()
    vc = torch.from_numpy(init.copy()).cuda()
    kg = torch.as_strided(wide.to(tdt).cuda(), (T, Hkv, D),
                          (Hkv * D + 32, D, 1))
    vg = torch.as_strided(wide2.to(tdt).cuda(), (T, Hkv, D),
                          (Hkv * D + 32, D, 1))
    pa.pa_reshape_and_cache(kg, vg, kc, vc, torch.from_numpy(slots).cuda(),
                            k_scale=g[0], v_scale=g[1], cache_dtype=fmt)
    assert pa.pa_get_device_error() == 0
    ko, vo = init.copy(), init.copy()
    oracle.reshape_and_cache(key.contiguous(), value.contiguous(), ko, vo,
                             slots, cache_dtype=fmt, k_scale=g[0],
                             v_scale=g[1])
    assert np.array_equal(kc.cpu().numpy(), ko)
    assert np.array_equal(vc.cpu().numpy(), vo)


@pytest.mark.parametrize("fmt", FMTS)
def test_4bit_copy_blocks_bit_exact(fmt):
    rng = np.random.default_rng(5)
    pb = workloads.page_bytes_4bit(fmt, 128)
    kc = rng.integers(0, 256, size=(30, 8, pb), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(30, 8, pb), dtype=np.uint8)
    pairs = np.array([[3, 17], [8, 2], [25, 26], [3, 0]], dtype=np.int64)
    kg, vg = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    pa.pa_copy_blocks(kg, vg, torch.from_numpy(pairs).cuda(), cache_dtype=fmt)
    assert pa.pa_get_device_error() == 0
    oracle.copy_blocks(kc, vc, pairs, cache_dtype=fmt, head_dim=128)
    assert np.array_equal(kg.cpu().numpy(), kc)
    assert np.array_equal(vg.cpu().numpy(), vc)


def _lowbit(seq_q, Hq, Hkv, fmt, D=128, dtype="bf16", seed=3, write_new=True):
    lens = [L for L, _ in seq_q]
    need = sum(-(-L // 16) for L in lens)
    return workloads.decode_step(
        "lowbit", seed, seq_lens=lens, q_lens=[n for _, n in seq_q],
        num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, num_blocks=need + 5,
        dtype=dtype, cache_dtype=fmt, write_new=write_new,
        k_scale=0.5 if fmt == "nvfp4" else 1.0,
        v_scale=0.25 if fmt == "nvfp4" else 1.0)


RAGGED = [(L, 1) for L in (1, 2, 15, 16, 17, 33, 255, 257, 1500)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("case", ["hg_decode", "onehead_decode", "mixed",
                                  "f16_q", "d64"])
def test_4bit_attention(fmt, case):
    if case == "hg_decode":        # KV heads a multiple of 4, 4 rows each
        wl = _lowbit(RAGGED, 32, 8, fmt)
    elif case == "onehead_decode":  # 6 KV heads, 1+k rows
        wl = _lowbit([(300, 4), (40, 3), (900, 1), (17, 2)], 12, 6, fmt)
    elif case == "mixed":          # decodes next to a prefill chunk
        wl = _lowbit([(700, 300), (64, 1), (1200, 1), (90, 90)], 32, 8, fmt)
    elif case == "f16_q":
        wl = _lowbit([(333, 1), (64, 7)], 32, 8, fmt, dtype="f16")
    else:
        wl = _lowbit([(100, 1), (50, 9)], 8, 2, fmt, D=64)
    _check_step(wl)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("case", ["g4_bf16", "g4_f16", "g8", "two_rows",
                                  "window", "split_long", "mha"])
def test_4bit_head_group_decode(fmt, case):
    """Decode-only steps whose KV heads come in groups of 4 run the
    head-group kernel on the 4-bit pages (bulk copies, f16 MMAs)."""
    rng = np.random.default_rng([FMTS.index(fmt), len(case)])
    lens = [int(L) for L in rng.integers(1, 3000, size=37)] + [1, 16, 17]
    if case == "g4_bf16":
        wl = _lowbit([(L, 1) for L in lens], 32, 8, fmt)
    elif case == "g4_f16":
        wl = _lowbit([(L, 1) for L in lens], 32, 8, fmt, dtype="f16")
    elif case == "g8":
        wl = _lowbit([(L, 1) for L in lens], 64, 8, fmt)
    elif case == "two_rows":       # 1 + 1 draft token at 4 heads: 8 rows
        wl = _lowbit([(max(L, 2), 2) for L in lens], 32, 8, fmt)
    elif case == "window":
        wl = _lowbit([(L, 1) for L in lens], 32, 8, fmt)
        wl.sliding_window = 300
    elif case == "split_long":     # one segment cut by dozens of CTAs
        wl = _lowbit([(40000, 1), (5, 1)], 32, 8, fmt)
    else:                          # 16 KV heads, one query head each
        wl = _lowbit([(L, 1) for L in lens[:12]], 16, 16, fmt)
    _check_step(wl)


@pytest.mark.parametrize("fmt", FMTS)
def test_4bit_decode_full_size_sampled(fmt):
    """The Llama-3.1-8B decode batch over a 4-bit cache (the bench's
    workload): sampled rows against the oracle's row function.  The random
    codes give outputs near 1, so the bar includes half an ulp of the bf16
    output (its final rounding), as for the small steps."""
    wl = workloads.config2(cache_dtype=fmt)
    out, kc, vc, md, flags = gpu_step(wl)
    assert flags == 0
    g = out.float().cpu().double().numpy()
    rng = np.random.default_rng(11)
    for r in rng.choice(len(wl.requests), size=10, replace=False):
        h = int(rng.integers(0, 32))
        row = oracle.paged_attention_row(
            wl.q, wl.k_cache, wl.v_cache, md["block_tables"], md["seq_lens"],
            md["query_start_loc"], int(r), 0, h, scale=wl.scale,
            cache_dtype=fmt, k_scale=wl.k_scale, v_scale=wl.v_scale)
        err = np.abs(g[md["query_start_loc"][r], h] - row)
        assert (err <= 2e-3 + half_ulp(row, "bf16")).all(), float(err.max())


def test_4bit_routing():
    """Decode-only steps in KV-head groups take the head-group kernel plus
    its merge (2 launches); others the generic kernel (1 launch)."""
    n0 = pa.pa_launch_count()
    gpu_step(_lowbit([(300, 1), (40, 1)], 32, 8, "int4", write_new=False))
    assert pa.pa_launch_count() - n0 == 2
    n0 = pa.pa_launch_count()
    gpu_step(_lowbit([(300, 1), (40, 1)], 12, 6, "int4", write_new=False))
    assert pa.pa_launch_count() - n0 == 1


@pytest.mark.parametrize("fmt", FMTS)
def test_4bit_window_and_untouched_rows(fmt):
    wl = _lowbit([(2000, 1), (500, 40), (41, 2)], 32, 8, fmt)
    wl.sliding_window = 100
    _check_step(wl)
