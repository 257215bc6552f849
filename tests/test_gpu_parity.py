"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Cache writes and block copies must be bit-exact.  Attention outputs must be
within max-abs 2e-3 (bf16 / fp16 / fp32 caches) or 2e-2 (FP8 cache) of the
fp64 oracle; on small shapes, whose outputs are not small, the half-ulp of
the final rounding to the output type is added to that bar (that rounding is
part of the definition of the output, not an error of the computation).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_82_gb300 as pa
import workloads
from paged_kv_cache_82_gb300.metadata import build_step_metadata
from tests._gpu_step import (ATOL, assert_close, cache_bits, gpu_step,
                             oracle_cache_bits)
from tests._helpers import Req

pytestmark = pytest.mark.gpu


def _oracle_full(wl):
    out, kc, vc, md = oracle.run_step(wl)
    return out, kc, vc, md


def _check_step(wl, with_rounding=True):
    out, kc, vc, md, flags = gpu_step(wl)
    assert flags == 0, f"device error flags 0x{flags:x}"
    ref, kco, vco, mdo = _oracle_full(wl)
    for k in ("query_start_loc", "seq_lens", "block_tables", "slot_mapping"):
        np.testing.assert_array_equal(md[k], mdo[k])
    assert np.array_equal(cache_bits(kc), oracle_cache_bits(kco).reshape(
        cache_bits(kc).shape))
    assert np.array_equal(cache_bits(vc), oracle_cache_bits(vco).reshape(
        cache_bits(vc).shape))
    return assert_close(out, ref, md, wl.cache_dtype, wl.q_dtype,
                        with_rounding)


# ---------------------------------------------------------------------------
# the five step shapes, small enough for the whole-step oracle
# ---------------------------------------------------------------------------
def test_cfg1_fig2_tiny_fp32():
    err = _check_step(workloads.config1())
    assert err <= 1e-5


SMALL = {
    "cfg2_small": lambda: workloads.config2(batch=8, lo=17, hi=700,
                                           num_blocks=600),
    "cfg3_small": lambda: workloads.config3(batch=4, seq_len=1000),
    "cfg4_small": lambda: workloads.config4(num_decodes=10, lo=100, hi=400,
                                           prefix=80, chunk=150,
                                           num_blocks=600),
    "cfg5_small": lambda: workloads.config5(batch=4, lo=300, hi=2000,
                                           num_blocks=700),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_configs(name):
    _check_step(SMALL[name]())


def test_cfg2_full_size_elementwise():
    wl = workloads.config2()
    err = _check_step(wl, with_rounding=False)
    assert err <= ATOL["bf16"]


def _sampled_check(wl, n_rows, seed, cascade_blocks=None):
    """Full-size step: caches compared where the step wrote, attention on
    sampled output rows the oracle computes one by one."""
    out, kc, vc, md, flags = gpu_step(wl, cascade_blocks=cascade_blocks)
    assert flags == 0, f"device error flags 0x{flags:x}"
    # oracle side: copies and writes on host copies of the initial caches
    kco = oracle._as_np(wl.k_cache)[0].copy()
    vco = oracle._as_np(wl.v_cache)[0].copy()
    if wl.copy_pairs:
        oracle.copy_blocks(kco, vco, np.asarray(wl.copy_pairs),
                           cache_dtype=wl.cache_dtype)
    if wl.write_new:
        oracle.reshape_and_cache(wl.key, wl.value, kco, vco,
                                 md["slot_mapping"],
                                 cache_dtype=wl.cache_dtype,
                                 k_scale=wl.k_scale, v_scale=wl.v_scale)
    touched = sorted({int(s) // 16 for s in md["slot_mapping"]} |
                     {d for _, d in wl.copy_pairs})
    if touched:
        idx = torch.tensor(touched, device=kc.device)
        assert np.array_equal(cache_bits(kc[idx]),
                              oracle_cache_bits(kco[touched]))
        assert np.array_equal(cache_bits(vc[idx]),
                              oracle_cache_bits(vco[touched]))
    rng = np.random.default_rng(seed)
    qsl = md["query_start_loc"]
    B = len(wl.requests)
    picks = [(r, int(rng.integers(0, qsl[r + 1] - qsl[r])),
              int(rng.integers(0, wl.num_q_heads)))
             for r in rng.choice(B, size=min(n_rows, B), replace=False)]
    # always include the longest prefill chunk's last query (most keys)
    big = int(np.argmax(np.diff(qsl)))
    picks.append((big, int(qsl[big + 1] - qsl[big] - 1), 0))
    g = out.float().cpu().double().numpy()
    worst = 0.0
    for r, i, h in picks:
        row = oracle.paged_attention_row(
            wl.q, kco, vco, md["block_tables"], md["seq_lens"], qsl, r, i, h,
            scale=wl.scale, cache_dtype=wl.cache_dtype, k_scale=wl.k_scale,
            v_scale=wl.v_scale)
        t = qsl[r] + i
        err = float(np.abs(g[t, h] - row).max())
        worst = max(worst, err)
        assert err <= ATOL[wl.cache_dtype], (r, i, h, err)
    return worst


def test_cfg3_full_size_sampled():
    _sampled_check(workloads.config3(), 48, 3)


def test_cfg4_full_size_sampled():
    wl = workloads.config4()
    _sampled_check(wl, 48, 4)


def test_cfg5_full_size_sampled():
    _sampled_check(workloads.config5(), 16, 5)


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------
def _custom(seq_q, Hq, Hkv, D=128, dtype="bf16", cache_dtype=None, seed=1,
            write_new=False, nb=None):
    lens = [L for L, _ in seq_q]
    qs = [n for _, n in seq_q]
    need = sum(-(-L // 16) for L in lens)
    return workloads.decode_step(
        "edge", seed, seq_lens=lens, q_lens=qs, num_q_heads=Hq,
        num_kv_heads=Hkv, head_dim=D, num_blocks=nb or need + 7,
        dtype=dtype, cache_dtype=cache_dtype, write_new=write_new,
        k_scale=0.02 if cache_dtype == "e4m3" else 1.0,
        v_scale=0.03 if cache_dtype == "e4m3" else 1.0)


@pytest.mark.parametrize("cache_dtype", ["bf16", "e4m3"])
def test_ragged_lengths(cache_dtype):
    seq_q = [(L, 1) for L in (1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257)]
    _check_step(_custom(seq_q, 32, 8, cache_dtype=cache_dtype,
                        write_new=cache_dtype == "e4m3"))


@pytest.mark.parametrize("batch", [1024, 1100])
def test_decode_batch_around_in_kernel_plan_limit(batch):
    # up to 1024 decode requests the attention kernel plans its own split-K
    # ranges; beyond that the planner kernel does
    rng = np.random.default_rng(batch)
    seq_q = [(int(L), 1) for L in rng.integers(1, 120, size=batch)]
    _check_step(_custom(seq_q, 32, 8, write_new=True))


@pytest.mark.parametrize("Hq,Hkv,cache_dtype", [
    (16, 4, "bf16"), (8, 8, "f16"), (36, 12, "bf16"), (64, 8, "e4m3"),
])
def test_decode_head_groups(Hq, Hkv, cache_dtype):
    # decode steps whose KV head count is a multiple of 4 run four KV heads
    # per work item (one TMA box for the four pages of a block), with 4, 1,
    # 3 and 8 query rows per KV head
    rng = np.random.default_rng(Hq * Hkv)
    seq_q = [(int(L), 1) for L in rng.integers(1, 900, size=37)]
    dtype = "f16" if cache_dtype == "f16" else "bf16"
    _check_step(_custom(seq_q, Hq, Hkv, dtype=dtype, cache_dtype=cache_dtype,
                        write_new=True))


@pytest.mark.parametrize("batch", [511, 600])
def test_mixed_batch_around_in_kernel_plan_limit(batch):
    # decodes next to one prefill chunk: up to 512 requests both kernels
    # plan themselves, beyond that the planner lists the prefill tiles for
    # the tensor-core kernel and cuts the decode work
    rng = np.random.default_rng(batch)
    seq_q = [(int(L), int(n)) for L, n in zip(rng.integers(20, 150, size=batch),
                                              rng.integers(1, 5, size=batch))]
    seq_q.append((700, 300))
    _check_step(_custom(seq_q, 32, 8, write_new=True))


@pytest.mark.parametrize("cache_dtype", ["bf16", "e4m3"])
def test_one_long_sequence_split_over_many_ctas(cache_dtype):
    # every KV head's segment is cut by dozens of CTA boundaries
    _check_step(_custom([(40000, 1)], 32, 8, cache_dtype=cache_dtype,
                        write_new=True))


@pytest.mark.parametrize("Hq,Hkv,seq_q", [
    (32, 8, [(300, 4), (40, 3), (17, 2)]),      # 16, 12, 8 rows: decode class
    (32, 8, [(300, 5), (100, 64)]),             # 20 / 256 rows: prefill tiles
    (16, 1, [(500, 1), (90, 2), (33, 33)]),     # group 16
    (8, 8, [(700, 100), (64, 1), (5, 5)]),      # MHA prefill, whole prompt
    (4, 2, [(1, 1), (16, 16), (47, 30)]),       # prompts without history
])
def test_query_shapes(Hq, Hkv, seq_q):
    _check_step(_custom(seq_q, Hq, Hkv, write_new=True))


@pytest.mark.parametrize("Hq,Hkv,seq_q,dtype", [
    (12, 4, [(1500, 300), (200, 1)], "bf16"),   # group 3: 126-row tiles
    (32, 8, [(3022, 1022), (90, 1)], "bf16"),   # a 1022-token chunk
    (8, 8, [(900, 257)], "f16"),                # MHA: 128-token tiles, f16
    (64, 4, [(650, 90), (77, 77)], "bf16"),     # group 16: 8-token tiles
])
def test_prefill_tiles(Hq, Hkv, seq_q, dtype):
    # bf16 / f16 prefill tiles run on the tensor-core kernel: several tiles
    # per request, several 128-key chunks, a partial last page (its free
    # slots hold NaN) and a prefill next to decodes
    _check_step(_custom(seq_q, Hq, Hkv, dtype=dtype, write_new=True))


@pytest.mark.parametrize("Hq,Hkv,seq_q,dtype", [
    (12, 4, [(1500, 300), (200, 1)], "bf16"),   # group 3: 126-row tiles
    (32, 8, [(3022, 1022), (90, 1)], "bf16"),   # a 1022-token chunk
    (8, 8, [(900, 257)], "f16"),                # MHA, f16 q
    (64, 4, [(650, 90), (77, 77)], "bf16"),     # group 16: 8-token tiles
    (24, 6, [(700, 300), (40, 2), (64, 1)], "bf16"),  # no head groups
])
def test_prefill_tiles_fp8_cache(Hq, Hkv, seq_q, dtype):
    # FP8 caches: the tiles' E4M3 pages are widened to f16 in shared memory
    # and run on the tensor cores with Q widened to f16
    _check_step(_custom(seq_q, Hq, Hkv, dtype=dtype, cache_dtype="e4m3",
                        write_new=True))


def test_prefill_tiles_fp8_cache_large_queries():
    # bf16 queries beyond the f16 range: their rows are shifted by a power of
    # two when widened, and the shift is undone on the scores
    wl = _custom([(1200, 400), (300, 1)], 32, 8, cache_dtype="e4m3",
                 write_new=True)
    big = torch.ones(wl.q.shape[0], 32, 1)
    big[::3] = 3.0e5
    big[1::7] = 7.0e4
    wl.q = (wl.q.float() * big).to(torch.bfloat16)
    wl.scale = wl.scale / 3.0e5
    _check_step(wl)


@pytest.mark.parametrize("cache_dtype,dtype", [("bf16", "bf16"), ("f16", "f16")])
def test_mixed_step_routing_by_rows(cache_dtype, dtype):
    # KV heads a multiple of 4 with a long prefill: requests of <= 8 rows run
    # on the head-group decode kernel, a 12-row (3-token) request and the
    # prefill on the tensor-core kernel
    seq_q = [(300, 3), (500, 1), (33, 2), (900, 40), (64, 1), (1200, 200)]
    _check_step(_custom(seq_q, 32, 8, dtype=dtype, cache_dtype=cache_dtype,
                        write_new=True))


def test_mixed_step_prefill_heavy():
    # a long chunk next to two decodes: the prefill grid ahead of the decode
    # kernel takes its largest share of the SMs and most tiles, the grid
    # behind the decode kernel the rest
    seq_q = [(4000, 2000), (300, 1), (777, 1)]
    _check_step(_custom(seq_q, 32, 8, write_new=True))


def test_prefill_row_max_growing_across_chunks():
    # with scores 11x larger than 1/sqrt(D) gives, row maxima keep growing
    # from chunk to chunk, so the running output is rescaled many times
    wl = _custom([(2000, 700), (50, 1)], 32, 8, write_new=True)
    wl.scale = 1.0
    _check_step(wl)


def test_f16_and_fp8_f16_query():
    _check_step(_custom([(333, 1), (64, 7)], 32, 8, dtype="f16",
                        write_new=True))
    _check_step(_custom([(333, 1), (64, 7)], 32, 8, dtype="f16",
                        cache_dtype="e4m3", write_new=True))


@pytest.mark.parametrize("case", ["g4_bf16", "g4_f16", "g8", "two_rows",
                                  "split_long", "window", "mha"])
def test_head_dim_64_head_group_decode(case):
    """head_dim 64, bf16 / f16, decode-only steps with KV heads in groups of
    4: the head-group kernel on 128-byte page rows."""
    rng = np.random.default_rng(len(case))
    lens = [int(L) for L in rng.integers(1, 3000, size=37)] + [1, 16, 17]
    if case == "g4_bf16":
        wl = _custom([(L, 1) for L in lens], 32, 8, D=64)
    elif case == "g4_f16":
        wl = _custom([(L, 1) for L in lens], 16, 4, D=64, dtype="f16")
    elif case == "g8":
        wl = _custom([(L, 1) for L in lens], 64, 8, D=64)
    elif case == "two_rows":
        wl = _custom([(max(L, 2), 2) for L in lens], 32, 8, D=64,
                     write_new=True)
    elif case == "split_long":
        wl = _custom([(40000, 1), (5, 1)], 32, 8, D=64, write_new=True)
    elif case == "window":
        wl = _custom([(L, 1) for L in lens], 32, 8, D=64)
        wl.sliding_window = 100
    else:
        wl = _custom([(L, 1) for L in lens[:12]], 16, 16, D=64)
    _check_step(wl)
    # the head-group kernel and its merge
    n0 = pa.pa_launch_count()
    gpu_step(_custom([(300, 1), (40, 1)], 32, 8, D=64))
    assert pa.pa_launch_count() - n0 == 2


def test_head_dim_64_and_fp32_generic_path():
    _check_step(_custom([(100, 1), (50, 9)], 8, 2, D=64, write_new=True))
    _check_step(_custom([(100, 1), (50, 9)], 8, 2, D=64, dtype="f32",
                        write_new=True))
    _check_step(_custom([(70, 3)], 4, 1, D=128, dtype="f32", write_new=True))


def test_zero_length_requests_and_unowned_rows():
    wl = _custom([(40, 1), (30, 2), (50, 1)], 8, 2, write_new=False)
    # request 1 schedules nothing this step; q keeps 4 rows, so the last row
    # belongs to no request and must stay untouched
    wl.requests[1].num_computed += wl.requests[1].num_new
    wl.requests[1].num_new = 0
    md = build_step_metadata(wl.requests)
    assert md["query_start_loc"].tolist() == [0, 1, 1, 2]
    sentinel = torch.full((4, 8, 128), 7.0, dtype=torch.bfloat16,
                          device="cuda")
    out, *_ = gpu_step(wl, out=sentinel)
    ref, *_ = _oracle_full(wl)
    assert_close(out, ref, md, "bf16", "bf16")
    assert (sentinel[2:] == 7.0).all()


def test_empty_step_launches_nothing():
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    n0 = pa.pa_launch_count()
    out = pa.pa_attention(q, kc, kc.clone(), torch.zeros(0, 1, **i32),
                          torch.zeros(0, **i32), torch.zeros(1, **i32), 0, 0,
                          0.1)
    assert out.shape == (0, 8, 128)
    assert pa.pa_launch_count() == n0
    assert pa.pa_get_device_error() == 0


def test_launches_per_step_kind():
    # decode-only step: the attention kernel plans itself, then the merge
    n0 = pa.pa_launch_count()
    gpu_step(_custom([(300, 1), (40, 1)], 32, 8))
    assert pa.pa_launch_count() - n0 == 2
    # one request of more than 8 rows per KV head: no decode work, the
    # tensor-core kernel alone (no decode kernel, no merge); two query
    # tokens at G = 4 (8 rows) are a decode
    n0 = pa.pa_launch_count()
    gpu_step(_custom([(300, 64)], 32, 8))
    assert pa.pa_launch_count() - n0 == 1
    n0 = pa.pa_launch_count()
    gpu_step(_custom([(300, 2)], 32, 8))
    assert pa.pa_launch_count() - n0 == 2
    # K/V write + a step with bf16 prefill tiles: a tensor-core prefill grid
    # beside the decode kernel, a second one behind it (both plan
    # themselves), then the merge
    n0 = pa.pa_launch_count()
    gpu_step(_custom([(300, 1), (100, 64)], 32, 8, write_new=True))
    assert pa.pa_launch_count() - n0 == 5
    # FP8 cache with prefill tiles: the same five launches, the tiles on the
    # tensor cores (E4M3 pages widened to f16 in shared memory)
    n0 = pa.pa_launch_count()
    gpu_step(_custom([(300, 1), (100, 64)], 32, 8, cache_dtype="e4m3",
                     write_new=True))
    assert pa.pa_launch_count() - n0 == 5
    # FP8 cache, 6 KV heads (no head groups): the write, the prefill tiles
    # on the tensor cores, the one-head attention kernel, the merge (both
    # attention kernels plan themselves)
    n0 = pa.pa_launch_count()
    gpu_step(_custom([(300, 1), (100, 64)], 24, 6, cache_dtype="e4m3",
                     write_new=True))
    assert pa.pa_launch_count() - n0 == 4


def test_bitwise_determinism_and_block_relabelling():
    wl = workloads.config4(num_decodes=6, lo=50, hi=300, prefix=48, chunk=70,
                           num_blocks=300)
    a, kc, vc, md, _ = gpu_step(wl)
    b, *_ = gpu_step(wl)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # relabel every physical block; outputs must not change by one bit
    perm = torch.randperm(wl.num_blocks, generator=torch.Generator().manual_seed(0))
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[perm.cuda()] = kc
    vc2[perm.cuda()] = vc
    tables = torch.from_numpy(md["block_tables"]).long()
    tables2 = perm[tables].to(torch.int32)
    for r, req in enumerate(wl.requests):
        tables2[r, len(req.block_ids):] = 0
    c = pa.pa_attention(wl.q.cuda(), kc2, vc2, tables2.cuda(),
                        torch.from_numpy(md["seq_lens"]).cuda(),
                        torch.from_numpy(md["query_start_loc"]).cuda(),
                        md["max_query_len"], md["max_seq_len"], wl.scale)
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_shared_blocks_equal_private_copies_bitwise():
    wl = _custom([(200, 1), (200, 1)], 32, 8, nb=40)
    # second request points at the first one's blocks (shared prefix), except
    # its last block; a private-copy version of the same step
    r0, r1 = wl.requests
    kc = wl.k_cache.clone()
    vc = wl.v_cache.clone()
    kc[r1.block_ids[:-1]] = kc[r0.block_ids[:-1]]
    vc[r1.block_ids[:-1]] = vc[r0.block_ids[:-1]]
    md = build_step_metadata(wl.requests)
    dev = lambda x: torch.from_numpy(x).cuda()  # noqa: E731
    args = (dev(md["seq_lens"]), dev(md["query_start_loc"]),
            md["max_query_len"], md["max_seq_len"], wl.scale)
    private = pa.pa_attention(wl.q.cuda(), kc.cuda(), vc.cuda(),
                              dev(md["block_tables"]), *args)
    shared_tables = md["block_tables"].copy()
    shared_tables[1, :len(r1.block_ids) - 1] = r0.block_ids[:-1]
    shared = pa.pa_attention(wl.q.cuda(), kc.cuda(), vc.cuda(),
                             dev(shared_tables), *args)
    assert torch.equal(private.view(torch.int16), shared.view(torch.int16))


# ---------------------------------------------------------------------------
# cache kernels: bit-exact
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("kv,cache", [("f32", "f32"), ("f16", "f16"),
                                      ("bf16", "bf16"), ("bf16", "e4m3"),
                                      ("f16", "e4m3"), ("f32", "e4m3")])
@pytest.mark.parametrize("strided", [False, True])
def test_reshape_and_cache_bit_exact(kv, cache, strided):
    rng = np.random.default_rng(17)
    T, H, D, NB = 37, 4, 128, 20
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
    src = torch.from_numpy(rng.standard_normal((T, 3, H, D)).astype(
        np.float32) * 3).to(tdt[kv])
    # strided: K and V are slices of a fused [T, 3, H, D] (row stride 3*H*D)
    key = src[:, 1] if strided else src[:, 1].contiguous()
    value = src[:, 2] if strided else src[:, 2].contiguous()
    slots = rng.choice(NB * 16, size=T, replace=False).astype(np.int64)
    slots[[3, 20]] = -1
    if cache == "e4m3":
        kc = torch.full((NB, H, 16, D), 0x7F, dtype=torch.uint8)
    else:
        kc = torch.full((NB, H, 16, D), float("nan"), dtype=tdt[cache])
    vc = kc.clone()
    kcg, vcg = kc.cuda(), vc.cuda()
    pa.pa_reshape_and_cache(key.cuda(), value.cuda(), kcg, vcg,
                            torch.from_numpy(slots).cuda(), k_scale=0.0125,
                            v_scale=0.015, cache_dtype=cache)
    assert pa.pa_get_device_error() == 0
    kco = oracle._as_np(kc)[0].copy()
    vco = oracle._as_np(vc)[0].copy()
    oracle.reshape_and_cache(key.contiguous(), value.contiguous(), kco, vco,
                             slots, cache_dtype=cache, k_scale=0.0125,
                             v_scale=0.015)
    assert np.array_equal(cache_bits(kcg), oracle_cache_bits(kco))
    assert np.array_equal(cache_bits(vcg), oracle_cache_bits(vco))


def test_fp8_write_of_every_bf16_value():
    """All 65,536 bf16 bit patterns (NaN, inf, subnormals, +-0 included),
    written to an FP8 cache with two scales, equal the oracle's encoder."""
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).view(512, 1, 128)
    NB = 32
    slots = torch.arange(512, dtype=torch.int64)
    kc = torch.zeros(NB, 1, 16, 128, dtype=torch.uint8)
    kcg, vcg = kc.cuda(), kc.clone().cuda()
    pa.pa_reshape_and_cache(x.cuda(), x.cuda(), kcg, vcg, slots.cuda(),
                            k_scale=1.0, v_scale=0.0125, cache_dtype="e4m3")
    kco, vco = kc.numpy().copy(), kc.numpy().copy()
    oracle.reshape_and_cache(x, x, kco, vco, slots.numpy(),
                             cache_dtype="e4m3", k_scale=1.0, v_scale=0.0125)
    assert np.array_equal(kcg.cpu().numpy(), kco)
    assert np.array_equal(vcg.cpu().numpy(), vco)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "e4m3"])
def test_copy_blocks_bit_exact(dtype):
    rng = np.random.default_rng(5)
    NB, H, D = 30, 8, 128
    if dtype == "e4m3":
        kc = torch.from_numpy(rng.integers(0, 256, (NB, H, 16, D), dtype=np.uint8))
    else:
        t = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
        kc = torch.from_numpy(rng.standard_normal((NB, H, 16, D)).astype(
            np.float32)).to(t)
    vc = kc.flip(0).contiguous()
    pairs = np.array([[3, 17], [8, 2], [25, 26], [3, 0]], dtype=np.int64)
    kg, vg = kc.cuda(), vc.cuda()
    pa.pa_copy_blocks(kg, vg, torch.from_numpy(pairs).cuda(), cache_dtype=dtype)
    assert pa.pa_get_device_error() == 0
    kco = oracle._as_np(kc)[0].copy()
    vco = oracle._as_np(vc)[0].copy()
    oracle.copy_blocks(kco, vco, pairs, cache_dtype=dtype)
    assert np.array_equal(cache_bits(kg), oracle_cache_bits(kco))
    assert np.array_equal(cache_bits(vg), oracle_cache_bits(vco))


# ---------------------------------------------------------------------------
# errors: host validation and device-side flags (no fault, no hang)
# ---------------------------------------------------------------------------
def test_device_flags_for_bad_indices():
    wl = _custom([(40, 1), (20, 1)], 8, 2, nb=10)
    md = build_step_metadata(wl.requests)
    kc, vc = wl.k_cache.cuda(), wl.v_cache.cuda()
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa
    # block id out of range: flagged, nothing faults
    bad = md["block_tables"].copy()
    bad[0, 1] = 10 + 5
    pa.pa_attention(wl.q.cuda(), kc, vc, dev(bad), dev(md["seq_lens"]),
                    dev(md["query_start_loc"]), 1, 40, wl.scale)
    assert pa.pa_get_device_error() & pa.PA_DEV_ERR_BLOCK_ID
    # a seq_len above the declared maximum: flagged, request skipped
    pa.pa_attention(wl.q.cuda(), kc, vc, dev(md["block_tables"]),
                    dev(md["seq_lens"]), dev(md["query_start_loc"]), 1, 30,
                    wl.scale)
    assert pa.pa_get_device_error() & pa.PA_DEV_ERR_METADATA
    # slot beyond the cache: flagged, not written
    key = torch.zeros(2, 2, 128, dtype=torch.bfloat16, device="cuda")
    before = kc.clone()
    pa.pa_reshape_and_cache(key, key, kc, vc,
                            torch.tensor([10 * 16, -1], device="cuda"))
    assert pa.pa_get_device_error() & pa.PA_DEV_ERR_SLOT
    assert torch.equal(before.view(torch.int16), kc.view(torch.int16))
    # copy pair out of range
    pa.pa_copy_blocks(kc, vc, torch.tensor([[0, 99]], device="cuda"))
    assert pa.pa_get_device_error() & pa.PA_DEV_ERR_BLOCK_ID
    assert pa.pa_get_device_error() == 0


def test_host_validation_rejects_before_launch():
    lib = pa.load_library()
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    bt, sl, qsl = (torch.zeros(2, 4, **i32), torch.ones(2, **i32),
                   torch.tensor([0, 1, 2], **i32))
    s = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(pa.pa_attention_workspace_size(2, 8, 2, 128, 2, 1, 1),
                     dtype=torch.uint8, device="cuda")

    def call(**kw):
        a = dict(q=q.data_ptr(), qdt=pa.PA_BF16, kc=kc.data_ptr(),
                 vc=vc.data_ptr(),
                 cdt=pa.PA_BF16, nb=4, bs=16, hq=8, hkv=2, d=128,
                 bt=bt.data_ptr(), mb=4, sl=sl.data_ptr(),
                 qsl=qsl.data_ptr(), B=2, T=2, mq=1, ms=1, scale=0.1,
                 ks=1.0, vs=1.0, out=torch.empty_like(q).data_ptr(),
                 ws=ws.data_ptr(), wsb=ws.numel(), s=s)
        a.update(kw)
        return lib.pa_attention(*a.values())

    assert call() == pa.PA_OK
    assert call(bs=32) == pa.PA_ERR_UNSUPPORTED
    assert call(hq=7) == pa.PA_ERR_INVALID_ARG
    assert call(d=96) == pa.PA_ERR_UNSUPPORTED
    assert call(out=q.data_ptr()) == pa.PA_ERR_INVALID_ARG       # alias q
    assert call(out=kc.data_ptr()) == pa.PA_ERR_INVALID_ARG      # alias cache
    assert call(wsb=16) == pa.PA_ERR_INVALID_ARG                 # workspace
    assert call(ms=100) == pa.PA_ERR_INVALID_ARG                 # > 4 blocks
    assert call(cdt=pa.PA_FP8_E4M3, ks=0.0) == pa.PA_ERR_INVALID_ARG
    assert call(qdt=pa.PA_F16) == pa.PA_ERR_UNSUPPORTED          # q != cache
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_output_16_byte_aligned(dtype):
    # an output view 16 bytes past a 32-byte boundary: the prefill tiles
    # write it with 16-byte stores instead of 32-byte ones
    wl = _custom([(300, 1), (700, 300), (90, 64)], 32, 8, dtype=dtype)
    T = int(wl.q.shape[0])
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    base = torch.full((T * 32 * 128 + 8,), float("nan"), dtype=tdt, device="cuda")
    out_view = base[8:].view(T, 32, 128)
    assert out_view.data_ptr() % 32 == 16
    out, kc, vc, md, flags = gpu_step(wl, out=out_view)
    assert flags == 0
    assert out.data_ptr() == out_view.data_ptr()
    ref, *_ = _oracle_full(wl)
    assert_close(out, ref, md, dtype, dtype)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (36, 3)])
def test_fp8_cache_every_code(Hq, Hkv):
    # cache bytes cover every E4M3 code but the two NaNs (subnormals, both
    # zeros, +-448): the kernels widen each exactly as the oracle decodes it.
    # 32/8 heads run the head-group kernel, 36/3 (12 rows per KV head) the
    # one-head kernel's 16-row path
    wl = _custom([(700, 1), (300, 1), (45, 1)], Hq, Hkv, cache_dtype="e4m3")
    codes = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)],
                         dtype=torch.uint8)
    for t, mul in ((wl.k_cache, 7), (wl.v_cache, 11)):
        idx = (torch.arange(t.numel(), dtype=torch.int64) * mul) % codes.numel()
        t.view(-1).copy_(codes[idx])
    wl.k_scale, wl.v_scale = 0.004, 0.005
    _check_step(wl)
