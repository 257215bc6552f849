"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test names the passage it rests on.  Values from the pages live in
tests/golden/*.json with their citation; everything else is a closed form, an
invariant, a library routine (torch / numpy) or a brute-force second
formulation.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests._helpers import (BS, Req, random_paged_step, scatter_paged,
                            sdpa_reference)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# "vLLM engine anatomy", PagedAttention section, Figure 2
# ---------------------------------------------------------------------------
def test_fig2_block_tables_and_next_slots():
    g = _golden("fig2_layout.json")
    A, B = g["sequences"]["A"], g["sequences"]["B"]
    reqs = [Req(A["block_table"], A["prompt_tokens"], 1),
            Req(B["block_table"], B["prompt_tokens"], 1)]
    md = oracle.step_metadata(reqs, g["block_size"])
    assert md["slot_mapping"].tolist() == [g["next_token_slot"]["A"],
                                           g["next_token_slot"]["B"]]
    assert md["seq_lens"].tolist() == [41, 21]
    assert md["query_start_loc"].tolist() == [0, 1, 2]
    assert md["block_tables"][0].tolist() == [0, 1, 2]
    assert md["block_tables"][1][:2].tolist() == [3, 4]
    # block contents: block k of a sequence holds tokens [first, last]
    for seq in (A, B):
        for blk, (first, last) in seq["block_contents"].items():
            for t in range(first, last + 1):
                s = oracle.slot_of(seq["block_table"], t, g["block_size"])
                assert s // g["block_size"] == int(blk)


def test_fig2_reshape_writes_only_the_new_slots():
    """cfg-1 write: the two new tokens land at (block 2, offset 8) and
    (block 4, offset 4); free blocks 5..11 and the other empty offsets stay
    untouched (NaN)."""
    import workloads
    wl = workloads.config1()
    g = _golden("fig2_layout.json")
    md = oracle.step_metadata(wl.requests)
    kc = wl.k_cache.numpy().copy()
    vc = wl.v_cache.numpy().copy()
    before_k = kc.copy()
    oracle.reshape_and_cache(wl.key, wl.value, kc, vc, md["slot_mapping"],
                             cache_dtype="f32")
    key = wl.key.numpy()
    value = wl.value.numpy()
    np.testing.assert_array_equal(kc[2, :, 8, :], key[0])
    np.testing.assert_array_equal(vc[4, :, 4, :], value[1])
    changed = ~((kc == before_k) | (np.isnan(kc) & np.isnan(before_k)))
    assert changed.sum() == 2 * wl.num_kv_heads * wl.head_dim
    for b in g["free_blocks"]:
        assert np.isnan(kc[b]).all() and np.isnan(vc[b]).all()
    assert np.isnan(kc[2, :, 9:, :]).all() and np.isnan(kc[4, :, 5:, :]).all()


# ---------------------------------------------------------------------------
# Table 1 ("vLLM engine anatomy"): per-token KV bytes
# ---------------------------------------------------------------------------
def test_table1_kv_bytes_per_token():
    g = _golden("table1_kv_bytes.json")
    eb = g["fp16_elem_bytes"]
    for row in g["rows"]:
        b = oracle.kv_bytes_per_token(eb, row["layers"], row["kv_heads"],
                                      row["head_dim"])
        assert b == row["bytes_per_token"], row["model"]
        assert b * 8192 == row["at_8k_bytes"], row["model"]
    b8 = oracle.kv_bytes_per_token(eb, 32, 8, 128)
    assert b8 * 131072 == g["llama31_8b_128k_bytes"]
    n = g["titan_rtx_kv_budget_bytes"] // b8
    assert n == g["titan_rtx_tokens_at_128KiB"]
    lo, hi = g["titan_rtx_tokens_range_stated"]
    assert lo <= n <= hi
    # FP8 halves it ("01. vLLM", --kv-cache-dtype fp8 row)
    assert oracle.kv_bytes_per_token(1, 32, 8, 128) * 2 == b8


def test_prefix_is_whole_blocks():
    g = _golden("prefix_blocks.json")
    assert g["prefix_tokens"] // g["block_size"] == g["full_blocks"]
    assert g["prefix_tokens"] % g["block_size"] == 0


def test_unified_step_metadata():
    """{"req-A": 1, "req-B": 1, "req-C": 1022} in a 1024-token budget."""
    g = _golden("unified_step.json")
    step = g["step"]
    assert sum(step.values()) <= g["token_budget"]
    assert g["prompt_tokens_of_C"] - g["scheduled_now_C"] == \
        g["left_for_next_step_C"]
    # A, B decode after 10 and 20 tokens; C's first chunk of a long prompt
    reqs = [Req([0], 10, 1), Req([1, 2], 20, 1),
            Req(list(range(3, 3 + 64)), 0, 1022)]
    md = oracle.step_metadata(reqs)
    assert md["query_start_loc"].tolist() == [0, 1, 2, 1024]
    assert md["max_query_len"] == 1022
    assert md["seq_lens"].tolist() == [11, 21, 1022]
    assert md["slot_mapping"].shape == (1024,)
    # C's chunk fills blocks 3.. in order: slot of token t is 3*16 + t
    assert md["slot_mapping"][2:].tolist() == list(range(48, 48 + 1022))


# ---------------------------------------------------------------------------
# number formats: IEEE binary16, bfloat16, OCP FP8 E4M3FN
# ---------------------------------------------------------------------------
def test_f16_decode_matches_numpy_for_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_bits_to_double(int(b)) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(ref[~both_nan], got[~both_nan])
    assert np.isnan(got).sum() == np.isnan(ref).sum()


def test_bf16_decode_matches_torch_for_all_patterns():
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_bits_to_double(int(b) & 0xFFFF)
                    for b in bits.tolist()])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(ref[~both_nan], got[~both_nan])
    assert np.isnan(got).sum() == np.isnan(ref).sum()


def test_e4m3_decode_spec_points_and_torch():
    # OCP FP8 E4M3: bias 7, max normal 448 = S.1111.110, min normal 2^-6,
    # min subnormal 2^-9, S.1111.111 is NaN, no infinities
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0xFE) == -448.0
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_double(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_to_double(0x38) == 1.0
    assert math.isnan(oracle.e4m3_to_double(0x7F))
    assert math.isnan(oracle.e4m3_to_double(0xFF))
    z = oracle.e4m3_to_double(0x80)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], got[fin])
    assert np.array_equal(np.isnan(ref), np.isnan(got))


def test_e4m3_encode_roundtrip_and_ties():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        v = oracle.e4m3_to_double(c)
        assert oracle.e4m3_encode(v) == c, hex(c)
    # midpoints between neighbouring positive codes go to the even code
    for c in range(0, 0x7E):
        a, b = oracle.e4m3_to_double(c), oracle.e4m3_to_double(c + 1)
        mid = np.float32((a + b) / 2)
        assert float(mid) == (a + b) / 2  # exact in fp32
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(mid)) == want, hex(c)
        assert oracle.e4m3_encode(-float(mid)) == want | 0x80
    # saturation and special values
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("-inf")) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(2.0 ** -11) == 0x00   # below half the min subnormal
    assert oracle.e4m3_encode(-(2.0 ** -11)) == 0x80


def test_e4m3_encode_matches_torch_on_all_bf16_inputs():
    """fl32(x / scale) then the nearest code, for every bf16 x, compared with
    torch's float8_e4m3fn cast (round to nearest even) wherever that cast is
    defined (|y| <= 448; torch does not saturate)."""
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).to(torch.float32)
    for scale in (1.0, 0.0125, 0.015, 3.0):
        y = x / torch.tensor(scale, dtype=torch.float32)   # fp32 division
        ok = torch.isfinite(y) & (y.abs() <= 448.0)
        ref = y[ok].to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = np.array([oracle.e4m3_encode(float(v)) for v in y[ok].tolist()],
                       dtype=np.uint8)
        assert np.array_equal(ref, got), scale
        big = y[torch.isfinite(y) & (y.abs() > 448.0)].tolist()
        for v in big[:2000]:
            assert oracle.e4m3_encode(v) == (0x7E if v > 0 else 0xFE)


def test_reshape_fp8_uses_fp32_division():
    """The FP8 write encodes fl32(x / scale): compare with numpy's float32
    division followed by torch's fp8 cast (independent of the oracle)."""
    rng = np.random.default_rng(5)
    T, H, D = 7, 2, 8
    key = torch.from_numpy(rng.standard_normal((T, H, D)).astype(np.float32)
                           ).to(torch.bfloat16)
    value = torch.from_numpy(rng.standard_normal((T, H, D)).astype(np.float32)
                             ).to(torch.bfloat16)
    kc = np.full((4, H, BS, D), 0x7F, dtype=np.uint8)
    vc = kc.copy()
    slots = np.array([0, 17, 35, -1, 50, 63, 3], dtype=np.int64)
    ks, vs = 0.0125, 0.015
    oracle.reshape_and_cache(key, value, kc, vc, slots, cache_dtype="e4m3",
                             k_scale=ks, v_scale=vs)
    kx = key.to(torch.float32).numpy()
    vx = value.to(torch.float32).numpy()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        yk = (kx[t] / np.float32(ks)).astype(np.float32)
        yv = (vx[t] / np.float32(vs)).astype(np.float32)
        wk = torch.from_numpy(np.clip(yk, -448, 448)).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
        wv = torch.from_numpy(np.clip(yv, -448, 448)).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(kc[s // BS, :, s % BS, :], wk)
        np.testing.assert_array_equal(vc[s // BS, :, s % BS, :], wv)
    # the padding token (slot -1) wrote nothing: 7 slots minus one
    assert (kc != 0x7F).any(axis=(1, 3)).sum() == 6


# ---------------------------------------------------------------------------
# copy-on-write block copies ("vLLM engine anatomy", CoW item; "V0 vs V1"
# blocks_to_copy)
# ---------------------------------------------------------------------------
def test_copy_blocks_copies_whole_blocks_only():
    rng = np.random.default_rng(11)
    kc = rng.standard_normal((9, 3, BS, 8)).astype(np.float32)
    vc = rng.standard_normal((9, 3, BS, 8)).astype(np.float32)
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[2, 7], [5, 1]], dtype=np.int64)
    oracle.copy_blocks(kc, vc, pairs, cache_dtype="f32")
    for s, d in pairs:
        np.testing.assert_array_equal(kc[d], k0[s])
        np.testing.assert_array_equal(vc[d], v0[s])
    untouched = [b for b in range(9) if b not in (7, 1)]
    np.testing.assert_array_equal(kc[untouched], k0[untouched])
    np.testing.assert_array_equal(vc[untouched], v0[untouched])


# ---------------------------------------------------------------------------
# attention: equality with contiguous attention via a library routine
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4), (6, 1)])
def test_paged_equals_contiguous_sdpa(Hq, Hkv):
    rng = np.random.default_rng(100 + Hq + Hkv)
    shapes = [(1, 37), (5, 21), (17, 53), (1, 1), (3, 3), (16, 80)]
    D = 16
    q, kc, vc, reqs, qs, ks, vs = random_paged_step(rng, shapes, Hq, Hkv, D,
                                                    40)
    md = oracle.step_metadata(reqs)
    scale = 0.3
    out = oracle.paged_attention(q, kc, vc, md["block_tables"],
                                 md["seq_lens"], md["query_start_loc"],
                                 scale=scale)
    ref = sdpa_reference([x.astype(np.float64) for x in qs],
                         [x.astype(np.float64) for x in ks],
                         [x.astype(np.float64) for x in vs], Hq // Hkv, scale)
    np.testing.assert_allclose(out, np.concatenate(ref, axis=0), rtol=0,
                               atol=1e-12)


def test_paged_bf16_and_fp8_match_sdpa_on_decoded_values():
    """Stored-format inputs are decoded exactly; FP8 values are scaled by
    k_scale / v_scale ("01. vLLM", fp8 KV cache)."""
    rng = np.random.default_rng(7)
    shapes = [(1, 45), (4, 33), (2, 16)]
    Hq, Hkv, D = 4, 2, 16
    q, kc, vc, reqs, qs, ks, vs = random_paged_step(rng, shapes, Hq, Hkv, D,
                                                    12)
    md = oracle.step_metadata(reqs)
    qb = torch.from_numpy(q).to(torch.bfloat16)
    q64 = qb.to(torch.float64).numpy()
    # bf16 cache
    kb = torch.from_numpy(kc).to(torch.bfloat16)
    vb = torch.from_numpy(vc).to(torch.bfloat16)
    out = oracle.paged_attention(qb, kb, vb, md["block_tables"],
                                 md["seq_lens"], md["query_start_loc"],
                                 scale=0.25)
    kd = kb.to(torch.float64).numpy()
    vd = vb.to(torch.float64).numpy()
    # fp8 cache with scales
    ks_, vs_ = 0.0125, 0.015
    k8 = torch.from_numpy(np.clip(kc / ks_, -448, 448).astype(np.float32)
                          ).to(torch.float8_e4m3fn)
    v8 = torch.from_numpy(np.clip(vc / vs_, -448, 448).astype(np.float32)
                          ).to(torch.float8_e4m3fn)
    out8 = oracle.paged_attention(qb, k8, v8, md["block_tables"],
                                  md["seq_lens"], md["query_start_loc"],
                                  scale=0.25, k_scale=ks_, v_scale=vs_)
    k8d = k8.to(torch.float64).numpy() * ks_
    v8d = v8.to(torch.float64).numpy() * vs_
    for o, kk, vv in ((out, kd, vd), (out8, k8d, v8d)):
        qsl = md["query_start_loc"]
        refs = sdpa_reference(
            [q64[qsl[i]:qsl[i + 1]] for i in range(len(reqs))],
            [np.stack([kk[r.block_ids[j // BS], :, j % BS] for j in
                       range(r.num_computed + r.num_new)]) for r in reqs],
            [np.stack([vv[r.block_ids[j // BS], :, j % BS] for j in
                       range(r.num_computed + r.num_new)]) for r in reqs],
            Hq // Hkv, 0.25)
        np.testing.assert_allclose(o, np.concatenate(refs, 0), rtol=0,
                                   atol=1e-12)


# ---------------------------------------------------------------------------
# invariants: block relabelling, sharing, copy-on-write
# ---------------------------------------------------------------------------
def test_permutation_invariance_bitwise():
    rng = np.random.default_rng(3)
    shapes = [(1, 70), (9, 40), (1, 16)]
    q, kc, vc, reqs, *_ = random_paged_step(rng, shapes, 8, 2, 16, 20)
    md = oracle.step_metadata(reqs)
    out = oracle.paged_attention(q, kc, vc, md["block_tables"],
                                 md["seq_lens"], md["query_start_loc"],
                                 scale=0.2)
    perm = rng.permutation(20)          # new id of physical block b
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    reqs2 = [Req([int(perm[b]) for b in r.block_ids], r.num_computed,
                 r.num_new) for r in reqs]
    md2 = oracle.step_metadata(reqs2)
    out2 = oracle.paged_attention(q, kc2, vc2, md2["block_tables"],
                                  md2["seq_lens"], md2["query_start_loc"],
                                  scale=0.2)
    assert np.array_equal(out, out2)


def test_shared_prefix_equals_private_copies_bitwise():
    """Block contents are a pure function of their tokens, so sequences may
    point at the same physical blocks ("vLLM engine anatomy", sharing)."""
    rng = np.random.default_rng(4)
    Hq, Hkv, D = 4, 2, 8
    prefix_k = rng.standard_normal((32, Hkv, D)).astype(np.float32)
    prefix_v = rng.standard_normal((32, Hkv, D)).astype(np.float32)
    tails = [rng.standard_normal((t, 2, Hkv, D)).astype(np.float32)
             for t in (5, 19)]
    seqs_k = [np.concatenate([prefix_k, t[:, 0]]) for t in tails]
    seqs_v = [np.concatenate([prefix_v, t[:, 1]]) for t in tails]
    # shared: both tables start with blocks 0, 1
    shared_lists = [[0, 1, 2], [0, 1, 3, 4]]
    private_lists = [[5, 6, 2], [7, 8, 3, 4]]
    q = rng.standard_normal((2, Hq, D)).astype(np.float32)
    outs = []
    for lists in (shared_lists, private_lists):
        kc = scatter_paged(seqs_k, lists, 9)
        vc = scatter_paged(seqs_v, lists, 9)
        reqs = [Req(lists[i], seqs_k[i].shape[0] - 1, 1) for i in range(2)]
        md = oracle.step_metadata(reqs)
        outs.append(oracle.paged_attention(
            q, kc, vc, md["block_tables"], md["seq_lens"],
            md["query_start_loc"], scale=0.5))
    assert np.array_equal(outs[0], outs[1])


def test_copy_on_write_leaves_other_reader_untouched():
    """r1 forks r0 (same blocks, shared partial last block).  r1 copies the
    block, rewrites only its own table, both write their next token.  r0's
    output and the source block's other bytes equal a run without r1."""
    rng = np.random.default_rng(9)
    Hq, Hkv, D, NB = 4, 2, 8, 8
    ctx = 37                                   # 2 full blocks + 5 tokens
    seq_k = rng.standard_normal((ctx, Hkv, D)).astype(np.float32)
    seq_v = rng.standard_normal((ctx, Hkv, D)).astype(np.float32)
    blocks0 = [4, 1, 6]
    kc = scatter_paged([seq_k], [blocks0], NB)
    vc = scatter_paged([seq_v], [blocks0], NB)
    new_k = rng.standard_normal((2, Hkv, D)).astype(np.float32)
    new_v = rng.standard_normal((2, Hkv, D)).astype(np.float32)
    q = rng.standard_normal((2, Hq, D)).astype(np.float32)

    # run with the fork
    kcf, vcf = kc.copy(), vc.copy()
    oracle.copy_blocks(kcf, vcf, np.array([[6, 3]]), cache_dtype="f32")
    reqs = [Req(blocks0, ctx, 1), Req([4, 1, 3], ctx, 1)]
    md = oracle.step_metadata(reqs)
    assert md["slot_mapping"].tolist() == [6 * 16 + 5, 3 * 16 + 5]
    oracle.reshape_and_cache(new_k, new_v, kcf, vcf, md["slot_mapping"],
                             cache_dtype="f32")
    out_f = oracle.paged_attention(q, kcf, vcf, md["block_tables"],
                                   md["seq_lens"], md["query_start_loc"],
                                   scale=0.4)
    # run without r1
    kc1, vc1 = kc.copy(), vc.copy()
    reqs1 = [Req(blocks0, ctx, 1)]
    md1 = oracle.step_metadata(reqs1)
    oracle.reshape_and_cache(new_k[:1], new_v[:1], kc1, vc1,
                             md1["slot_mapping"], cache_dtype="f32")
    out_1 = oracle.paged_attention(q[:1], kc1, vc1, md1["block_tables"],
                                   md1["seq_lens"], md1["query_start_loc"],
                                   scale=0.4)
    assert np.array_equal(out_f[0], out_1[0])
    np.testing.assert_array_equal(kcf[6], kc1[6])   # source block
    np.testing.assert_array_equal(vcf[6], vc1[6])
    # the copy got r1's token and the shared history
    np.testing.assert_array_equal(kcf[3, :, :5], kc[6, :, :5])
    np.testing.assert_array_equal(kcf[3, :, 5], new_k[1])


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
def _single(q, k_seq, v_seq, n, scale=1.0, Hkv=1):
    q, k_seq, v_seq = (np.asarray(a, dtype=np.float32) for a in
                       (q, k_seq, v_seq))
    L = k_seq.shape[0]
    nb = -(-L // BS)
    blocks = list(range(nb))
    kc = scatter_paged([k_seq], [blocks], nb)
    vc = scatter_paged([v_seq], [blocks], nb)
    md = oracle.step_metadata([Req(blocks, L - n, n)])
    return oracle.paged_attention(q, kc, vc, md["block_tables"],
                                  md["seq_lens"], md["query_start_loc"],
                                  scale=scale)


def test_closed_forms():
    rng = np.random.default_rng(21)
    D = 8
    k = rng.standard_normal((41, 1, D)).astype(np.float32)
    v = rng.standard_normal((41, 1, D)).astype(np.float32).astype(np.float64)
    # q = 0: uniform weights -> mean of the visible values
    out = _single(np.zeros((1, 1, D)), k, v, 1)
    np.testing.assert_allclose(out[0, 0], v[:, 0].mean(0), atol=1e-14)
    # a single visible key -> that value
    out = _single(rng.standard_normal((1, 1, D)), k[:1], v[:1], 1)
    np.testing.assert_allclose(out[0, 0], v[0, 0], atol=0)
    # identical keys -> mean of the values
    kk = np.repeat(k[:1], 41, axis=0)
    out = _single(rng.standard_normal((1, 1, D)), kk, v, 1)
    np.testing.assert_allclose(out[0, 0], v[:, 0].mean(0), atol=1e-14)
    # one key with a huge score dominates
    q = np.ones((1, 1, D))
    kh = k.copy()
    kh[23, 0] = 1e3
    out = _single(q, kh, v, 1)
    np.testing.assert_allclose(out[0, 0], v[23, 0], atol=1e-12)
    # first token of a chunk with no history sees only itself -> v_0; the
    # i-th sees tokens 0..i -> causal prefix means when q = 0
    n = 19
    out = _single(np.zeros((n, 1, D)), k[:n], v[:n], n)
    for i in range(n):
        np.testing.assert_allclose(out[i, 0], v[:i + 1, 0].mean(0),
                                   atol=1e-14)


# ---------------------------------------------------------------------------
# brute force: a second, naive formulation on tiny shapes
# ---------------------------------------------------------------------------
def _brute(q, kc, vc, reqs, Hq, Hkv, scale, window=0):
    out = {}
    t = 0
    G = Hq // Hkv
    for r in reqs:
        L = r.num_computed + r.num_new
        for i in range(r.num_new):
            limit = L - r.num_new + i
            for h in range(Hq):
                g = h // G
                keys, vals = [], []
                start = max(0, limit - window + 1) if window else 0
                for j in range(start, limit + 1):
                    b = r.block_ids[j // BS]
                    keys.append([float(x) for x in kc[b, g, j % BS]])
                    vals.append([float(x) for x in vc[b, g, j % BS]])
                scores = [scale * sum(a * b for a, b in
                                      zip(q[t + i, h].tolist(), kj))
                          for kj in keys]
                m = max(scores)
                w = [math.exp(s - m) for s in scores]
                z = sum(w)
                out[(t + i, h)] = [sum(w[j] * vals[j][d] for j in
                                       range(len(w))) / z
                                   for d in range(len(vals[0]))]
        t += r.num_new
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 4))
    shapes = []
    for _ in range(B):
        L = int(rng.integers(1, 41))
        n = int(rng.integers(1, L + 1))
        shapes.append((n, L))
    Hq, Hkv = [(2, 1), (4, 2), (3, 3)][seed]
    q, kc, vc, reqs, *_ = random_paged_step(rng, shapes, Hq, Hkv, 8, 12)
    md = oracle.step_metadata(reqs)
    out = oracle.paged_attention(q, kc, vc, md["block_tables"],
                                 md["seq_lens"], md["query_start_loc"],
                                 scale=0.7)
    ref = _brute(q, kc, vc, reqs, Hq, Hkv, 0.7)
    for (t, h), row in ref.items():
        np.testing.assert_allclose(out[t, h], row, rtol=0, atol=1e-12)


def test_row_function_equals_full_step():
    rng = np.random.default_rng(8)
    q, kc, vc, reqs, *_ = random_paged_step(rng, [(3, 50), (1, 17)], 8, 2,
                                            16, 10)
    md = oracle.step_metadata(reqs)
    args = (q, kc, vc, md["block_tables"], md["seq_lens"],
            md["query_start_loc"])
    out = oracle.paged_attention(*args, scale=0.3)
    for (r, i) in [(0, 0), (0, 2), (1, 0)]:
        for h in (0, 5, 7):
            row = oracle.paged_attention_row(*args, r, i, h, scale=0.3)
            t = md["query_start_loc"][r] + i
            assert np.array_equal(row, out[t, h])


def test_zero_length_request_produces_nothing():
    rng = np.random.default_rng(12)
    q, kc, vc, reqs, *_ = random_paged_step(rng, [(2, 20)], 2, 1, 8, 4)
    reqs = [Req([3], 5, 0)] + reqs
    md = oracle.step_metadata(reqs)
    out = oracle.paged_attention(q, kc, vc, md["block_tables"],
                                 md["seq_lens"], md["query_start_loc"],
                                 scale=1.0)
    assert md["query_start_loc"].tolist() == [0, 0, 2]
    assert np.isfinite(out).all()


# ---------------------------------------------------------------------------
# sliding window ("01. vLLM", hybrid KV cache manager paragraph: layers with
# sliding-window attention; their blocks outside the window can be released)
# ---------------------------------------------------------------------------
def _window_step(seed=31, shapes=((1, 70), (9, 40), (1, 16), (20, 53)),
                 Hq=8, Hkv=2, D=16, NB=24):
    rng = np.random.default_rng(seed)
    q, kc, vc, reqs, qs, ks, vs = random_paged_step(rng, list(shapes), Hq, Hkv,
                                                    D, NB)
    return q, kc, vc, reqs, qs, ks, vs, oracle.step_metadata(reqs)


def _attn(q, kc, vc, md, window, scale=0.4):
    return oracle.paged_attention(q, kc, vc, md["block_tables"],
                                  md["seq_lens"], md["query_start_loc"],
                                  scale=scale, window=window)


def test_window_wider_than_the_context_is_no_window():
    q, kc, vc, reqs, *_, md = _window_step()
    base = _attn(q, kc, vc, md, 0)
    for w in (70, 71, 1000):
        assert np.array_equal(_attn(q, kc, vc, md, w), base)


def test_window_of_one_key_is_the_own_value():
    q, kc, vc, reqs, qs, ks, vs, md = _window_step()
    out = _attn(q, kc, vc, md, 1)
    G = 4
    t = 0
    for r, v in zip(reqs, vs):
        L = r.num_computed + r.num_new
        for i in range(r.num_new):
            for h in range(8):
                assert np.array_equal(out[t + i, h],
                                      v[L - r.num_new + i, h // G].astype(
                                          np.float64))
        t += r.num_new


@pytest.mark.parametrize("window", [2, 7, 16, 17, 33])
def test_window_matches_banded_sdpa(window):
    q, kc, vc, reqs, qs, ks, vs, md = _window_step()
    out = _attn(q, kc, vc, md, window)
    ref = sdpa_reference([x.astype(np.float64) for x in qs],
                         [x.astype(np.float64) for x in ks],
                         [x.astype(np.float64) for x in vs], 4, 0.4,
                         window=window)
    np.testing.assert_allclose(out, np.concatenate(ref, 0), rtol=0,
                               atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_window_brute_force_tiny(seed):
    rng = np.random.default_rng(2000 + seed)
    shapes = [(int(rng.integers(1, 6)), int(rng.integers(6, 41)))
              for _ in range(3)]
    q, kc, vc, reqs, *_ = random_paged_step(rng, shapes, 4, 2, 8, 12)
    md = oracle.step_metadata(reqs)
    for window in (3, 16, 21):
        out = _attn(q, kc, vc, md, window, scale=0.7)
        ref = _brute(q, kc, vc, reqs, 4, 2, 0.7, window=window)
        for (t, h), row in ref.items():
            np.testing.assert_allclose(out[t, h], row, rtol=0, atol=1e-12)


def test_blocks_outside_the_window_are_never_read():
    """The blocks a request's queries cannot see may be released: poisoning
    them, or pointing the table at a block that does not exist, changes
    nothing."""
    q, kc, vc, reqs, *_, md = _window_step()
    window = 17
    base = _attn(q, kc, vc, md, window)
    bt = md["block_tables"].copy()
    kc2, vc2 = kc.copy(), vc.copy()
    for b, r in enumerate(reqs):
        first = max(0, r.num_computed - window + 1)  # first query's first key
        for k in range(first // 16):
            kc2[bt[b, k]] = np.nan
            vc2[bt[b, k]] = np.nan
            bt[b, k] = 10 ** 6
    md2 = dict(md, block_tables=bt)
    assert np.array_equal(_attn(q, kc2, vc2, md2, window), base)
    # without the window the same table is out of range
    with pytest.raises(oracle.OracleError):
        _attn(q, kc2, vc2, md2, 0)


def test_window_row_function_equals_full_step():
    q, kc, vc, reqs, *_, md = _window_step()
    out = _attn(q, kc, vc, md, 9)
    args = (q, kc, vc, md["block_tables"], md["seq_lens"],
            md["query_start_loc"])
    for r, i in ((0, 0), (1, 8), (3, 19), (3, 0)):
        for h in (0, 7):
            row = oracle.paged_attention_row(*args, r, i, h, scale=0.4,
                                             window=9)
            assert np.array_equal(row, out[md["query_start_loc"][r] + i, h])


# ---------------------------------------------------------------------------
# lower-bit KV caches ("01. vLLM", KV cache options table: nvfp4 and
# int4_per_token_head).  Pages of one (block, KV head): 16 * D / 2 bytes of
# codes (element 2i in the low nibble of byte i of its token), then the
# scales: 16 fp32 (int4, one per token) or 16 * D / 16 E4M3 (nvfp4).
# ---------------------------------------------------------------------------
E2M1 = json.load(open(os.path.join(GOLDEN, "e2m1_values.json")))["values"]


def _parse_page(page, fmt, D, bs=16):
    """Independent reading of one 4-bit page: [bs, D] decoded values
    (without the per-tensor scale), the codes, and the scales."""
    page = np.asarray(page, dtype=np.uint8)
    codes_b = page[:bs * D // 2].reshape(bs, D // 2)
    nib = np.stack([codes_b & 0xF, codes_b >> 4], axis=-1).reshape(bs, D)
    if fmt == "int4":
        sc = page[bs * D // 2:].view(np.float32)
        assert sc.shape == (bs,)
        signed = np.where(nib >= 8, nib.astype(np.int64) - 16, nib)
        return sc.astype(np.float64)[:, None] * signed, signed, sc
    bsc = page[bs * D // 2:].reshape(bs, D // 16)
    bval = torch.from_numpy(bsc.copy()).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()
    vals = np.asarray(E2M1, dtype=np.float64)[nib]
    return np.repeat(bval, 16, axis=1) * vals, nib, bsc


def test_e2m1_decode_matches_the_spec_table():
    for c in range(16):
        v = oracle.e2m1_to_double(c)
        assert v == E2M1[c] and np.signbit(v) == np.signbit(E2M1[c])


def test_e2m1_encode_nearest_ties_to_even_saturating():
    for c in range(16):
        assert oracle.e2m1_encode(E2M1[c]) == c               # round trip
    # midpoints go to the code whose mantissa bit is 0
    for y, c in ((0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4),
                 (3.5, 6), (5.0, 6), (-0.75, 10), (-5.0, 14)):
        assert oracle.e2m1_encode(y) == c, y
    for y, c in ((0.2501, 1), (0.7499, 1), (4.99, 6), (5.01, 7), (6.5, 7),
                 (1e30, 7), (-1e30, 15)):
        assert oracle.e2m1_encode(y) == c, y


def test_int4_encode_nearest_ties_to_even_clamped():
    for y, c in ((0.5, 0), (1.5, 2), (2.5, 2), (-0.5, 0), (-1.5, -2),
                 (6.5, 6), (7.4, 7), (7.6, 7), (-9.0, -7), (3.49, 3)):
        assert oracle.int4_encode(y) == c, y


def _write_4bit(fmt, x, D, scale=1.0):
    """Write tokens x [T, Hkv, D] (float32) into slots 0..T-1 of a fresh
    4-bit cache with the oracle; returns the cache."""
    T, Hkv, _ = x.shape
    nb = -(-T // 16)
    pb = oracle.page_bytes_4bit(fmt, D)
    kc = np.full((nb, Hkv, pb), 0xA5, dtype=np.uint8)
    vc = kc.copy()
    oracle.reshape_and_cache(x, x, kc, vc, np.arange(T), cache_dtype=fmt,
                             k_scale=scale, v_scale=scale)
    assert np.array_equal(kc, vc)
    return kc


def test_int4_write_properties():
    rng = np.random.default_rng(71)
    D = 64
    x = (rng.standard_normal((16, 2, D)) * rng.uniform(0.01, 100, (16, 2, 1))
         ).astype(np.float32)
    x[3, 1] = 0.0                                  # an all-zero token-head
    x[5, 0, :15] = 0.5 * np.arange(-7, 8)          # multiples of amax / 7
    x[5, 0, 15:] = 0.0
    kc = _write_4bit("int4", x, D)
    for h in range(2):
        deq, codes, sc = _parse_page(kc[0, h], "int4", D)
        for t in range(16):
            amax = float(np.abs(x[t, h]).max())
            if amax == 0.0:
                assert sc[t] == 0 and (codes[t] == 0).all()
                continue
            assert sc[t] == np.float32(amax) / np.float32(7.0)
            assert np.abs(codes[t]).max() == 7          # the extreme element
            err = np.abs(deq[t] - x[t, h].astype(np.float64))
            assert (err <= 0.5 * float(sc[t]) * (1 + 1e-6)).all()
            neg = _write_4bit("int4", -x[t:t + 1, h:h + 1], D)
            assert np.array_equal(_parse_page(neg[0, 0], "int4", D)[1][0],
                                  -codes[t])           # sign symmetric
    deq, _, _ = _parse_page(kc[0, 0], "int4", D)
    np.testing.assert_array_equal(deq[5], x[5, 0])


def test_nvfp4_write_properties():
    rng = np.random.default_rng(72)
    D, g = 128, 2.0 ** -6
    x = (rng.standard_normal((16, 1, D)) * rng.uniform(0.01, 5, (16, 1, 1))
         ).astype(np.float32)
    # a token whose values are on the grid: decoded exactly
    grid = np.asarray(E2M1[:8], dtype=np.float32)
    x[7, 0] = (g * 2.0 * grid[np.arange(D) % 8]).astype(np.float32)
    kc = _write_4bit("nvfp4", x, D, scale=g)
    deq, codes, bsc = _parse_page(kc[0, 0], "nvfp4", D)
    for t in range(16):
        for b in range(D // 16):
            blk = x[t, 0, 16 * b:16 * b + 16]
            amax = float(np.abs(blk).max())
            want = torch.tensor((np.float32(amax) / np.float32(6.0)) /
                                np.float32(g)).to(torch.float8_e4m3fn)
            assert bsc[t, b] == int(want.view(torch.uint8))
            r = np.float32(float(want.to(torch.float64)) * g)
            # each element decodes to the grid point nearest to x / r (a
            # tie may go either way here; the encoder pin fixes ties)
            y = blk / r
            got = deq[t, 16 * b:16 * b + 16] / float(want.to(torch.float64))
            dist = np.abs(np.abs(y)[:, None] - grid[None, :])
            nearest = grid[np.argmin(dist, axis=1)] * np.sign(y)
            assert (np.abs(np.abs(got) - np.abs(nearest)) <=
                    (np.sort(dist, 1)[:, 1] - np.sort(dist, 1)[:, 0] < 1e-6)
                    * 2.0 + 1e-12).all()
    np.testing.assert_allclose(deq[7] * g, x[7, 0], rtol=0, atol=0)


@pytest.mark.parametrize("fmt", ["int4", "nvfp4"])
def test_4bit_attention_equals_sdpa_on_decoded_values(fmt):
    rng = np.random.default_rng(73)
    Hq, Hkv, D, NB = 8, 2, 32, 20
    shapes = [(1, 45), (4, 33), (2, 16), (9, 40)]
    q, kc_f, vc_f, reqs, qs, ks, vs = random_paged_step(rng, shapes, Hq, Hkv,
                                                        D, NB)
    md = oracle.step_metadata(reqs)
    g = 0.01 if fmt == "nvfp4" else 1.0
    pb = oracle.page_bytes_4bit(fmt, D)
    kc = np.zeros((NB, Hkv, pb), dtype=np.uint8)
    vc = np.zeros((NB, Hkv, pb), dtype=np.uint8)
    kk = np.concatenate(ks, 0)
    vv = np.concatenate(vs, 0)
    slots = np.concatenate([[oracle.slot_of(r.block_ids, j) for j in
                             range(r.num_computed + r.num_new)] for r in reqs])
    oracle.reshape_and_cache(kk, vv, kc, vc, slots, cache_dtype=fmt,
                             k_scale=g, v_scale=g)
    out = oracle.paged_attention(q, kc, vc, md["block_tables"],
                                 md["seq_lens"], md["query_start_loc"],
                                 scale=0.3, cache_dtype=fmt, k_scale=g,
                                 v_scale=g)

    def decoded(cache, r):
        L = r.num_computed + r.num_new
        rows = []
        for j in range(L):
            b, o = r.block_ids[j // 16], j % 16
            rows.append([_parse_page(cache[b, h], fmt, D)[0][o] for h in
                         range(Hkv)])
        return np.asarray(rows) * g

    ref = sdpa_reference([x.astype(np.float64) for x in qs],
                         [decoded(kc, r) for r in reqs],
                         [decoded(vc, r) for r in reqs], Hq // Hkv, 0.3)
    np.testing.assert_allclose(out, np.concatenate(ref, 0), rtol=0,
                               atol=1e-12)


@pytest.mark.parametrize("fmt", ["int4", "nvfp4"])
def test_4bit_copy_blocks_copies_whole_pages(fmt):
    rng = np.random.default_rng(74)
    pb = oracle.page_bytes_4bit(fmt, 128)
    kc = rng.integers(0, 256, size=(9, 4, pb), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(9, 4, pb), dtype=np.uint8)
    k0, v0 = kc.copy(), vc.copy()
    oracle.copy_blocks(kc, vc, np.array([[2, 7], [0, 5]]), cache_dtype=fmt,
                       head_dim=128)
    np.testing.assert_array_equal(kc[7], k0[2])
    np.testing.assert_array_equal(vc[5], v0[0])
    keep = [0, 1, 2, 3, 4, 6, 8]
    np.testing.assert_array_equal(kc[keep], k0[keep])
    np.testing.assert_array_equal(vc[keep], v0[keep])
