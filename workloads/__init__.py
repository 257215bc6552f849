"""Seeded synthetic inputs for the paged-KV attention step.

This module is the only code shared by the CUDA path's tests/benchmark and
the CPU oracle.  It draws inputs and lays them out; it computes nothing the
method computes (no attention, no slot metadata, no block copies): it decides
which physical blocks each request owns, fills the cache pages that hold
cached tokens with N(0, 1) values and poisons every other cache slot with
NaN so that a read of an unowned slot cannot go unnoticed.

The five named workloads follow the shapes the pages' discussion uses
("vLLM engine anatomy": Figure 2 layout, Table 1 model shapes, Figure 3 mixed
steps; "vLLM V1 engine architecture": the 1022-token chunk in a 1024-token
budget; "01. vLLM": the 2,000-token shared prefix = 125 blocks of 16, FP8 KV
cache).  Seeds are 82000 + config number.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

BLOCK_SIZE = 16

_TORCH_DT = {"f32": torch.float32, "f16": torch.float16,
             "bf16": torch.bfloat16}
FOUR_BIT = ("int4", "nvfp4")


def page_bytes_4bit(cache_dtype: str, head_dim: int) -> int:
    """Bytes of one (block, KV head) page of a 4-bit cache: 16 tokens x
    head_dim / 2 bytes of codes, then 16 fp32 scales (int4) or 16 x
    head_dim / 16 E4M3 block scales (nvfp4)."""
    return 8 * head_dim + (64 if cache_dtype == "int4" else head_dim)
# NaN bit patterns used to poison unowned cache slots
_NAN_BITS = {"f32": 0x7FC00000, "f16": 0x7E00, "bf16": 0x7FC0, "e4m3": 0x7F}
_ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}


@dataclass
class Request:
    """One entry of the step {request_id: num_tokens}.

    block_ids    -- physical blocks of the request's block table (after this
                    step's allocations and copy-on-write remapping)
    num_computed -- tokens whose K/V are already in the cache
    num_new      -- tokens scheduled in this step
    """
    block_ids: List[int]
    num_computed: int
    num_new: int

    @property
    def seq_len(self) -> int:
        return self.num_computed + self.num_new


@dataclass
class Workload:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    q_dtype: str            # "f32" | "f16" | "bf16"
    cache_dtype: str        # "f32" | "f16" | "bf16" | "e4m3" | "int4" | "nvfp4"
    scale: float
    k_scale: float
    v_scale: float
    requests: List[Request]
    copy_pairs: List[Tuple[int, int]]
    write_new: bool         # True: this step's K/V still have to be written
    q: torch.Tensor         # [T, Hq, D]  (CPU)
    key: Optional[torch.Tensor]    # [T, Hkv, D] new tokens' K (CPU) or None
    value: Optional[torch.Tensor]  # [T, Hkv, D]
    k_cache: torch.Tensor   # [NB, Hkv, 16, D] (uint8 bit patterns for e4m3)
    v_cache: torch.Tensor
    block_size: int = BLOCK_SIZE
    shared_blocks: List[int] = field(default_factory=list)
    description: str = ""
    sliding_window: int = 0  # keys a query sees through a window (0: all)

    @property
    def num_tokens(self) -> int:
        return sum(r.num_new for r in self.requests)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def kv_bytes(self, unique: bool = True) -> int:
        """Bytes of K and V the step's attention must read: every key some
        query of a request sees, once (a block shared by several requests
        counted once when unique=True); a 4-bit cache's scales included.
        With a sliding window of W keys a request of n new tokens after L - n
        cached sees keys max(0, L - n - W + 1) .. L - 1."""
        if self.cache_dtype in FOUR_BIT:
            per_token = 2 * self.num_kv_heads * page_bytes_4bit(
                self.cache_dtype, self.head_dim) // BLOCK_SIZE
        else:
            per_token = (2 * _ELEM_BYTES[self.cache_dtype] *
                         self.num_kv_heads * self.head_dim)
        W = self.sliding_window

        def first_key(r):
            return max(0, r.seq_len - r.num_new - W + 1) if W > 0 else 0
        if not unique:
            return per_token * sum(r.seq_len - first_key(r)
                                   for r in self.requests)
        seen = {}
        for r in self.requests:
            L, lo = r.seq_len, first_key(r)
            for k, b in enumerate(r.block_ids):
                n = min(BLOCK_SIZE, L - k * BLOCK_SIZE) - max(0, lo - k * BLOCK_SIZE)
                if n > 0:
                    seen[b] = max(seen.get(b, 0), n)
        return per_token * sum(seen.values())

    def qo_bytes(self) -> int:
        eb = _ELEM_BYTES[self.q_dtype]
        return 2 * self.num_tokens * self.num_q_heads * self.head_dim * eb


# --------------------------------------------------------------------------
# fast, reproducible N(0,1) draws: fixed-size chunks, each from its own child
# seed, so the values do not depend on the number of threads.
# --------------------------------------------------------------------------
_CHUNK = 1 << 22


def normal_f32(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    nchunks = max(1, -(-n // _CHUNK))
    children = np.random.SeedSequence([seed, stream]).spawn(nchunks)

    def fill(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        if hi > lo:
            np.random.default_rng(children[i]).standard_normal(
                out=out[lo:hi], dtype=np.float32)

    workers = min(nchunks, os.cpu_count() or 1)
    if workers > 1:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    else:
        for i in range(nchunks):
            fill(i)
    return out


def _to_dtype(x: np.ndarray, dtype: str, scale: float = 1.0) -> torch.Tensor:
    t = torch.from_numpy(x)
    if dtype == "e4m3":
        # input bytes for an FP8 cache: N(0,1) values quantised with torch's
        # own fp8 cast (clamped to the finite range first)
        return (t / scale).clamp_(-448.0, 448.0).to(
            torch.float8_e4m3fn).view(torch.uint8)
    return t.to(_TORCH_DT[dtype])


def _nan_tensor(shape, dtype: str) -> torch.Tensor:
    if dtype == "e4m3":
        return torch.full(shape, _NAN_BITS["e4m3"], dtype=torch.uint8)
    return torch.full(shape, float("nan"), dtype=_TORCH_DT[dtype])


def _fill_cache(cache: torch.Tensor, filled: dict, dtype: str, seed: int,
                stream: int, scale: float) -> None:
    """Give the first n tokens of each listed block N(0,1) contents.

    filled: {physical block: number of leading tokens holding data}.
    """
    if not filled:
        return
    _, H, bs, D = cache.shape
    blocks = np.fromiter(filled.keys(), dtype=np.int64, count=len(filled))
    counts = np.fromiter(filled.values(), dtype=np.int64, count=len(filled))
    per_block = H * bs * D
    step = max(1, (1 << 24) // per_block)
    for s in range(0, len(blocks), step):
        bsel = blocks[s:s + step]
        vals = normal_f32(seed, stream * 1_000_003 + s, len(bsel) * per_block)
        vals = _to_dtype(vals, dtype, scale).view(len(bsel), H, bs, D)
        # tokens past each block's count stay NaN
        cnt = torch.from_numpy(counts[s:s + step])
        keep = torch.arange(bs)[None, :] < cnt[:, None]          # [n, bs]
        dst = cache[torch.from_numpy(bsel)]
        dst = torch.where(keep[:, None, :, None], vals, dst)
        cache[torch.from_numpy(bsel)] = dst


def _fill_cache_4bit(cache: torch.Tensor, filled: dict, fmt: str,
                     head_dim: int, seed: int, stream: int) -> None:
    """4-bit pages (see page_bytes_4bit): random codes in every token slot
    of the listed blocks; scales random for the first n tokens of each block
    (int4: 0.05 + 0.25 |N(0,1)|; nvfp4: E4M3 codes of 0.25 .. 0.94) and NaN
    for the rest (int4: fp32 NaN; nvfp4: the E4M3 NaN code), so that a read
    of an unwritten slot shows."""
    if not filled:
        return
    NB, H, pb = cache.shape
    cb = BLOCK_SIZE * head_dim // 2
    blocks = np.fromiter(filled.keys(), dtype=np.int64, count=len(filled))
    counts = np.fromiter(filled.values(), dtype=np.int64, count=len(filled))
    step = max(1, (1 << 22) // (H * pb))
    for s0 in range(0, len(blocks), step):
        bsel = blocks[s0:s0 + step]
        n = len(bsel)
        rng = np.random.default_rng(np.random.SeedSequence([seed, stream, s0]))
        pages = np.empty((n, H, pb), dtype=np.uint8)
        pages[:, :, :cb] = rng.integers(0, 256, size=(n, H, cb), dtype=np.uint8)
        keep = (np.arange(BLOCK_SIZE)[None, :] <
                counts[s0:s0 + step][:, None])                  # [n, 16]
        if fmt == "int4":
            sc = (0.05 + 0.25 * np.abs(rng.standard_normal(
                (n, H, BLOCK_SIZE)))).astype(np.float32)
            sc = np.where(keep[:, None, :], sc, np.float32(np.nan))
            pages[:, :, cb:] = sc.view(np.uint8).reshape(n, H, 4 * BLOCK_SIZE)
        else:
            nsc = BLOCK_SIZE * head_dim // 16
            sc = rng.integers(0x28, 0x38, size=(n, H, BLOCK_SIZE, head_dim // 16),
                              dtype=np.uint8)
            sc = np.where(keep[:, None, :, None], sc, np.uint8(0x7F))
            pages[:, :, cb:] = sc.reshape(n, H, nsc)
        cache[torch.from_numpy(bsel)] = torch.from_numpy(pages)


def make_workload(name: str, seed: int, *, num_q_heads: int,
                  num_kv_heads: int, head_dim: int, num_blocks: int,
                  q_dtype: str, cache_dtype: str, requests: Sequence[Request],
                  filled: dict, write_new: bool,
                  copy_pairs: Sequence[Tuple[int, int]] = (),
                  scale: Optional[float] = None, k_scale: float = 1.0,
                  v_scale: float = 1.0, shared_blocks=(),
                  description: str = "") -> Workload:
    """Draw q, the new tokens' K/V and the cache contents for a step whose
    block ownership is already decided (`filled` lists the cached tokens per
    physical block)."""
    T = sum(r.num_new for r in requests)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    q = _to_dtype(normal_f32(seed, 1, T * num_q_heads * head_dim),
                  q_dtype).view(T, num_q_heads, head_dim)
    key = value = None
    if write_new:
        key = _to_dtype(normal_f32(seed, 2, T * num_kv_heads * head_dim),
                        q_dtype).view(T, num_kv_heads, head_dim)
        value = _to_dtype(normal_f32(seed, 3, T * num_kv_heads * head_dim),
                          q_dtype).view(T, num_kv_heads, head_dim)
    if cache_dtype in FOUR_BIT:
        shape4 = (num_blocks, num_kv_heads,
                  page_bytes_4bit(cache_dtype, head_dim))
        k_cache = torch.zeros(shape4, dtype=torch.uint8)
        v_cache = torch.zeros(shape4, dtype=torch.uint8)
        # every slot starts unwritten: NaN scales
        for c in (k_cache, v_cache):
            view = c.view(num_blocks * num_kv_heads, -1)
            cb = BLOCK_SIZE * head_dim // 2
            if cache_dtype == "int4":
                view[:, cb:] = torch.full((BLOCK_SIZE,), float("nan"),
                                          dtype=torch.float32).view(torch.uint8)
            else:
                view[:, cb:] = 0x7F
        _fill_cache_4bit(k_cache, filled, cache_dtype, head_dim, seed, 4)
        _fill_cache_4bit(v_cache, filled, cache_dtype, head_dim, seed, 5)
    else:
        shape = (num_blocks, num_kv_heads, BLOCK_SIZE, head_dim)
        k_cache = _nan_tensor(shape, cache_dtype)
        v_cache = _nan_tensor(shape, cache_dtype)
        _fill_cache(k_cache, filled, cache_dtype, seed, 4, k_scale)
        _fill_cache(v_cache, filled, cache_dtype, seed, 5, v_scale)
    return Workload(name=name, seed=seed, num_q_heads=num_q_heads,
                    num_kv_heads=num_kv_heads, head_dim=head_dim,
                    num_blocks=num_blocks, q_dtype=q_dtype,
                    cache_dtype=cache_dtype, scale=float(scale),
                    k_scale=float(k_scale), v_scale=float(v_scale),
                    requests=list(requests), copy_pairs=list(copy_pairs),
                    write_new=write_new, q=q, key=key, value=value,
                    k_cache=k_cache, v_cache=v_cache,
                    shared_blocks=list(shared_blocks),
                    description=description)


def _blocks_for(n_tokens: int) -> int:
    return -(-n_tokens // BLOCK_SIZE)


class _Pool:
    """Hands out physical blocks in the order of a seeded permutation."""

    def __init__(self, rng, num_blocks: int, permute: bool = True):
        self.order = rng.permutation(num_blocks) if permute else \
            np.arange(num_blocks)
        self.next = 0

    def take(self, n: int) -> List[int]:
        if self.next + n > len(self.order):
            raise ValueError("block pool exhausted")
        out = [int(b) for b in self.order[self.next:self.next + n]]
        self.next += n
        return out


def _leading(filled: dict, blocks: Sequence[int], n_tokens: int) -> None:
    """Mark the first n_tokens positions of a block list as cached."""
    for k, b in enumerate(blocks):
        n = min(BLOCK_SIZE, n_tokens - k * BLOCK_SIZE)
        if n > 0:
            filled[b] = max(filled.get(b, 0), n)


def decode_step(name: str, seed: int, *, seq_lens: Sequence[int],
                num_q_heads: int, num_kv_heads: int, head_dim: int,
                num_blocks: int, dtype: str, cache_dtype: Optional[str] = None,
                permute: bool = True, write_new: bool = False,
                k_scale: float = 1.0, v_scale: float = 1.0,
                q_lens: Optional[Sequence[int]] = None,
                description: str = "") -> Workload:
    """A step where request i has seq_lens[i] keys and q_lens[i] (default 1)
    new tokens; blocks consecutive from a seeded permutation of the pool.
    write_new=False: the cache already holds all keys (the new tokens were
    written earlier); True: only the first seq_len - q_len are cached."""
    rng = np.random.default_rng(seed)
    pool = _Pool(rng, num_blocks, permute)
    cache_dtype = cache_dtype or dtype
    if q_lens is None:
        q_lens = [1] * len(seq_lens)
    reqs, filled = [], {}
    for L, n in zip(seq_lens, q_lens):
        blocks = pool.take(_blocks_for(L))
        cached = L - n if write_new else L
        _leading(filled, blocks, cached)
        reqs.append(Request(blocks, L - n, n))
    return make_workload(name, seed, num_q_heads=num_q_heads,
                         num_kv_heads=num_kv_heads, head_dim=head_dim,
                         num_blocks=num_blocks, q_dtype=dtype,
                         cache_dtype=cache_dtype, requests=reqs,
                         filled=filled, write_new=write_new, k_scale=k_scale,
                         v_scale=v_scale, description=description)


def shared_prefix_step(name: str, seed: int, *, prefix_blocks: int,
                       private: Sequence[int], q_lens: Sequence[int],
                       num_q_heads: int, num_kv_heads: int, head_dim: int = 128,
                       dtype: str = "bf16", cache_dtype: Optional[str] = None,
                       num_blocks: Optional[int] = None, k_scale: float = 1.0,
                       v_scale: float = 1.0, description: str = "") -> Workload:
    """A step whose requests all begin with the same `prefix_blocks` full
    blocks (a cached shared prefix, "01. vLLM", prefix caching): request i
    has `private[i]` more cached tokens of its own after the prefix, then
    q_lens[i] new tokens (written by the step).  Blocks come from a seeded
    permutation of the pool."""
    rng = np.random.default_rng(seed)
    cache_dtype = cache_dtype or dtype
    prefix = prefix_blocks * BLOCK_SIZE
    if num_blocks is None:
        num_blocks = prefix_blocks + sum(
            _blocks_for(prefix + p + n) - prefix_blocks
            for p, n in zip(private, q_lens)) + 5
    pool = _Pool(rng, num_blocks, True)
    shared = pool.take(prefix_blocks)
    filled: dict = {}
    _leading(filled, shared, prefix)
    reqs = []
    for p_, n in zip(private, q_lens):
        ctx = prefix + int(p_)
        blocks = shared + pool.take(_blocks_for(ctx + n) - prefix_blocks)
        _leading(filled, blocks, ctx)
        reqs.append(Request(blocks, ctx, int(n)))
    return make_workload(name, seed, num_q_heads=num_q_heads,
                         num_kv_heads=num_kv_heads, head_dim=head_dim,
                         num_blocks=num_blocks, q_dtype=dtype,
                         cache_dtype=cache_dtype, requests=reqs, filled=filled,
                         write_new=True, k_scale=k_scale, v_scale=v_scale,
                         shared_blocks=shared, description=description)


# --------------------------------------------------------------------------
# the five named configurations
# --------------------------------------------------------------------------
def config1() -> Workload:
    """Tiny decode on the layout of Figure 2 ("vLLM engine anatomy"): 12
    blocks of 16; A has 40 cached tokens in blocks [0,1,2], B has 20 in
    [3,4]; one new token each; 4 query heads / 2 KV heads, head_dim 64,
    fp32, scale 1/8."""
    seed = 82001
    reqs = [Request([0, 1, 2], 40, 1), Request([3, 4], 20, 1)]
    filled = {}
    _leading(filled, [0, 1, 2], 40)
    _leading(filled, [3, 4], 20)
    return make_workload("cfg1_fig2_tiny", seed, num_q_heads=4,
                         num_kv_heads=2, head_dim=64, num_blocks=12,
                         q_dtype="f32", cache_dtype="f32", requests=reqs,
                         filled=filled, write_new=True, scale=1.0 / 8.0,
                         description="Figure-2 layout, fp32, 2 decodes")


def config2(batch: int = 64, lo: int = 512, hi: int = 4096,
            num_blocks: int = 20000, cache_dtype: str = "bf16",
            head_dim: int = 128) -> Workload:
    """Llama-3.1-8B-shaped decode: 32q/8kv heads, head_dim 128, bf16, batch
    64, context uniform in [512, 4096], 20,000-block permuted pool.  With
    cache_dtype "int4" / "nvfp4" the same batch over a 4-bit cache (NVFP4
    tensor scales 0.5 for K, 0.25 for V)."""
    seed = 82002
    rng = np.random.default_rng([seed, 7])
    lens = rng.integers(lo, hi, size=batch, endpoint=True).tolist()
    nv = cache_dtype == "nvfp4"
    return decode_step("cfg2_llama31_8b_decode", seed, seq_lens=lens,
                       num_q_heads=32, num_kv_heads=8, head_dim=head_dim,
                       num_blocks=num_blocks, dtype="bf16",
                       cache_dtype=cache_dtype,
                       k_scale=0.5 if nv else 1.0, v_scale=0.25 if nv else 1.0,
                       description=(f"{batch} decodes, L~U[{lo},{hi}], "
                                    f"{cache_dtype} KV, head_dim {head_dim}"))


def config3(batch: int = 32, seq_len: int = 8192,
            num_blocks: Optional[int] = None) -> Workload:
    """Llama-2-7B-shaped MHA decode: 32 = 32 heads, head_dim 128, fp16,
    batch 32 x 8192 keys; pool = exactly the blocks needed, permuted."""
    seed = 82003
    need = batch * _blocks_for(seq_len)
    return decode_step("cfg3_llama2_7b_mha_decode", seed,
                       seq_lens=[seq_len] * batch, num_q_heads=32,
                       num_kv_heads=32, head_dim=128,
                       num_blocks=num_blocks or need, dtype="f16",
                       description=f"{batch} x {seq_len} keys, MHA, fp16")


def config4(num_decodes: int = 120, lo: int = 1024, hi: int = 8192,
            prefix: int = 2000, chunk: int = 1022,
            num_blocks: int = 65536) -> Workload:
    """Mixed unified step, Llama-3.1-8B shape, bf16.

    All requests share a `prefix`-token prefix held in the same physical
    blocks.  `num_decodes` one-token decodes with a private context of
    U[lo, hi] tokens after the prefix; request 1 is a fork of request 0
    (same blocks, last block partial and shared) and gets its own copy of
    that block by copy-on-write before the step writes; one chunked prefill
    of `chunk` new tokens after the prefix."""
    seed = 82004
    rng = np.random.default_rng(seed)
    pool = _Pool(rng, num_blocks, True)
    n_pref_blocks = _blocks_for(prefix)
    prefix_blocks = pool.take(n_pref_blocks)
    filled = {}
    _leading(filled, prefix_blocks, prefix)
    priv = rng.integers(lo, hi, size=num_decodes, endpoint=True)
    while (prefix + int(priv[0])) % BLOCK_SIZE == 0:
        priv[0] = rng.integers(lo, hi, endpoint=True)
    if num_decodes > 1:
        priv[1] = priv[0]
    reqs, copy_pairs = [], []
    r0_blocks = None
    for i in range(num_decodes):
        ctx = prefix + int(priv[i])
        L = ctx + 1
        if i == 1 and r0_blocks is not None:
            # fork of request 0: same table; its last block is copied on write
            dst = pool.take(1)[0]
            copy_pairs.append((r0_blocks[-1], dst))
            reqs.append(Request(r0_blocks[:-1] + [dst], ctx, 1))
            continue
        own = pool.take(_blocks_for(L) - n_pref_blocks)
        blocks = prefix_blocks + own
        _leading(filled, blocks, ctx)
        reqs.append(Request(blocks, ctx, 1))
        if i == 0:
            r0_blocks = blocks
    own = pool.take(_blocks_for(prefix + chunk) - n_pref_blocks)
    reqs.append(Request(prefix_blocks + own, prefix, chunk))
    return make_workload("cfg4_mixed_step", seed, num_q_heads=32,
                         num_kv_heads=8, head_dim=128, num_blocks=num_blocks,
                         q_dtype="bf16", cache_dtype="bf16", requests=reqs,
                         filled=filled, write_new=True,
                         copy_pairs=copy_pairs, shared_blocks=prefix_blocks,
                         description=(f"{num_decodes} decodes + {chunk}-token "
                                      f"chunk after a {prefix}-token shared "
                                      "prefix, 1 copy-on-write, bf16"))


def config5(batch: int = 16, lo: int = 32768, hi: int = 131072,
            num_blocks: Optional[int] = None) -> Workload:
    """Llama-3.1-70B-shaped long-context decode: 64q/8kv heads, head_dim
    128, bf16 q, FP8 E4M3 cache (k_scale 0.0125, v_scale 0.015), batch 16,
    context U[32768, 131072], one new token each written bf16 -> fp8."""
    seed = 82005
    rng = np.random.default_rng([seed, 7])
    ctx = rng.integers(lo, hi, size=batch, endpoint=True)
    lens = (ctx + 1).tolist()
    nb = num_blocks or batch * _blocks_for(hi + 1)
    return decode_step("cfg5_llama31_70b_fp8_longctx", seed, seq_lens=lens,
                       num_q_heads=64, num_kv_heads=8, head_dim=128,
                       num_blocks=nb, dtype="bf16", cache_dtype="e4m3",
                       write_new=True, k_scale=0.0125, v_scale=0.015,
                       description=(f"{batch} decodes, ctx~U[{lo},{hi}], "
                                    "FP8 E4M3 KV"))


def prefill_chunk(ctx: int = 4096, new: int = 4096,
                  cache_dtype: str = "bf16") -> Workload:
    """One chunked prefill, Llama-3.1-8B shape (32q/8kv heads, head_dim 128,
    bf16 q): `new` prompt tokens after `ctx` cached ones, already in the cache
    (the step attends only).  Used to measure the prefill tiles alone.  With
    cache_dtype "e4m3" the cache is FP8 (scales 0.0125 / 0.015)."""
    seed = 82006
    L = ctx + new
    fp8 = cache_dtype == "e4m3"
    return decode_step("prefill_chunk_llama31_8b", seed, seq_lens=[L],
                       q_lens=[new], num_q_heads=32, num_kv_heads=8,
                       head_dim=128, num_blocks=_blocks_for(L) + 8,
                       dtype="bf16", cache_dtype=cache_dtype, write_new=False,
                       k_scale=0.0125 if fp8 else 1.0,
                       v_scale=0.015 if fp8 else 1.0,
                       description=(f"1 prefill chunk: {new} new after {ctx}, "
                                    f"{cache_dtype} KV"))


def shared_prefix_decode(num_decodes: int = 32, prefix_blocks: int = 1024,
                         lo: int = 256, hi: int = 2048,
                         seed: Optional[int] = None,
                         cache_dtype: str = "bf16") -> Workload:
    """Decodes behind one long shared prompt prefix (prefix caching hands
    every request the same `prefix_blocks` full blocks, "01. vLLM", prefix
    caching), Llama-3.1-8B shape, bf16: each request has a private context of
    U[lo, hi) tokens after the prefix, then one new token (written by the
    step).  The default is 32 decodes behind a 16,384-token prefix.  With
    cache_dtype "e4m3" the cache is FP8 (scales 0.02 / 0.03)."""
    seed = 82007 + num_decodes + 7 * prefix_blocks if seed is None else seed
    rng = np.random.default_rng(seed)
    private = [int(x) for x in rng.integers(lo, hi, size=num_decodes)]
    fp8 = cache_dtype == "e4m3"
    return shared_prefix_step(
        "shared_prefix_decode_llama31_8b", seed, prefix_blocks=prefix_blocks,
        private=private, q_lens=[1] * num_decodes, num_q_heads=32,
        num_kv_heads=8, head_dim=128, dtype="bf16", cache_dtype=cache_dtype,
        k_scale=0.02 if fp8 else 1.0, v_scale=0.03 if fp8 else 1.0,
        description=(f"{num_decodes} decodes behind a shared "
                     f"{prefix_blocks * BLOCK_SIZE}-token prefix, private "
                     f"context U[{lo},{hi}), {cache_dtype} KV"))


def sliding_window_decode(batch: int = 64, lo: int = 2048, hi: int = 12288,
                          window: int = 1024) -> Workload:
    """Decodes of a sliding-window layer ("01. vLLM", the hybrid KV cache
    manager paragraph: layers whose queries see only the last `window`
    keys), Llama-3.1-8B shape, bf16: `batch` requests with contexts U[lo,
    hi], each query seeing its last `window` keys."""
    seed = 82008
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(lo, hi, size=batch, endpoint=True)]
    wl = decode_step("sliding_window_decode_llama31_8b", seed, seq_lens=lens,
                     num_q_heads=32, num_kv_heads=8, head_dim=128,
                     num_blocks=sum(_blocks_for(L) for L in lens) + 64,
                     dtype="bf16",
                     description=(f"{batch} decodes, L~U[{lo},{hi}], window "
                                  f"{window}, bf16"))
    wl.sliding_window = window
    return wl


def attention_flops(wl: Workload) -> int:
    """Multiply-adds x 2 of Q.K^T and P.V over the visible (row, key) pairs
    of the step: query i of a request with n new tokens and L keys sees
    L - n + i + 1 keys."""
    pairs = 0
    for r in wl.requests:
        L = r.num_computed + r.num_new
        n = r.num_new
        pairs += n * (L - n) + n * (n + 1) // 2
    return pairs * wl.num_q_heads * wl.head_dim * 2 * 2


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}
