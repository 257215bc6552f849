"""CPU fp64 oracle for the paged-KV attention step.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library in ``paged_kv_cache_82_gb300`` and imports nothing from
it; the two meet only in the seeded input generators of ``workloads``.

The arithmetic lives in ``pa_oracle.c`` (plain C, double precision, compiled
here with gcc).  This module marshals numpy / torch-CPU arrays into it and adds
the host-side step metadata (slot numbers, query offsets) written out from
the same definitions:

* "vLLM engine anatomy", section "PagedAttention: paging the KV cache",
  Figure 2 -- 16-token physical blocks; token j of a sequence is at offset
  j % 16 of block ``block_table[j // 16]``.
* "vLLM V1 engine architecture ...", "Scheduler forms one round of work" and
  "A 1024-token budget example" -- a step is ``{request: num_tokens}``.
* "vLLM V0 vs V1", section 3.1 -- per request: query length, context length,
  block table.

Parity status of every function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# element type codes of pa_oracle.c
F32, F16, BF16, E4M3, INT4, NVFP4 = 0, 1, 2, 3, 4, 5
_DT_NAMES = {"f32": F32, "f16": F16, "bf16": BF16, "e4m3": E4M3,
             "int4": INT4, "nvfp4": NVFP4}
_ELEM_BYTES = {F32: 4, F16: 2, BF16: 2, E4M3: 1}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc (ISO C11, no fast-math, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-D_POSIX_C_SOURCE=200809L", "-o", tmp, _SRC,
           "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    i64, i32, f32, f64 = (ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                          ctypes.c_double)
    lib.orc_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_f16_to_double.restype = f64
    lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_double.restype = f64
    lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_to_double.restype = f64
    lib.orc_e4m3_encode.argtypes = [f32]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_e2m1_to_double.argtypes = [ctypes.c_uint8]
    lib.orc_e2m1_to_double.restype = f64
    lib.orc_e2m1_encode.argtypes = [f32]
    lib.orc_e2m1_encode.restype = ctypes.c_uint8
    lib.orc_int4_encode.argtypes = [f32]
    lib.orc_int4_encode.restype = i32
    lib.orc_reshape_and_cache.argtypes = [P, P, i32, i64, i64, i64, P, P,
                                          i32, i64, i32, i32, i32, P, f32,
                                          f32]
    lib.orc_reshape_and_cache.restype = i32
    lib.orc_copy_blocks.argtypes = [P, P, i32, i64, i32, i32, i32, P, i64]
    lib.orc_copy_blocks.restype = i32
    lib.orc_paged_attention.argtypes = [P, i32, P, P, i32, i64, i32, i32,
                                        i32, i32, P, i32, P, P, i32, f64,
                                        f64, f64, P, i32, i32]
    lib.orc_paged_attention.restype = i32
    lib.orc_paged_attention_row.argtypes = [P, i32, P, P, i32, i64, i32,
                                            i32, i32, i32, P, i32, P, P,
                                            i32, i32, i32, f64, f64, f64, P,
                                            i32]
    lib.orc_paged_attention_row.restype = i32
    lib.orc_kv_bytes_per_token.argtypes = [i64, i64, i64, i64]
    lib.orc_kv_bytes_per_token.restype = i64
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def swap_library(path):
    """Use the oracle compiled at `path` instead of the default one (the
    tests use this to plant mistakes in copies of pa_oracle.c).  Returns the
    previous library object; pass it to restore_library."""
    global _lib
    old = _load()
    with _lock:
        _lib = _bind(ctypes.CDLL(path))
    return old


def restore_library(lib):
    global _lib
    with _lock:
        _lib = lib


class OracleError(RuntimeError):
    pass


def _check(status: int, what: str) -> None:
    if status != 0:
        raise OracleError(f"{what}: oracle status {status}")


# --------------------------------------------------------------------------
# array marshalling: numpy arrays, or torch CPU tensors (bf16 / fp8 stored
# as their bit patterns).
# --------------------------------------------------------------------------
def _as_np(x):
    """Return (contiguous numpy array, dtype code or None) for x."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        if x.device.type != "cpu":
            raise OracleError("oracle inputs must live in host memory")
        x = x.contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), BF16
        if x.dtype == torch.float16:
            return x.numpy(), F16
        if x.dtype == torch.float32:
            return x.numpy(), F32
        if x.dtype == getattr(torch, "float8_e4m3fn", None):
            return x.view(torch.uint8).numpy(), E4M3
        return x.numpy(), None
    x = np.ascontiguousarray(x)
    code = {np.dtype(np.float32): F32, np.dtype(np.float16): F16}.get(x.dtype)
    return x, code


def _dt(code_or_name, fallback):
    if code_or_name is None:
        if fallback is None:
            raise OracleError("element type must be given for this array")
        return fallback
    if isinstance(code_or_name, str):
        return _DT_NAMES[code_or_name]
    return int(code_or_name)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# scalar format helpers (exact)
# --------------------------------------------------------------------------
def f16_bits_to_double(bits: int) -> float:
    return _load().orc_f16_to_double(bits & 0xFFFF)


def bf16_bits_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(bits & 0xFFFF)


def e4m3_to_double(code: int) -> float:
    return _load().orc_e4m3_to_double(code & 0xFF)


def e4m3_encode(y: float) -> int:
    """E4M3 code nearest to the fp32 value y (ties to even, saturating)."""
    return int(_load().orc_e4m3_encode(float(np.float32(y))))


def e2m1_to_double(code: int) -> float:
    return _load().orc_e2m1_to_double(code & 0xF)


def e2m1_encode(y: float) -> int:
    """E2M1 code nearest to the fp32 value y (ties to even, saturating)."""
    return int(_load().orc_e2m1_encode(float(np.float32(y))))


def int4_encode(y: float) -> int:
    """Nearest integer to the fp32 value y (ties to even) in [-7, 7]."""
    return int(_load().orc_int4_encode(float(np.float32(y))))


def page_bytes_4bit(cache_dtype, head_dim: int, block_size: int = 16) -> int:
    """Bytes of one (block, KV head) page of a 4-bit cache: the codes, then
    one fp32 scale per token (int4) or one E4M3 scale per 16 elements
    (nvfp4)."""
    codes = block_size * head_dim // 2
    dt = _dt(cache_dtype, None)
    return codes + (4 * block_size if dt == INT4 else
                    block_size * head_dim // 16)


def _geometry(cache, head_dim=None, block_size=16):
    """(num_blocks, kv_heads, block_size, head_dim) of a cache array:
    [NB, Hkv, bs, D] elements, or [NB, Hkv, page_bytes] for the 4-bit
    formats (head_dim given)."""
    if cache.ndim == 4:
        return cache.shape
    if head_dim is None:
        raise OracleError("a 4-bit cache needs head_dim")
    return cache.shape[0], cache.shape[1], block_size, head_dim


def kv_bytes_per_token(elem_bytes: int, layers: int, kv_heads: int,
                       head_dim: int) -> int:
    """Table 1 of "vLLM engine anatomy": 2 x elem bytes x layers x KV heads x
    head dim."""
    return int(_load().orc_kv_bytes_per_token(elem_bytes, layers, kv_heads,
                                              head_dim))


# --------------------------------------------------------------------------
# step metadata (host) -- "vLLM engine anatomy" Figure 2; "vLLM V0 vs V1" 3.1
# --------------------------------------------------------------------------
def slot_of(block_table, position: int, block_size: int = 16) -> int:
    """Slot of the token at `position` of a sequence: its block is
    block_table[position // block_size], its offset position % block_size."""
    return int(block_table[position // block_size]) * block_size + \
        position % block_size


def step_metadata(requests, block_size: int = 16):
    """Attention metadata of one step, written out literally.

    ``requests`` is a sequence of objects with ``block_ids`` (the physical
    blocks of the request's block table), ``num_computed`` (tokens already in
    the cache) and ``num_new`` (tokens scheduled this step).  Returns a dict
    of numpy arrays: query_start_loc int32 [B+1], seq_lens int32 [B],
    block_tables int32 [B, max_blocks] (unused entries 0), slot_mapping int64
    [T] (slots of the new tokens), and the host ints max_query_len,
    max_seq_len.
    """
    B = len(requests)
    qsl = [0]
    seq_lens = []
    slots = []
    max_blocks = max([len(r.block_ids) for r in requests] + [1])
    tables = np.zeros((B, max_blocks), dtype=np.int32)
    for b, r in enumerate(requests):
        L = r.num_computed + r.num_new
        seq_lens.append(L)
        qsl.append(qsl[-1] + r.num_new)
        for k, blk in enumerate(r.block_ids):
            tables[b, k] = blk
        for pos in range(r.num_computed, L):
            slots.append(slot_of(r.block_ids, pos, block_size))
    return {
        "query_start_loc": np.asarray(qsl, dtype=np.int32),
        "seq_lens": np.asarray(seq_lens, dtype=np.int32),
        "block_tables": tables,
        "slot_mapping": np.asarray(slots, dtype=np.int64),
        "max_query_len": max([r.num_new for r in requests] + [0]),
        "max_seq_len": max(seq_lens + [0]),
    }


# --------------------------------------------------------------------------
# the three operations
# --------------------------------------------------------------------------
def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, *,
                      cache_dtype=None, kv_dtype=None, k_scale=1.0,
                      v_scale=1.0, block_size=16):
    """In-place write of new tokens' K/V into numpy caches of shape
    [NB, Hkv, block_size, D] (see pa_oracle.c).  key/value: [T, Hkv, D]."""
    k, kdt = _as_np(key)
    v, _ = _as_np(value)
    if not (isinstance(k_cache, np.ndarray) and isinstance(v_cache, np.ndarray)
            and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise OracleError("caches must be C-contiguous numpy arrays (in place)")
    kdt = _dt(kv_dtype, kdt)
    cdt = _dt(cache_dtype, None)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = sm.shape[0]
    NB, Hkv, bs, D = _geometry(k_cache, k.shape[-1], block_size)
    _check(_load().orc_reshape_and_cache(
        _ptr(k), _ptr(v), kdt, T, Hkv * D, Hkv * D, _ptr(k_cache),
        _ptr(v_cache), cdt, NB, bs, Hkv, D, _ptr(sm), k_scale, v_scale),
        "reshape_and_cache")


def copy_blocks(k_cache, v_cache, block_mapping, *, cache_dtype,
                head_dim=None):
    """In-place block copies; block_mapping int64 [P, 2] of (src, dst)."""
    bm = np.ascontiguousarray(block_mapping, dtype=np.int64).reshape(-1, 2)
    NB, Hkv, bs, D = _geometry(k_cache, head_dim)
    _check(_load().orc_copy_blocks(
        _ptr(k_cache), _ptr(v_cache), _dt(cache_dtype, None), NB, bs, Hkv, D,
        _ptr(bm), bm.shape[0]), "copy_blocks")


def paged_attention(q, k_cache, v_cache, block_tables, seq_lens,
                    query_start_loc, *, scale, cache_dtype=None, q_dtype=None,
                    k_scale=1.0, v_scale=1.0, num_threads=None, window=0):
    """fp64 output [T, Hq, D] of the step (rows of unowned tokens are NaN).
    window > 0: each query sees only its own key and the window - 1 keys
    before it (sliding-window attention)."""
    qa, qdt = _as_np(q)
    kc, kcdt = _as_np(k_cache)
    vc, _ = _as_np(v_cache)
    qdt = _dt(q_dtype, qdt)
    cdt = _dt(cache_dtype, kcdt)
    T, Hq, D = qa.shape
    NB, Hkv, bs, _ = _geometry(kc, D)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    out = np.full((T, Hq, D), np.nan, dtype=np.float64)
    if num_threads is None:
        num_threads = os.cpu_count() or 1
    _check(_load().orc_paged_attention(
        _ptr(qa), qdt, _ptr(kc), _ptr(vc), cdt, NB, bs, Hq, Hkv, D, _ptr(bt),
        bt.shape[1], _ptr(sl), _ptr(qsl), sl.shape[0], float(scale),
        float(k_scale), float(v_scale), _ptr(out), int(num_threads),
        int(window)), "paged_attention")
    return out


def paged_attention_row(q, k_cache, v_cache, block_tables, seq_lens,
                        query_start_loc, r: int, i: int, h: int, *, scale,
                        cache_dtype=None, q_dtype=None, k_scale=1.0,
                        v_scale=1.0, window=0):
    """fp64 output row of request r, query i, head h (same definition)."""
    qa, qdt = _as_np(q)
    kc, kcdt = _as_np(k_cache)
    vc, _ = _as_np(v_cache)
    qdt = _dt(q_dtype, qdt)
    cdt = _dt(cache_dtype, kcdt)
    T, Hq, D = qa.shape
    NB, Hkv, bs, _ = _geometry(kc, D)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    out = np.empty(D, dtype=np.float64)
    _check(_load().orc_paged_attention_row(
        _ptr(qa), qdt, _ptr(kc), _ptr(vc), cdt, NB, bs, Hq, Hkv, D, _ptr(bt),
        bt.shape[1], _ptr(sl), _ptr(qsl), r, i, h, float(scale),
        float(k_scale), float(v_scale), _ptr(out), int(window)),
        "paged_attention_row")
    return out


def run_step(wl, num_threads=None):
    """The whole step of a workload on the CPU, in the order the engine runs
    it: copy-on-write block copies, then the new tokens' K/V writes, then
    attention.  Returns (fp64 output [T, Hq, D], k_cache, v_cache, metadata).
    The caches are fresh numpy copies of the workload's initial caches."""
    md = step_metadata(wl.requests, wl.block_size)
    kc, kcdt = _as_np(wl.k_cache)
    vc, _ = _as_np(wl.v_cache)
    kc = kc.copy()
    vc = vc.copy()
    cdt = _DT_NAMES[wl.cache_dtype]
    if wl.copy_pairs:
        copy_blocks(kc, vc, np.asarray(wl.copy_pairs, dtype=np.int64),
                    cache_dtype=cdt, head_dim=wl.head_dim)
    if wl.write_new:
        reshape_and_cache(wl.key, wl.value, kc, vc, md["slot_mapping"],
                          cache_dtype=cdt, k_scale=wl.k_scale,
                          v_scale=wl.v_scale, block_size=wl.block_size)
    out = paged_attention(wl.q, kc.reshape(wl.k_cache.shape),
                          vc.reshape(wl.v_cache.shape), md["block_tables"],
                          md["seq_lens"], md["query_start_loc"],
                          scale=wl.scale, cache_dtype=cdt,
                          k_scale=wl.k_scale, v_scale=wl.v_scale,
                          num_threads=num_threads,
                          window=getattr(wl, "sliding_window", 0))
    return out, kc, vc, md
