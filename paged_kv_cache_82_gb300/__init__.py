"""paged_kv_cache_82_gb300 -- Python binding of libpa (paged-KV attention on
GB300).

Thin ctypes marshalling over the C ABI declared in ``include/pa.h``: the
functions here have the same names and the same semantics; they only turn
torch tensors into pointers, sizes and the current CUDA stream.  Every step of
the computation runs in the CUDA kernels of ``libpa.so``; there is no other
implementation.  If the library is missing or no CUDA device is present the
calls raise; nothing falls back.

    pa_reshape_and_cache  -- write this step's K/V into their cache slots
    pa_copy_blocks        -- block-granular copy-on-write
    pa_attention          -- unified decode + chunked-prefill paged attention
    pa_attention_workspace_size, pa_get_device_error
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import metadata  # noqa: F401  (host step metadata builder)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_DEVICE = \
    range(5)
PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3, PA_INT4, PA_NVFP4 = range(6)
PA_DEV_ERR_SLOT, PA_DEV_ERR_BLOCK_ID, PA_DEV_ERR_METADATA, \
    PA_DEV_ERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8
BLOCK_SIZE = 16

EXPORTED = ("pa_status_string", "pa_reshape_and_cache", "pa_copy_blocks",
            "pa_attention_workspace_size", "pa_attention",
            "pa_get_device_error", "pa_set_profile_events",
            "pa_launch_count", "pa_attention_noalloc",
            "pa_set_debug_bounds", "pa_attention_window",
            "pa_attention_window_workspace_size", "pa_set_wait_limit_ns",
            "pa_test_skip_copy", "pa_attention_cascade",
            "pa_attention_cascade_workspace_size")

_DT = {"f32": PA_F32, "f16": PA_F16, "bf16": PA_BF16, "e4m3": PA_FP8_E4M3,
       "int4": PA_INT4, "nvfp4": PA_NVFP4}


def page_bytes_4bit(cache_dtype: str, head_dim: int) -> int:
    """PA_PAGE_BYTES of pa.h: bytes of one (block, KV head) page of a 4-bit
    cache (int4: codes + 16 fp32 scales; nvfp4: codes + E4M3 block scales)."""
    return 8 * head_dim + (64 if cache_dtype == "int4" else head_dim)


def _cache_geometry(cache: torch.Tensor, cache_dtype: Optional[str],
                    head_dim: Optional[int] = None):
    """(num_blocks, kv_heads, block_size, head_dim) of a cache tensor:
    [NB, Hkv, 16, D] elements, or [NB, Hkv, page_bytes] uint8 for the 4-bit
    formats (head_dim from the page size when not given)."""
    if cache_dtype in ("int4", "nvfp4"):
        if cache.dim() != 3 or cache.dtype != torch.uint8:
            raise ValueError("a 4-bit cache is a uint8 [NB, Hkv, page_bytes] "
                             "tensor")
        NB, H, pb = cache.shape
        D = (pb - 64) // 8 if cache_dtype == "int4" else pb // 9
        if head_dim is not None and head_dim != D:
            raise ValueError("head_dim does not match the cache's pages")
        if page_bytes_4bit(cache_dtype, D) != pb:
            raise ValueError("page size matches no head_dim")
        return NB, H, BLOCK_SIZE, D
    if cache.dim() != 4:
        raise ValueError("the caches must be [NB, Hkv, 16, D]")
    return tuple(cache.shape)
_lib = None


class PaError(RuntimeError):
    def __init__(self, status: int, what: str, flags: int = 0):
        self.status = status
        self.flags = flags
        name = _load().pa_status_string(status).decode() if _lib else str(status)
        super().__init__(f"{what}: {name}" + (f" (flags 0x{flags:x})"
                                              if flags else ""))


def load_library(path: str = LIB_PATH):
    """Load libpa.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                            ctypes.c_float, ctypes.c_size_t)
    lib.pa_status_string.argtypes = [i32]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_reshape_and_cache.argtypes = [P, P, i32, i64, i64, i64, P, P, i32,
                                         i64, i32, i32, i32, P, f32, f32, P]
    lib.pa_reshape_and_cache.restype = i32
    lib.pa_copy_blocks.argtypes = [P, P, i32, i64, i32, i32, i32, P, i64, P]
    lib.pa_copy_blocks.restype = i32
    lib.pa_attention_workspace_size.argtypes = [i64, i32, i32, i32, i32, i32,
                                                i32, ctypes.POINTER(sz)]
    lib.pa_attention_workspace_size.restype = i32
    lib.pa_attention.argtypes = [P, i32, P, P, i32, i64, i32, i32, i32, i32, P,
                                 i32, P, P, i32, i64, i32, i32, f32, f32, f32,
                                 P, P, sz, P]
    lib.pa_attention.restype = i32
    lib.pa_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.pa_get_device_error.restype = i32
    lib.pa_set_profile_events.argtypes = [P, P]
    lib.pa_set_profile_events.restype = i32
    lib.pa_launch_count.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
    lib.pa_launch_count.restype = i32
    lib.pa_attention_window.argtypes = [P, i32, P, P, i32, i64, i32, i32, i32,
                                        i32, P, i32, P, P, i32, i64, i32, i32,
                                        f32, f32, f32, i32, P, P, sz, P]
    lib.pa_attention_window.restype = i32
    lib.pa_attention_window_workspace_size.argtypes = [
        i64, i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
    lib.pa_attention_window_workspace_size.restype = i32
    lib.pa_attention_cascade.argtypes = [P, i32, P, P, i32, i64, i32, i32, i32,
                                         i32, P, i32, P, P, i32, i64, i32, i32,
                                         f32, f32, f32, i32, P, P, sz, P]
    lib.pa_attention_cascade.restype = i32
    lib.pa_attention_cascade_workspace_size.argtypes = [
        i64, i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
    lib.pa_attention_cascade_workspace_size.restype = i32
    lib.pa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.pa_set_wait_limit_ns.restype = i32
    lib.pa_test_skip_copy.argtypes = [i64]
    lib.pa_test_skip_copy.restype = i32
    lib.pa_set_debug_bounds.argtypes = [i32]
    lib.pa_set_debug_bounds.restype = i32
    lib.pa_attention_noalloc.argtypes = [P, i32, P, P, i32, i64, i32, i32, i32,
                                         i32, P, i32, P, P, i32, i64, i32, i32,
                                         f32, f32, f32, P, P]
    lib.pa_attention_noalloc.restype = i32
    _lib = lib
    return lib


def _load():
    return _lib if _lib is not None else load_library()


def _dtype_code(t: torch.Tensor, override: Optional[str] = None) -> int:
    if override is not None:
        return _DT[override]
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        return PA_FP8_E4M3
    raise TypeError(f"unsupported tensor dtype {t.dtype}")


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PaError(status, what)


def _step_shapes(q, k_cache, v_cache, block_tables, seq_lens,
                 query_start_loc, out, cache_dtype=None):
    """Check the tensors of one attention step the way the C ABI reads them
    (contiguous, int32 metadata, consistent sizes) and return (T, Hq, D, NB,
    Hkv, block_size, B).  Runs before any pointer is taken, so a strided q or
    an int64 length array is refused instead of being read as raw bytes."""
    if q.dim() != 3 or v_cache.shape != k_cache.shape:
        raise ValueError("q must be [T, Hq, D] and both caches alike")
    T, Hq, D = q.shape
    NB, Hkv, bs, Dc = _cache_geometry(k_cache, cache_dtype)
    if Dc != D:
        raise ValueError("head_dim of q and of the caches differ")
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for t, n in ((block_tables, "block_tables"), (seq_lens, "seq_lens"),
                 (query_start_loc, "query_start_loc")):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 tensor")
    B = seq_lens.numel()
    if (query_start_loc.numel() != B + 1 or block_tables.dim() != 2
            or block_tables.shape[0] != B):
        raise ValueError("inconsistent number of sequences")
    if out is not None and (out.shape != q.shape or out.dtype != q.dtype
                            or not out.is_contiguous()):
        raise ValueError("out must be a contiguous tensor like q")
    return T, Hq, D, NB, Hkv, bs, B


def pa_reshape_and_cache(key: torch.Tensor, value: torch.Tensor,
                         k_cache: torch.Tensor, v_cache: torch.Tensor,
                         slot_mapping: torch.Tensor, k_scale: float = 1.0,
                         v_scale: float = 1.0, cache_dtype: Optional[str] = None,
                         stream=None) -> None:
    """key/value [T, Hkv, D] (row stride may exceed Hkv*D), caches
    [NB, Hkv, 16, D], slot_mapping int64 [T]."""
    T, Hkv, D = key.shape
    if value.shape != key.shape or key.stride(2) != 1 or key.stride(1) != D \
            or value.stride(2) != 1 or value.stride(1) != D:
        raise ValueError("key/value must be [T, Hkv, D] with contiguous rows")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T:
        raise ValueError("slot_mapping must be int64 [num_tokens]")
    NB, Hc, bs, Dc = _cache_geometry(k_cache, cache_dtype, D)
    if (Hc, Dc) != (Hkv, D) or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape does not match key/value")
    lib = _load()
    st = lib.pa_reshape_and_cache(
        _dev(key, "key"), _dev(value, "value"), _dtype_code(key), T,
        key.stride(0), value.stride(0), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dtype_code(k_cache, cache_dtype), NB, bs,
        Hkv, D, _dev(slot_mapping, "slot_mapping"), float(k_scale),
        float(v_scale), _stream(stream))
    _check(st, "pa_reshape_and_cache")


def pa_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor,
                   block_mapping: torch.Tensor,
                   cache_dtype: Optional[str] = None, stream=None) -> None:
    """block_mapping int64 [P, 2] of (src, dst) pairs."""
    if block_mapping.dtype != torch.int64 or not block_mapping.is_contiguous():
        raise ValueError("block_mapping must be a contiguous int64 [P, 2]")
    NB, Hkv, bs, D = _cache_geometry(k_cache, cache_dtype)
    lib = _load()
    st = lib.pa_copy_blocks(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                            _dtype_code(k_cache, cache_dtype), NB, bs, Hkv, D,
                            _dev(block_mapping, "block_mapping"),
                            block_mapping.numel() // 2, _stream(stream))
    _check(st, "pa_copy_blocks")


def pa_attention_workspace_size(num_tokens: int, num_q_heads: int,
                                num_kv_heads: int, head_dim: int,
                                num_seqs: int, max_query_len: int,
                                max_seq_len: int) -> int:
    out = ctypes.c_size_t(0)
    st = _load().pa_attention_workspace_size(num_tokens, num_q_heads,
                                             num_kv_heads, head_dim, num_seqs,
                                             max_query_len, max_seq_len,
                                             ctypes.byref(out))
    _check(st, "pa_attention_workspace_size")
    return int(out.value)


def pa_attention(q: torch.Tensor, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, block_tables: torch.Tensor,
                 seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                 max_query_len: int, max_seq_len: int, scale: float,
                 k_scale: float = 1.0, v_scale: float = 1.0,
                 out: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None,
                 cache_dtype: Optional[str] = None, stream=None) -> torch.Tensor:
    """q [T, Hq, D]; caches [NB, Hkv, 16, D]; block_tables int32 [B, M];
    seq_lens int32 [B]; query_start_loc int32 [B+1].  Returns out [T, Hq, D]
    (allocated if not given; the workspace too)."""
    T, Hq, D, NB, Hkv, bs, B = _step_shapes(q, k_cache, v_cache, block_tables,
                                            seq_lens, query_start_loc, out,
                                            cache_dtype)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = pa_attention_workspace_size(T, Hq, Hkv, D, B, max_query_len,
                                             max_seq_len)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8,
                                device=q.device)
    lib = _load()
    st = lib.pa_attention(
        _dev(q, "q"), _dtype_code(q), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dtype_code(k_cache, cache_dtype), NB, bs, Hq,
        Hkv, D, _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(seq_lens, "seq_lens"), _dev(query_start_loc, "query_start_loc"),
        B, T, int(max_query_len), int(max_seq_len), float(scale),
        float(k_scale), float(v_scale), _dev(out, "out"),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check(st, "pa_attention")
    return out


def pa_attention_window_workspace_size(num_tokens: int, num_q_heads: int,
                                       num_kv_heads: int, head_dim: int,
                                       num_seqs: int, max_query_len: int,
                                       max_seq_len: int,
                                       sliding_window: int) -> int:
    out = ctypes.c_size_t(0)
    st = _load().pa_attention_window_workspace_size(
        num_tokens, num_q_heads, num_kv_heads, head_dim, num_seqs,
        max_query_len, max_seq_len, sliding_window, ctypes.byref(out))
    _check(st, "pa_attention_window_workspace_size")
    return int(out.value)


def pa_attention_window(q: torch.Tensor, k_cache: torch.Tensor,
                        v_cache: torch.Tensor, block_tables: torch.Tensor,
                        seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                        max_query_len: int, max_seq_len: int, scale: float,
                        sliding_window: int, k_scale: float = 1.0,
                        v_scale: float = 1.0,
                        out: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None,
                        cache_dtype: Optional[str] = None,
                        stream=None) -> torch.Tensor:
    """pa_attention with a sliding window of `sliding_window` keys (each
    query sees its own key and the window - 1 keys before it; 0: none)."""
    T, Hq, D, NB, Hkv, bs, B = _step_shapes(q, k_cache, v_cache, block_tables,
                                            seq_lens, query_start_loc, out,
                                            cache_dtype)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = pa_attention_window_workspace_size(
            T, Hq, Hkv, D, B, max_query_len, max_seq_len, sliding_window)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8,
                                device=q.device)
    st = _load().pa_attention_window(
        _dev(q, "q"), _dtype_code(q), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dtype_code(k_cache, cache_dtype), NB, bs, Hq,
        Hkv, D, _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(seq_lens, "seq_lens"), _dev(query_start_loc, "query_start_loc"),
        B, T, int(max_query_len), int(max_seq_len), float(scale),
        float(k_scale), float(v_scale), int(sliding_window), _dev(out, "out"),
        _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "pa_attention_window")
    return out


def pa_attention_cascade_workspace_size(num_tokens: int, num_q_heads: int,
                                        num_kv_heads: int, head_dim: int,
                                        num_seqs: int, max_query_len: int,
                                        max_seq_len: int) -> int:
    out = ctypes.c_size_t(0)
    st = _load().pa_attention_cascade_workspace_size(
        num_tokens, num_q_heads, num_kv_heads, head_dim, num_seqs,
        max_query_len, max_seq_len, ctypes.byref(out))
    _check(st, "pa_attention_cascade_workspace_size")
    return int(out.value)


def pa_attention_cascade(q: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, block_tables: torch.Tensor,
                         seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                         max_query_len: int, max_seq_len: int, scale: float,
                         common_prefix_blocks: int, k_scale: float = 1.0,
                         v_scale: float = 1.0,
                         out: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         cache_dtype: Optional[str] = None,
                         stream=None) -> torch.Tensor:
    """pa_attention for a step whose requests all begin with the same
    `common_prefix_blocks` block ids (the shared prefix is read once per KV
    head and merged with each request's own part)."""
    T, Hq, D, NB, Hkv, bs, B = _step_shapes(q, k_cache, v_cache, block_tables,
                                            seq_lens, query_start_loc, out,
                                            cache_dtype)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = pa_attention_cascade_workspace_size(
            T, Hq, Hkv, D, B, max_query_len, max_seq_len)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8,
                                device=q.device)
    st = _load().pa_attention_cascade(
        _dev(q, "q"), _dtype_code(q), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dtype_code(k_cache, cache_dtype), NB, bs, Hq,
        Hkv, D, _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(seq_lens, "seq_lens"), _dev(query_start_loc, "query_start_loc"),
        B, T, int(max_query_len), int(max_seq_len), float(scale),
        float(k_scale), float(v_scale), int(common_prefix_blocks),
        _dev(out, "out"), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "pa_attention_cascade")
    return out


def pa_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error flags."""
    flags = ctypes.c_uint32(0)
    st = _load().pa_get_device_error(_stream(stream), ctypes.byref(flags))
    if st not in (PA_OK, PA_ERR_DEVICE):
        raise PaError(st, "pa_get_device_error")
    return int(flags.value)


def pa_set_profile_events(start: Optional[torch.cuda.Event],
                          stop: Optional[torch.cuda.Event]) -> None:
    """Record `start` / `stop` around the attention kernels of every later
    pa_attention call of this thread (measurement hook); None, None turns it
    off."""
    def handle(ev):
        if ev is None:
            return None
        ev.record()  # make sure the event object exists on the device
        return ev.cuda_event
    _check(_load().pa_set_profile_events(handle(start), handle(stop)),
           "pa_set_profile_events")


def pa_set_debug_bounds(enable: bool) -> None:
    """The device-side index checks are always on: True is accepted, False
    raises (PA_ERR_UNSUPPORTED)."""
    _check(_load().pa_set_debug_bounds(1 if enable else 0),
           "pa_set_debug_bounds")


def pa_set_wait_limit_ns(ns: int) -> None:
    """Longest one pipeline wait in the kernels may last (0: the default
    2 s); a wait that runs out is reported as PA_DEV_ERR_TIMEOUT."""
    _check(_load().pa_set_wait_limit_ns(int(ns)), "pa_set_wait_limit_ns")


def pa_test_skip_copy(stage: int) -> None:
    """Testing hook: CTA 0 of the pipelined kernels leaves out the copy of
    pipeline stage `stage` (-1: off), so that the waits on it run out."""
    _check(_load().pa_test_skip_copy(int(stage)), "pa_test_skip_copy")


def pa_launch_count() -> int:
    """Kernels the library has launched from this thread so far."""
    n = ctypes.c_uint64(0)
    _check(_load().pa_launch_count(ctypes.byref(n)), "pa_launch_count")
    return int(n.value)


def pa_attention_noalloc(q: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, block_tables: torch.Tensor,
                         seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                         max_query_len: int, max_seq_len: int, scale: float,
                         k_scale: float = 1.0, v_scale: float = 1.0,
                         out: Optional[torch.Tensor] = None,
                         cache_dtype: Optional[str] = None,
                         stream=None) -> torch.Tensor:
    """pa_attention with the library's fixed device scratch instead of a
    workspace, for callers that cannot allocate device memory per step (the
    output tensor is still the caller's)."""
    if out is None:
        raise ValueError("pa_attention_noalloc needs a caller-provided out")
    T, Hq, D, NB, Hkv, bs, B = _step_shapes(q, k_cache, v_cache, block_tables,
                                            seq_lens, query_start_loc, out,
                                            cache_dtype)
    st = _load().pa_attention_noalloc(_dev(q, "q"), _dtype_code(q), _dev(k_cache, "k_cache"),
           _dev(v_cache, "v_cache"), _dtype_code(k_cache, cache_dtype), NB, bs,
           Hq, Hkv, D, _dev(block_tables, "block_tables"),
           block_tables.shape[1], _dev(seq_lens, "seq_lens"),
           _dev(query_start_loc, "query_start_loc"), B, T, int(max_query_len),
           int(max_seq_len), float(scale), float(k_scale), float(v_scale),
           _dev(out, "out"), _stream(stream))
    _check(st, "pa_attention_noalloc")
    return out
