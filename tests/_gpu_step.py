"""Run one workload step through the C ABI (via the package binding) and
through the oracle, for the parity tests."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_82_gb300 as pa
from paged_kv_cache_82_gb300.metadata import build_step_metadata

# bar for attention outputs against the fp64 oracle (max-abs), per cache type
ATOL = {"bf16": 2e-3, "f16": 2e-3, "f32": 2e-3, "e4m3": 2e-2,
        # the 4-bit formats decode exactly to 16-bit values; the oracle
        # reads the same codes, so the 16-bit bar applies
        "int4": 2e-3, "nvfp4": 2e-3}
# bits of precision of the output type (for the unavoidable final rounding)
OUT_MANT = {"bf16": 8, "f16": 11, "f32": 24}


def half_ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of `dtype` at |ref|: the error that the
    final round-to-nearest of the output alone may add."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, 1e-30)))
    return np.ldexp(1.0, (e - OUT_MANT[dtype]).astype(np.int64))


def gpu_step(wl, device="cuda", out=None, workspace=None, cascade_blocks=None):
    """cascade_blocks: run the step through pa_attention_cascade with that
    many shared leading blocks (None: pa_attention / pa_attention_window)."""
    md = build_step_metadata(wl.requests, wl.block_size)
    kc = wl.k_cache.to(device)
    vc = wl.v_cache.to(device)
    cdt = wl.cache_dtype
    if wl.copy_pairs:
        pairs = torch.tensor(wl.copy_pairs, dtype=torch.int64, device=device)
        pa.pa_copy_blocks(kc, vc, pairs, cache_dtype=cdt)
    if wl.write_new:
        pa.pa_reshape_and_cache(
            wl.key.to(device), wl.value.to(device), kc, vc,
            torch.from_numpy(md["slot_mapping"]).to(device),
            k_scale=wl.k_scale, v_scale=wl.v_scale, cache_dtype=cdt)
    q = wl.q.to(device)
    meta = (torch.from_numpy(md["block_tables"]).to(device),
            torch.from_numpy(md["seq_lens"]).to(device),
            torch.from_numpy(md["query_start_loc"]).to(device),
            md["max_query_len"], md["max_seq_len"], wl.scale)
    if cascade_blocks is not None:
        res = pa.pa_attention_cascade(
            q, kc, vc, *meta, cascade_blocks, wl.k_scale, wl.v_scale,
            out=out, workspace=workspace, cache_dtype=cdt)
    elif wl.sliding_window:
        res = pa.pa_attention_window(
            q, kc, vc, *meta, wl.sliding_window, wl.k_scale, wl.v_scale,
            out=out, workspace=workspace, cache_dtype=cdt)
    else:
        res = pa.pa_attention(q, kc, vc, *meta, wl.k_scale, wl.v_scale,
                              out=out, workspace=workspace, cache_dtype=cdt)
    flags = pa.pa_get_device_error()
    return res, kc, vc, md, flags


def owned_rows(md) -> np.ndarray:
    """Token indices that belong to some request."""
    qsl = md["query_start_loc"]
    return np.concatenate([np.arange(qsl[i], qsl[i + 1])
                           for i in range(len(qsl) - 1)] + [np.zeros(0, int)])


def assert_close(gpu_out: torch.Tensor, ref: np.ndarray, md, cache_dtype,
                 out_dtype, with_rounding=True):
    rows = owned_rows(md)
    g = gpu_out.float().cpu().double().numpy()[rows]
    r = ref[rows]
    assert np.isfinite(g).all(), "non-finite GPU output"
    tol = ATOL[cache_dtype] + (half_ulp(r, out_dtype) if with_rounding else 0)
    err = np.abs(g - r)
    bad = err > tol
    assert not bad.any(), (
        f"max err {err.max():.3e} (bar {ATOL[cache_dtype]}), "
        f"{int(bad.sum())} elements over")
    return float(err.max())


def cache_bits(t) -> np.ndarray:
    t = t.cpu() if isinstance(t, torch.Tensor) else torch.from_numpy(t)
    if t.dtype in (torch.float32,):
        return t.view(torch.int32).numpy()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy()
    if t.dtype == torch.uint8:
        return t.numpy()
    raise TypeError(t.dtype)


def oracle_cache_bits(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.float32:
        return a.view(np.int32)
    if a.dtype in (np.float16, np.uint16):
        return a.view(np.int16)
    return a
