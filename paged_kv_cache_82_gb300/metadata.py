"""Host-side attention metadata of one scheduler step.

A step is ``{request: num_tokens}`` ("vLLM V1 engine architecture", "Scheduler
forms one round of work"); the model runner turns it, with each request's
block table and number of already computed tokens, into the per-step arrays
the attention kernels read ("vLLM V0 vs V1", section 3.1: query length,
context length, block table).  Slots follow Figure 2 of "vLLM engine
anatomy": position j of a request is in block ``block_table[j // 16]`` at
offset ``j % 16``.

Input: a sequence of requests with ``block_ids``, ``num_computed`` and
``num_new``.  Output (numpy):

* ``query_start_loc`` int32 [B+1] -- offsets of each request's new tokens
* ``seq_lens`` int32 [B] -- keys per request, this step's tokens included
* ``block_tables`` int32 [B, max_blocks] -- unused entries are 0
* ``slot_mapping`` int64 [T] -- cache slot of every new token
* ``max_query_len``, ``max_seq_len`` -- host upper bounds for the kernels

``common_prefix_blocks`` gives the number of leading block ids that every
request of the step shares and whose keys precede every request's queries:
the shared prefix a cascade step (pa_attention_cascade) reads once.
``cascade_prefix_blocks`` gives it only where the cascade is the faster way
to run the step (a measured crossover), else 0.
"""
from __future__ import annotations

import itertools

import numpy as np

BLOCK_SIZE = 16


def build_step_metadata(requests, block_size: int = BLOCK_SIZE,
                        block_tables=None) -> dict:
    """The step's metadata (module docstring).  block_tables: the requests'
    block-table rows already as an int32 array (a planner that keeps them,
    e.g. block_manager's StepPlan.block_tables); else built from the
    requests' block_ids."""
    n_new = np.fromiter((r.num_new for r in requests), dtype=np.int64,
                        count=len(requests))
    n_done = np.fromiter((r.num_computed for r in requests), dtype=np.int64,
                         count=len(requests))
    lens = n_done + n_new
    qsl = np.zeros(len(requests) + 1, dtype=np.int64)
    np.cumsum(n_new, out=qsl[1:])
    if block_tables is not None:
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    else:
        nb = np.fromiter((len(r.block_ids) for r in requests), dtype=np.int64,
                         count=len(requests))
        width = max(int(nb.max()) if len(requests) else 0, 1)
        tables = np.zeros((len(requests), width), dtype=np.int32)
        # every row's ids in one pass: the mask's row-major order is the
        # concatenated lists' order
        flat = np.fromiter(itertools.chain.from_iterable(r.block_ids for r in requests),
                           dtype=np.int32, count=int(nb.sum()))
        tables[np.arange(width)[None, :] < nb[:, None]] = flat
    T = int(qsl[-1])
    # request index and position of every new token
    req_of_tok = np.repeat(np.arange(len(requests)), n_new)
    pos = np.arange(T, dtype=np.int64) - qsl[req_of_tok] + n_done[req_of_tok]
    blocks = tables[req_of_tok, pos // block_size].astype(np.int64)
    slots = blocks * block_size + pos % block_size
    return {
        "query_start_loc": qsl.astype(np.int32),
        "seq_lens": lens.astype(np.int32),
        "block_tables": tables,
        "slot_mapping": slots.astype(np.int64),
        "max_query_len": int(n_new.max()) if len(requests) else 0,
        "max_seq_len": int(lens.max()) if len(requests) else 0,
    }


def to_device(md: dict, device) -> dict:
    """Copy the metadata arrays to `device` (torch tensors); host ints kept."""
    import torch
    out = {}
    for k, v in md.items():
        out[k] = torch.from_numpy(v).to(device) if isinstance(v, np.ndarray) \
            else v
    return out


def common_prefix_blocks(requests) -> int:
    """Leading block ids that all requests share (prefix caching hands the
    same full blocks to requests with the same prompt prefix, "01. vLLM",
    KV cache management and prefix caching), cut to the full blocks before
    every request's first new token; 0 for an empty step."""
    if not requests:
        return 0
    first = requests[0].block_ids
    n = min(len(first), min(r.num_computed // BLOCK_SIZE for r in requests))
    for r in requests[1:]:
        k = 0
        lim = min(n, len(r.block_ids))
        while k < lim and r.block_ids[k] == first[k]:
            k += 1
        n = k
    return int(n)


# Where a cascade step beats the plain step (decode steps of the
# Llama-3.1-8B shape on a GB300, private contexts of 256 - 8192 tokens after
# the prefix), in prefix blocks N and decode requests n.  16-bit caches: N of
# at least CASCADE_MIN_BLOCKS, or N x n of at least CASCADE_MIN_BLOCK_READS.
# FP8 caches (the prefix tiles widen E4M3 pages on the way, the plain step
# reads half the bytes): N x n of at least CASCADE_MIN_BLOCK_READS_FP8 only.
# Below that the plain step re-reads the prefix from L2 for less than the
# cascade's fixed costs (the prefix tiles' start-up and the extra merge
# parts).  Caches without a cascade path (4-bit) never take it.
CASCADE_MIN_BLOCKS = 512
CASCADE_MIN_BLOCK_READS = 8192
CASCADE_MIN_BLOCK_READS_FP8 = 16384


def cascade_prefix_blocks(requests, group: int, cache_dtype: str = "bf16") -> int:
    """The shared prefix to run as a cascade (pa_attention_cascade's
    cascade_blocks), or 0 where the plain step is faster.  Only the
    decode-class requests (at most 8 query rows: q_len x group <= 8) read the
    prefix once through the cascade; prefill requests read their whole row
    either way.  Needs at least two of them."""
    if cache_dtype not in ("bf16", "f16", "e4m3"):
        return 0
    n = common_prefix_blocks(requests)
    dec = sum(1 for r in requests if 0 < r.num_new and r.num_new * group <= 8)
    if n <= 0 or dec < 2:
        return 0
    if cache_dtype == "e4m3":
        return int(n) if n * dec >= CASCADE_MIN_BLOCK_READS_FP8 else 0
    if n >= CASCADE_MIN_BLOCKS or n * dec >= CASCADE_MIN_BLOCK_READS:
        return int(n)
    return 0
