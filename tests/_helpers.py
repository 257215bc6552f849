"""Test-side helpers: contiguous ground truth, its scatter into pages, and a
library reference (torch scaled_dot_product_attention in float64)."""
from __future__ import annotations

import numpy as np
import torch

BS = 16


def scatter_paged(seqs, block_lists, num_blocks, fill=np.nan):
    """Place contiguous per-sequence arrays [L, H, D] into a paged cache
    [NB, H, 16, D]: token j of a sequence goes to block_list[j // 16],
    offset j % 16.  Unused slots get `fill`."""
    H, D = seqs[0].shape[1], seqs[0].shape[2]
    cache = np.full((num_blocks, H, BS, D), fill, dtype=seqs[0].dtype)
    for s, blocks in zip(seqs, block_lists):
        for j in range(s.shape[0]):
            cache[blocks[j // BS], :, j % BS, :] = s[j]
    return cache


def sdpa_reference(q_seqs, k_seqs, v_seqs, group, scale, window=0):
    """Per request: q [n, Hq, D], k/v [L, Hkv, D] (float64) -> [n, Hq, D].

    Query i of a request with n queries and L keys sees keys 0..L-n+i
    (bottom-right causal alignment), and with window > 0 only the last
    `window` of those; GQA by repeating each KV head `group` times."""
    outs = []
    for q, k, v in zip(q_seqs, k_seqs, v_seqs):
        n, L = q.shape[0], k.shape[0]
        Q = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))
        K = torch.from_numpy(np.ascontiguousarray(k.transpose(1, 0, 2)))
        V = torch.from_numpy(np.ascontiguousarray(v.transpose(1, 0, 2)))
        K = K.repeat_interleave(group, dim=0)
        V = V.repeat_interleave(group, dim=0)
        i = torch.arange(n)[:, None]
        j = torch.arange(L)[None, :]
        mask = j <= (L - n + i)
        if window > 0:
            mask = mask & (j > (L - n + i - window))
        o = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, attn_mask=mask, scale=scale)
        outs.append(o.numpy().transpose(1, 0, 2))
    return outs


class Req:
    def __init__(self, block_ids, num_computed, num_new):
        self.block_ids = list(block_ids)
        self.num_computed = num_computed
        self.num_new = num_new


def random_paged_step(rng, shapes, Hq, Hkv, D, num_blocks, dtype=np.float32,
                      permute=True):
    """shapes: list of (n, L).  Returns (q, k_cache, v_cache, requests,
    contiguous q/k/v lists) with blocks drawn from a permutation."""
    order = rng.permutation(num_blocks) if permute else np.arange(num_blocks)
    nxt = 0
    reqs, qs, ks, vs = [], [], [], []
    for n, L in shapes:
        nb = -(-L // BS)
        blocks = [int(b) for b in order[nxt:nxt + nb]]
        nxt += nb
        reqs.append(Req(blocks, L - n, n))
        qs.append(rng.standard_normal((n, Hq, D)).astype(dtype))
        ks.append(rng.standard_normal((L, Hkv, D)).astype(dtype))
        vs.append(rng.standard_normal((L, Hkv, D)).astype(dtype))
    kc = scatter_paged(ks, [r.block_ids for r in reqs], num_blocks)
    vc = scatter_paged(vs, [r.block_ids for r in reqs], num_blocks)
    q = np.concatenate(qs, axis=0)
    return q, kc, vc, reqs, qs, ks, vs
