"""Host-side KV block manager and step planner.

The bookkeeping that decides, step by step, which physical blocks hold each
request's keys and values, and which `{request: num_tokens}` step the GPU
runs next.  Its output is what the C ABI consumes: per request the block
table, the number of tokens already in the cache and the number scheduled
now, plus the block copies to make before the step's writes.

What it follows (the pages this project is built from):

* "01. vLLM: a general inference engine that grew out of paged KV", section
  "KV cache management and prefix caching": the manager only keeps the
  accounts, the K/V tensors live on the GPU; the unit is a block of 16
  tokens; every free block sits in one doubly linked queue in LRU order,
  taken from the head when allocated and put back at the tail when released,
  with its hash and contents left in place; each full block has a hash over
  its parent block's hash, its token ids and extra keys (a cache salt goes
  into the first block's hash only); a new request looks its blocks up from
  the first one until the first miss; only full blocks are cached; a block
  with references is never reclaimed, a block with none waits in the free
  queue and stops being valid only when it is handed out again.
* Same page, scheduler section: when the next block of a running request
  cannot be allocated, a request is preempted -- under first-come
  first-served the one that joined the running queue last; it releases all
  its blocks, its progress goes back to zero and it returns to the front of
  the waiting queue; its released full blocks may still be hit later.
* "vLLM V0 vs V1", section 3.1: a request's pending tokens are its target
  tokens minus its computed tokens; the step takes 0 <= S_i <= pending with
  sum S_i within the token budget, and the output is {request_id: S_i};
  section 4: KVCacheBlock keeps the reference count, the block hash and the
  free-list links, and FreeKVCacheBlockQueue removes a block from the middle
  in O(1) without creating list nodes.
* "vLLM engine anatomy", "PagedAttention" (blocks shared between sequences;
  a shared block is copied before one of its readers writes into it) and
  "V1: unified scheduling", Figure 3 (prefill chunks and decodes in one
  step; requests join and leave independently).

Readings where the pages leave a step open: a request's blocks are released
tail first, so the blocks deepest in a hash chain are evicted before the
prefix blocks other requests may hit; a prompt that is cached in full still
computes its last block (at least one token must run to produce the next
token); a block is registered in the prefix cache when its 16 tokens have
been computed; two requests that computed the same block independently keep
the first registration.
"""
from __future__ import annotations

import hashlib
import struct
from dataclasses import dataclass, field
from typing import Dict, Iterator, List, Optional, Sequence, Tuple

import numpy as np

BLOCK_SIZE = 16


class KVBlock:
    """One physical block: its id, how many requests reference it, the hash
    it is cached under (None if not cached) and its links in the free
    queue."""

    __slots__ = ("block_id", "ref_cnt", "block_hash", "prev_free", "next_free")

    def __init__(self, block_id: int):
        self.block_id = block_id
        self.ref_cnt = 0
        self.block_hash: Optional[bytes] = None
        self.prev_free: Optional["KVBlock"] = None
        self.next_free: Optional["KVBlock"] = None

    def __repr__(self) -> str:
        return f"KVBlock({self.block_id}, ref={self.ref_cnt})"


class FreeBlockQueue:
    """Doubly linked list of the blocks nobody references, least recently
    released first.  The links live in the blocks themselves, so removing a
    block from the middle (a prefix hit on a free cached block) is O(1) and
    creates nothing."""

    def __init__(self, blocks: Sequence[KVBlock]):
        self._head = KVBlock(-1)   # sentinels
        self._tail = KVBlock(-1)
        self._head.next_free = self._tail
        self._tail.prev_free = self._head
        self._n = 0
        for b in blocks:
            self.append(b)

    def __len__(self) -> int:
        return self._n

    def popleft(self) -> KVBlock:
        b = self._head.next_free
        if b is self._tail:
            raise RuntimeError("no free block")
        self.remove(b)
        return b

    def remove(self, b: KVBlock) -> None:
        if b.prev_free is None or b.next_free is None:
            raise RuntimeError(f"block {b.block_id} is not in the free queue")
        b.prev_free.next_free = b.next_free
        b.next_free.prev_free = b.prev_free
        b.prev_free = b.next_free = None
        self._n -= 1

    def append(self, b: KVBlock) -> None:
        if b.prev_free is not None or b.next_free is not None:
            raise RuntimeError(f"block {b.block_id} is already free")
        last = self._tail.prev_free
        last.next_free = b
        b.prev_free = last
        b.next_free = self._tail
        self._tail.prev_free = b
        self._n += 1

    def __iter__(self) -> Iterator[KVBlock]:
        b = self._head.next_free
        while b is not self._tail:
            yield b
            b = b.next_free


def hash_block(parent: Optional[bytes], token_ids: Sequence[int],
               extra: Optional[Tuple] = None) -> bytes:
    """SHA-256 over the parent block's hash, the block's token ids and its
    extra keys, in a fixed encoding (a present parent and an absent one, or
    different extra keys, never encode alike)."""
    ids = np.asarray(token_ids, dtype="<i8")
    return _hash_encoded(parent, struct.pack("<I", len(ids)) + ids.tobytes(), extra)


def _hash_encoded(parent: Optional[bytes], ids: bytes,
                  extra: Optional[Tuple] = None) -> bytes:
    """hash_block with the token ids already encoded (count, then each id as
    a little-endian int64)."""
    h = hashlib.sha256(b"\x00" if parent is None else b"\x01" + parent)
    h.update(ids)
    if extra:
        h.update(b"\x02" + repr(tuple(extra)).encode())
    return h.digest()


class BlockPool:
    """All physical blocks, allocated once; the free queue and the map from
    block hash to cached block."""

    def __init__(self, num_blocks: int, order: Optional[Sequence[int]] = None):
        if num_blocks <= 0:
            raise ValueError("num_blocks must be positive")
        self.blocks = [KVBlock(i) for i in range(num_blocks)]
        ids = range(num_blocks) if order is None else order
        if sorted(ids) != list(range(num_blocks)):
            raise ValueError("order must be a permutation of the block ids")
        self.free_queue = FreeBlockQueue([self.blocks[i] for i in ids])
        self.cached: Dict[bytes, KVBlock] = {}

    @property
    def num_free(self) -> int:
        return len(self.free_queue)

    def allocate(self) -> KVBlock:
        """A block from the head of the free queue, referenced once; if it was
        cached under a hash, that cache entry ends here."""
        b = self.free_queue.popleft()
        if b.block_hash is not None:
            if self.cached.get(b.block_hash) is b:
                del self.cached[b.block_hash]
            b.block_hash = None
        b.ref_cnt = 1
        return b

    def touch(self, b: KVBlock) -> None:
        """One more reference; a free block leaves the free queue."""
        if b.ref_cnt == 0:
            self.free_queue.remove(b)
        b.ref_cnt += 1

    def release(self, b: KVBlock) -> None:
        """One reference fewer; at zero the block goes to the tail of the free
        queue, keeping its hash and contents."""
        if b.ref_cnt <= 0:
            raise RuntimeError(f"block {b.block_id} released too often")
        b.ref_cnt -= 1
        if b.ref_cnt == 0:
            self.free_queue.append(b)

    def register(self, b: KVBlock, h: bytes) -> None:
        """Cache a full block under its hash (the first registration of a
        hash stays)."""
        if h not in self.cached and b.block_hash is None:
            self.cached[h] = b
            b.block_hash = h

    def lookup(self, h: bytes) -> Optional[KVBlock]:
        return self.cached.get(h)


@dataclass
class SeqState:
    """A request as the manager sees it."""
    request_id: str
    token_ids: List[int]          # prompt, then the sampled tokens
    num_prompt: int
    max_tokens: int
    cache_salt: Optional[str] = None
    num_computed: int = 0         # tokens whose K/V are in the cache
    blocks: List[KVBlock] = field(default_factory=list)
    block_hashes: List[bytes] = field(default_factory=list)
    num_cached_blocks: int = 0    # leading blocks registered in the cache
    arrival: int = 0
    # the ids of `blocks`, kept alongside it (a step's block-table row is a
    # copy of this list, not a walk over the blocks) and as an int32 array
    # whose first len(blocks) entries are valid (the step's block table is
    # filled from it row by row)
    block_ids: List[int] = field(default_factory=list)
    ids: np.ndarray = field(default_factory=lambda: np.zeros(16, dtype=np.int32))

    def _set_ids(self, ids: Sequence[int]) -> None:
        self.block_ids = list(ids)
        cap = max(16, 1 << max(0, len(self.block_ids) - 1).bit_length())
        self.ids = np.zeros(cap, dtype=np.int32)
        self.ids[:len(self.block_ids)] = self.block_ids

    def _append_id(self, block_id: int) -> None:
        n = len(self.block_ids)
        if n == len(self.ids):
            grown = np.zeros(2 * n, dtype=np.int32)
            grown[:n] = self.ids
            self.ids = grown
        self.ids[n] = block_id
        self.block_ids.append(block_id)

    @property
    def num_tokens(self) -> int:
        return len(self.token_ids)

    @property
    def num_output(self) -> int:
        return len(self.token_ids) - self.num_prompt

    @property
    def finished(self) -> bool:
        return self.num_output >= self.max_tokens


class KVCacheManager:
    """Blocks per request on top of a BlockPool, with prefix caching and
    copy-on-write for forked requests."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE,
                 enable_prefix_caching: bool = True,
                 order: Optional[Sequence[int]] = None):
        if block_size != BLOCK_SIZE:
            raise ValueError("the attention kernels take 16-token blocks")
        self.block_size = block_size
        self.pool = BlockPool(num_blocks, order)
        self.enable_prefix_caching = enable_prefix_caching

    # -- hashes --------------------------------------------------------------
    def _extend_hashes(self, seq: SeqState) -> None:
        bs = self.block_size
        k0, k1 = len(seq.block_hashes), seq.num_tokens // bs
        if k1 <= k0:
            return
        # the new full blocks' ids, encoded once (hash_block's encoding)
        ids = np.asarray(seq.token_ids[k0 * bs:k1 * bs], dtype="<i8").tobytes()
        count = struct.pack("<I", bs)
        step = 8 * bs
        for k in range(k0, k1):
            parent = seq.block_hashes[-1] if k else None
            extra = (("salt", seq.cache_salt),) if (k == 0 and seq.cache_salt) \
                else None
            off = (k - k0) * step
            seq.block_hashes.append(
                _hash_encoded(parent, count + ids[off:off + step], extra))

    # -- admission -----------------------------------------------------------
    def computed_blocks(self, seq: SeqState) -> List[KVBlock]:
        """The longest run of leading full blocks found in the cache, at most
        (num_tokens - 1) // 16 of them (the last token always runs)."""
        if not self.enable_prefix_caching:
            return []
        self._extend_hashes(seq)
        hits = []
        for h in seq.block_hashes[:(seq.num_tokens - 1) // self.block_size]:
            b = self.pool.lookup(h)
            if b is None:
                break
            hits.append(b)
        return hits

    def admit(self, seq: SeqState, hits: Sequence[KVBlock]) -> None:
        """Take the prefix hits of a request that had no blocks."""
        assert not seq.blocks and seq.num_computed == 0
        for b in hits:
            self.pool.touch(b)
        seq.blocks = list(hits)
        seq._set_ids([b.block_id for b in hits])
        seq.num_computed = len(hits) * self.block_size
        seq.num_cached_blocks = len(hits)

    # -- slots for one step --------------------------------------------------
    def blocks_needed(self, seq: SeqState, num_new: int) -> int:
        bs = self.block_size
        total = -(-(seq.num_computed + num_new) // bs)
        need = max(0, total - len(seq.blocks))
        if self._write_hits_shared_block(seq, num_new):
            need += 1
        return need

    def _write_hits_shared_block(self, seq: SeqState, num_new: int) -> bool:
        k = seq.num_computed // self.block_size
        return (num_new > 0 and k < len(seq.blocks)
                and seq.blocks[k].ref_cnt > 1)

    def allocate_slots(self, seq: SeqState, num_new: int,
                       copies: List[Tuple[int, int]]) -> bool:
        """Blocks for the request's next num_new tokens.  A block the write
        lands in that others still reference is replaced by a private copy
        first ((src, dst) appended to `copies`).  False, with nothing
        changed, if the pool has too few free blocks."""
        if self.blocks_needed(seq, num_new) > self.pool.num_free:
            return False
        if self._write_hits_shared_block(seq, num_new):
            k = seq.num_computed // self.block_size
            old = seq.blocks[k]
            new = self.pool.allocate()
            copies.append((old.block_id, new.block_id))
            seq.blocks[k] = new
            seq.block_ids[k] = new.block_id
            seq.ids[k] = new.block_id
            self.pool.release(old)
        total = -(-(seq.num_computed + num_new) // self.block_size)
        while len(seq.blocks) < total:
            b = self.pool.allocate()
            seq.blocks.append(b)
            seq._append_id(b.block_id)
        return True

    def commit(self, seq: SeqState, num_new: int) -> None:
        """The step computed num_new more tokens: register the blocks that
        are now full."""
        seq.num_computed += num_new
        if not self.enable_prefix_caching:
            return
        self._extend_hashes(seq)
        full = seq.num_computed // self.block_size
        while seq.num_cached_blocks < min(full, len(seq.block_hashes)):
            k = seq.num_cached_blocks
            self.pool.register(seq.blocks[k], seq.block_hashes[k])
            seq.num_cached_blocks += 1

    def free(self, seq: SeqState) -> None:
        """Release every block of the request, last block first."""
        for b in reversed(seq.blocks):
            self.pool.release(b)
        seq.blocks = []
        seq._set_ids([])
        seq.num_computed = 0
        seq.num_cached_blocks = 0

    def fork(self, parent: SeqState, child_id: str,
             max_tokens: Optional[int] = None) -> SeqState:
        """A second sequence sharing all of the parent's blocks (parallel
        sampling): same tokens and progress, every block referenced once
        more."""
        child = SeqState(child_id, list(parent.token_ids), parent.num_prompt,
                         parent.max_tokens if max_tokens is None else max_tokens,
                         parent.cache_salt, parent.num_computed,
                         list(parent.blocks), list(parent.block_hashes),
                         parent.num_cached_blocks, parent.arrival,
                         list(parent.block_ids), parent.ids.copy())
        for b in child.blocks:
            self.pool.touch(b)
        return child


@dataclass
class StepRequest:
    """One request of a planned step, in the form the attention metadata is
    built from (see metadata.build_step_metadata): its block-table row is
    row[:num_blocks] of the plan's block table, `block_ids` as a list."""
    request_id: str
    row: np.ndarray
    num_blocks: int
    num_computed: int
    num_new: int

    @property
    def block_ids(self) -> List[int]:
        return self.row[:self.num_blocks].tolist()


@dataclass
class StepPlan:
    step: int
    scheduled: Dict[str, int]                 # {request_id: num_tokens}
    requests: List[StepRequest]
    copy_pairs: List[Tuple[int, int]]         # block copies before the writes
    new_token_ids: List[int]                  # ids of the step's tokens, in order
    new_positions: List[int]                  # their positions in their sequences
    preempted: List[str]
    # the requests' block-table rows, int32 [len(requests), max blocks]
    # (unused entries 0): build_step_metadata's block_tables
    block_tables: Optional[np.ndarray] = None


class Scheduler:
    """First-come first-served planner of unified steps: running requests
    first (their remaining prompt chunk or one decode token), then waiting
    requests in order, all within a token budget; a prompt chunk is capped at
    `long_prefill_threshold` tokens (0: no cap)."""

    def __init__(self, manager: KVCacheManager, token_budget: int = 2048,
                 max_num_seqs: int = 256, long_prefill_threshold: int = 0,
                 watermark: float = 0.0):
        self.kv = manager
        self.token_budget = token_budget
        self.max_num_seqs = max_num_seqs
        self.long_prefill_threshold = long_prefill_threshold
        self.watermark_blocks = int(watermark * len(manager.pool.blocks))
        self.waiting: List[SeqState] = []
        self.running: List[SeqState] = []
        self.finished: List[SeqState] = []
        self.step_no = 0

    def add_request(self, request_id: str, prompt: Sequence[int],
                    max_tokens: int, cache_salt: Optional[str] = None) -> SeqState:
        seq = SeqState(request_id, [int(t) for t in prompt], len(prompt),
                       max_tokens, cache_salt, arrival=self.step_no + 1)
        self.waiting.append(seq)
        return seq

    def fork(self, parent_id: str, child_id: str,
             max_tokens: Optional[int] = None) -> SeqState:
        """A running request gets a sibling that shares its blocks."""
        parent = next(s for s in self.running if s.request_id == parent_id)
        child = self.kv.fork(parent, child_id, max_tokens)
        self.running.append(child)
        return child

    def _chunk(self, seq: SeqState, budget: int) -> int:
        n = seq.num_tokens - seq.num_computed
        if seq.num_computed < seq.num_prompt and self.long_prefill_threshold:
            n = min(n, self.long_prefill_threshold)
        return min(n, budget)

    def _preempt(self, victim: SeqState, preempted: List[str]) -> None:
        self.running.remove(victim)
        self.kv.free(victim)
        self.waiting.insert(0, victim)
        preempted.append(victim.request_id)

    def schedule(self) -> StepPlan:
        self.step_no += 1
        budget = self.token_budget
        scheduled: Dict[str, int] = {}
        copies: List[Tuple[int, int]] = []
        preempted: List[str] = []
        order: List[SeqState] = []
        # running requests, in the order they joined
        i = 0
        while i < len(self.running) and budget > 0:
            seq = self.running[i]
            n = self._chunk(seq, budget)
            if n <= 0:
                i += 1
                continue
            while not self.kv.allocate_slots(seq, n, copies):
                victim = self.running[-1]
                self._preempt(victim, preempted)
                if victim is seq:
                    break
            else:
                scheduled[seq.request_id] = n
                order.append(seq)
                budget -= n
                i += 1
                continue
            # the request preempted itself; the ones after it are gone too
        # waiting requests, first come first served
        while (self.waiting and budget > 0 and not preempted
               and len(self.running) < self.max_num_seqs):
            seq = self.waiting[0]
            hits = self.kv.computed_blocks(seq)
            # blocks of its first chunk beyond the hits (before touching them)
            n_hit = len(hits) * self.kv.block_size
            n = min(seq.num_tokens - n_hit, budget)
            if self.long_prefill_threshold:
                n = min(n, self.long_prefill_threshold)
            fresh = sum(1 for b in hits if b.ref_cnt == 0)
            need = -(-(n_hit + n) // self.kv.block_size) - len(hits)
            if need + fresh + self.watermark_blocks > self.kv.pool.num_free:
                break
            self.waiting.pop(0)
            self.kv.admit(seq, hits)
            ok = self.kv.allocate_slots(seq, n, copies)
            assert ok
            self.running.append(seq)
            scheduled[seq.request_id] = n
            order.append(seq)
            budget -= n
        reqs, toks, poss = [], [], []
        width = max([len(seq.blocks) for seq in order] + [1])
        table = np.zeros((len(order), width), dtype=np.int32)
        for i, seq in enumerate(order):
            n = scheduled[seq.request_id]
            nb = len(seq.blocks)
            table[i, :nb] = seq.ids[:nb]
            reqs.append(StepRequest(seq.request_id, table[i], nb,
                                    seq.num_computed, n))
            toks += seq.token_ids[seq.num_computed:seq.num_computed + n]
            poss += list(range(seq.num_computed, seq.num_computed + n))
        return StepPlan(self.step_no, scheduled, reqs, copies, toks, poss,
                        preempted, table)

    def update(self, plan: StepPlan, sampled: Dict[str, int]) -> List[str]:
        """After the step ran: commit the computed tokens; a request whose
        tokens are all computed appends its sampled token (`sampled[id]`)
        and finishes when it has max_tokens outputs.  Returns the ids of the
        requests that finished."""
        done = []
        by_id = {s.request_id: s for s in self.running}
        for rid, n in plan.scheduled.items():
            seq = by_id.get(rid)
            if seq is None:
                continue
            self.kv.commit(seq, n)
            if seq.num_computed == seq.num_tokens:
                seq.token_ids.append(int(sampled[rid]))
                if seq.finished:
                    self.running.remove(seq)
                    self.kv.free(seq)
                    self.finished.append(seq)
                    done.append(rid)
        return done
