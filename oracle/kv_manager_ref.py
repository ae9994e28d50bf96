"""Oracle for the allocator: KVCacheManager, single-type managers, shared blocks.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and bench.py's
cpu_baseline / reference leg may import this module; the product library never
does. Plain Python (deques, dicts, loops) written from the pages:

* "KV Cache 管理设计文档" (cann-recipes-infer), §2.2 KVCacheManager
  (allocate_slots, get_block_ids, free, format_usage), §2.3 SingleTypeKVCacheManager
  (get_num_blocks_to_allocate, allocate_new_blocks, remove_skipped_blocks, free,
  get_num_skipped_tokens), §2.3.2 SlidingWindowManager (null-padded logical layout),
  §2.4 BlockPool, §3.1-3.3 the two-phase allocate_slots;
* "KV Cache 笔记" (the HF continuous-batching section): block fingerprints chained
  from the parent block, the tokens and the layer group; prefix match; fork_blocks
  sharing full blocks by reference count and copying the incomplete last block;
  a process-independent hash (blake2b with an 8-byte digest).

Readings where the pages leave a step open (each listed in the design notes):

* The leading null blocks of a sliding-window layout come from the tokens already
  computed: logical block j is null when it lies wholly before position
  ``computed - W + 1``. Every position a query of this step can see (a paged prefill
  reads the cache through the table) is then backed by a real block.
* Freed blocks go back to the queue tail in the request's logical order.
* A block's fingerprint is forgotten when its reference count drops to zero:
  prefixes are shared while some request holds them.
* The hashed bytes are: the parent fingerprint (8 bytes, little-endian; absent for
  the first block), the block's token ids (int32, little-endian), the group id
  (int32, little-endian). The fingerprint is the 8-byte blake2b digest read
  little-endian.
* Prefix matching covers full blocks only and never the block holding the last
  token, so at least one token of the request is computed.
* One manager per attention type: at most one full-attention manager and one
  sliding-window manager, each with its own pool; the group id of a manager is its
  index.
"""
from __future__ import annotations

import hashlib
from collections import deque

import numpy as np


class OutOfBlocks(Exception):
    """The pool holds fewer free blocks than requested (nothing was allocated)."""


class DoubleFree(Exception):
    """A block was released more times than it is referenced (or is the null block)."""


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def block_hash(parent, tokens, group_id: int) -> int:
    """Fingerprint of one full block: blake2b-64 of parent | tokens | group id."""
    data = b"" if parent is None else int(parent).to_bytes(8, "little")
    data += np.asarray(tokens, dtype="<i4").tobytes()
    data += int(group_id).to_bytes(4, "little", signed=True)
    return int.from_bytes(hashlib.blake2b(data, digest_size=8).digest(), "little")


class RefBlockPool:
    """BlockPool of §2.4 (FIFO queue, first popped id is the null block) whose
    blocks carry a reference count, so that forked requests can share them."""

    def __init__(self, num_blocks: int, initial_order=None):
        order = list(range(num_blocks)) if initial_order is None else [int(x) for x in initial_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("initial_order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.queue = deque(order)
        self.null_block = self.queue.popleft()
        self.ref = [0] * num_blocks

    def num_free(self) -> int:
        return len(self.queue)

    def get_new_blocks(self, n: int) -> list[int]:
        if n > len(self.queue):
            raise OutOfBlocks(f"need {n}, have {len(self.queue)}")
        out = [self.queue.popleft() for _ in range(n)]
        for b in out:
            self.ref[b] = 1
        return out

    def share(self, blocks) -> None:
        for b in blocks:
            if b == self.null_block or self.ref[b] <= 0:
                raise ValueError(f"block {b} is not held")
        for b in blocks:
            self.ref[b] += 1

    def free_blocks(self, blocks) -> list[int]:
        """Drop one reference per listed id; ids that reach zero go to the queue
        tail in the listed order. Returns those ids."""
        blocks = [int(b) for b in blocks]
        count: dict[int, int] = {}
        for b in blocks:
            if not 0 <= b < self.num_blocks or b == self.null_block:
                raise DoubleFree(f"block {b}")
            count[b] = count.get(b, 0) + 1
            if count[b] > self.ref[b]:
                raise DoubleFree(f"block {b} released more often than referenced")
        released = []
        for b in blocks:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.queue.append(b)
                released.append(b)
        return released


class SingleTypeManager:
    """Logical block lists of one attention type (§2.3). window 0 = full attention."""

    def __init__(self, pool: RefBlockPool, block_size: int, max_model_len: int, window: int = 0,
                 group_id: int = 0, prefix_caching: bool = False):
        self.pool = pool
        self.block_size = block_size
        self.max_model_len = max_model_len
        self.window = window
        self.group_id = group_id
        self.prefix_caching = prefix_caching and window == 0
        self.req_to_blocks: dict[int, list[int]] = {}
        self.req_hashes: dict[int, list[int]] = {}
        self.hash_to_block: dict[int, int] = {}
        self.block_to_hash: dict[int, int] = {}

    @property
    def null(self) -> int:
        return self.pool.null_block

    def num_skipped_tokens(self, num_computed_tokens: int) -> int:
        """0 for full attention; max(0, n - W + 1) for a sliding window (§2.3)."""
        if self.window <= 0:
            return 0
        return max(0, num_computed_tokens - self.window + 1)

    def _release(self, blocks) -> None:
        for b in self.pool.free_blocks(blocks):
            h = self.block_to_hash.pop(b, None)
            if h is not None:
                del self.hash_to_block[h]

    def remove_skipped_blocks(self, req: int, total_computed: int) -> None:
        """Blocks wholly before the first position still visible become the null
        block and go back to the pool (§2.3, §2.3.2)."""
        blocks = self.req_to_blocks.get(req)
        if not blocks:
            return
        n_skip = self.num_skipped_tokens(total_computed) // self.block_size
        freed = []
        for j in range(min(n_skip, len(blocks))):
            if blocks[j] != self.null:
                freed.append(blocks[j])
                blocks[j] = self.null
        self._release(freed)

    def _layout(self, num_tokens: int, total_computed: int) -> tuple[int, int]:
        """(logical entries, leading null entries) covering num_tokens."""
        nblk = ceil_div(num_tokens, self.block_size)
        n_null = min(self.num_skipped_tokens(total_computed) // self.block_size, nblk)
        return nblk, n_null

    def get_num_blocks_to_allocate(self, req: int, num_tokens: int, total_computed: int) -> int:
        """New real blocks needed so the list covers num_tokens (§3.3.1)."""
        nblk, n_null = self._layout(num_tokens, total_computed)
        held = len(self.req_to_blocks.get(req, []))
        return sum(1 for j in range(held, nblk) if j >= n_null)

    def allocate_new_blocks(self, req: int, num_tokens: int, total_computed: int) -> None:
        nblk, n_null = self._layout(num_tokens, total_computed)
        blocks = self.req_to_blocks.setdefault(req, [])
        n_new = self.get_num_blocks_to_allocate(req, num_tokens, total_computed)
        fresh = deque(self.pool.get_new_blocks(n_new))
        for j in range(len(blocks), nblk):
            blocks.append(self.null if j < n_null else fresh.popleft())

    def free(self, req: int) -> None:
        blocks = self.req_to_blocks.pop(req, [])
        self.req_hashes.pop(req, None)
        self._release([b for b in blocks if b != self.null])

    # ---- prefix sharing ("KV Cache 笔记", HF continuous batching) ----
    def cache_full_blocks(self, req: int, tokens) -> None:
        """Fingerprint every full block of the request not fingerprinted yet."""
        if not self.prefix_caching:
            return
        blocks = self.req_to_blocks.get(req, [])
        hashes = self.req_hashes.setdefault(req, [])
        n_full = min(len(tokens) // self.block_size, len(blocks))
        for j in range(len(hashes), n_full):
            parent = hashes[j - 1] if j else None
            h = block_hash(parent, tokens[j * self.block_size:(j + 1) * self.block_size], self.group_id)
            hashes.append(h)
            b = blocks[j]
            if h not in self.hash_to_block and b not in self.block_to_hash:
                self.hash_to_block[h] = b
                self.block_to_hash[b] = h

    def match_prefix(self, tokens) -> list[int]:
        """Held blocks whose fingerprint chain equals the leading full blocks of
        `tokens`, never including the block of the last token."""
        if not self.prefix_caching:
            return []
        out, parent = [], None
        j = 0
        while (j + 1) * self.block_size <= len(tokens) - 1:
            h = block_hash(parent, tokens[j * self.block_size:(j + 1) * self.block_size], self.group_id)
            if h not in self.hash_to_block:
                break
            out.append(self.hash_to_block[h])
            parent = h
            j += 1
        return out

    def attach_prefix(self, req: int, blocks, tokens) -> None:
        self.pool.share(blocks)
        self.req_to_blocks[req] = list(blocks)
        hashes, parent = [], None
        for j in range(len(blocks)):
            parent = block_hash(parent, tokens[j * self.block_size:(j + 1) * self.block_size], self.group_id)
            hashes.append(parent)
        self.req_hashes[req] = hashes

    def fork_plan(self, parent: int, num_tokens: int, shareable: bool) -> list[tuple[int, str]]:
        """Per logical entry of the forked list: (parent block, action) with action
        'null', 'share' (full block, one more reference) or 'copy' (new block whose
        contents are copied). Shared: only the incomplete last block is copied;
        not shared: every real block is copied ("KV Cache 笔记", fork_blocks)."""
        blocks = self.req_to_blocks[parent]
        nblk = ceil_div(num_tokens, self.block_size)
        if nblk > len(blocks):
            raise ValueError("parent holds fewer blocks than num_tokens needs")
        n_full = num_tokens // self.block_size
        plan = []
        for j in range(nblk):
            b = blocks[j]
            if b == self.null:
                plan.append((b, "null"))
            elif shareable and j < n_full:
                plan.append((b, "share"))
            else:
                plan.append((b, "copy"))
        return plan

    def fork(self, parent: int, children, num_tokens: int, shareable: bool) -> list[tuple[int, int]]:
        """Give each child the parent's first ceil(num_tokens / bs) entries; returns
        the (source, destination) block copies, child by child."""
        plan = self.fork_plan(parent, num_tokens, shareable)
        copies = []
        for child in children:
            row = []
            for b, action in plan:
                if action == "null":
                    row.append(self.null)
                elif action == "share":
                    self.pool.share([b])
                    row.append(b)
                else:
                    nb = self.pool.get_new_blocks(1)[0]
                    copies.append((b, nb))
                    row.append(nb)
            self.req_to_blocks[child] = row
            if shareable and self.prefix_caching:
                n_full = num_tokens // self.block_size
                self.req_hashes[child] = list(self.req_hashes.get(parent, [])[:n_full])
        return copies


class KVCacheManager:
    """Request-level coordinator over the single-type managers (§2.2, §3)."""

    def __init__(self, windows, num_blocks, block_size: int, max_model_len: int,
                 prefix_caching: bool = False, initial_orders=None):
        kinds = [w > 0 for w in windows]
        if len(windows) == 0 or len(kinds) != len(set(kinds)):
            raise ValueError("one manager per attention type: at most one full and one sliding")
        self.block_size = block_size
        self.max_model_len = max_model_len
        self.managers = []
        for i, (w, n) in enumerate(zip(windows, num_blocks)):
            order = None if initial_orders is None else initial_orders[i]
            self.managers.append(SingleTypeManager(RefBlockPool(n, order), block_size, max_model_len,
                                                   window=w, group_id=i,
                                                   prefix_caching=prefix_caching))

    def allocate_slots(self, req: int, computed_tokens: int, num_new_tokens: int,
                       lookahead_tokens: int = 0) -> bool:
        """Two phases (§3.3): per manager, recycle skipped blocks and check the pool
        can supply the new blocks (False at the first that cannot, nothing
        allocated); then allocate in every manager."""
        total_computed = min(computed_tokens, self.max_model_len)
        need = min(computed_tokens + num_new_tokens + lookahead_tokens, self.max_model_len)
        for m in self.managers:
            m.remove_skipped_blocks(req, total_computed)
            if m.pool.num_free() < m.get_num_blocks_to_allocate(req, need, total_computed):
                return False
        for m in self.managers:
            m.allocate_new_blocks(req, need, total_computed)
        return True

    def get_block_ids(self, req: int) -> list[list[int]]:
        return [list(m.req_to_blocks.get(req, [])) for m in self.managers]

    def free(self, req: int) -> None:
        for m in self.managers:
            m.free(req)

    def format_usage(self) -> str:
        """"full:used/total,sliding:used/total": used = blocks handed out (the null
        block not counted), total = the pool's size."""
        parts = []
        for m in self.managers:
            name = "sliding" if m.window > 0 else "full"
            used = m.pool.num_blocks - 1 - m.pool.num_free()
            parts.append(f"{name}:{used}/{m.pool.num_blocks}")
        return ",".join(parts)

    def block_table(self, type_idx: int, reqs, max_blocks_per_seq: int) -> np.ndarray:
        """prepare_block_tables (§4.2.2): rows of the requests' lists, padded with
        the manager's null block."""
        m = self.managers[type_idx]
        table = np.full((len(reqs), max_blocks_per_seq), m.null, dtype=np.int32)
        for i, r in enumerate(reqs):
            row = m.req_to_blocks.get(r, [])
            if len(row) > max_blocks_per_seq:
                raise ValueError("row longer than max_blocks_per_seq")
            table[i, :len(row)] = row
        return table

    def match_prefix(self, req: int, tokens) -> int:
        """Attach the longest fingerprinted prefix common to every manager to a new
        request; returns the number of cached tokens (0 when any manager is a
        sliding window or prefix caching is off)."""
        if any(m.window > 0 or not m.prefix_caching for m in self.managers):
            return 0
        matches = [m.match_prefix(tokens) for m in self.managers]
        n = min(len(x) for x in matches)
        if n == 0:
            return 0
        for m, blocks in zip(self.managers, matches):
            m.attach_prefix(req, blocks[:n], tokens)
        return n * self.block_size

    def cache_blocks(self, req: int, tokens) -> None:
        for m in self.managers:
            m.cache_full_blocks(req, tokens)

    def fork(self, parent: int, children, num_tokens: int, shareable: bool) -> list[list[tuple[int, int]]]:
        """All-or-nothing over the managers: checks every pool can supply the copies
        for all children first (OutOfBlocks, nothing changed), then forks."""
        for m in self.managers:
            plan = m.fork_plan(parent, num_tokens, shareable)
            need = sum(1 for _, a in plan if a == "copy") * len(children)
            if need > m.pool.num_free():
                raise OutOfBlocks(f"fork needs {need}, have {m.pool.num_free()}")
        return [m.fork(parent, children, num_tokens, shareable) for m in self.managers]


def copy_blocks(cache: np.ndarray, pairs) -> np.ndarray:
    """Cache after copying block src to block dst for each pair in order (the
    device side of a fork). cache is [num_blocks, ...]; rows are bit copies."""
    out = cache.copy()
    for s, d in pairs:
        out[d] = out[s]
    return out
