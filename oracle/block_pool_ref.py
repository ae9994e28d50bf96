"""Oracle for the host side of the paged KV cache: addressing, block pool, tables.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and bench.py's
cpu_baseline / reference leg may import this module; the product library never
does. It is plain Python (deques, sets, loops) written from the pages:

* "KVCache 优化技能" (model-infer-kvcache skill note), §3.1 logical -> physical
  mapping, §3.2 static block_table, §3.3 slot_mapping, §3.4 actual_seq_lengths;
* "KV Cache 管理设计文档", §2.3 SingleTypeKVCacheManager (skipped tokens,
  Full / SlidingWindow managers), §2.4 BlockPool, §3.3.1 the blocks-to-allocate
  formula, §4.2.1 calculate_block_num, §4.2.2 prepare_block_tables /
  prepare_slot_mapping;
* "昇腾 NPU 独立部署模式 KVCache 自管完整指南", 模式二 (runner-owned slot_mapping
  for prefill and decode; the two slot formulas agree when the table is arange).
"""
from __future__ import annotations

from collections import deque

import numpy as np


class OutOfBlocks(Exception):
    """The pool holds fewer free blocks than requested (nothing was allocated)."""


class DoubleFree(Exception):
    """A block that is already free (or the null block) was freed again."""


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


# --------------------------------------------------------------------------
# Logical -> physical mapping ("KVCache 优化技能" §3.1)
# --------------------------------------------------------------------------
def logical_to_physical(block_table, batch_idx: int, seq_pos: int, block_size: int):
    """Return (logical block, offset in block, physical block id, physical slot).

    logical block = seq_pos // block_size; offset = seq_pos % block_size;
    physical block = block_table[batch_idx, logical block];
    slot = physical block * block_size + offset.
    """
    lb = seq_pos // block_size
    off = seq_pos % block_size
    pb = int(block_table[batch_idx][lb])
    return lb, off, pb, pb * block_size + off


def slot_mapping(block_table, start_pos, num_new, block_size: int) -> np.ndarray:
    """General slot_mapping: one slot per new token, sequences concatenated.

    Sequence b writes positions start_pos[b] .. start_pos[b] + num_new[b] - 1; each
    slot is block_table[b, pos // bs] * bs + pos % bs ("KV Cache 管理设计文档"
    §4.2.2 prepare_slot_mapping; skill note §3.1 formula).
    """
    out = []
    for b in range(len(num_new)):
        for i in range(int(num_new[b])):
            pos = int(start_pos[b]) + i
            out.append(logical_to_physical(block_table, b, pos, block_size)[3])
    return np.asarray(out, dtype=np.int32)


def slot_mapping_contiguous_prefill(kv_len, max_seq_len: int) -> np.ndarray:
    """Skill note §3.3 prefill form: concat of arange(b*max_seq_len, b*max_seq_len + len_b)."""
    parts = [np.arange(b * max_seq_len, b * max_seq_len + int(n)) for b, n in enumerate(kv_len)]
    return np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)


def slot_mapping_contiguous_decode(kv_len, max_seq_len: int) -> np.ndarray:
    """Skill note §3.3 decode form: kv_len.view(B, 1) + arange(0, B*max_seq_len, max_seq_len)."""
    kv_len = np.asarray(kv_len, dtype=np.int64)
    offset = np.arange(0, len(kv_len) * max_seq_len, max_seq_len).reshape(-1, 1)
    return (kv_len.reshape(-1, 1) + offset).astype(np.int32)


def block_table_arange(batch: int, blocks_per_seq: int) -> np.ndarray:
    """Static table of the skill note §3.2: arange(total).reshape(batch, -1), int32."""
    return np.arange(batch * blocks_per_seq, dtype=np.int32).reshape(batch, blocks_per_seq)


def actual_seq_lengths(kv_len, layout: str, phase: str) -> np.ndarray:
    """actual_seq_lengths per layout and phase (skill note §3.4; standalone guide table).

    TND prefill: cumulative sums (KV and Q alike); decode KV: the direct lengths;
    TND decode Q: cumulative sums of ones. BSH uses the direct lengths throughout.
    """
    kv_len = np.asarray(kv_len, dtype=np.int64)
    if phase == "prefill":
        return np.cumsum(kv_len) if layout == "TND" else kv_len.copy()
    if phase == "decode_kv":
        return kv_len.copy()
    if phase == "decode_q":
        ones = np.ones_like(kv_len)
        return np.cumsum(ones) if layout == "TND" else ones
    raise ValueError(phase)


# --------------------------------------------------------------------------
# BlockPool ("KV Cache 管理设计文档" §2.4)
# --------------------------------------------------------------------------
class BlockPool:
    """FIFO free queue plus a set for O(1) double-free detection.

    The queue starts as ``initial_order`` (default 0..num_blocks-1); the first id
    popped becomes the null block, which is never handed out.
    """

    def __init__(self, num_blocks: int, initial_order=None):
        order = list(range(num_blocks)) if initial_order is None else [int(x) for x in initial_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("initial_order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.free_queue = deque(order)
        self.free_set = set(order)
        self.null_block = self.free_queue.popleft()
        self.free_set.discard(self.null_block)

    def num_free(self) -> int:
        return len(self.free_queue)

    def get_new_blocks(self, n: int) -> list[int]:
        if n > len(self.free_queue):
            raise OutOfBlocks(f"need {n}, have {len(self.free_queue)}")
        out = [self.free_queue.popleft() for _ in range(n)]
        for blk in out:
            self.free_set.discard(blk)
        return out

    def free_blocks(self, blocks) -> None:
        blocks = [int(b) for b in blocks]
        for blk in blocks:
            if blk == self.null_block or blk in self.free_set or not 0 <= blk < self.num_blocks:
                raise DoubleFree(f"block {blk}")
        if len(set(blocks)) != len(blocks):
            raise DoubleFree("duplicate ids in one free call")
        for blk in blocks:
            self.free_queue.append(blk)
            self.free_set.add(blk)


# --------------------------------------------------------------------------
# Single-type managers ("KV Cache 管理设计文档" §2.3, §3.3.1)
# --------------------------------------------------------------------------
def num_skipped_tokens(num_computed_tokens: int, window: int) -> int:
    """Full attention skips nothing; a sliding window skips max(0, n - W + 1)."""
    if window <= 0:
        return 0
    return max(0, num_computed_tokens - window + 1)


def num_blocks_to_allocate(num_tokens_need_slot: int, existing: int, block_size: int) -> int:
    """max(0, ceil(tokens / bs) - blocks already held) (§3.3.1)."""
    return max(0, ceil_div(num_tokens_need_slot, block_size) - existing)


def block_table_row(pool: BlockPool, seq_len: int, block_size: int, window: int) -> list[int]:
    """Logical table row of one sequence of total length ``seq_len``.

    The row has ceil(seq_len / bs) entries. For a sliding window the tokens
    computed before the newest one are n = seq_len - 1; the leading
    floor(skipped / bs) blocks, wholly outside the window, are the null block and
    take nothing from the pool (§2.3.2); the rest come from the pool in FIFO order.
    """
    nblk = ceil_div(seq_len, block_size)
    skipped = num_skipped_tokens(seq_len - 1, window)
    n_null = min(skipped // block_size, nblk)
    return [pool.null_block] * n_null + pool.get_new_blocks(nblk - n_null)


def prepare_block_tables(pool: BlockPool, seq_lens, block_size: int, window: int,
                         max_blocks_per_seq: int) -> np.ndarray:
    """Batch table [B, max_blocks_per_seq], rows padded with the null block (§4.2.2)."""
    table = np.full((len(seq_lens), max_blocks_per_seq), pool.null_block, dtype=np.int32)
    for b, n in enumerate(seq_lens):
        row = block_table_row(pool, int(n), block_size, window)
        if len(row) > max_blocks_per_seq:
            raise ValueError("sequence longer than max_blocks_per_seq * block_size")
        table[b, : len(row)] = row
    return table


# --------------------------------------------------------------------------
# Pool sizing ("KV Cache 管理设计文档" §4.2.1 calculate_block_num)
# --------------------------------------------------------------------------
def block_num_fixed(max_concurrency: int, sliding_window: int, next_n: int, block_size: int) -> int:
    """Sliding-window types: max_conc * (ceil((W + 2*next_n) / bs) + 1) + 1 (the +1: null)."""
    return max_concurrency * (ceil_div(sliding_window + 2 * next_n, block_size) + 1) + 1


def block_num_full_offline(max_len: int, block_size: int, max_concurrency: int) -> int:
    """Full attention, offline: ceil(max_len / bs) * max_conc + 1."""
    return ceil_div(max_len, block_size) * max_concurrency + 1


def block_num_full_online(available_bytes: int, per_token_bytes: int, block_size: int) -> int:
    """Full attention, online: floor(floor(budget / per_token_bytes) / bs) + 1."""
    return (available_bytes // per_token_bytes) // block_size + 1
