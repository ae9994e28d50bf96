"""Oracle work for one sequence of a full-size FP8 parity case, run in a pool worker.

Imports numpy and the oracle only (the workers are spawned processes). Each step is
an oracle function, called in the order the test applies them on the GPU:

1. quantise the sequence's live blocks of the bf16 cache (``fp8_ref.quantize_rows``);
   the null block, which the GPU test fills with NaN, is never quantised or read;
2. the quantising write of the sequence's new rows (``fp8_ref.cache_write_fp8``);
3. compare codes and scales bit for bit with the GPU's;
4. NaN codes and scales past the sequence's end in its last block (never read);
5. dequantise (``fp8_ref.dequantize_cache``) and decode (``paged_ref.paged_decode``).

The blocks a sequence reads are copied into a compact cache whose block 0 is the
null block and whose block i + 1 is the sequence's i-th live block; its table row is
remapped to match. Paging makes the result independent of physical block ids (paged
attention equals contiguous attention under any table), so this is the same problem
the GPU solved, at a fraction of the memory of the whole cache in float64.
"""
from __future__ import annotations

import numpy as np

from oracle import fp8_ref as f8
from oracle import paged_ref as ref


def fp8_sequence(k_pre, v_pre, gpu_kc, gpu_ks, gpu_vc, gpu_vs, q_row, table_row, seq_len,
                 slots, k_new, v_new, block_size, scale, window):
    """Returns (o [1, H, d], lse [1, H], mismatching code/scale entries)."""
    n = int(seq_len)
    nblk = -(-n // block_size)
    ids = [int(x) for x in table_row[:nblk]]
    live = [x for x in ids if x != 0]
    index = {x: i + 1 for i, x in enumerate(live)}
    sub_table = np.zeros((1, max(nblk, 1)), dtype=np.int32)
    for j, x in enumerate(ids):
        sub_table[0, j] = index.get(x, 0)
    phys = np.array([0] + live, dtype=np.int64)
    mismatches = 0
    dq = []
    for pre, new, gc, gs in ((k_pre, k_new, gpu_kc, gpu_ks), (v_pre, v_new, gpu_vc, gpu_vs)):
        # The live blocks are quantised; the compact block 0 stands for the null block
        # (its rows are only ever masked), with zero codes and scales.
        live_codes, live_scales = f8.quantize_rows(np.asarray(pre[phys[1:]]))
        codes = np.zeros((len(phys),) + live_codes.shape[1:], dtype=live_codes.dtype)
        codes[1:] = live_codes
        scales = np.zeros((len(phys), live_scales.shape[2], live_scales.shape[1]),
                          dtype=live_scales.dtype)
        scales[1:] = live_scales.transpose(0, 2, 1)
        # new rows of this sequence, their slots remapped to the compact cache
        sub_slots = []
        for s in np.asarray(slots).reshape(-1):
            s = int(s)
            sub_slots.append(index[s // block_size] * block_size + s % block_size)
        if sub_slots:
            codes, scales = f8.cache_write_fp8(codes, scales, new, np.array(sub_slots))
        got_c = np.asarray(gc[phys[1:]])
        got_s = np.asarray(gs[phys[1:]])
        mismatches += int((got_c != codes[1:]).sum())
        mismatches += int((got_s.view(np.uint32) != scales[1:].view(np.uint32)).sum())
        if n % block_size:
            blk = int(sub_table[0, n // block_size])
            codes[blk, n % block_size:] = 0x7F
            scales[blk, :, n % block_size:] = np.nan
        dq.append(f8.dequantize_cache(codes, scales))
    o, lse = ref.paged_decode(np.asarray(q_row), dq[0], dq[1], sub_table, np.array([n]),
                              block_size, scale, window)
    return o, lse, mismatches
