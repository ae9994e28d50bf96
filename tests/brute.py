"""Brute-force attention with nested Python loops and math.exp, for tiny inputs.

Independent of the oracle's numpy code: it builds every score, normaliser and
weighted sum element by element, reading keys through the block table itself.
"""
import math


def row_attention(qvec, keys, values, visible, scale):
    """keys/values: lists of lists (one per position); visible: list of bool."""
    scores = []
    for j in range(len(keys)):
        if visible[j]:
            s = 0.0
            for i in range(len(qvec)):
                s += qvec[i] * keys[j][i]
            scores.append((j, scale * s))
    if not scores:
        return [0.0] * (len(values[0]) if values else 0), -math.inf
    m = max(s for _, s in scores)
    denom = 0.0
    for _, s in scores:
        denom += math.exp(s - m)
    out = [0.0] * len(values[0])
    for j, s in scores:
        w = math.exp(s - m) / denom
        for i in range(len(out)):
            out[i] += w * values[j][i]
    return out, m + math.log(denom)


def read_positions(cache, table_row, length, bs, head):
    """Key or value rows of one head for positions 0..length-1 via the block table."""
    rows = []
    for pos in range(length):
        blk = table_row[pos // bs]
        rows.append([float(x) for x in cache[blk][pos % bs][head]])
    return rows
