"""Split-KV schedule: a plain restatement of the policy, and its invariants.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The pages fix only the shapes: ``get_mla_metadata`` returns
``tile_scheduler_metadata`` (num_sm_parts, TileSchedulerMetaDataSize) int32 and
``num_splits`` (batch_size + 1) int32 (FlashMLA-PyTorch page,
flash_mla_interface.py, get_mla_metadata docstring; vLLM page, get_mla_metadata
return table).  The record layout and the partition policy are this library's
choice; the reading of ``num_splits`` as the exclusive prefix sum of the
per-sequence split counts follows from its batch_size + 1 length.

Record (8 int32 per part):
  [0] begin_b   [1] begin_blk   [2] end_b   [3] end_blk
  [4] first_slot (partial-result slot of the part's first segment)
  [5] num_blocks (blocks of KV the part processes)   [6], [7] zero
A part covers, for b in [begin_b, end_b] (b < batch), the blocks
  [begin_blk if b == begin_b else 0,  end_blk if b == end_b else n_b)
where n_b = ceil(max(L_b, 0) / 64); an empty range is no segment.

Policy (greedy contiguous walk with a fixed cost per segment):
  c = blocks charged for every segment a part opens: segment_cost(R, kv_bytes)
      = 6 for R >= 64 query rows per KV head, 4 below, plus 1 for a one-byte
      (e4m3) cache; FIXED_COST = 6 is the bf16 value for R >= 64
  W = sum over b with n_b > 0 of (n_b + c)
  T = max(1, ceil((W + (parts - 1) * c) / parts))
  parts take the blocks in (b, blk) order; part p stops opening segments once
  T - load - c <= 0, takes min(remaining, T - load - c) blocks when it opens
  one, and the last part takes whatever remains.
Every part boundary either splits a sequence (one more segment, cost c) or
falls between sequences (the part left at most c of its budget unused), so
the (parts - 1) * c term makes every part's load, the last one's included,
at most T.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

PAGE = 64
# The per-segment cost, in 64-row blocks: a part's fixed work for each
# sequence it opens (loading that sequence's queries, storing its output)
# measured on the decode kernel as about six pages' time.
FIXED_COST = 6
RECORD = 8


def segment_cost(rows_per_head_k: int, kv_bytes: int = 2) -> int:
    """Blocks charged per segment: a part's fixed work for a sequence it takes up,
    in page times -- larger with many query rows (more output to store), and one more
    for an e4m3 cache, whose pages take less time than bf16 ones."""
    return (6 if rows_per_head_k >= 64 else 4) + (1 if kv_bytes == 1 else 0)


def n_blocks(seqlens: Sequence[int]) -> List[int]:
    return [(max(0, int(L)) + PAGE - 1) // PAGE for L in seqlens]


def schedule(seqlens: Sequence[int], parts: int, fixed_cost: int = FIXED_COST
             ) -> Tuple[np.ndarray, np.ndarray]:
    """The policy walk; returns (metadata (parts, 8) int32, num_splits (B+1) int32)."""
    nb = n_blocks(seqlens)
    B = len(nb)
    W = sum(n + fixed_cost for n in nb if n > 0)
    T = max(1, -(-(W + (parts - 1) * fixed_cost) // parts))
    md = np.zeros((parts, RECORD), dtype=np.int32)
    splits = [0] * B
    seg_index_of_first = []   # (b of first segment, index among b's segments) per part
    b, k = 0, 0
    for p in range(parts):
        begin = (b, k)
        load = 0
        total = 0
        first = None
        while b < B:
            if nb[b] == 0:
                b, k = b + 1, 0
                continue
            rem = nb[b] - k
            if p == parts - 1:
                take = rem
            else:
                avail = T - load - fixed_cost
                if avail <= 0:
                    break
                take = min(rem, avail)
            if first is None:
                first = (b, splits[b])
            splits[b] += 1
            load += fixed_cost + take
            total += take
            k += take
            if k == nb[b]:
                b, k = b + 1, 0
            if p != parts - 1 and load >= T:
                break
        md[p, 0], md[p, 1] = begin
        md[p, 2], md[p, 3] = b, k
        md[p, 5] = total
        seg_index_of_first.append(first)
    num_splits = np.zeros(B + 1, dtype=np.int32)
    num_splits[1:] = np.cumsum(splits)
    for p, first in enumerate(seg_index_of_first):
        if first is not None:
            md[p, 4] = num_splits[first[0]] + first[1]
    return md, num_splits


def part_segments(md_row, seqlens: Sequence[int]) -> List[Tuple[int, int, int]]:
    """(b, blk_begin, blk_end) segments of one part, by the record's rule."""
    nb = n_blocks(seqlens)
    B = len(nb)
    b0, k0, b1, k1 = (int(x) for x in md_row[:4])
    segs = []
    b = b0
    while b <= b1 and b < B:
        lo = k0 if b == b0 else 0
        hi = k1 if b == b1 else nb[b]
        if lo < hi:
            segs.append((b, lo, hi))
        b += 1
    return segs


def check_metadata(seqlens: Sequence[int], md: np.ndarray, num_splits: np.ndarray) -> None:
    """Raise AssertionError unless (md, num_splits) is a valid schedule.

    Checked: every block (b, blk < n_b) is covered exactly once and in order;
    no segment touches a block >= n_b; num_splits is the prefix sum of the
    per-sequence segment counts; each part's first_slot and num_blocks agree
    with its segments.
    """
    md = np.asarray(md)
    num_splits = np.asarray(num_splits)
    nb = n_blocks(seqlens)
    B = len(nb)
    assert md.ndim == 2 and md.shape[1] == RECORD, md.shape
    assert num_splits.shape == (B + 1,), num_splits.shape
    seq = []
    count = [0] * B
    first_of = []
    for p in range(md.shape[0]):
        segs = part_segments(md[p], seqlens)
        for (b, lo, hi) in segs:
            assert 0 <= lo < hi <= nb[b], (p, b, lo, hi, nb[b])
            seq.extend((b, k) for k in range(lo, hi))
        first_of.append((segs[0][0], count[segs[0][0]]) if segs else None)
        for (b, _, _) in segs:
            count[b] += 1
        assert int(md[p, 5]) == sum(hi - lo for (_, lo, hi) in segs), (p, md[p])
        assert int(md[p, 6]) == 0 and int(md[p, 7]) == 0
    expect = [(b, k) for b in range(B) for k in range(nb[b])]
    assert seq == expect, "blocks not covered exactly once in order"
    assert int(num_splits[0]) == 0
    for b in range(B):
        assert int(num_splits[b + 1]) - int(num_splits[b]) == count[b], (b, count[b])
        if nb[b] > 0:
            assert count[b] >= 1
    for p, first in enumerate(first_of):
        if first is not None:
            assert int(md[p, 4]) == int(num_splits[first[0]]) + first[1], (p, md[p], first)


def max_part_load(seqlens: Sequence[int], md: np.ndarray, fixed_cost: int = FIXED_COST) -> int:
    loads = []
    for p in range(md.shape[0]):
        segs = part_segments(md[p], seqlens)
        loads.append(sum(hi - lo + fixed_cost for (_, lo, hi) in segs))
    return max(loads) if loads else 0
