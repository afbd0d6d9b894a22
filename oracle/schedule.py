"""Oracle schedule tables for one decode step of the two-phase partition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What the pages fix [CA-summary §3.2, §3.3]:
  * chunk-first phase: the queries of all sequences that share a chunk are
    batched against it and partial results are kept;
  * sequence-first phase: each query restores its partials and goes through
    its remaining chunks;
  * the tables the kernel reads (the "context") are rebuilt only when the tree
    changes, i.e. when a chunk fills, a sequence joins or a sequence leaves.

Readings where the pages leave the step open:
  R3  a chunk goes to the chunk-first phase iff two or more sequences *of the
      scheduled batch* pass through it; every other chunk of a batch sequence
      is sequence-first, even if sequences outside the batch also hold it.
  R4  ordering: children are visited in insertion order (depth first); at a
      node, the sequences whose path ends there come before those in its
      children, and among themselves by ascending seq_id; chunk-first rows are
      listed in DFS pre-order.  In this order every chunk's sharers are one
      contiguous range [lo, hi) of batch positions.

Tables (all int32, positions are DFS batch positions 0..b-1):
  seq_perm[b]          position -> index into the caller's seq_ids (Q/out row)
  cf_rows[R, 4]        (slot, ntok, lo, hi) per chunk-first chunk, pre-order
  cf_runs[U, 4]        (row0, nrows, lo, hi): maximal stretches of consecutive
                       rows on one path with the same [lo, hi)
  sf_offsets[b+1]      CSR over positions into sf_chunks
  sf_chunks[S, 2]      (slot, ntok) of each position's sequence-first chunks,
                       in path order
  merge_offsets[b+1]   CSR over positions into merge_runs
  merge_runs[M]        indices of the runs whose [lo, hi) holds the position
"""
from __future__ import annotations

import numpy as np

from .pakv import OracleError, OracleTrie


def build_schedule(trie: OracleTrie, seq_ids) -> dict[str, np.ndarray]:
    seq_ids = [int(s) for s in seq_ids]
    b = len(seq_ids)
    if b <= 0:
        raise OracleError("invalid", "empty batch")
    if len(set(seq_ids)) != b:
        raise OracleError("invalid", "duplicate seq_id")
    for s in seq_ids:
        if s not in trie.paths:
            raise OracleError("not_found", str(s))

    # How many batch sequences pass through each node, and where each ends.
    count: dict[int, int] = {}
    ending: dict[int, list[int]] = {}
    for s in seq_ids:
        path = trie.paths[s]
        for node in path:
            count[id(node)] = count.get(id(node), 0) + 1
        ending.setdefault(id(path[-1]), []).append(s)

    # Depth-first walk (R4), iterative so that long chains need no recursion.
    order: list[int] = []
    rows: list[list[int]] = []
    row_node: list = []
    stack = [(trie.root, None, 0)]   # (node, row index or None, next child)
    while stack:
        node, row, ci = stack.pop()
        if ci == 0 and node is not trie.root:
            # pre-visit: open the node's range, emit its row, then its enders
            lo = len(order)
            if count[id(node)] >= 2:
                row = len(rows)
                rows.append([node.slot, node.ntok, lo, -1])
                row_node.append(node)
            order.extend(sorted(ending.get(id(node), [])))
        # next active child
        while ci < len(node.children) and count.get(id(node.children[ci]), 0) == 0:
            ci += 1
        if ci < len(node.children):
            stack.append((node, row, ci + 1))
            stack.append((node.children[ci], None, 0))
        elif row is not None:
            rows[row][3] = len(order)       # close the range after the subtree
    assert len(order) == b

    pos_of = {s: p for p, s in enumerate(order)}
    caller = {s: i for i, s in enumerate(seq_ids)}
    seq_perm = np.array([caller[s] for s in order], dtype=np.int32)

    # Runs: consecutive rows, parent then child, with the same [lo, hi).
    runs: list[list[int]] = []
    for r, row in enumerate(rows):
        if (runs and row_node[r].parent is row_node[r - 1]
                and rows[r - 1][2:] == row[2:]):
            runs[-1][1] += 1
        else:
            runs.append([r, 1, row[2], row[3]])

    # Sequence-first chunks: the chunks only this batch sequence holds (R3).
    sf_offsets, sf_chunks = [0], []
    for s in order:
        for node in trie.paths[s]:
            if count[id(node)] == 1:
                sf_chunks.append([node.slot, node.ntok])
        sf_offsets.append(len(sf_chunks))

    merge_offsets, merge_runs = [0], []
    for p in range(b):
        for u, run in enumerate(runs):
            if run[2] <= p < run[3]:
                merge_runs.append(u)
        merge_offsets.append(len(merge_runs))

    as2 = lambda x, w: np.array(x, dtype=np.int32).reshape(-1, w)
    return {
        "seq_perm": seq_perm,
        "cf_rows": as2(rows, 4),
        "cf_runs": as2(runs, 4),
        "sf_offsets": np.array(sf_offsets, dtype=np.int32),
        "sf_chunks": as2(sf_chunks, 2),
        "merge_offsets": np.array(merge_offsets, dtype=np.int32),
        "merge_runs": np.array(merge_runs, dtype=np.int32),
        "order": np.array(order, dtype=np.int64),
        "pos_of": pos_of,
    }
