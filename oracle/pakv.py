"""Oracle prefix-aware KV cache (PAKV): a trie of fixed-size KV chunks.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What the pages fix [CA-summary §3.1; CA-blog, Prefix-Aware KV Cache]:
  * key/value tensors are cut into chunks of c tokens; a chunk's K/V is kept
    once in memory and every sequence that shares it refers to it;
  * the chunks form a prefix tree in which every root-to-leaf path is one
    sequence; a new sequence adds a path, a finished one removes it;
  * a sequence's prompt is matched against the tree when it arrives, matched
    chunks gain a reference, a finishing sequence drops its references, and a
    chunk with no references left is collected [CA-blog, 動的プレフィックス検出].

Readings where the pages leave the step open (each one is the plainest reading
the rest supports):
  R2  a chunk is shared only when its full c tokens and the whole path before
      it match; the trailing partial chunk (< c tokens) of a sequence is always
      a private leaf and is never matched; children are matched by their exact
      c-token tuple.
  R5  slots are taken lowest index first (a min-heap of free slots); a freed
      slot goes back to the heap at once.
  R6  a matched chunk keeps the K/V rows of its first inserter; later
      inserters' rows for matched tokens are not read.
  R7  a sequence's context is exactly the tokens inserted for it.
  NS  with ``no_sharing`` nothing is ever matched, so every sequence owns a
      private chain of chunks (the flat paged layout used as the control).
  R13 decode-time append [CA-summary §3.1: decoding appends tokens to leaf
      chunks or grows new chunks; §3.3: a full chunk triggers a context
      copy]: the appended tokens first fill the sequence's partial last chunk
      (always private, R2), then grow new private chunks (lowest slots first);
      an append never matches existing chunks.  A chunk that becomes full
      this way becomes matchable for later inserts unless its parent already
      has a matchable child with the same tokens.  Only growing a new chunk
      changes the tree's structure (bumps the generation); filling the
      partial chunk in place does not.
"""
from __future__ import annotations

import heapq

import numpy as np


class OracleError(Exception):
    """Raised with one of: 'invalid', 'oom', 'exists', 'not_found'."""

    def __init__(self, code: str, msg: str = ""):
        super().__init__(f"{code}: {msg}")
        self.code = code


class Node:
    __slots__ = ("slot", "tokens", "k", "v", "children", "match", "parent", "refcount")

    def __init__(self, slot, tokens, k, v, parent):
        self.slot = slot          # chunk slot in the pool (root: -1)
        self.tokens = tokens      # tuple of the chunk's token ids
        self.k = k                # [L, ntok, H, D] float16 view, or None
        self.v = v
        self.children = []        # every child, in insertion order
        self.match = {}           # token tuple -> child, full shareable chunks only
        self.parent = parent
        self.refcount = 0         # live sequences whose path holds this chunk

    @property
    def ntok(self) -> int:
        return len(self.tokens)


class OracleTrie:
    def __init__(self, chunk: int, capacity: int, no_sharing: bool = False):
        if chunk <= 0 or capacity < 0:
            raise OracleError("invalid", "chunk and capacity")
        self.chunk = chunk
        self.capacity = capacity
        self.no_sharing = no_sharing
        self.root = Node(-1, (), None, None, None)
        self.free = list(range(capacity))
        heapq.heapify(self.free)
        self.paths: dict[int, list[Node]] = {}
        self.lengths: dict[int, int] = {}
        self.generation = 0

    # -- queries -----------------------------------------------------------
    def match_prefix(self, tokens) -> int:
        """Leading tokens of ``tokens`` whose chunks already sit in the tree."""
        if self.no_sharing:
            return 0
        c, node, matched = self.chunk, self.root, 0
        for i in range(len(tokens) // c):
            key = tuple(int(t) for t in tokens[i * c:(i + 1) * c])
            child = node.match.get(key)
            if child is None:
                break
            node, matched = child, matched + c
        return matched

    def slots(self, seq_id: int) -> list[int]:
        return [n.slot for n in self.paths[seq_id]]

    def live_slots(self) -> int:
        return self.capacity - len(self.free)

    def refcount_sum(self) -> int:
        seen, total = set(), 0
        for path in self.paths.values():
            for n in path:
                if id(n) not in seen:
                    seen.add(id(n))
                    total += n.refcount
        return total

    # -- insert / remove ---------------------------------------------------
    def insert(self, seq_id: int, tokens, k=None, v=None) -> int:
        """Add a sequence's path; returns how many leading tokens were shared.

        ``k``/``v`` are [L, n, H, D] arrays (or None for a table-only trie);
        rows of matched tokens are not read (R6).  On any error the trie is
        left exactly as it was.
        """
        tokens = [int(t) for t in tokens]
        n, c = len(tokens), self.chunk
        if n <= 0:
            raise OracleError("invalid", "empty sequence")
        if seq_id in self.paths:
            raise OracleError("exists", str(seq_id))
        n_full, rem = divmod(n, c)
        pieces = [tuple(tokens[i * c:(i + 1) * c]) for i in range(n_full)]
        if rem:
            pieces.append(tuple(tokens[n_full * c:]))

        # Walk the matched prefix (R2).
        node, n_matched = self.root, 0
        if not self.no_sharing:
            for key in pieces[:n_full]:
                child = node.match.get(key)
                if child is None:
                    break
                node, n_matched = child, n_matched + 1
        n_new = len(pieces) - n_matched
        if n_new > len(self.free):
            raise OracleError("oom", f"need {n_new} slots, {len(self.free)} free")

        path, node = [], self.root
        for i, key in enumerate(pieces):
            if i < n_matched:
                node = node.match[key]
            else:
                slot = heapq.heappop(self.free)           # R5: lowest free slot
                a = i * c
                kk = None if k is None else k[:, a:a + len(key)]
                vv = None if v is None else v[:, a:a + len(key)]
                child = Node(slot, key, kk, vv, node)
                node.children.append(child)
                if len(key) == c and not self.no_sharing:
                    node.match[key] = child
                node = child
            node.refcount += 1
            path.append(node)
        self.paths[seq_id] = path
        self.lengths[seq_id] = n
        self.generation += 1
        return n_matched * c

    def append(self, seq_id: int, tokens, k=None, v=None) -> int:
        """Append decoded tokens to a sequence (R13).  ``k``/``v`` are
        [L, n, H, D] for the appended tokens (or None).  Returns the number of
        new chunks; on error the trie is unchanged."""
        if seq_id not in self.paths:
            raise OracleError("not_found", str(seq_id))
        tokens = [int(t) for t in tokens]
        n, c = len(tokens), self.chunk
        if n <= 0:
            raise OracleError("invalid", "empty append")
        path = self.paths[seq_id]
        last = path[-1]
        fill = min(c - last.ntok, n)
        n_new = -(-(n - fill) // c)
        if n_new > len(self.free):
            raise OracleError("oom", f"need {n_new} slots, {len(self.free)} free")
        if fill:
            last.tokens = last.tokens + tuple(tokens[:fill])
            if k is not None:
                last.k = np.concatenate([last.k, k[:, :fill]], axis=1)
                last.v = np.concatenate([last.v, v[:, :fill]], axis=1)
            if last.ntok == c and not self.no_sharing:
                last.parent.match.setdefault(last.tokens, last)
        node = last
        for i in range(n_new):
            a = fill + i * c
            key = tuple(tokens[a:a + c])
            slot = heapq.heappop(self.free)
            child = Node(slot, key, None if k is None else k[:, a:a + len(key)],
                         None if v is None else v[:, a:a + len(key)], node)
            node.children.append(child)
            if len(key) == c and not self.no_sharing:
                node.match.setdefault(key, child)
            child.refcount = 1
            path.append(child)
            node = child
        self.lengths[seq_id] += n
        if n_new:
            self.generation += 1
        return n_new

    def remove(self, seq_id: int) -> None:
        """Drop a sequence's references; chunks left with none are freed."""
        if seq_id not in self.paths:
            raise OracleError("not_found", str(seq_id))
        path = self.paths.pop(seq_id)
        del self.lengths[seq_id]
        for node in path:
            node.refcount -= 1
            if node.refcount == 0:
                heapq.heappush(self.free, node.slot)
                parent = node.parent
                if parent is not None and node in parent.children:
                    parent.children.remove(node)
                    if parent.match.get(node.tokens) is node:
                        del parent.match[node.tokens]
        self.generation += 1

    # -- materialisation -----------------------------------------------------
    def materialize(self, seq_id: int, layer: int = 0) -> tuple[np.ndarray, np.ndarray]:
        """The sequence's full K and V, [n, H, D] float64, read chunk by chunk
        along its path (each request refers to its chunks [CA-blog,
        Prefix-Aware KV Cache])."""
        path = self.paths[seq_id]
        k = np.concatenate([n.k[layer] for n in path], axis=0).astype(np.float64)
        v = np.concatenate([n.v[layer] for n in path], axis=0).astype(np.float64)
        return k, v
