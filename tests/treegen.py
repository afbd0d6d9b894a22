"""Random prefix trees for tests: token lists only (no attention arithmetic)."""
import numpy as np


def random_token_lists(seed: int, n_seqs: int, chunk: int, alphabet: int = 3,
                       max_len: int = 24, n_stems: int = 3):
    """Sequences built from a few random stems plus random tails.  A small
    alphabet makes chunk tuples collide across branches, so the tree gets
    shared chunks, branch points, sequences ending at inner nodes and partial
    leaves."""
    rng = np.random.default_rng(seed)
    stems = [rng.integers(0, alphabet, size=int(rng.integers(0, max_len))).tolist()
             for _ in range(n_stems)]
    out = []
    for _ in range(n_seqs):
        stem = stems[int(rng.integers(0, n_stems))]
        cut = int(rng.integers(0, len(stem) + 1))
        tail = rng.integers(0, alphabet, size=int(rng.integers(0, max_len // 2))).tolist()
        toks = stem[:cut] + tail
        if not toks:
            toks = [int(rng.integers(0, alphabet))]
        out.append(toks)
    return out


def lcp_chunks(a, b, c):
    """Longest common prefix of two token lists, in whole chunks."""
    k = 0
    while (k + 1) * c <= min(len(a), len(b)) and a[k * c:(k + 1) * c] == b[k * c:(k + 1) * c]:
        k += 1
    return k


def random_segment_sequences(seed: int, n_seqs: int, chunk: int, n_segments: int = 8):
    """Sequences that walk a random tree of token segments, plus random
    private tails.  Segment lengths mix whole chunks with ragged lengths, so
    branch points fall both on and inside chunk boundaries; an empty tail
    makes identical sequences that end at the same node."""
    rng = np.random.default_rng(seed)
    parent, length = [-1], [0]
    for s in range(1, n_segments + 1):
        parent.append(int(rng.integers(0, s)))
        length.append(int(rng.choice([chunk, 2 * chunk, 3 * chunk, chunk // 2, chunk + 3,
                                      2 * chunk - 1])))
    out = []
    for i in range(n_seqs):
        s = int(rng.integers(0, n_segments + 1))
        path = []
        while s > 0:
            path.append(s)
            s = parent[s]
        toks = []
        for seg in reversed(path):
            toks += [seg * 1000 + j for j in range(length[seg])]
        tail = int(rng.integers(0, 2 * chunk + 1))
        toks += [500_000 + i * 1000 + j for j in range(tail)]
        if not toks:
            toks = [900_000 + i]
        out.append(toks)
    return out
