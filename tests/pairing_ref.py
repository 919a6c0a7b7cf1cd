"""Plain restatement of the fine stage's query-cube pairing (csrc/pair.cu).

The fine kernel takes query cubes two at a time and walks the union of their
selections, so a pair (i, j) costs ceil(|sel(i) | sel(j)| / 2) steps.  The
pairing pass picks, per (batch, head), pairs with large overlaps.  It is a
scheduling choice: the attention results do not depend on it.  This module
states the same deterministic integer procedure with numpy and plain loops so
that the GPU pass can be checked for exact agreement on small cases.

  1. overlap(i, j) = |sel(i) & sel(j)| for j in sel(i); the candidates of i
     are the TOPC cubes j != i of sel(i) of largest overlap (ties: smaller j);
  2. ROUNDS1 rounds: every unpaired cube proposes to its unpaired candidate of
     largest overlap (ties: smaller j), if any; mutual proposals pair up;
  3. the still-unpaired cubes, in index order (the first max_left(n) of them),
     run ROUNDS2 rounds of the same matching where each proposes to the
     unpaired cube of largest overlap among the next WINDOW entries of that
     list and the WINDOW entries before it;
  4. cubes still unpaired pair in index order; with N odd one stays single.
Units are listed by their smaller cube index: (i, j) or (i, -1).
"""
import numpy as np

TOPC = 16
ROUNDS1 = 4
ROUNDS2 = 4
MAX_LEFT = 640
WINDOW = 64


def words(n):
    """Bitmap words per cube, rounded up to a multiple of 4."""
    return ((n + 31) // 32 + 3) & ~3


def max_left(n):
    """Length cap of the leftover list."""
    return MAX_LEFT


def overlap_matrix(sel_rows, n):
    s = np.zeros((len(sel_rows), n), np.int64)
    for i, row in enumerate(sel_rows):
        s[i, np.asarray(row)] = 1
    return s @ s.T


def _round(cands, ov_of, partner):
    n = len(partner)
    prop = [-1] * n
    for i in range(n):
        if partner[i] >= 0:
            continue
        best, bv = -1, -1
        for j in cands(i):
            if j == i or partner[j] >= 0:
                continue
            o = ov_of(i, j)
            if o > bv or (o == bv and j < best):
                best, bv = j, o
        prop[i] = best
    for i in range(n):
        j = prop[i]
        if j > i and prop[j] == i:
            partner[i] = j
            partner[j] = i


def pair_cubes(sel_rows, n):
    """sel_rows: list of n index arrays (one head). Returns the unit list."""
    ov = overlap_matrix(sel_rows, n)
    partner = [-1] * n
    cand = []
    for i in range(n):
        js = sorted({int(j) for j in sel_rows[i] if 0 <= int(j) < n and int(j) != i},
                    key=lambda j: (-int(ov[i, j]), j))
        cand.append(js[:TOPC])
    for _ in range(ROUNDS1):
        _round(lambda i: cand[i], lambda i, j: int(ov[i, j]), partner)
    left = [i for i in range(n) if partner[i] < 0][:max_left(n)]
    pos = {c: a for a, c in enumerate(left)}
    for _ in range(ROUNDS2):
        def cands(i):
            if i not in pos:
                return []
            a = pos[i]
            return left[max(0, a - WINDOW):a] + left[a + 1:a + 1 + WINDOW]
        _round(cands, lambda i, j: int(ov[i, j]), partner)
    rest = [i for i in range(n) if partner[i] < 0]
    for a in range(0, len(rest) - 1, 2):
        partner[rest[a]] = rest[a + 1]
        partner[rest[a + 1]] = rest[a]
    if len(rest) % 2:
        partner[rest[-1]] = rest[-1]
    return [(i, -1 if partner[i] == i else partner[i]) for i in range(n) if partner[i] >= i]


def union_steps(units, sel_rows):
    tot = 0
    for i, j in units:
        u = set(int(x) for x in sel_rows[i])
        if j >= 0:
            u |= set(int(x) for x in sel_rows[j])
        tot += (len(u) + 1) // 2
    return tot
