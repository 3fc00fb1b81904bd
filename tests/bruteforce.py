"""Pure-Python brute-force restatements used to pin the oracle.

Each function reaches the same result as the oracle by a different route, so
that a slip in the oracle's loops (a wrong chunk index, a swapped rank, an
off-by-one boundary) shows up as a mismatch:

  * ``l2g_by_ownership``: give every global token its owner from the chunk it
    falls in, then list each rank's tokens in ascending global position.
    Under DualChunkSwap rank r's two chunks r < 2P-1-r already lie in
    ascending order, so this equals the oracle's chunk-by-chunk walk without
    sharing its structure.
  * ``metadata_by_runs``: walk rank r's local tokens one at a time and split
    them into runs of equal document id.
  * ``compositions``: every way to write T as an ordered sum of document
    lengths that are multiples of ``unit`` (zero-length documents included),
    for exhaustive checks on tiny T.
"""
from __future__ import annotations


def doc_of_token(cu, g):
    """Document index of global token g (linear scan, skips empty docs)."""
    for i in range(len(cu) - 1):
        if cu[i] <= g < cu[i + 1]:
            return i
    raise IndexError(g)


def owner_dsc(cu, P, g):
    """Rank owning token g under DualChunkSwap (chunk k -> k or 2P-1-k)."""
    i = doc_of_token(cu, g)
    L = cu[i + 1] - cu[i]
    m = L // (2 * P)
    k = (g - cu[i]) // m
    return k if k < P else 2 * P - 1 - k


def owner_packed(T, P, g):
    return g // (T // P)


def l2g_by_ownership(layout, cu, P, T):
    owners = []
    for g in range(T):
        owners.append(owner_dsc(cu, P, g) if layout == 0 else owner_packed(T, P, g))
    out = []
    for r in range(P):
        out.extend(g for g in range(T) if owners[g] == r)
    return out


def metadata_by_runs(layout, cu, P, T):
    """(num_segs, seg_doc_first, cu_local rows, seg_offsets) by token walk.

    DSC: a rank's segment for document i is the run of its local tokens that
    come from document i; documents it holds no tokens of (length 0) still
    count as empty segments, one per document, as the per-document layout
    keeps every document on every rank. Packed: runs of equal document id
    inside the rank's contiguous chunk; only non-empty runs exist.
    """
    n = len(cu) - 1
    Tp = T // P
    l2g = l2g_by_ownership(layout, cu, P, T)
    num_segs, first, rows = [], [], []
    for r in range(P):
        local_docs = [doc_of_token(cu, l2g[r * Tp + j]) for j in range(Tp)]
        if layout == 0:
            counts = [0] * n
            for d in local_docs:
                counts[d] += 1
            row = [0]
            for c in counts:
                row.append(row[-1] + c)
            num_segs.append(n)
            first.append(0 if n > 0 else -1)
            rows.append(row)
        else:
            starts, docs = [], []
            for j, d in enumerate(local_docs):
                if j == 0 or d != local_docs[j - 1]:
                    starts.append(j)
                    docs.append(d)
            row = starts + [Tp] * (n + 1 - len(starts))
            num_segs.append(len(starts))
            first.append(docs[0] if docs else -1)
            rows.append(row)
    offs = [0]
    for s in num_segs:
        offs.append(offs[-1] + s)
    return num_segs, first, rows, offs


def compositions(T, unit, max_docs=None):
    """All tuples of lengths (multiples of unit, >= 0) summing to T.

    Zero-length documents are allowed but not two in a row, and at most
    ``max_docs`` documents, to keep the set finite.
    """
    out = []

    def rec(rem, acc):
        if rem == 0 and acc:
            out.append(tuple(acc))
        if max_docs is not None and len(acc) >= max_docs:
            return
        for L in range(0, rem + 1, unit):
            if L == 0 and acc and acc[-1] == 0:
                continue
            rec(rem - L, acc + [L])

    rec(T, [])
    return out
