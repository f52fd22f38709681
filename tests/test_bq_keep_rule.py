"""CPU pin of the rule by which the fused kNN + Ball Query pass keeps a
query's Ball Query hits (``bq_keep`` in ``csrc/pc_knn.cu``) while it visits
the references in its own order (the seed tile outwards from the query's
place, then tiles outwards from the block's home tile).

The operator (mps-pointops project page, "Ball Query: first K within a
radius"; "Numerical contracts", "Selection and output"): the first K
references in input order with s32 < R2, i.e. the K smallest indices among
the hits, then (-1, 0) padding.  The pass keeps K slots in no order: while
fewer than K are full a hit takes the next slot; afterwards a hit with a
smaller index than the largest kept one replaces it and the slots are
scanned for the new largest.  A finish step sorts each row by index.

The restatement below follows those steps on random hit sequences in random
visiting orders and checks the sorted row against the K smallest indices;
the planted-mistake tests drop one step and show that it is caught.
"""
import numpy as np
import pytest


def keep_row(hits, K, mutant=None):
    """hits: (j, s) in visiting order.  Returns the K slots after the pass."""
    row = []
    maxj, maxpos, n = -1, 0, 0
    for j, s in hits:
        if n < K:
            row.append((j, s))
            if j > maxj and mutant != "no_fill_max":
                maxj, maxpos = j, n
        elif j < maxj:
            row[maxpos] = (j, s)
            if mutant == "no_rescan":
                maxj = j
            else:
                maxj = -1
                for e, (je, _) in enumerate(row):
                    if je > maxj:
                        maxj, maxpos = je, e
        n += 1
    return row, n


def finish(row, n, K):
    """Sort by index and pad with (-1, 0)."""
    out = sorted(row)[:K]
    return out + [(-1, 0.0)] * (K - len(out)), n


def cases():
    rng = np.random.default_rng(20262)
    out = []
    for trial in range(400):
        K = int(rng.choice([1, 2, 3, 8, 32, 64]))
        nh = int(rng.choice([0, 1, K - 1, K, K + 1, 2 * K, 5 * K, 300]))
        nh = max(nh, 0)
        js = rng.choice(100000, size=nh, replace=False)
        s = rng.random(nh).astype(np.float32)
        kind = trial % 4
        if kind == 1:    # descending indices: every later hit replaces
            order = np.argsort(-js)
        elif kind == 2:  # ascending: nothing is replaced
            order = np.argsort(js)
        else:            # random visiting order
            order = rng.permutation(nh)
        out.append((K, [(int(js[i]), float(s[i])) for i in order]))
    return out


def expected(hits, K):
    kept = sorted(hits)[:K]
    return kept + [(-1, 0.0)] * (K - len(kept))


def test_keeps_the_K_smallest_indices_in_any_order():
    for K, hits in cases():
        row, n = keep_row(hits, K)
        got, n = finish(row, n, K)
        assert got == expected(hits, K), (K, len(hits))
        assert n == len(hits)


@pytest.mark.parametrize("mutant", ["no_rescan", "no_fill_max"])
def test_planted_mistakes_are_caught(mutant):
    """Without the rescan the new largest is not found; without tracking the
    largest while the slots fill, the first K hits in visiting order stay."""
    bad = 0
    for K, hits in cases():
        row, n = keep_row(hits, K, mutant)
        got, _ = finish(row, n, K)
        bad += int(got != expected(hits, K))
    assert bad > 0
