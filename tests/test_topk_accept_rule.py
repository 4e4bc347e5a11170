"""The acceptance rule of the seeded top-k (dsa_decode_step_hist), on the CPU.

The seeded top-k starts its radix digits from a first-digit histogram counted by the
indexer. Whatever that histogram held, the digits end in some prefix, mask and count
`rem` still to take from the entries equal to the prefix under the mask; the kernel
keeps the selection only if the exact totals of its placement scan (tg entries above
the prefix, te equal to it) satisfy

    rem >= 0  and  tg + min(rem, te) == k  and  (rem >= te  or  the mask covers all 32 bits)

and otherwise selects the segment again without the histogram. These tests check that
rule as stated, independently of the CUDA code: over any (prefix, mask, rem) the digits
might leave, an accepted selection is the oracle's top-k (ties to the lower position);
the digits of the true histogram are always accepted; and a weakened rule without the
mask clause accepts a wrong selection, so the property test can tell the difference.
"""
import numpy as np
import pytest

import oracle

FULL = 0xFFFFFFFF


def _orderable(x32: np.ndarray) -> np.ndarray:
    """32-bit keys whose unsigned order is the float order, -0 folded onto +0."""
    u = x32.astype(np.float32).view(np.uint32).astype(np.uint64)
    u[u == 0x80000000] = 0
    return np.where(u & 0x80000000, (~u) & FULL, u | 0x80000000).astype(np.uint64)


def _select(keys, prefix, pmask, rem):
    """Every entry above the prefix under the mask, then the first `rem` equal ones by
    position; the totals tg and te."""
    m = keys & pmask
    gt = np.flatnonzero(m > prefix)
    eq = np.flatnonzero(m == prefix)
    sel = np.sort(np.concatenate([gt, eq[: max(rem, 0)]]))
    return sel, gt.size, eq.size


def _accept(tg, te, rem, k, pmask, weak=False):
    if rem < 0 or tg + min(rem, te) != k:
        return False
    return weak or rem >= te or pmask == FULL


def _true_digits(keys, k):
    """Digits of 11, 11 and 10 bits from the top bit over exact histograms, stopping as
    soon as the threshold bin holds exactly the count still to take."""
    rem, prefix, pmask, consumed = k, 0, 0, 0
    while consumed < 32:
        w = min(11, 32 - consumed)
        sh = 32 - consumed - w
        sub = keys[(keys & pmask) == prefix]
        h = np.bincount(((sub >> sh) & ((1 << w) - 1)).astype(np.int64), minlength=1 << w)
        above = 0
        for b in range((1 << w) - 1, -1, -1):
            if above + h[b] >= rem:
                break
            above += h[b]
        rem -= above
        prefix |= b << sh
        pmask |= ((1 << w) - 1) << sh
        consumed += w
        if h[b] == rem:
            break
    return prefix, pmask, rem


def _rows(rng):
    """Score rows of the kinds the selection meets: both signs, one sign in a narrow
    range (long shared key prefixes), many exact ties, zeros of both signs."""
    n = int(rng.integers(300, 3000))
    yield rng.normal(0, 50, n).astype(np.float32)
    yield (1.0 + rng.random(n) * 1e-3).astype(np.float32)
    yield rng.integers(-4, 5, n).astype(np.float32)
    z = rng.normal(0, 1, n).astype(np.float32)
    z[rng.random(n) < 0.3] = 0.0
    z[rng.random(n) < 0.3] = -0.0
    yield z


def _truth(x, k):
    t = oracle.topk_row(x.astype(np.float64), k)
    return t[t >= 0]


@pytest.mark.parametrize("seed", range(6))
def test_true_digits_are_accepted(seed):
    rng = np.random.default_rng(seed)
    for x in _rows(rng):
        for k in (1, 7, len(x) // 3, len(x) - 1):
            keys = _orderable(x)
            prefix, pmask, rem = _true_digits(keys, k)
            sel, tg, te = _select(keys, prefix, pmask, rem)
            assert _accept(tg, te, rem, k, pmask)
            assert np.array_equal(sel, _truth(x, k))


@pytest.mark.parametrize("seed", range(6))
def test_any_accepted_selection_is_the_top_k(seed):
    """(prefix, mask, rem) drawn around the true ones and at random: whenever the rule
    accepts, the selection is the exact top-k."""
    rng = np.random.default_rng(100 + seed)
    accepted = 0
    for x in _rows(rng):
        n = len(x)
        keys = _orderable(x)
        for k in (1, 5, n // 2, n - 1):
            tp, tm, tr = _true_digits(keys, k)
            truth = _truth(x, k)
            for _ in range(60):
                bits = int(rng.choice([11, 22, 32]))
                pmask = (FULL << (32 - bits)) & FULL
                src = int(keys[rng.integers(n)]) if rng.random() < 0.7 else int(rng.integers(0, 1 << 32))
                prefix = src & pmask
                if rng.random() < 0.3:           # the true threshold, cut to this mask
                    prefix = tp & pmask
                rem = int(rng.integers(-2, n + 3))
                sel, tg, te = _select(keys, prefix, pmask, rem)
                if rng.random() < 0.5:           # the count the prefix implies
                    rem = k - tg
                    sel, tg, te = _select(keys, prefix, pmask, rem)
                if _accept(tg, te, rem, k, pmask):
                    accepted += 1
                    assert np.array_equal(sel, truth), (k, hex(prefix), bits, rem)
    assert accepted > 50   # the property was exercised, not vacuous


def test_mask_clause_is_needed():
    """Without `rem >= te or full mask`, a prefix that stops inside a bin holding both
    selected and unselected keys takes the lower positions instead of the larger keys."""
    # keys share their top 22 bits in pairs; the larger key of the pair sits later
    x = np.array([1.0, 1.0000001, 3.0, 3.0000002], dtype=np.float32)
    keys = _orderable(x)
    k = 3
    pmask = (FULL << 10) & FULL                  # top 22 bits: 1.0 and 1.0000001 share them
    prefix = int(keys[0]) & pmask
    assert (int(keys[1]) & pmask) == prefix
    sel, tg, te = _select(keys, prefix, pmask, k - 2)
    assert (tg, te) == (2, 2)
    assert _accept(tg, te, k - 2, k, pmask, weak=True)
    assert not np.array_equal(sel, _truth(x, k))
    assert not _accept(tg, te, k - 2, k, pmask)
