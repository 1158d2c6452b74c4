"""The grouped decode kernel's work split, recomputed on the host: no CTA's
share of the weighted split meets more sequences than its shared-memory window
holds (640), whatever the length mix, once the start weight per sequence follows
the kernel's rule

    sw = max(least, ceil((T + grid - 638 grid) / (638 grid - NE)))

(T tiles of the batch, NE non-empty sequences; least = 1 for head groups whose
Q and P' are double-buffered, 3 for those with one buffer), for batches of up to
638 grid / 2 sequences (the host's admission bound).  CPU only: the arithmetic of
the split, checked by brute force over random and adversarial batches; the GPU
test with 700 one-token sequences beside a 3.2M-token one runs the kernel on
such a batch."""
import math

import numpy as np
import pytest

KWIN = 640


LEAST = (1, 3)


def start_weight(T: int, NE: int, grid: int, least: int = 1) -> int:
    num = T + grid - (KWIN - 2) * grid
    den = (KWIN - 2) * grid - NE
    assert den > 0
    return max(least, -(-num // den)) if num > 0 else least


def max_sequences_per_share(tiles, grid: int, sw: int) -> int:
    """Largest number of sequences with at least one tile in one CTA's share."""
    tiles = [t for t in tiles if t > 0]
    W = sum(tiles) + sw * len(tiles)
    starts = [c * W // grid for c in range(grid + 1)]
    # tile units of each sequence: [pos + sw, pos + sw + nt)
    spans, pos = [], 0
    for nt in tiles:
        spans.append((pos + sw, pos + sw + nt))
        pos += sw + nt
    best = 0
    j = 0
    for c in range(grid):
        x0, x1 = starts[c], starts[c + 1]
        if x0 == x1:
            continue
        while j < len(spans) and spans[j][1] <= x0:
            j += 1
        k, n = j, 0
        while k < len(spans) and spans[k][0] < x1:
            if spans[k][1] > x0:
                n += 1
            k += 1
        best = max(best, n)
    return best


def check(tiles, grid, least=1):
    T = int(sum(tiles))
    NE = int(sum(1 for t in tiles if t > 0))
    assert 2 * len(tiles) <= (KWIN - 2) * grid
    sw = start_weight(T, NE, grid, least)
    assert sw >= least
    # the rule's own inequality, then the window by brute force
    W = T + sw * NE
    assert math.ceil(W / grid) <= (KWIN - 2) * (sw + 1)
    assert max_sequences_per_share(tiles, grid, sw) <= KWIN
    # the host's admission bound keeps the batch's weight an int
    tmax = max(tiles) if tiles else 0
    assert W <= 2 * len(tiles) * (tmax + 1)
    return sw


@pytest.mark.parametrize("least", LEAST)
@pytest.mark.parametrize("grid", [148, 152, 160])
def test_short_sequences_beside_very_long_ones(grid, least):
    """The batch that overflows the window with the least start weight: with the
    rule the start weight rises and every share fits."""
    tiles = [1] * 700 + [240_000] if least == 1 else [1] * 700 + [1_500_000]
    assert max_sequences_per_share(tiles, grid, least) > KWIN    # the hazard is real
    assert check(tiles, grid, least) > least
    # the long sequences first, the short ones last, and interleaved
    check([tiles[-1]] + [1] * 700, grid, least)
    check([1] * 350 + [tiles[-1]] + [1] * 350, grid, least)


@pytest.mark.parametrize("least", LEAST)
def test_the_rule_keeps_the_least_weight_below_its_threshold(least):
    """Batches of fewer than ~194K tiles plus sequences (about 6 GB of K/V) keep
    the least start weight."""
    g = np.random.default_rng(7)
    for B, hi in ((64, 300), (256, 600), (2048, 90), (16_384, 10)):
        tiles = [int(x) for x in g.integers(1, hi, size=B)]
        assert sum(tiles) + B < 194_000
        assert check(tiles, 152, least) == least


@pytest.mark.parametrize("least", LEAST)
def test_a_raised_start_weight_costs_little_balance_on_long_batches(least):
    """The rule assumes the shortest sequences, so a very long batch of medium
    sequences also gets a start weight above the least; the extra start weight
    is then a small share of each CTA's units (the split's balance moves by
    about that)."""
    g = np.random.default_rng(9)
    tiles = [int(x) for x in g.integers(100, 300, size=2048)]
    T, NE = sum(tiles), len(tiles)
    sw = check(tiles, 152, least)
    assert sw > least
    assert (sw - least) * NE / (T + sw * NE) < 0.02


@pytest.mark.parametrize("least", LEAST)
def test_random_skewed_batches(least):
    g = np.random.default_rng(11)
    for trial in range(300):
        n_short = int(g.integers(1, 20_000))
        n_long = int(g.integers(0, 4))
        tiles = [int(x) for x in g.integers(0, 3, size=n_short)]       # empty and 1-2 tiles
        for _ in range(n_long):
            pos = int(g.integers(0, len(tiles) + 1))
            tiles.insert(pos, int(g.integers(10_000, 2_000_000)))
        if 2 * len(tiles) > (KWIN - 2) * 152:
            continue
        check(tiles, 152, least)


def test_largest_admitted_batch_of_single_tiles():
    """32,768 sequences of one tile each (the kernel's batch cap) beside the
    longest sequences the weight's int range allows."""
    tiles = [1] * 32_768 + [30_000_000]
    check(tiles, 152)
    check(tiles, 152, 3)
