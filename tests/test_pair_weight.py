"""Host model of the tile pair's slab stream (no kernels run).

The attention kernel runs the block-sparse attention of a pair of 128-row
query tiles over the slabs (64 key rows of one frame) that either tile
selected (Hybrid Forcing, English technical summary, section 2.A.2), in an
order that keeps both tiles busy: slabs both tiles need two per round, then
rounds of two slabs of tile A alone alternating with rounds of two of tile B
alone, then the rest of the longer side, then the odd shared slab.  The
prologue writes each pair's weight for the kernel's work division in closed
form from the three counts (both / A only / B only); the kernel checks it
against the weight of the list it builds.  These tests restate the kernel's
placement formulas and the prologue's closed form and check that the
placement is a permutation and that both weights agree for every count up to
40 of each kind."""

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "hybrid_sparse_linear_scores_b300", "csrc")


def test_round_weight_definition_is_the_restated_one():
    src = open(os.path.join(CSRC, "hf_internal.h")).read()
    assert "return 15u + (sa ? 2u * (uint32_t)sa + 4u : 0u) + (sb ? 2u * (uint32_t)sb + 4u : 0u);" in src


def round_weight(sa, sb):
    return 15 + (2 * sa + 4 if sa else 0) + (2 * sb + 4 if sb else 0)


def placement(nI, nA, nB):
    """List position of the q-th slab of each category (1: both tiles, 2:
    tile A only, 3: tile B only), as the attention kernel's list build places
    it; returns the list of categories by position."""
    n = nI + nA + nB
    nI2 = nI & ~1
    mp = 2 * min(nA >> 1, nB >> 1)
    out = [None] * n
    for cat, count in ((1, nI), (2, nA), (3, nB)):
        for q in range(count):
            if cat == 1:
                pos = q if q < nI2 else n - 1
            elif cat == 2:
                pos = nI2 + 2 * (q & ~1) + (q & 1) if q < mp else nI2 + mp + q
            else:
                pos = nI2 + 2 * (q & ~1) + 2 + (q & 1) if q < mp else nI2 + nA + q
            assert out[pos] is None, f"position {pos} placed twice ({nI}, {nA}, {nB})"
            out[pos] = cat
    assert None not in out, f"hole in the list ({nI}, {nA}, {nB})"
    return out


def list_weight(cats):
    w = 0
    for r in range(0, len(cats), 2):
        rnd = cats[r:r + 2]
        sa = sum(c in (1, 2) for c in rnd)
        sb = sum(c in (1, 3) for c in rnd)
        w += round_weight(sa, sb)
    return w


def pair_weight(nI, nA, nB):
    """The prologue's closed form (restated)."""
    nI2, mp = nI & ~1, 2 * min(nA >> 1, nB >> 1)
    w = (nI2 // 2) * round_weight(2, 2) + (mp // 2) * (round_weight(2, 0) + round_weight(0, 2))
    a, c, b = nA - mp, nI & 1, nB - mp
    w += (a // 2) * round_weight(2, 0)
    if a & 1:
        if b > 0:
            w += round_weight(1, 1)
            b -= 1
        else:
            return w + (round_weight(2, 1) if c else round_weight(1, 0))
    w += (b // 2) * round_weight(0, 2)
    if b & 1:
        return w + (round_weight(1, 2) if c else round_weight(0, 1))
    return w + (round_weight(1, 1) if c else 0)


def test_closed_form_is_the_prologues():
    """The restated closed form follows the prologue's source line by line
    (the same round_weight terms in the same branches)."""
    src = open(os.path.join(CSRC, "hf_select.cu")).read()
    body = src[src.index("__device__ uint32_t pair_weight(int nI, int nA, int nB)"):]
    body = body[:body.index("\n}\n")]
    terms = re.findall(r"round_weight\((\d), (\d)\)", body)
    assert terms == [("2", "2"), ("2", "0"), ("0", "2"), ("2", "0"), ("1", "1"), ("2", "1"), ("1", "0"),
                     ("0", "2"), ("1", "2"), ("0", "1"), ("1", "1")]


@pytest.mark.parametrize("nI", range(0, 41))
def test_prologue_weight_is_the_lists_weight(nI):
    for nA in range(0, 41):
        for nB in range(0, 41):
            cats = placement(nI, nA, nB)
            assert list_weight(cats) == pair_weight(nI, nA, nB), (nI, nA, nB)


def test_alternating_rounds_keep_one_tile_per_round():
    """In the alternating part every round is two slabs of one tile, A and B
    in turn; the shared slabs come first, two per round."""
    cats = placement(6, 5, 8)
    rounds = [tuple(cats[r:r + 2]) for r in range(0, len(cats), 2)]
    assert rounds[:3] == [(1, 1)] * 3
    assert rounds[3:7] == [(2, 2), (3, 3), (2, 2), (3, 3)]
    assert cats[-1] in (1, 2, 3)
