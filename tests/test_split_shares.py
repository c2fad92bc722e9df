"""Host model of the attention kernel's split mode (no kernels run).

In split mode the attention kernel gives every CTA an equal share of the
weighted units of all tile pairs' slab streams: pair i counts kPartWeight
units ahead of its rounds, then the weights of its rounds; CTA c takes units
[c T / G, (c + 1) T / G).  A CTA takes a part of every pair whose rounds
start in its share; a pair cut between CTAs leaves a partial result per part
in a per-CTA slot, and the part that arrives last merges the parts of the
CTAs it enumerates from the owners of the pair's first and last round units.
These tests restate that arithmetic (share starts, round owners, the part
loop's conditions, the rounds a part takes, the partial-result slots) and
check the invariants the merge relies on, for random pair and round weights:
every round of every pair is taken by exactly one CTA, the CTAs that take a
part of a pair are exactly those the merge enumerates, and no CTA uses one
partial-result slot for two cut pairs.  (Work division for the block-sparse
attention of Hybrid Forcing, English technical summary, section 2.A.2.)"""

import os
import random
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _part_weight() -> int:
    src = open(os.path.join(ROOT, "hybrid_sparse_linear_scores_b300", "csrc", "hf_internal.h")).read()
    return int(re.search(r"constexpr uint32_t kPartWeight = (\d+);", src).group(1))


KPW = _part_weight()


def share_start(c, T, G):
    return c * T // G


def round_owner(x, T, G):
    return ((x + 1) * G - 1) // T


def share_nonempty(c, T, G):
    return share_start(c, T, G) < share_start(c + 1, T, G)


def simulate(round_weights, G):
    """Per CTA, the parts it runs as the kernel's part loop finds them:
    [(pair, [rounds taken])]."""
    R = [sum(w) for w in round_weights]
    NP = len(R)
    T = sum(r + KPW for r in R)
    starts, P = [], 0
    for r in R:
        starts.append(P)
        P += r + KPW
    parts = {}
    for c in range(G):
        s_c, e_c = share_start(c, T, G), share_start(c + 1, T, G)
        # the first pair: the one whose units contain s_c
        pair = next((i for i in range(NP) if starts[i] <= s_c < starts[i] + R[i] + KPW), NP)
        P = starts[pair] if pair < NP else 0
        mine = []
        while pair < NP and P + KPW < e_c and s_c < e_c:
            Pr = P + KPW
            lo, hi = max(s_c, Pr) - Pr, min(e_c, Pr + R[pair]) - Pr
            taken, st = [], 0
            for r, w in enumerate(round_weights[pair]):
                if lo <= st < hi:
                    taken.append(r)
                st += w
            mine.append((pair, taken))
            P += R[pair] + KPW
            pair += 1
        parts[c] = mine
    return parts, R, starts, T


def _random_case(rng, n_pairs, small):
    rw = []
    for _ in range(n_pairs):
        n_rounds = rng.randint(1, 3) if small else rng.randint(10, 70)
        # weights of rounds with 1 or 2 slabs of one or both tiles (15 + 2s + 4 per tile)
        rw.append([rng.choice([21, 23, 27, 29, 31, 25]) for _ in range(n_rounds)])
    return rw


CASES = [(1, 148, False), (2, 148, False), (7, 148, False), (228, 148, False), (456, 148, False),
         (760, 148, False), (3, 148, True), (40, 148, True), (5, 4, False), (33, 16, True)]


@pytest.mark.parametrize("n_pairs,G,small", CASES)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_every_round_has_one_owner(n_pairs, G, small, seed):
    rw = _random_case(random.Random(1000 * seed + n_pairs), n_pairs, small)
    parts, R, starts, T = simulate(rw, G)
    owners = {}
    for c, mine in parts.items():
        for pair, taken in mine:
            for r in taken:
                assert (pair, r) not in owners, f"round {r} of pair {pair} taken twice"
                owners[(pair, r)] = c
    for i, w in enumerate(rw):
        for r in range(len(w)):
            assert (i, r) in owners, f"round {r} of pair {i} taken by no CTA"
    # and each CTA's rounds are one contiguous run of the global order
    order = [(i, r) for i, w in enumerate(rw) for r in range(len(w))]
    for c in range(G):
        got = [k for k in order if owners[k] == c]
        if got:
            a, b = order.index(got[0]), order.index(got[-1])
            assert b - a + 1 == len(got)


@pytest.mark.parametrize("n_pairs,G,small", CASES)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merge_enumerates_exactly_the_parts(n_pairs, G, small, seed):
    """The merge counts the CTAs c0..c1 with a non-empty share, c0 and c1 the
    owners of the pair's first and last round units; those are exactly the
    CTAs whose part loop runs a part of the pair (a part may take no round
    when its share holds no round start: it then leaves an empty result)."""
    rw = _random_case(random.Random(7 + 1000 * seed + n_pairs), n_pairs, small)
    parts, R, starts, T = simulate(rw, G)
    runners = {i: [] for i in range(n_pairs)}
    for c, mine in parts.items():
        for pair, _ in mine:
            runners[pair].append(c)
    for i in range(n_pairs):
        Pr = starts[i] + KPW
        c0, c1 = round_owner(Pr, T, G), round_owner(Pr + R[i] - 1, T, G)
        expect = [c for c in range(c0, c1 + 1) if share_nonempty(c, T, G)]
        assert runners[i] == expect, (i, runners[i], expect)
        assert c0 in runners[i] and c1 in runners[i]


@pytest.mark.parametrize("n_pairs,G,small", CASES)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_partial_slots_do_not_collide(n_pairs, G, small, seed):
    """CTA c writes a cut pair's partial result to slot 1 when it is the
    owner of the pair's round 0 but its share starts before the pair, else to
    slot 0: no CTA uses one slot for two cut pairs."""
    rw = _random_case(random.Random(13 + 1000 * seed + n_pairs), n_pairs, small)
    parts, R, starts, T = simulate(rw, G)
    for c, mine in parts.items():
        used = {}
        for pair, _ in mine:
            Pr = starts[pair] + KPW
            c0, c1 = round_owner(Pr, T, G), round_owner(Pr + R[pair] - 1, T, G)
            nparts = sum(share_nonempty(k, T, G) for k in range(c0, c1 + 1))
            if nparts < 2:
                continue
            slot = 1 if (c == c0 and share_start(c0, T, G) != Pr) else 0
            assert slot not in used, f"CTA {c}: slot {slot} for pairs {used[slot]} and {pair}"
            used[slot] = pair


def test_head_part_ends_its_share():
    """The part holding a cut pair's round 0 is the last part of its CTA (its
    share ends inside the pair), while the other parts start the following
    shares: the head part is the one that usually arrives last."""
    rw = _random_case(random.Random(5), 228, False)
    parts, R, starts, T = simulate(rw, 148)
    for c, mine in parts.items():
        for k, (pair, taken) in enumerate(mine):
            Pr = starts[pair] + KPW
            c0, c1 = round_owner(Pr, T, 148), round_owner(Pr + R[pair] - 1, T, 148)
            if c0 != c1 and c == c0:
                assert k == len(mine) - 1
            if c0 != c1 and c != c0:
                assert k == 0
