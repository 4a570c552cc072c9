"""moe_tier_plan, the ranking behind the expert tiers (experts beyond HBM), on
a machine without a GPU: checked against a brute-force restatement of its
rule on random and hand-made cases.

Rule: experts that have a host copy, or already hold a slot, are ranked by
heat (descending), then resident before not resident, then id (ascending);
the first n_slots are kept; kept residents stay in their slot and the others
take the free slots in ascending order."""
import numpy as np
import pytest

from quantized_expert_ffn_score_gb300 import moe


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_expert_ffn_score_gb300 import build
    build.build()


def brute(heat, has, cur, n_slots):
    E = len(heat)
    cand = [e for e in range(E) if has[e] or 0 <= cur[e] < n_slots]
    cand.sort(key=lambda e: (-float(heat[e]), 0 if cur[e] >= 0 else 1, e))
    kept = cand[:n_slots]
    new = np.full(E, -1, dtype=np.int32)
    used = set()
    for e in kept:
        if 0 <= cur[e] < n_slots:
            new[e] = cur[e]
            used.add(int(cur[e]))
    free = [s for s in range(n_slots) if s not in used]
    moves = 0
    for e in kept:
        if new[e] < 0:
            new[e] = free.pop(0)
            moves += 1
    return new, moves


def test_hottest_fill_empty_slots_in_heat_order():
    heat = np.array([1, 9, 3, 7, 5], dtype=np.float32)
    new, n = moe.tier_plan(heat, np.ones(5), np.full(5, -1), 3)
    assert n == 3 and list(new) == [-1, 0, -1, 1, 2]


def test_ties_prefer_residents_then_lower_ids():
    heat = np.array([2, 2, 2, 2], dtype=np.float32)
    cur = np.array([-1, -1, -1, 0])
    new, n = moe.tier_plan(heat, np.ones(4), cur, 2)
    assert list(new) == [1, -1, -1, 0] and n == 1  # expert 3 keeps slot 0; expert 0 takes slot 1


def test_expert_without_host_copy_stays_only_if_resident():
    heat = np.array([10, 9, 1], dtype=np.float32)
    has = np.array([0, 1, 1])
    new, _ = moe.tier_plan(heat, has, np.full(3, -1), 2)
    assert list(new) == [-1, 0, 1]  # expert 0 is hottest but has nothing to load from
    new, n = moe.tier_plan(heat, has, np.array([1, -1, -1]), 2)
    assert list(new) == [1, 0, -1] and n == 1


def test_no_slots_and_bad_arguments():
    new, n = moe.tier_plan(np.ones(4), np.ones(4), np.full(4, -1), 0)
    assert n == 0 and np.all(new == -1)
    with pytest.raises(moe.MoeError):
        moe.tier_plan(np.ones(4), np.ones(4), np.full(4, -1), -1)


@pytest.mark.parametrize("seed", range(40))
def test_random_cases_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 60))
    n_slots = int(rng.integers(0, E + 1))
    heat = rng.integers(0, 6, size=E).astype(np.float32)  # many ties
    has = (rng.random(E) < 0.8).astype(np.uint8)
    cur = np.full(E, -1, dtype=np.int32)
    occupied = rng.permutation(E)[:int(rng.integers(0, n_slots + 1))]
    slots = rng.permutation(n_slots)[:len(occupied)]
    for e, s in zip(occupied, slots):
        cur[e] = s
    new, n = moe.tier_plan(heat, has, cur, n_slots)
    want, wn = brute(heat, has, cur, n_slots)
    np.testing.assert_array_equal(new, want)
    assert n == wn
    # a valid residency: distinct slots in range, at most n_slots experts
    s = new[new >= 0]
    assert len(set(s.tolist())) == len(s) and np.all(s < n_slots) and len(s) <= n_slots
