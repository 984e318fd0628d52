"""Pins for the load-balancing part of the oracle: the auxiliary-loss-free bias
update ("05 - Expert Parallelism (MoE)", "Load balancing" (b), and its exercise
with counts [100, 50, 200, 50]) and replicate-then-pack placement of redundant
experts ("Expert parallelism", "Load imbalance becomes idle time", with its
hand-checkable eight-expert case).  CPU only."""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import moe_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "eplb_example.json")) as fh:
        return json.load(fh)


# --------------------------------------------------------------------------
# Bias update
# --------------------------------------------------------------------------

def test_bias_update_page_exercise():
    """Counts [100, 50, 200, 50] after a step: the average load is 100, so the
    two under-loaded experts gain 50 lr, the over-loaded one loses 100 lr and
    the balanced one is unchanged."""
    lr = 1e-3
    new = oracle.bias_update(np.zeros(4), [100, 50, 200, 50], lr)
    assert np.allclose(new, [0.0, 50 * lr, -100 * lr, 50 * lr], rtol=0, atol=1e-15)


def test_bias_update_is_additive_and_zero_sum():
    rng = np.random.default_rng(0)
    c = rng.integers(0, 500, size=64)
    b0 = rng.normal(size=64)
    b1 = oracle.bias_update(b0, c, 0.01)
    assert abs((b1 - b0).sum()) < 1e-9                  # deviations from the mean sum to 0
    assert (np.sign(b1 - b0) == np.sign(c.mean() - c)).all()
    assert np.allclose(oracle.bias_update(b0, np.full(64, 7), 0.5), b0)   # balanced: no change


# --------------------------------------------------------------------------
# Replicate then pack
# --------------------------------------------------------------------------

def test_eplb_page_example():
    g = _golden()
    plan = oracle.eplb_plan(g["loads"], 4, 3)
    # all four spare slots go to expert 0: five copies of 18
    assert plan["copies"].tolist() == [5, 1, 1, 1, 1, 1, 1, 1]
    assert plan["rank_load"].tolist() == g["greedy_gpu_loads"]
    assert oracle.imbalance_eta(np.array([plan["rank_load"]])) == pytest.approx(g["greedy_eta"],
                                                                                abs=0.005)
    # greedy is a heuristic: the page's better plan beats it
    assert g["better_eta"] > oracle.imbalance_eta(np.array([plan["rank_load"]]))
    # the plain layout (experts 2g, 2g+1 on rank g)
    plain = np.add.reduceat(np.array(g["loads"]), [0, 2, 4, 6])
    assert plain.tolist() == g["plain_gpu_loads"]


def test_eplb_replicate_trace():
    """Expert 0's load per copy goes 90 -> 45 -> 30 -> 22.5 -> 18 as the spare
    slots arrive one by one, always above the cold experts' 10."""
    loads = [90, 10, 10, 10, 10, 10, 10, 10]
    per = []
    for spare in range(5):
        q = oracle.eplb_replicate(loads, 8 + spare)
        assert q[1:].tolist() == [1] * 7
        per.append(Fraction(90, int(q[0])))
    assert per == [90, 45, 30, Fraction(45, 2), 18]


def _makespan_opt(weights, n):
    best = None
    for assign in itertools.product(range(n), repeat=len(weights)):
        m = max(sum(w for w, a in zip(weights, assign) if a == r) for r in range(n))
        best = m if best is None or m < best else best
    return best


@pytest.mark.parametrize("seed", range(12))
def test_eplb_pack_within_graham_bound(seed):
    """Without a slot limit, longest-processing-time-first finishes within 4/3
    of the best makespan (Graham 1969); brute force gives the best."""
    rng = np.random.default_rng(seed)
    E = int(rng.integers(2, 7))
    n = int(rng.integers(2, 4))
    loads = rng.integers(1, 60, size=E)
    q = np.ones(E, np.int64)
    _, _, rank_load = oracle.eplb_pack(loads, q, n, E)
    opt = _makespan_opt([float(v) for v in loads], n)
    assert rank_load.max() <= (4 / 3 - 1 / (3 * n)) * opt + 1e-9


@pytest.mark.parametrize("seed", range(6))
def test_eplb_plan_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    E, n = 32, 8
    slots = E // n + int(rng.integers(0, 3))
    loads = rng.integers(0, 400, size=E)
    loads[rng.integers(0, E)] += 2000                  # one hot expert
    plan = oracle.eplb_plan(loads, n, slots)
    q = plan["copies"]
    assert q.sum() == n * slots and (q >= 1).all()
    if n * slots > E:                                  # spare slots: the hot expert got them
        assert q[loads.argmax()] == q.max() > 1
    se = plan["slot_expert"]
    assert ((se >= 0).sum(axis=1) <= slots).all()
    assert np.bincount(se[se >= 0], minlength=E).tolist() == q.tolist()
    assert plan["rank_load"].sum() == pytest.approx(loads.sum())
    # every copy's rank is consistent with the slot table
    for e in range(E):
        for j in range(q[e]):
            r = plan["copy_rank"][plan["copy_offset"][e] + j]
            assert e in se[r].tolist()


def test_eplb_dispatch_without_copies_is_the_plain_layout():
    """One copy per expert, on rank floor(e*n/E): the dispatch count matrix is
    the expert-parallel layout's (computed independently by ep_layout)."""
    rng = np.random.default_rng(5)
    T, E, k, n = 64, 16, 3, 4
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    p = oracle.permute(idx, E)
    lay = oracle.ep_layout(idx, p["inv"], E, n, T)
    plan = {"copies": np.ones(E, np.int64), "copy_offset": np.arange(E),
            "copy_rank": np.arange(E) * n // E}
    dest, C = oracle.eplb_dispatch(idx, p["inv"], p["offsets"], p["counts"], plan, n, T)
    assert np.array_equal(C, lay["C"])
    assert (dest == (idx.reshape(-1) * n // E)).all()


def test_eplb_dispatch_splits_each_expert_evenly():
    rng = np.random.default_rng(6)
    T, E, k, n = 128, 8, 2, 4
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    p = oracle.permute(idx, E)
    plan = oracle.eplb_plan(p["counts"], n, 3)
    dest, C = oracle.eplb_dispatch(idx, p["inv"], p["offsets"], p["counts"], plan, n, T)
    assert C.sum() == T * k
    flat = idx.reshape(-1)
    for e in range(E):
        qe = plan["copies"][e]
        got = np.zeros(n, np.int64)
        np.add.at(got, dest[flat == e], 1)
        sizes = [((j + 1) * p["counts"][e]) // qe - (j * p["counts"][e]) // qe for j in range(qe)]
        assert max(sizes) - min(sizes) <= 1
        want = np.zeros(n, np.int64)
        for j in range(qe):
            want[plan["copy_rank"][plan["copy_offset"][e] + j]] += sizes[j]
        assert got.tolist() == want.tolist()
    # realised rank loads track the plan (each copy within one row of c/q)
    assert np.abs(C.sum(axis=0) - plan["rank_load"]).max() <= 3


def test_planted_replicate_by_total_load_is_caught(monkeypatch):
    """A replicate step that ranks experts by total load instead of load per
    copy keeps giving copies to expert 0 regardless: the trace pin still holds,
    but with a second hot expert the page's rule must share the spares."""
    loads = [60, 50, 10, 10]
    q = oracle.eplb_replicate(loads, 6)
    assert q.tolist() == [2, 2, 1, 1]           # 60 -> 30 < 50, so expert 1 gets the 2nd

    def by_total(loads, n_slots):
        q = np.ones(len(loads), np.int64)
        for _ in range(n_slots - len(loads)):
            q[int(np.argmax(loads))] += 1
        return q
    monkeypatch.setattr(oracle, "eplb_replicate", by_total)
    assert oracle.eplb_replicate(loads, 6).tolist() != [2, 2, 1, 1]


def test_planted_pack_smallest_first_is_caught():
    """Packing in increasing load order (the reverse of the page's rule) misses
    the hand example's (46, 38, 38, 38)."""
    g = _golden()
    q = oracle.eplb_replicate(g["loads"], 12)
    loads = list(g["loads"])
    # a mutant: sort ascending by passing negated loads for the ordering only
    order_loads = [-v for v in loads]
    copy_rank, _, _ = oracle.eplb_pack(order_loads, q, 4, 3)
    rank_load = np.zeros(4)
    off = np.concatenate([[0], np.cumsum(q)])[:-1]
    for e in range(8):
        for j in range(q[e]):
            rank_load[copy_rank[off[e] + j]] += loads[e] / q[e]
    assert rank_load.tolist() != g["greedy_gpu_loads"]
