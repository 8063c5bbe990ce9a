"""Pins for the oracle's hardware-aware prefix scheduler ("DSpark Speculative
Decoding Explained: Block Drafting and Confidence Checks", "Survival
probability" and "Picking the budget"; the DSpark post's "Hardware aware
prefix scheduler").

Each pin checks the oracle against something other than itself: the pages'
printed survivals, a brute force over every subset of slots (no ranking,
no prefix rule), the marginal rule that characterises the optimum of a
linear cost, and the special cases of flat and prohibitive costs."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dspark_survival.txt")


def golden():
    out = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, *vals = line.split()
        out[name] = [float(v) for v in vals]
    return out


def survivals(conf):
    return np.cumprod(np.clip(np.nan_to_num(conf, nan=0.0), 0.0, 1.0), axis=1)


def theta_of(conf, cost, n_keep):
    """tokens per ms of a kept set given as per-request prefix lengths"""
    s = survivals(conf)
    R = conf.shape[0]
    tokens = R + sum(s[r, :n_keep[r]].sum() for r in range(R))
    return tokens / cost[int(np.sum(n_keep))], tokens


@pytest.mark.parametrize("name", ["chances_0.9_0.8", "prefix_example"])
def test_printed_survivals(name):
    surv = golden()[name]
    # chances that give the printed survivals (each the ratio of consecutive ones)
    chances = [surv[0]] + [surv[k] / surv[k - 1] for k in range(1, len(surv))]
    conf = np.array([chances])
    L = len(surv)
    flat = np.ones(L + 1)  # a flat cost keeps every guess
    n_keep, n, theta, tokens, st = oracle.schedule_prefix(conf, flat)
    assert st == 0 and n == L and list(n_keep) == [L]
    assert tokens == pytest.approx(1 + sum(surv), abs=1e-12)
    # the survival of each position alone: keep exactly k guesses with a cost
    # that makes only n = k affordable
    for k in range(1, L + 1):
        cost = np.full(L + 1, 1e30)
        cost[k] = 1.0
        _, n, _, tokens, _ = oracle.schedule_prefix(conf, cost)
        assert n == k
        assert tokens - 1 - sum(surv[:k - 1]) == pytest.approx(surv[k - 1], abs=1e-12)


def cost_tables(rng, R, N):
    n = np.arange(N + 1, dtype=np.float64)
    tables = {
        "toy": 25.0 + 0.1 * (R + n),  # the page's toy: 25 ms plus 0.1 ms per token checked
        "flat": np.full(N + 1, 3.0),
        "steep": 1.0 + 2.0 * n,
        "convex": 5.0 + 0.05 * n + 0.04 * n ** 2,
        "steps": 10.0 + 4.0 * (n // 3),
        "random": rng.uniform(0.5, 2.0, size=N + 1),
        "holes": np.where(rng.random(N + 1) < 0.3, -1.0, rng.uniform(1.0, 3.0, size=N + 1)),
    }
    return tables


@pytest.mark.parametrize("seed", range(12))
def test_matches_brute_force_over_all_subsets(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 5))
    L = int(rng.integers(1, max(2, 12 // R) + 1))
    L = min(L, 20 // R)
    conf = rng.uniform(0.0, 1.0, size=(R, L))
    if seed % 3 == 0:
        conf[rng.random((R, L)) < 0.2] = 1.0  # survivals that stay level
    for name, cost in cost_tables(rng, R, R * L).items():
        n_keep, n, theta, tokens, st = oracle.schedule_prefix(conf, cost)
        best = oracle.schedule_bruteforce(conf, cost)
        assert theta == pytest.approx(best, rel=1e-12, abs=1e-15), name
        assert n == int(n_keep.sum()) and (n_keep >= 0).all() and (n_keep <= L).all()
        if n > 0 or cost[0] > 0:
            t2, tok2 = theta_of(conf, cost, n_keep)
            assert t2 == pytest.approx(theta, rel=1e-12), name
            assert tok2 == pytest.approx(tokens, rel=1e-12), name


@pytest.mark.parametrize("seed", range(6))
def test_linear_cost_marginal_rule(seed):
    """For cost a + b n the optimum keeps adding the next-best slot while its
    survival exceeds b times the current tokens per ms (the ratio rises
    exactly then), and stops at the first slot that does not."""
    rng = np.random.default_rng(100 + seed)
    R, L = 16, 5
    base = rng.uniform(0.5, 0.95, size=(R, 1))
    conf = np.clip(base - 0.05 * np.arange(L) + 0.05 * rng.standard_normal((R, L)), 0.01, 1.0)
    a, b = 25.0, float(rng.uniform(0.05, 0.6))
    N = R * L
    cost = a + b * np.arange(N + 1)
    s = np.sort(survivals(conf).ravel())[::-1]
    n, tokens = 0, float(R)
    while n < N and s[n] > b * tokens / cost[n]:
        tokens += s[n]
        n += 1
    n_keep, n_orc, theta, tok_orc, _ = oracle.schedule_prefix(conf, cost)
    assert n_orc == n
    assert tok_orc == pytest.approx(tokens, rel=1e-12)
    assert theta == pytest.approx(tokens / cost[n], rel=1e-12)


def test_flat_and_prohibitive_costs():
    rng = np.random.default_rng(7)
    conf = rng.uniform(0.1, 0.9, size=(6, 4))
    conf[2, 1] = 0.0  # request 2 can commit nothing past its first guess
    N = conf.size
    n_keep, n, *_ = oracle.schedule_prefix(conf, np.full(N + 1, 2.0))
    assert list(n_keep) == [4, 4, 1, 4, 4, 4]  # every slot with positive survival
    n_keep, n, theta, tokens, _ = oracle.schedule_prefix(conf, 1.0 + 1e9 * np.arange(N + 1))
    assert n == 0 and (n_keep == 0).all() and theta == 6.0 and tokens == 6.0


def test_ties_go_to_earlier_positions_then_lower_requests():
    conf = np.full((3, 2), 0.5)  # survivals 0.5, 0.25 in every request
    for n_want, expect in [(1, [1, 0, 0]), (2, [1, 1, 0]), (3, [1, 1, 1]), (4, [2, 1, 1]),
                           (5, [2, 2, 1])]:
        cost = np.full(7, 1e30)
        cost[n_want] = 1.0
        n_keep, n, *_ = oracle.schedule_prefix(conf, cost)
        assert n == n_want and list(n_keep) == expect
    # equal survivals at different positions: the earlier position first
    # (request 1's first guess before request 0's second)
    conf = np.array([[1.0, 0.5], [0.5, 0.5]])
    cost = np.full(5, 1e30)
    cost[2] = 1.0
    n_keep, n, *_ = oracle.schedule_prefix(conf, cost)
    assert n == 2 and list(n_keep) == [1, 1]
    # equal ratios: the smaller n wins (a zero-survival slot adds nothing)
    conf = np.array([[0.5, 0.0]])
    n_keep, n, *_ = oracle.schedule_prefix(conf, np.ones(3))
    assert n == 1 and list(n_keep) == [1]


def test_invalid_inputs():
    conf = np.array([[np.nan, 0.5], [1.5, -0.2]])
    n_keep, n, theta, tokens, st = oracle.schedule_prefix(conf, np.ones(5))
    assert st & oracle.NAN_SEEN
    # NaN counts as 0 (request 0 keeps nothing); 1.5 -> 1 and -0.2 -> 0
    assert list(n_keep) == [0, 1] and tokens == pytest.approx(3.0)
    # no valid cost at all: nothing is verified
    n_keep, n, theta, tokens, st = oracle.schedule_prefix(np.full((2, 2), 0.9), -np.ones(5))
    assert n == 0 and theta == 0.0 and tokens == 2.0
    # no requests
    n_keep, n, theta, tokens, st = oracle.schedule_prefix(np.zeros((0, 3)), np.ones(1))
    assert n == 0 and n_keep.size == 0
