"""Pins for the oracle's best-first tree (step a2).

Algorithm 1 of "DDTree Explained ..." (section 4) and the heap loop of
"SparklingTree ..." (Step 3). Pinned against: a hand-worked example, an
independent sort-every-prefix construction, Lemma 1 (K = min(B, V) loses
nothing), Prop. 2 (the tree is prefix-closed and maximises the sum of prefix
probabilities among all prefix-closed B-sets, by exhaustive search) and
Prop. 1 (sum of prefix probabilities = expected accepted depth under the
drafter's factorised distribution, by enumerating every draft path).
"""
import itertools
import os

import numpy as np
import pytest

from speculative_decoding_draft_depth_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_worked_example(fname):
    lp, ids, out = {}, {}, {}
    with open(os.path.join(GOLDEN, fname)) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            if line[0] == "lp":
                lp[int(line[1])] = [float(x) for x in line[2:]]
            elif line[0] == "id":
                ids[int(line[1])] = [int(x) for x in line[2:]]
            else:
                out[line[0]] = [int(x) for x in line[1:]]
    L = len(lp)
    return (np.array([lp[d] for d in range(L)]), np.array([ids[d] for d in range(L)], np.int32),
            out)


@pytest.mark.parametrize("fname", ["heap_worked_example.txt", "heap_worked_example_ties.txt"])
def test_hand_worked_example(orc, fname):
    lp, ids, want = _read_worked_example(fname)
    B = want["budget"][0]
    t = orc.build_tree(lp[None], ids[None], B)
    assert t.n_nodes[0] == B
    np.testing.assert_array_equal(t.tokens[0], want["tree_tokens"])
    np.testing.assert_array_equal(t.parents[0], want["parents"])
    np.testing.assert_array_equal(t.depths[0], want["depths"])


def _assert_same_tree(a, b, r=0):
    np.testing.assert_array_equal(a.n_nodes[r], b.n_nodes[0])
    np.testing.assert_array_equal(a.tokens[r], b.tokens[0])
    np.testing.assert_array_equal(a.parents[r], b.parents[0])
    np.testing.assert_array_equal(a.depths[r], b.depths[0])
    np.testing.assert_array_equal(a.ranks[r], b.ranks[0])
    np.testing.assert_array_equal(a.S[r], b.S[0])


@pytest.mark.parametrize("L,K,B,quant", [(4, 8, 8, 0), (3, 5, 20, 0), (4, 4, 40, 0.5),
                                         (5, 3, 60, 0.25), (2, 6, 12, 1.0), (6, 2, 30, 0)])
def test_heap_equals_sorted_enumeration(orc, L, K, B, quant):
    rng = np.random.default_rng(L * 100 + K * 10 + B)
    for trial in range(5):
        z = rng.standard_normal((L, 50)) * 2
        if quant:
            z = np.round(z / quant) * quant  # many exact ties in lp
        lp, ids, _, _ = orc.topk_logprobs(z.astype(np.float32), K)
        heap = orc.build_tree(lp[None], ids[None], B)
        brute = orc.build_tree_bruteforce(lp, ids, B)
        _assert_same_tree(heap, brute)


def test_short_tree_when_prefix_space_is_small(orc):
    # L=2, K=2 has 6 prefixes; a budget of 10 yields 6 nodes and -1 padding
    lp = np.log(np.array([[0.6, 0.4], [0.7, 0.3]]))
    ids = np.array([[4, 1], [2, 3]], np.int32)
    t = orc.build_tree(lp[None], ids[None], 10)
    assert t.n_nodes[0] == 6
    assert np.all(t.tokens[0, 6:] == -1)
    assert np.all(t.parents[0, 7:] == -1)


def test_lemma1_topk_truncation_is_lossless(orc):
    """The tree from K = min(B, V) equals the tree from the full vocabulary
    (every one of the V^L = 32^4 paths' prefixes enumerated and sorted)."""
    cfg = synth.config("tiny")
    inp = synth.draw_round_inputs(cfg)
    z = inp["draft_logits"][0]
    lpK, idsK, _, _ = orc.topk_logprobs(z, cfg.K)
    lpV, idsV, _, _ = orc.topk_logprobs(z, cfg.V)
    small = orc.build_tree(lpK[None], idsK[None], cfg.B)
    full = orc.build_tree_bruteforce(lpV, idsV, cfg.B, max_prefixes=2_000_000)
    _assert_same_tree(small, full)


def _prefix_closed_subsets(V, L, B):
    """All prefix-closed sets of B token paths (each a tuple) over V tokens,
    depth <= L, by growing sets one frontier node at a time in canonical
    (sorted) order."""
    out = []

    def grow(chosen, frontier_min):
        if len(chosen) == B:
            out.append(tuple(chosen))
            return
        # candidates: children of the root or of chosen nodes, not chosen
        cands = set()
        for t in range(V):
            cands.add((t,))
        for u in chosen:
            if len(u) < L:
                for t in range(V):
                    cands.add(u + (t,))
        cands = sorted(c for c in cands if c not in chosen and c > frontier_min)
        for c in cands:
            grow(chosen + [c], c)

    grow([], ())
    return out


@pytest.mark.parametrize("V,L,B", [(3, 3, 4), (4, 2, 5), (2, 3, 6)])
def test_prop2_optimal_among_prefix_closed_sets(orc, V, L, B):
    rng = np.random.default_rng(V * 7 + L * 3 + B)
    z = rng.standard_normal((L, V)) * 1.5
    lp, ids, _, _ = orc.topk_logprobs(z.astype(np.float32), V)
    t = orc.build_tree(lp[None], ids[None], B)
    # token-level marginal log-probs for scoring arbitrary paths
    lpt = np.empty((L, V))
    for d in range(L):
        lpt[d, ids[d]] = lp[d]
    # the tree is prefix-closed: every parent is a node one level up
    n = t.n_nodes[0]
    for node in range(1, n + 1):
        p = t.parents[0, node]
        assert 0 <= p < node
        assert t.depths[0, node] == t.depths[0, p] + 1
    tree_value = np.exp(t.S[0, 1:n + 1]).sum()
    best = -1.0
    for subset in _prefix_closed_subsets(V, L, B):
        val = sum(np.exp(sum(lpt[i, tok] for i, tok in enumerate(u))) for u in subset)
        best = max(best, val)
    assert abs(tree_value - best) < 1e-12


def test_prop1_expected_acceptance_equals_sum_of_prefix_probabilities(orc):
    """E_{Y~Q}[alpha_T(Y)] by enumerating all 32^4 draft paths y, where
    alpha_T(y) is the number of tree nodes whose token path is a prefix of y."""
    cfg = synth.config("tiny")
    inp = synth.draw_round_inputs(cfg)
    z = inp["draft_logits"][0]
    L, V = cfg.L, cfg.V
    lpK, idsK, _, _ = orc.topk_logprobs(z, cfg.K)
    t = orc.build_tree(lpK[None], idsK[None], cfg.B)
    lpV, idsV, _, _ = orc.topk_logprobs(z, V)
    logq = np.empty((L, V))
    for d in range(L):
        logq[d, idsV[d]] = lpV[d]
    # token path of every node
    n = t.n_nodes[0]
    paths = {0: ()}
    for node in range(1, n + 1):
        paths[node] = paths[t.parents[0, node]] + (int(t.tokens[0, node - 1]),)
    nodes_by_depth = {}
    for node in range(1, n + 1):
        nodes_by_depth.setdefault(len(paths[node]), set()).add(paths[node])
    # enumerate y in V^L with numpy: alpha(y) = sum_d [y[:d] is a node]
    grid = np.array(list(itertools.product(range(V), repeat=L)), np.int64)  # [V^L, L]
    logQ = sum(logq[d, grid[:, d]] for d in range(L))
    alpha = np.zeros(grid.shape[0])
    for d, pset in nodes_by_depth.items():
        keys = grid[:, :d] @ (V ** np.arange(d - 1, -1, -1))
        want = np.array([sum(tok * V ** (d - 1 - i) for i, tok in enumerate(p)) for p in pset])
        alpha += np.isin(keys, want)
    expectation = float(np.sum(np.exp(logQ) * alpha))
    prefix_sum = float(np.exp(t.S[0, 1:n + 1]).sum())
    assert abs(expectation - prefix_sum) < 1e-12


def test_tree_structure_invariants_at_full_vocab(orc):
    """Budget-sized trees on a 'single'-shaped drafter: depths in 1..L,
    parents before children, siblings carry distinct tokens, S decreases
    along the pop order (best-first)."""
    cfg = synth.config("single", V=4096)
    inp = synth.draw_round_inputs(cfg)
    lp, ids, _, _ = orc.topk_logprobs(inp["draft_logits"], cfg.K)
    t = orc.build_tree(lp, ids, cfg.B)
    n = t.n_nodes[0]
    assert n == cfg.B
    S = t.S[0, 1:n + 1]
    assert np.all(np.diff(S) <= 0)
    for node in range(1, n + 1):
        assert 1 <= t.depths[0, node] <= cfg.L
        assert t.parents[0, node] < node
    sib = {}
    for node in range(1, n + 1):
        key = (int(t.parents[0, node]), int(t.tokens[0, node - 1]))
        assert key not in sib
        sib[key] = node


@pytest.mark.parametrize("L,K,quant,seed", [(3, 3, False, 1), (4, 3, True, 2), (2, 5, True, 3)])
def test_prefixes_at_least_matches_full_enumeration(orc, L, K, quant, seed):
    """The pruned walk returns exactly the prefixes a full enumeration of the
    K + K^2 + ... + K^L prefixes scores at or above the cut, with the same
    fp64 scores (quantised log-probs make many exact ties at the cut)."""
    rng = np.random.default_rng(seed)
    lp = -np.sort(rng.exponential(1.0, (L, K)), axis=1)
    if quant:
        lp = np.round(lp * 2) / 2
    lp = -np.sort(-lp, axis=1)  # descending per depth
    ids = np.stack([rng.permutation(50)[:K] for _ in range(L)]).astype(np.int32)
    full = {}
    for depth in range(1, L + 1):
        for ranks in itertools.product(range(K), repeat=depth):
            path = tuple(int(ids[d, j]) for d, j in enumerate(ranks))
            full[path] = float(sum(lp[d, j] for d, j in enumerate(ranks)))
    for smin in sorted(set(full.values()))[::max(1, len(full) // 7)] + [-1e9, 0.0]:
        want = {p: s for p, s in full.items() if s >= smin}
        got = dict(orc.prefixes_at_least(lp, ids, smin))
        assert set(got) == set(want)
        for p in want:
            assert got[p] == pytest.approx(want[p], abs=1e-12)


def test_tree_nodes_lie_in_the_prefix_set_of_its_last_score(orc):
    """The heap's B nodes all score at least the B-th score, and every prefix
    strictly above it is one of them."""
    rng = np.random.default_rng(5)
    L, K, B = 5, 4, 24
    lp = -np.sort(np.round(rng.exponential(1.0, (1, L, K)) * 2) / 2, axis=2)
    ids = np.stack([rng.permutation(100)[:K] for _ in range(L)])[None].astype(np.int32)
    t = orc.build_tree(lp, ids, B)
    n = int(t.n_nodes[0])
    SB = t.S[0, 1:n + 1].min()
    above = {p for p, s in orc.prefixes_at_least(lp[0], ids[0], SB) if s > SB}
    paths = {}
    for node in range(1, n + 1):
        paths[node] = paths.get(int(t.parents[0, node]), ()) + (int(t.tokens[0, node - 1]),)
    assert above <= set(paths.values())
    assert set(paths.values()) <= {p for p, _ in orc.prefixes_at_least(lp[0], ids[0], SB)}
