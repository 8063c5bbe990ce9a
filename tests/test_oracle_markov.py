"""Pins of the oracle's SparklingTree table tree ("SparklingTree ...",
"Building SparklingTree" and "Solving the candidate tree construction"): a
top-C prefilter per depth, a table of the Markov head's conditional
log-probs, and Algorithm 1 reading each parent's list from the table.

  * with no bias and a prefilter that keeps the whole vocabulary, the tree is
    DDTree's best-first tree of the same logits (the oracle's independent
    Algorithm 1 on per-depth top-K lists);
  * the prefilter and table equal numpy's stable argsort, matmul and
    log-softmax;
  * the heap equals a brute-force sort of every prefix (Prop. 2 with a list
    per parent), for weak and strong biases;
  * bf16 inputs widen exactly; equal log-probs go to the lower token id;
  * invariants (prefix-closed, scores non-increasing along edges) and the
    page's printed policy numbers.
"""
import os

import numpy as np
import pytest

import oracle
from speculative_decoding_draft_depth_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _inputs(R=2, L=3, V=40, H=8, seed=0, wscale=0.5):
    rng = np.random.default_rng(seed)
    ell = (rng.standard_normal((R, L, V)) * 3).astype(np.float32)
    W = (rng.standard_normal((V, H)) * wscale).astype(np.float32)
    E = (rng.standard_normal((V, H)) * wscale).astype(np.float32)
    anchors = rng.integers(0, V, size=R).astype(np.int32)
    return ell, W, E, anchors


def test_no_bias_full_prefilter_is_ddtree():
    for seed in range(4):
        R, L, V, B = 3, 4, 12, 20
        ell, W, E, anchors = _inputs(R=R, L=L, V=V, seed=seed)
        W[:] = 0.0
        cand, tab = oracle.markov_table(ell, W, E, anchors, C=V)
        t = oracle.markov_tree(cand, tab, B)
        lp, ids, _, _ = oracle.topk_logprobs(ell, min(B, V))
        d = oracle.build_tree(lp, ids, B)
        np.testing.assert_array_equal(t.n_nodes, d.n_nodes)
        np.testing.assert_array_equal(t.tokens, d.tokens)
        np.testing.assert_array_equal(t.parents, d.parents)
        np.testing.assert_array_equal(t.depths, d.depths)
        np.testing.assert_allclose(t.S, d.S, rtol=0, atol=1e-12)


@pytest.mark.parametrize("quantized", [False, True])
def test_table_matches_numpy(quantized):
    R, L, V, H, C = 2, 3, 50, 8, 7
    ell, W, E, anchors = _inputs(R=R, L=L, V=V, H=H, seed=5)
    if quantized:  # many equal logits: the prefilter keeps the lower ids
        ell = np.round(ell).astype(np.float32)
    cand, tab = oracle.markov_table(ell, W, E, anchors, C)
    e64, W64, E64 = ell.astype(np.float64), W.astype(np.float64), E.astype(np.float64)
    for r in range(R):
        for d in range(L):
            want_cand = np.argsort(-e64[r, d], kind="stable")[:C]
            np.testing.assert_array_equal(cand[r, d], want_cand)
            parents = [anchors[r]] if d == 0 else list(want_cand_prev)
            for a in range(C):
                if d == 0 and a > 0:
                    assert np.all(np.isneginf(tab[r, d, a]))
                    continue
                z = e64[r, d, want_cand] + W64[want_cand] @ E64[parents[a]]
                lse = z.max() + np.log(np.exp(z - z.max()).sum())
                np.testing.assert_allclose(tab[r, d, a], z - lse, rtol=0, atol=1e-12)
            want_cand_prev = want_cand


@pytest.mark.parametrize("seed,wscale", [(0, 0.1), (1, 0.5), (2, 1.5), (3, 3.0)])
def test_heap_equals_bruteforce(seed, wscale):
    L, V, C, B = 3, 30, 5, 25
    ell, W, E, anchors = _inputs(R=1, L=L, V=V, seed=seed, wscale=wscale)
    cand, tab = oracle.markov_table(ell, W, E, anchors, C)
    t = oracle.markov_tree(cand, tab, B)
    b = oracle.markov_tree_bruteforce(cand, tab, B)
    np.testing.assert_array_equal(t.n_nodes, b.n_nodes)
    np.testing.assert_array_equal(t.tokens, b.tokens)
    np.testing.assert_array_equal(t.parents, b.parents)
    np.testing.assert_array_equal(t.depths, b.depths)
    np.testing.assert_allclose(t.S, b.S, rtol=0, atol=0)


def test_small_budget_covers_every_prefix():
    # fewer prefixes than the budget: the tree holds them all
    L, V, C = 2, 10, 3
    ell, W, E, anchors = _inputs(R=1, L=L, V=V, seed=9)
    cand, tab = oracle.markov_table(ell, W, E, anchors, C)
    t = oracle.markov_tree(cand, tab, 50)
    assert t.n_nodes[0] == C + C * C
    assert (t.tokens[0, C + C * C:] == -1).all()


def test_bf16_widens_exactly_and_ties_go_to_lower_ids():
    rng = np.random.default_rng(11)
    R, L, V, H, C = 2, 3, 64, 8, 9
    f = lambda a: synth.bf16_bits_to_f32(synth.to_bf16_bits(a))
    ell = f((rng.standard_normal((R, L, V)) * 3).astype(np.float32))
    ell[:, :, 10:20] = ell[:, :, 5:6]   # equal logits: a tie run
    W = f((rng.standard_normal((V, H)) * 0.3).astype(np.float32))
    E = f((rng.standard_normal((V, H)) * 0.3).astype(np.float32))
    anchors = rng.integers(0, V, size=R).astype(np.int32)
    c1, t1 = oracle.markov_table(synth.to_bf16_bits(ell), synth.to_bf16_bits(W),
                                 synth.to_bf16_bits(E), anchors, C)
    c2, t2 = oracle.markov_table(ell, W, E, anchors, C)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(t1, t2)
    # with W = 0 every row of a depth is the same: equal lp, lower token first
    W0 = np.zeros_like(W)
    cand, tab = oracle.markov_table(ell, W0, E, anchors, C)
    t = oracle.markov_tree(cand, tab, 30)
    for r in range(R):
        kids = [t.tokens[r, n - 1] for n in range(1, t.n_nodes[r] + 1) if t.parents[r, n] == 0]
        lps = [tab[r, 0, 0, list(cand[r, 0]).index(k)] for k in kids]
        for i in range(len(kids) - 1):
            assert lps[i] > lps[i + 1] or (lps[i] == lps[i + 1] and kids[i] < kids[i + 1])


@pytest.mark.parametrize("seed", [21, 22])
def test_invariants(seed):
    R, L, V, C, B = 3, 5, 60, 8, 40
    ell, W, E, anchors = _inputs(R=R, L=L, V=V, seed=seed, wscale=1.0)
    cand, tab = oracle.markov_table(ell, W, E, anchors, C)
    t = oracle.markov_tree(cand, tab, B)
    for r in range(R):
        n = t.n_nodes[r]
        assert n == B
        for i in range(1, n + 1):
            p = t.parents[r, i]
            assert 0 <= p < i
            assert t.depths[r, i] == t.depths[r, p] + 1
            assert t.S[r, i] <= t.S[r, p]
            # the node's token is its candidate at its depth, and its score
            # is the parent's plus the table entry
            d, b = t.depths[r, i] - 1, t.cand[r, i]
            assert cand[r, d, b] == t.tokens[r, i - 1]
            a = 0 if p == 0 else t.cand[r, p]
            assert t.S[r, i] == t.S[r, p] + tab[r, d, a, b]
        # popped in order: scores non-increasing
        assert np.all(np.diff(t.S[r, 1:n + 1]) <= 0)


def test_page_policy_numbers():
    rows = [l.split() for l in open(os.path.join(HERE, "golden", "sparkling_policy_numbers.txt"))
            if l.strip() and not l.startswith("#")]
    C, B, depths = map(int, rows[0])
    cfg = synth.config("sparkling")
    assert (cfg.prefilter, cfg.B, cfg.L) == (C, B, depths)
    assert cfg.B + 1 == cfg.P
