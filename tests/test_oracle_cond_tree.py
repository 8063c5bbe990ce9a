"""Pins of the oracle's parent-conditioned tree ("Robot2050/TreeSpark",
items 1 and 2): a Markov bias W e(t_u) on per-depth logits, per-parent top-k,
frontier pruning by path score, top-N packing.

  * with W = 0 and no pruning the packed tree is the best-first DDTree tree
    of the same logits at K = k (an independent construction: the heap of
    Algorithm 1 in the oracle's other function);
  * depth 1's lists equal numpy's matmul + log-softmax + stable top-k;
  * the page's printed policy numbers (100 candidates, 33 positions);
  * invariants: prefix-closed packing, scores non-increasing along edges,
    each frontier the best F candidates of its depth, replay reproduces.
"""
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _inputs(R=2, D=3, V=40, H=8, seed=0, wscale=0.5):
    rng = np.random.default_rng(seed)
    ell = (rng.standard_normal((R, D, V)) * 3).astype(np.float32)
    W = (rng.standard_normal((V, H)) * wscale).astype(np.float32)
    E = (rng.standard_normal((V, H)) * wscale).astype(np.float32)
    anchors = rng.integers(0, V, size=R).astype(np.int32)
    return ell, W, E, anchors


def test_no_bias_no_pruning_is_the_best_first_tree():
    ell, W, E, anchors = _inputs(R=3, D=3, V=30, seed=1)
    W[:] = 0.0
    k, N = 4, 20
    t = oracle.cond_tree(ell, W, E, anchors, k=k, F=k ** 2, N=N)
    lp, ids, _, _ = oracle.topk_logprobs(ell, k)
    ref = oracle.build_tree(lp, ids, N)
    np.testing.assert_array_equal(t.n_nodes, ref.n_nodes)
    np.testing.assert_array_equal(t.tokens, ref.tokens)
    np.testing.assert_array_equal(t.parents, ref.parents)
    np.testing.assert_array_equal(t.depths, ref.depths)
    np.testing.assert_allclose(t.S, ref.S, rtol=0, atol=1e-12)


def test_depth_one_lists_match_numpy():
    ell, W, E, anchors = _inputs(R=3, D=2, V=64, H=16, seed=2)
    k = 5
    t = oracle.cond_tree(ell, W, E, anchors, k=k, F=4, N=12)
    for r in range(3):
        z = ell[r, 0].astype(np.float64) + W.astype(np.float64) @ E[anchors[r]].astype(np.float64)
        lse = z.max() + np.log(np.exp(z - z.max()).sum())
        order = np.argsort(-z, kind="stable")[:k]
        np.testing.assert_array_equal(t.cand_ids[r, 0, 0], order)
        np.testing.assert_allclose(t.cand_lp[r, 0, 0], z[order] - lse, rtol=0, atol=1e-12)
        assert t.frontier_tok[r, 0, 0] == anchors[r]
        assert (t.frontier_tok[r, 0, 1:] == -1).all()


def test_page_policy_numbers():
    rows = [l.split() for l in open(os.path.join(HERE, "golden", "treespark_policy_numbers.txt"))
            if l.strip() and not l.startswith("#")]
    k, depths, N, cands, positions = map(int, rows[0])
    assert k + (depths - 1) * k * k == cands  # frontier width F = k
    assert N + 1 == positions
    ell, W, E, anchors = _inputs(R=2, D=depths, V=50, H=8, seed=3)
    t = oracle.cond_tree(ell, W, E, anchors, k=k, F=k, N=N)
    # every candidate slot is filled: depth 1 has one parent, later depths F
    assert (t.cand_ids[:, 0, 0] >= 0).all() and (t.cand_ids[:, 0, 1:] == -1).all()
    assert (t.cand_ids[:, 1:] >= 0).all()
    n_cand = int((t.cand_ids[0] >= 0).sum())
    assert n_cand == cands
    assert (t.n_nodes == N).all()


@pytest.mark.parametrize("seed", [4, 5, 6])
def test_invariants(seed):
    ell, W, E, anchors = _inputs(R=3, D=5, V=40, H=8, seed=seed)
    k, F, N = 3, 2, 14
    t = oracle.cond_tree(ell, W, E, anchors, k=k, F=F, N=N)
    for r in range(3):
        n = int(t.n_nodes[r])
        assert n == N
        assert t.parents[r, 0] == -1 and t.depths[r, 0] == 0
        for i in range(1, n + 1):
            p = int(t.parents[r, i])
            assert 0 <= p < i                                  # prefix-closed, parent first
            assert t.depths[r, i] == t.depths[r, p] + 1
            assert t.S[r, i] <= t.S[r, p]                      # lp <= 0 along an edge
        assert np.all(np.diff(t.S[r, 1:n + 1]) <= 0)           # packed by score
        # the frontier of depth d+1: the F best (S, creation order) of depth d's candidates
        S_par = {0: 0.0}
        for d in range(1, 5):
            lp = t.cand_lp[r, d - 1]
            ids = t.cand_ids[r, d - 1]
            # scores of depth d's candidates: parent score + lp, parent = frontier slot
            if d == 1:
                par_scores = [0.0]
            else:
                par_scores = S_prev_sorted[:F]
            scores = []
            for f, ps in enumerate(par_scores):
                for j in range(k):
                    scores.append((ps + lp[f, j], f * k + j, int(ids[f, j])))
            best = sorted(scores, key=lambda x: (-x[0], x[1]))[:F]
            S_prev_sorted = [b[0] for b in best]
            np.testing.assert_array_equal(t.frontier_tok[r, d, :len(best)], [b[2] for b in best])


def test_replay_reproduces():
    ell, W, E, anchors = _inputs(R=2, D=4, V=40, H=8, seed=7)
    t = oracle.cond_tree(ell, W, E, anchors, k=4, F=4, N=20)
    t2 = oracle.cond_tree(ell, W, E, anchors, k=4, F=4, N=20, replay_lp=t.cand_lp,
                          replay_ids=t.cand_ids)
    for name in ("tokens", "parents", "depths", "n_nodes", "frontier_tok"):
        np.testing.assert_array_equal(getattr(t2, name), getattr(t, name))
    np.testing.assert_array_equal(t2.S, t.S)


def test_parent_lists_match_the_tree_lists():
    ell, W, E, anchors = _inputs(R=2, D=3, V=40, H=8, seed=8)
    t = oracle.cond_tree(ell, W, E, anchors, k=4, F=2, N=10)
    req, dep, tok, want_lp, want_ids = [], [], [], [], []
    for r in range(2):
        for d in range(3):
            for f in range(2):
                if t.frontier_tok[r, d, f] >= 0:
                    req.append(r)
                    dep.append(d)
                    tok.append(t.frontier_tok[r, d, f])
                    want_lp.append(t.cand_lp[r, d, f])
                    want_ids.append(t.cand_ids[r, d, f])
    lp, ids = oracle.cond_parent_lists(ell, W, E, req, dep, tok, 4)
    np.testing.assert_array_equal(ids, np.array(want_ids))
    np.testing.assert_array_equal(lp, np.array(want_lp))


def test_tied_logits_list_the_lower_token_first():
    """Equal logits (integers, many ties) with no bias: each parent's list is
    numpy's stable descending order, lower token id first among equals."""
    rng = np.random.default_rng(11)
    R, D, V, H, k = 2, 2, 24, 4, 6
    ell = rng.integers(-2, 3, size=(R, D, V)).astype(np.float32)
    W = np.zeros((V, H), np.float32)
    E = rng.standard_normal((V, H)).astype(np.float32)
    anchors = rng.integers(0, V, size=R).astype(np.int32)
    t = oracle.cond_tree(ell, W, E, anchors, k=k, F=2, N=8)
    for r in range(R):
        z = ell[r, 0].astype(np.float64)
        np.testing.assert_array_equal(t.cand_ids[r, 0, 0], np.argsort(-z, kind="stable")[:k])


def test_score_ties_pack_the_parent_first():
    """A depth whose only likely token has log-prob 0 (the others 1000 below:
    exp underflows, log-partition exactly the max) gives each child the same
    score as its parent. Packing by (score desc, depth asc) keeps the tree
    prefix-closed: every node's parent comes before it."""
    R, D, V, H, k, N = 2, 3, 12, 4, 3, 10
    rng = np.random.default_rng(12)
    ell = (rng.standard_normal((R, D, V)) * 2).astype(np.float32)
    ell[:, 1, :] = -1000.0
    ell[:, 1, 5] = 0.0  # depth 2 is certain: token 5 with log-prob 0
    W = np.zeros((V, H), np.float32)
    E = rng.standard_normal((V, H)).astype(np.float32)
    anchors = rng.integers(0, V, size=R).astype(np.int32)
    t = oracle.cond_tree(ell, W, E, anchors, k=k, F=k, N=N)
    for r in range(R):
        n = int(t.n_nodes[r])
        for i in range(1, n + 1):
            p = int(t.parents[r, i])
            assert 0 <= p < i, (r, i, p)
            if t.depths[r, i] == 2:  # the certain child ties with its parent
                assert t.S[r, i] == t.S[r, p]
