"""Pins for the oracle's target argmax, greedy walk and KV compaction (a5-a7).

argmax: numpy's argmax (first index of the maximum) on random rows with
planted ties, and the signed-zero case.
walk: with a path-deterministic synthetic target, the committed tokens equal
plain autoregressive greedy decoding under that target ("Robot2050/TreeSpark"
item 4; "DDTree Explained ..." section 5, verifier walk); on a chain with a
constant per-token agreement a the mean acceptance length matches the closed
form (1 - a^(g+1)) / (1 - a), whose printed values are checked first.
compaction: cache bytes after compaction equal a hand-built expectation.
"""
import os

import numpy as np
import pytest

from speculative_decoding_draft_depth_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_argmax_matches_numpy_first_index(orc):
    rng = np.random.default_rng(2)
    t = rng.integers(-5, 6, size=(50, 777)).astype(np.float32)  # many ties
    out, flags = orc.argmax(t)
    assert flags == 0
    np.testing.assert_array_equal(out, np.argmax(t, axis=1))
    tb = synth.to_bf16_bits(t)
    outb, _ = orc.argmax(tb)
    np.testing.assert_array_equal(outb, np.argmax(t, axis=1))


def test_argmax_signed_zero_and_nan(orc):
    t = np.array([[-0.0, 0.0, -1.0], [-3.0, 0.0, -0.0]], np.float32)
    out, _ = orc.argmax(t)
    assert list(out) == [0, 1]
    t2 = np.array([[1.0, np.nan, 2.0]], np.float32)
    out2, flags = orc.argmax(t2)
    assert flags & orc.NAN_SEEN and out2[0] == 2


def _round_tree_and_targets(orc, cfg):
    inp = synth.draw_round_inputs(cfg)
    lp, ids, _, _ = orc.topk_logprobs(inp["draft_logits"], cfg.K)
    t = orc.build_tree(lp, ids, cfg.B)
    target = synth.GreedyTarget(cfg, inp["draft"], inp["agree"])
    tl = target.logits_for_tree(t.tokens, t.parents, t.n_nodes)
    a, _ = orc.argmax(tl)
    return inp, t, target, a


@pytest.mark.parametrize("name,overrides", [("tiny", {}), ("tiny", {"seed": 5, "B": 16}),
                                            ("single", {"V": 4096}),
                                            ("batch64", {"R": 6, "V": 4096})])
def test_walk_reproduces_autoregressive_greedy(orc, name, overrides):
    cfg = synth.config(name, **overrides)
    inp, t, target, a = _round_tree_and_targets(orc, cfg)
    acc_len, acc_nodes, acc_tokens, bonus = orc.walk(a, t.tokens, t.parents, t.n_nodes, cfg.L)
    for r in range(cfg.R):
        n = int(acc_len[r])
        assert 1 <= n <= cfg.L + 1
        greedy = target.greedy_decode(r, n)
        assert list(acc_tokens[r, :n]) == greedy
        assert bonus[r] == greedy[-1]
        assert np.all(acc_tokens[r, n:] == -1) and np.all(acc_nodes[r, n - 1:] == -1)
        # accepted nodes form a root path of increasing depth
        prev = 0
        for j in range(n - 1):
            node = int(acc_nodes[r, j])
            assert t.parents[r, node] == prev and t.depths[r, node] == j + 1
            assert t.tokens[r, node - 1] == acc_tokens[r, j]
            prev = node


def _chain_formula(a, g):
    return (1 - a ** (g + 1)) / (1 - a)


def test_chain_formula_printed_values():
    with open(os.path.join(GOLDEN, "chain_tokens_per_pass.txt")) as f:
        rows = [line.split() for line in f if line.strip() and not line.startswith("#")]
    for a, g, printed, dec in rows:
        val = _chain_formula(float(a), int(g))
        assert round(val, int(dec)) == pytest.approx(float(printed)), (a, g, val)


@pytest.mark.parametrize("a,g", [(0.5, 4), (0.8, 4), (0.5, 8)])
def test_chain_mean_acceptance_matches_closed_form(orc, a, g):
    """K=1 and B=L=g make the tree the drafter's top-1 chain; the synthetic
    target agrees with each top-1 with probability a and otherwise picks a
    token off the chain, so acc_len is a truncated geometric count."""
    R = 4000
    cfg = synth.config("tiny", R=R, L=g, B=g, K=1, V=16, agree_kind="const", agree_args=(a,),
                       seed=1000 + int(a * 10) + g)
    rng = np.random.default_rng(cfg.seed)
    z = rng.standard_normal((R, g, cfg.V)).astype(np.float32) * 3
    draft = synth.DraftLogits(z=z)
    agree = synth.draw_agreement(cfg, rng)
    lp, ids, _, _ = orc.topk_logprobs(z, 1)
    t = orc.build_tree(lp, ids, cfg.B)
    target = synth.GreedyTarget(cfg, draft, agree)
    tl = target.logits_for_tree(t.tokens, t.parents, t.n_nodes)
    amax, _ = orc.argmax(tl)
    acc_len, _, _, _ = orc.walk(amax, t.tokens, t.parents, t.n_nodes, g)
    mean = acc_len.mean()
    want = _chain_formula(a, g)
    sd = acc_len.std() / np.sqrt(R)
    assert abs(mean - want) < 4 * sd + 1e-9, (mean, want, sd)


def test_compaction_against_hand_built_cache(orc):
    cfg = synth.config("tiny", R=3, ctx_kind="uniform", ctx_args=(10, 40), seed=17, B=8)
    inp = synth.draw_round_inputs(cfg)
    kc, vc = inp["k_cache"].copy(), inp["v_cache"].copy()
    ctx = inp["ctx_lens"].copy()
    bt = inp["block_table"]
    P, L = cfg.P, cfg.L
    # an accepted path per request, chosen by hand
    acc_len = np.array([1, 3, 5], np.int32)
    acc_nodes = np.full((3, L), -1, np.int32)
    acc_nodes[1, :2] = [2, 6]
    acc_nodes[2, :4] = [1, 3, 4, 8]
    want_k, want_v = kc.copy(), vc.copy()
    for r in range(3):
        nodes = [0] + [int(x) for x in acc_nodes[r, :acc_len[r] - 1]]
        for j, node in enumerate(nodes):
            s = int(ctx[r]) + j
            want_k[bt[r, s // cfg.page], s % cfg.page] = inp["k_tree"][r, node]
            want_v[bt[r, s // cfg.page], s % cfg.page] = inp["v_tree"][r, node]
    flags = orc.compact(kc, vc, bt, ctx, inp["k_tree"], inp["v_tree"], acc_nodes, acc_len)
    assert flags == 0
    np.testing.assert_array_equal(kc, want_k)
    np.testing.assert_array_equal(vc, want_v)
    np.testing.assert_array_equal(ctx, inp["ctx_lens"] + acc_len)
    assert P == cfg.B + 1
