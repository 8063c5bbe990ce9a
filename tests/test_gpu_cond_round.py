"""The parent-conditioned round ("Robot2050/TreeSpark", items 1 and 2, then
the verification of "DDTree Explained ...", section 5) through the C ABI
(ddt_round_conditioned): the GPU's tree, mask, tree attention, target argmax,
greedy walk and KV compaction against the oracle, stage by stage."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_depth_gb300 import synth
from gpu_helpers import dev, host, make_ctx

pytestmark = pytest.mark.gpu

ATT_TOL = 1e-2

CASES = {
    "small": dict(name="treespark", R=3, L=4, V=5000, B=16, K=3, frontier=3, seed=31),
    "treespark": dict(name="treespark"),
}


class CondRoundCase:
    def __init__(self, cfg):
        self.cfg = cfg
        self.inp = inp = synth.draw_round_inputs(cfg)
        self.W, self.E, self.anchors = synth.draw_markov_head(cfg)
        # the oracle's tree; the synthetic target follows it
        self.o_tree = oracle.cond_tree(inp["draft_logits"], self.W, self.E, self.anchors, k=cfg.K,
                                       F=cfg.frontier, N=cfg.B)
        self.target = synth.GreedyTarget(cfg, inp["draft"], inp["agree"])
        self.target_logits = self.target.logits_for_tree(self.o_tree.tokens, self.o_tree.parents,
                                                         self.o_tree.n_nodes)
        ctx = self.ctx = make_ctx(cfg, inp)
        d = {k: dev(inp[k]) for k in ("draft_logits", "q", "k_tree", "v_tree", "k_cache",
                                       "v_cache", "block_table", "ctx_lens")}
        d["target_logits"] = dev(self.target_logits)
        self.out = ctx.alloc_outputs(cfg.R)
        bufs = dict(self.out)
        bufs.update(d)
        ctx.ddt_round_conditioned(cfg.R, bufs, dev(self.W), dev(self.E), dev(self.anchors))
        torch.cuda.synchronize()
        self.status = ctx.ddt_device_status()
        self.g = {k: host(v) for k, v in self.out.items()}
        self.g_k_cache = host(d["k_cache"], np.uint16)
        self.g_v_cache = host(d["v_cache"], np.uint16)
        self.g_ctx_lens = host(d["ctx_lens"])


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    kw = dict(CASES[request.param])
    return CondRoundCase(synth.config(kw.pop("name"), **kw))


def test_status_clean(case):
    assert case.status == 0


def test_tree_and_mask(case):
    t, g = case.o_tree, case.g
    np.testing.assert_array_equal(g["n_nodes"], t.n_nodes)
    np.testing.assert_array_equal(g["tree_tokens"], t.tokens)
    np.testing.assert_array_equal(g["parents"], t.parents)
    np.testing.assert_array_equal(g["depths"], t.depths)
    np.testing.assert_array_equal(g["mask"].view(np.uint32), oracle.build_mask(t.parents, t.n_nodes))


def test_attention(case):
    cfg, inp = case.cfg, case.inp
    mask = oracle.build_mask(case.o_tree.parents, case.o_tree.n_nodes)
    if cfg.R * cfg.P * cfg.Hq <= 4096:
        rr, ii, hh = np.meshgrid(np.arange(cfg.R), np.arange(cfg.P), np.arange(cfg.Hq),
                                 indexing="ij")
        sel = np.stack([rr.ravel(), ii.ravel(), hh.ravel()], 1).astype(np.int32)
    else:
        rng = np.random.default_rng(7)
        sel = np.array([(r, int(rng.integers(0, cfg.P)), int(rng.integers(0, cfg.Hq)))
                        for r in range(cfg.R) for _ in range(16)], np.int32)
    want, flags = oracle.tree_attention_rows(inp["q"], inp["k_tree"], inp["v_tree"],
                                             inp["k_cache"], inp["v_cache"], inp["block_table"],
                                             inp["ctx_lens"], mask, sel)
    assert flags == 0
    got = case.out["attn_out"].float().cpu().numpy()[sel[:, 0], sel[:, 1], sel[:, 2]]
    assert np.abs(got - want).max() <= ATT_TOL


def test_accept_walk_compaction(case):
    t, g, inp = case.o_tree, case.g, case.inp
    a, _ = oracle.argmax(case.target_logits)
    np.testing.assert_array_equal(g["target_argmax"], a)
    acc_len, acc_nodes, acc_tokens, bonus = oracle.walk(a, t.tokens, t.parents, t.n_nodes,
                                                        case.cfg.L)
    np.testing.assert_array_equal(g["acc_len"], acc_len)
    np.testing.assert_array_equal(g["acc_nodes"], acc_nodes)
    np.testing.assert_array_equal(g["acc_tokens"], acc_tokens)
    np.testing.assert_array_equal(g["bonus"], bonus)
    kc, vc, ctx = inp["k_cache"].copy(), inp["v_cache"].copy(), inp["ctx_lens"].copy()
    assert oracle.compact(kc, vc, inp["block_table"], ctx, inp["k_tree"], inp["v_tree"],
                          acc_nodes, acc_len) == 0
    np.testing.assert_array_equal(case.g_ctx_lens, ctx)
    assert np.array_equal(case.g_k_cache, kc) and np.array_equal(case.g_v_cache, vc)


def test_walk_reproduces_greedy_decoding(case):
    # the committed tokens are the first acc_len tokens of greedy decoding
    # under the target ("Robot2050/TreeSpark", item 4)
    g = case.g
    for r in range(case.cfg.R):
        n = int(g["acc_len"][r])
        assert list(g["acc_tokens"][r, :n]) == case.target.greedy_decode(r, n)
