"""GPU parity of the parent-conditioned tree ("Robot2050/TreeSpark", items 1
and 2) through ddt_build_tree_conditioned, against the oracle on the same
seeded inputs:

  * every frontier parent's children lists: ids exact (up to values within
    the log-prob tolerance of each other), log-probs within 1e-5 of the
    oracle's fp64 lists for the same (request, depth, parent token);
  * the frontier and packing logic stage-wise: the oracle replays the GPU's
    lists and must give the same frontiers and tree bit for bit;
  * the tree end to end against the oracle's own (fp64) tree, and the mask.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import dev, host, make_ctx
from speculative_decoding_draft_depth_gb300 import synth

pytestmark = pytest.mark.gpu

LP_TOL = 1e-5

CASES = {
    "treespark": dict(name="treespark"),
    "small": dict(name="treespark", R=3, L=4, V=1000, B=12, K=3, frontier=2, seed=21),
    "k1": dict(name="treespark", R=2, L=3, V=5000, B=5, K=1, frontier=4, seed=22),
    "wide_frontier": dict(name="treespark", R=4, L=5, V=3000, B=40, K=4, frontier=8, seed=23),
    # a head whose bias is half the logits' spread: the seeded bounds are weak
    "strong_head": dict(name="treespark", R=4, L=4, V=20000, B=24, K=4, frontier=4, seed=24,
                        head_scale=0.3),
    # V not a multiple of 8 (l by direct loads, a ragged last tile)
    "ragged_v": dict(name="treespark", R=3, L=4, V=3001, B=16, K=3, frontier=3, seed=25),
    # more requests than l stages hold, and seed rows that do not fit
    "many_requests": dict(name="treespark", R=60, L=3, V=4096, B=10, K=2, frontier=2, seed=26),
    # depth 2 is certain (one token at 0, the rest 60 below: their exp is
    # below one ulp of 1 in fp32 and fp64, so its log-prob is exactly 0):
    # each child's score ties with its parent's, and packing must keep
    # parents first
    "certain_depth": dict(name="treespark", R=3, L=4, V=2000, B=16, K=3, frontier=3, seed=27,
                          certain_depth=1),
}


class CondCase:
    def __init__(self, cfg, head_scale=0.02, certain_depth=None):
        self.cfg = cfg
        self.inp = inp = synth.draw_round_inputs(cfg)
        if certain_depth is not None:
            z = inp["draft_logits"]  # bf16 bits
            z[:, certain_depth, :] = synth.to_bf16_bits(np.array([-60.0], np.float32))[0]
            z[:, certain_depth, 5] = 0
        self.W, self.E, self.anchors = synth.draw_markov_head(cfg, scale=head_scale)
        ctx = self.ctx = make_ctx(cfg, inp)
        R, L, F, K, N = cfg.R, cfg.L, cfg.frontier, cfg.K, cfg.B
        P = N + 1
        i32 = dict(dtype=torch.int32, device="cuda")
        out = self.out = dict(
            tree_tokens=torch.empty((R, N), **i32), parents=torch.empty((R, P), **i32),
            depths=torch.empty((R, P), **i32), n_nodes=torch.empty((R,), **i32),
            mask=torch.empty((R, P, (P + 31) // 32), **i32),
            cand_lp=torch.empty((R, L, F, K), dtype=torch.float32, device="cuda"),
            cand_ids=torch.empty((R, L, F, K), **i32), frontier_tok=torch.empty((R, L, F), **i32))
        ctx.ddt_build_tree_conditioned(dev(inp["draft_logits"]), dev(self.W), dev(self.E),
                                       dev(self.anchors), R, out["tree_tokens"], out["parents"],
                                       out["depths"], out["n_nodes"], out["mask"], out["cand_lp"],
                                       out["cand_ids"], out["frontier_tok"])
        torch.cuda.synchronize()
        self.status = ctx.ddt_device_status()
        self.g = {k: host(v) for k, v in out.items()}


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    kw = dict(CASES[request.param])
    scale = kw.pop("head_scale", 0.02)
    certain = kw.pop("certain_depth", None)
    return CondCase(synth.config(kw.pop("name"), **kw), head_scale=scale, certain_depth=certain)


def test_status_clean(case):
    assert case.status == 0


def test_parent_lists(case):
    cfg, g = case.cfg, case.g
    ft = g["frontier_tok"]
    np.testing.assert_array_equal(ft[:, 0, 0], case.anchors)
    sel = np.argwhere(ft >= 0)
    lp, ids = oracle.cond_parent_lists(case.inp["draft_logits"], case.W, case.E, sel[:, 0],
                                       sel[:, 1], ft[sel[:, 0], sel[:, 1], sel[:, 2]], cfg.K)
    glp = g["cand_lp"][sel[:, 0], sel[:, 1], sel[:, 2]].astype(np.float64)
    gids = g["cand_ids"][sel[:, 0], sel[:, 1], sel[:, 2]]
    assert np.abs(glp - lp).max() <= LP_TOL
    # ids exact, except that entries whose oracle values lie within the
    # tolerance of each other may appear in either order
    for i in range(len(sel)):
        if not np.array_equal(gids[i], ids[i]):
            assert sorted(gids[i].tolist()) == sorted(ids[i].tolist()) or \
                np.min(np.abs(np.diff(lp[i]))) <= 2 * LP_TOL, (sel[i], gids[i], ids[i])
    # slots past the frontier are empty
    empty = np.argwhere(ft < 0)
    assert (g["cand_ids"][empty[:, 0], empty[:, 1], empty[:, 2]] == -1).all()


def test_frontier_and_packing_stagewise(case):
    cfg, g = case.cfg, case.g
    t = oracle.cond_tree(case.inp["draft_logits"], case.W, case.E, case.anchors, k=cfg.K,
                         F=cfg.frontier, N=cfg.B, replay_lp=g["cand_lp"].astype(np.float64),
                         replay_ids=g["cand_ids"])
    np.testing.assert_array_equal(g["frontier_tok"], t.frontier_tok)
    np.testing.assert_array_equal(g["n_nodes"], t.n_nodes)
    np.testing.assert_array_equal(g["tree_tokens"], t.tokens)
    np.testing.assert_array_equal(g["parents"], t.parents)
    np.testing.assert_array_equal(g["depths"], t.depths)
    np.testing.assert_array_equal(g["mask"].view(np.uint32), oracle.build_mask(t.parents, t.n_nodes))


def test_tree_end_to_end(case):
    cfg, g = case.cfg, case.g
    t = oracle.cond_tree(case.inp["draft_logits"], case.W, case.E, case.anchors, k=cfg.K,
                         F=cfg.frontier, N=cfg.B)
    np.testing.assert_array_equal(g["n_nodes"], t.n_nodes)
    np.testing.assert_array_equal(g["tree_tokens"], t.tokens)
    np.testing.assert_array_equal(g["parents"], t.parents)
    np.testing.assert_array_equal(g["depths"], t.depths)
