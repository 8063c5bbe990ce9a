"""The SparklingTree table tree on the GPU ("SparklingTree ...", "Solving the
candidate tree construction" and "Building SparklingTree") through the C ABI:
the prefilter, the Markov table, the tree over the table, and the whole round
(ddt_round_markov), each against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_depth_gb300 import synth
from gpu_helpers import dev, host, make_ctx, tree_paths

pytestmark = pytest.mark.gpu

LP_TOL = 1e-5
ATT_TOL = 1e-2
TIE = 1e-5

CASES = {
    "small": dict(R=3, L=4, V=3000, B=20, K=20, prefilter=16, seed=41),
    "ragged": dict(R=2, L=5, V=1001, B=12, K=12, prefilter=7, seed=42),
    "wide": dict(R=4, L=6, V=20000, B=64, K=64, prefilter=128, seed=43),
    "strong_head": dict(R=3, L=4, V=5000, B=30, K=30, prefilter=32, seed=44),
    "sparkling": dict(),
}
HEAD_SCALE = {"strong_head": 0.3}
ORACLE_REQUESTS = 4  # requests whose table the oracle recomputes at full size


class MarkovCase:
    def __init__(self, cfg, head_scale=0.02):
        self.cfg = cfg
        self.inp = inp = synth.draw_round_inputs(cfg)
        self.W, self.E, self.anchors = synth.draw_markov_head(cfg, scale=head_scale)
        R, L, C, B = cfg.R, cfg.L, cfg.prefilter, cfg.B
        P = B + 1
        ctx = self.ctx = make_ctx(cfg, inp)
        i32 = dict(dtype=torch.int32, device="cuda")
        self.cand = torch.empty((R, L, C), **i32)
        self.tab = torch.empty((R, L, C, C), dtype=torch.float32, device="cuda")
        out = self.out = dict(
            tree_tokens=torch.empty((R, B), **i32), parents=torch.empty((R, P), **i32),
            depths=torch.empty((R, P), **i32), n_nodes=torch.empty((R,), **i32),
            mask=torch.empty((R, P, (P + 31) // 32), **i32))
        ell, Wd, Ed, an = dev(inp["draft_logits"]), dev(self.W), dev(self.E), dev(self.anchors)
        ctx.ddt_markov_table(ell, Wd, Ed, an, R, self.cand, self.tab)
        ctx.ddt_build_tree_markov(self.cand, self.tab, R, out["tree_tokens"], out["parents"],
                                  out["depths"], out["n_nodes"], out["mask"])
        torch.cuda.synchronize()
        self.status = ctx.ddt_device_status()
        self.g = {k: host(v) for k, v in out.items()}
        self.g_cand = host(self.cand)
        self.g_tab = host(self.tab)
        # the oracle's table: every request, or the first few at full size
        n = R if R <= 8 else ORACLE_REQUESTS
        self.n_or = n
        self.o_cand, self.o_tab = oracle.markov_table(inp["draft_logits"][:n], self.W, self.E,
                                                      self.anchors[:n], C)


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    kw = dict(CASES[request.param])
    return MarkovCase(synth.config("sparkling", **kw), HEAD_SCALE.get(request.param, 0.02))


def test_status_clean(case):
    assert case.status == 0


def test_prefilter(case):
    n = case.n_or
    np.testing.assert_array_equal(case.g_cand[:n], case.o_cand)


def test_table(case):
    n, o, g = case.n_or, case.o_tab, case.g_tab[:case.n_or].astype(np.float64)
    inf = np.isneginf(o)
    np.testing.assert_array_equal(np.isneginf(g), inf)
    assert np.abs(g[~inf] - o[~inf]).max() <= LP_TOL


def test_tree_stagewise(case):
    # the oracle's heap on the GPU's own table: bit-exact
    t = oracle.markov_tree(case.g_cand, case.g_tab.astype(np.float64), case.cfg.B)
    g = case.g
    np.testing.assert_array_equal(g["n_nodes"], t.n_nodes)
    np.testing.assert_array_equal(g["tree_tokens"], t.tokens)
    np.testing.assert_array_equal(g["parents"], t.parents)
    np.testing.assert_array_equal(g["depths"], t.depths)
    np.testing.assert_array_equal(g["mask"].view(np.uint32), oracle.build_mask(t.parents, t.n_nodes))


def test_tree_end_to_end_tie_band(case):
    # against the oracle's own fp64 table: the node sets agree except for
    # nodes whose score is within TIE of the budget's last score
    n, B = case.n_or, case.cfg.B
    t = oracle.markov_tree(case.o_cand, case.o_tab, B)
    g = case.g
    for r in range(n):
        nn = int(t.n_nodes[r])
        assert int(g["n_nodes"][r]) == nn
        o_paths = tree_paths(t.tokens[r], t.parents[r], nn)
        g_paths = tree_paths(g["tree_tokens"][r], g["parents"][r], nn)
        S = {p: t.S[r, i + 1] for i, p in enumerate(o_paths)}
        cut = t.S[r, nn] if nn else 0.0
        for p in set(o_paths) ^ set(g_paths):
            if p in S:
                assert abs(S[p] - cut) <= TIE, (r, p, S[p], cut)
        if set(o_paths) == set(g_paths):
            continue
        # outside the band the sets agree
        keep = [p for p in o_paths if S[p] > cut + TIE]
        assert set(keep) <= set(g_paths)


# ------------------------------------------------------------------ the round
class MarkovRoundCase:
    """ddt_round_markov: the table, the tree, then a4..a7. The synthetic
    target follows the tree the GPU builds (checked stage-wise above)."""

    def __init__(self, cfg):
        self.cfg = cfg
        self.inp = inp = synth.draw_round_inputs(cfg)
        self.W, self.E, self.anchors = synth.draw_markov_head(cfg)
        ctx = self.ctx = make_ctx(cfg, inp)
        R, L, C = cfg.R, cfg.L, cfg.prefilter
        ell, Wd, Ed, an = dev(inp["draft_logits"]), dev(self.W), dev(self.E), dev(self.anchors)
        cand = torch.empty((R, L, C), dtype=torch.int32, device="cuda")
        tab = torch.empty((R, L, C, C), dtype=torch.float32, device="cuda")
        ctx.ddt_markov_table(ell, Wd, Ed, an, R, cand, tab)
        torch.cuda.synchronize()
        self.tree = oracle.markov_tree(host(cand), host(tab).astype(np.float64), cfg.B)
        self.target = synth.GreedyTarget(cfg, inp["draft"], inp["agree"])
        self.target_logits = self.target.logits_for_tree(self.tree.tokens, self.tree.parents,
                                                         self.tree.n_nodes)
        d = {k: dev(inp[k]) for k in ("q", "k_tree", "v_tree", "k_cache", "v_cache",
                                       "block_table", "ctx_lens")}
        d["draft_logits"] = ell
        d["target_logits"] = dev(self.target_logits)
        self.out = ctx.alloc_outputs(R)
        bufs = dict(self.out)
        bufs.update(d)
        ctx.ddt_round_markov(R, bufs, Wd, Ed, an)
        torch.cuda.synchronize()
        self.status = ctx.ddt_device_status()
        self.g = {k: host(v) for k, v in self.out.items()}
        self.g_k_cache = host(d["k_cache"], np.uint16)
        self.g_v_cache = host(d["v_cache"], np.uint16)
        self.g_ctx_lens = host(d["ctx_lens"])


ROUND_CASES = {"small": dict(R=3, L=4, V=3000, B=20, K=20, prefilter=16, seed=51),
               "sparkling": dict()}


@pytest.fixture(scope="module", params=list(ROUND_CASES))
def rcase(request):
    return MarkovRoundCase(synth.config("sparkling", **ROUND_CASES[request.param]))


def test_round_status_and_tree(rcase):
    assert rcase.status == 0
    t, g = rcase.tree, rcase.g
    np.testing.assert_array_equal(g["n_nodes"], t.n_nodes)
    np.testing.assert_array_equal(g["tree_tokens"], t.tokens)
    np.testing.assert_array_equal(g["parents"], t.parents)
    np.testing.assert_array_equal(g["mask"].view(np.uint32), oracle.build_mask(t.parents, t.n_nodes))


def test_round_attention(rcase):
    cfg, inp = rcase.cfg, rcase.inp
    mask = oracle.build_mask(rcase.tree.parents, rcase.tree.n_nodes)
    rng = np.random.default_rng(3)
    sel = np.array([(r, int(rng.integers(0, cfg.P)), int(rng.integers(0, cfg.Hq)))
                    for r in range(cfg.R) for _ in range(6)]
                   + [(r, cfg.P - 1, cfg.Hq - 1) for r in range(cfg.R)], np.int32)
    want, flags = oracle.tree_attention_rows(inp["q"], inp["k_tree"], inp["v_tree"],
                                             inp["k_cache"], inp["v_cache"], inp["block_table"],
                                             inp["ctx_lens"], mask, sel)
    assert flags == 0
    got = rcase.out["attn_out"].float().cpu().numpy()[sel[:, 0], sel[:, 1], sel[:, 2]]
    assert np.abs(got - want).max() <= ATT_TOL


def test_round_accept_walk_compaction(rcase):
    t, g, inp = rcase.tree, rcase.g, rcase.inp
    a, _ = oracle.argmax(rcase.target_logits)
    np.testing.assert_array_equal(g["target_argmax"], a)
    acc_len, acc_nodes, acc_tokens, bonus = oracle.walk(a, t.tokens, t.parents, t.n_nodes,
                                                        rcase.cfg.L)
    np.testing.assert_array_equal(g["acc_len"], acc_len)
    np.testing.assert_array_equal(g["acc_nodes"], acc_nodes)
    np.testing.assert_array_equal(g["acc_tokens"], acc_tokens)
    np.testing.assert_array_equal(g["bonus"], bonus)
    kc, vc, ctx = inp["k_cache"].copy(), inp["v_cache"].copy(), inp["ctx_lens"].copy()
    assert oracle.compact(kc, vc, inp["block_table"], ctx, inp["k_tree"], inp["v_tree"],
                          acc_nodes, acc_len) == 0
    np.testing.assert_array_equal(rcase.g_ctx_lens, ctx)
    assert np.array_equal(rcase.g_k_cache, kc) and np.array_equal(rcase.g_v_cache, vc)
