"""GPU parity of the wide workload at full size over consecutive rounds:
R=256 requests, B=K=64 (P=65), lognormal contexts up to 32768, 8 rounds with
compaction in between (the context lengths grow by each round's accepted
length, new draft logits and tree K/V every round).

Every round is checked against the oracle on the same seeded inputs: top-K
ids and log-probs (1e-5), trees stage-wise (bit-exact, oracle fed the GPU's
fp32 log-probs) and with the tie band end to end, the mask, attention on
sampled rows (1e-2), the argmax, the walk, and the compaction: the context
lengths and every cache row the round wrote, against the oracle's own
compaction of a host mirror of the cache.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_tie_band, dev, host, make_ctx
from speculative_decoding_draft_depth_gb300 import synth

pytestmark = pytest.mark.gpu

LP_TOL = 1e-5
ATT_TOL = 1e-2


def _check_round(cfg, k, inp, kc_host, vc_host, ctx_host, g):
    # a1
    o_lp, o_ids, _, _ = oracle.topk_logprobs(inp["draft_logits"], cfg.K)
    np.testing.assert_array_equal(g["top_ids"], o_ids)
    err = np.abs(g["top_lp"].astype(np.float64) - o_lp).max()
    assert err <= LP_TOL, (k, err)
    # a2 stage-wise (bit-exact) and a3
    t = oracle.build_tree(g["top_lp"].astype(np.float64), g["top_ids"], cfg.B)
    np.testing.assert_array_equal(g["n_nodes"], t.n_nodes)
    np.testing.assert_array_equal(g["tree_tokens"], t.tokens)
    np.testing.assert_array_equal(g["parents"], t.parents)
    np.testing.assert_array_equal(g["depths"], t.depths)
    mask = oracle.build_mask(t.parents, t.n_nodes)
    np.testing.assert_array_equal(g["mask"].view(np.uint32), mask)
    # a2 end to end: the node set agrees with the fp64 tree up to the tie band
    ot = oracle.build_tree(o_lp, o_ids, cfg.B)
    check_tie_band(cfg.B, o_lp, o_ids, ot, g["tree_tokens"], g["parents"], g["depths"],
                   g["n_nodes"], range(cfg.R))
    # a4 on sampled rows (2 per request, the tail position among them)
    rng = np.random.default_rng(1000 + k)
    sel = []
    for r in range(cfg.R):
        sel.append((r, int(rng.integers(0, cfg.P)), int(rng.integers(0, cfg.Hq))))
        sel.append((r, cfg.P - 1, int(rng.integers(0, cfg.Hq))))
    sel = np.array(sel, np.int32)
    want, flags = oracle.tree_attention_rows(inp["q"], inp["k_tree"], inp["v_tree"], kc_host,
                                             vc_host, inp["block_table"], ctx_host, mask, sel)
    assert flags == 0
    got = g["attn_out"][sel[:, 0], sel[:, 1], sel[:, 2]]
    assert np.abs(got - want).max() <= ATT_TOL, k
    return t


def test_wide256_eight_rounds():
    cfg = synth.config("wide256")
    inp = synth.draw_round_inputs(cfg)
    ctx = make_ctx(cfg, inp)
    # host mirror of the cache and context lengths (the oracle compacts it)
    kc_host, vc_host = inp["k_cache"], inp["v_cache"]
    ctx_host = inp["ctx_lens"].copy()
    d = {k: dev(inp[k]) for k in ("k_cache", "v_cache", "block_table", "ctx_lens")}
    out = ctx.alloc_outputs(cfg.R)
    page = cfg.page
    for k in range(cfg.rounds):
        if k > 0:
            nxt = synth.draw_next_round(cfg, k)
            nxt["block_table"] = inp["block_table"]
            inp = nxt
        # the target follows the oracle's fp64 tree of this round
        o_lp, o_ids, _, _ = oracle.topk_logprobs(inp["draft_logits"], cfg.K)
        otree = oracle.build_tree(o_lp, o_ids, cfg.B)
        target = synth.GreedyTarget(cfg, inp["draft"], inp["agree"], seed=cfg.seed + 1000 * k)
        tl = target.logits_for_tree(otree.tokens, otree.parents, otree.n_nodes)
        bufs = dict(out)
        bufs.update(d)
        for name in ("draft_logits", "q", "k_tree", "v_tree"):
            bufs[name] = dev(inp[name])
        bufs["target_logits"] = dev(tl)
        ctx.ddt_round(cfg.R, bufs)
        torch.cuda.synchronize()
        assert ctx.ddt_device_status() == 0, k
        g = {name: host(v) for name, v in out.items()}
        g["attn_out"] = out["attn_out"].cpu().numpy()
        del bufs["target_logits"]
        t = _check_round(cfg, k, inp, kc_host, vc_host, ctx_host, g)
        # a5..a7
        a, _ = oracle.argmax(tl)
        del tl
        np.testing.assert_array_equal(g["target_argmax"], a)
        acc_len, acc_nodes, acc_tokens, bonus = oracle.walk(a, t.tokens, t.parents, t.n_nodes,
                                                            cfg.L)
        np.testing.assert_array_equal(g["acc_len"], acc_len)
        np.testing.assert_array_equal(g["acc_nodes"], acc_nodes)
        np.testing.assert_array_equal(g["acc_tokens"], acc_tokens)
        np.testing.assert_array_equal(g["bonus"], bonus)
        before = ctx_host.copy()
        flags = oracle.compact(kc_host, vc_host, inp["block_table"], ctx_host, inp["k_tree"],
                               inp["v_tree"], acc_nodes, acc_len)
        assert flags == 0
        np.testing.assert_array_equal(host(d["ctx_lens"]), ctx_host)
        # every row this round wrote: slots before[r] .. before[r] + acc_len[r] - 1
        pages, offs = [], []
        for r in range(cfg.R):
            for slot in range(int(before[r]), int(before[r]) + int(acc_len[r])):
                pages.append(int(inp["block_table"][r, slot // page]))
                offs.append(slot % page)
        pi = torch.tensor(pages, device="cuda", dtype=torch.long)
        oi = torch.tensor(offs, device="cuda", dtype=torch.long)
        gk = host(d["k_cache"][pi, oi], np.uint16)
        gv = host(d["v_cache"][pi, oi], np.uint16)
        np.testing.assert_array_equal(gk, kc_host[pages, offs])
        np.testing.assert_array_equal(gv, vc_host[pages, offs])
