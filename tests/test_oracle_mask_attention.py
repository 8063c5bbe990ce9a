"""Pins for the oracle's ancestor mask (a3) and tree attention (a4).

Mask: every row equals the set of positions on the node's root path, found
by walking parent pointers; popcount = depth + 1.
Attention: along every root-to-leaf path, tree attention equals ordinary
causal attention over context + path computed by torch's
scaled_dot_product_attention in float64; a chain tree (K=1, B=L) is plain
causal decode attention; paging does not change the result.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_draft_depth_gb300 import synth


def _tree(orc, cfg, inp):
    lp, ids, _, _ = orc.topk_logprobs(inp["draft_logits"], cfg.K)
    return orc.build_tree(lp, ids, cfg.B)


def test_mask_hand_example(orc):
    # root 0; 1 under 0; 2 under 1; 3 under 1; 4 under 0
    parents = np.array([[-1, 0, 1, 1, 0]], np.int32)
    mask = orc.build_mask(parents, np.array([4], np.int32))
    rows = [int(w) for w in mask[0, :, 0]]
    assert rows == [0b00001, 0b00011, 0b00111, 0b01011, 0b10001]


@pytest.mark.parametrize("name,overrides", [("tiny", {}), ("single", {"V": 2048}),
                                            ("wide256", {"R": 3, "V": 2048, "rounds": 1})])
def test_mask_rows_are_root_paths(orc, name, overrides):
    cfg = synth.config(name, **overrides)
    inp = synth.draw_round_inputs(cfg)
    t = _tree(orc, cfg, inp)
    mask = orc.build_mask(t.parents, t.n_nodes)
    P, W = cfg.P, cfg.W
    assert mask.shape == (cfg.R, P, W)
    for r in range(cfg.R):
        for i in range(P):
            bits = {w * 32 + b for w in range(W) for b in range(32) if (int(mask[r, i, w]) >> b) & 1}
            if i > t.n_nodes[r]:
                assert bits == set()
                continue
            path, cur = set(), i
            while cur >= 0:
                path.add(cur)
                cur = int(t.parents[r, cur])
            assert bits == path
            assert len(bits) == t.depths[r, i] + 1


def _bf(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(torch.float64)


def _gather_ctx(kc, block_table, r, ctx, page):
    idx = np.arange(ctx)
    pg = block_table[r, idx // page]
    return kc[pg, idx % page]  # [ctx, Hkv, d]


def _sdpa_causal_rows(q_rows, k_seq, v_seq, n_ctx, Hq, Hkv):
    """q_rows [n, Hq, d] are the last n positions of a causal sequence whose
    keys/values are k_seq/v_seq [n_ctx + n, Hkv, d]."""
    n = q_rows.shape[0]
    group = Hq // Hkv
    q = _bf(q_rows).permute(1, 0, 2)  # [Hq, n, d]
    k = _bf(k_seq).permute(1, 0, 2).repeat_interleave(group, 0)
    v = _bf(v_seq).permute(1, 0, 2).repeat_interleave(group, 0)
    S = n_ctx + n
    allowed = torch.ones(n, S, dtype=torch.bool)
    allowed[:, n_ctx:] = torch.tril(torch.ones(n, n, dtype=torch.bool))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed)
    return o.permute(1, 0, 2).numpy()  # [n, Hq, d]


@pytest.mark.parametrize("name,overrides", [("tiny", {}),
                                            ("tiny", {"Hq": 4, "Hkv": 2, "B": 12, "seed": 9}),
                                            ("single", {"V": 1024, "Hq": 8, "Hkv": 2, "d": 64,
                                                        "ctx_args": (200,)})])
def test_tree_attention_equals_causal_attention_on_every_path(orc, name, overrides):
    cfg = synth.config(name, **overrides)
    inp = synth.draw_round_inputs(cfg)
    t = _tree(orc, cfg, inp)
    mask = orc.build_mask(t.parents, t.n_nodes)
    out, flags = orc.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"],
                                    inp["v_cache"], inp["block_table"], inp["ctx_lens"], mask)
    assert flags == 0
    r = 0
    n = t.n_nodes[r]
    children = {i: [] for i in range(n + 1)}
    for i in range(1, n + 1):
        children[int(t.parents[r, i])].append(i)
    leaves = [i for i in range(n + 1) if not children[i]]
    ctx = int(inp["ctx_lens"][r])
    kc = _gather_ctx(inp["k_cache"], inp["block_table"], r, ctx, cfg.page)
    vc = _gather_ctx(inp["v_cache"], inp["block_table"], r, ctx, cfg.page)
    for leaf in leaves:
        path, cur = [], leaf
        while cur >= 0:
            path.append(cur)
            cur = int(t.parents[r, cur])
        path = path[::-1]  # root first
        kseq = np.concatenate([kc, inp["k_tree"][r, path]], 0)
        vseq = np.concatenate([vc, inp["v_tree"][r, path]], 0)
        ref = _sdpa_causal_rows(inp["q"][r, path], kseq, vseq, ctx, cfg.Hq, cfg.Hkv)
        np.testing.assert_allclose(out[r, path], ref, rtol=0, atol=1e-12)


def test_chain_tree_is_plain_causal_decode(orc):
    # K=1, B=L: the tree is the top-1 chain, positions in depth order
    cfg = synth.config("tiny", K=1, B=4, seed=3)
    inp = synth.draw_round_inputs(cfg)
    t = _tree(orc, cfg, inp)
    assert list(t.parents[0]) == [-1, 0, 1, 2, 3]
    mask = orc.build_mask(t.parents, t.n_nodes)
    out, _ = orc.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"],
                                inp["v_cache"], inp["block_table"], inp["ctx_lens"], mask)
    ctx = int(inp["ctx_lens"][0])
    kc = _gather_ctx(inp["k_cache"], inp["block_table"], 0, ctx, cfg.page)
    vc = _gather_ctx(inp["v_cache"], inp["block_table"], 0, ctx, cfg.page)
    kseq = np.concatenate([kc, inp["k_tree"][0]], 0)
    vseq = np.concatenate([vc, inp["v_tree"][0]], 0)
    ref = _sdpa_causal_rows(inp["q"][0], kseq, vseq, ctx, cfg.Hq, cfg.Hkv)
    np.testing.assert_allclose(out[0], ref, atol=1e-12)


def test_paging_does_not_change_attention(orc):
    cfg = synth.config("tiny", R=2, ctx_kind="uniform", ctx_args=(1, 70), seed=21)
    inp = synth.draw_round_inputs(cfg)
    t = _tree(orc, cfg, inp)
    mask = orc.build_mask(t.parents, t.n_nodes)
    a, _ = orc.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"],
                              inp["v_cache"], inp["block_table"], inp["ctx_lens"], mask)
    # relocate every page to a new, reversed pool
    bt = inp["block_table"]
    used = bt[bt >= 0]
    npages = inp["k_cache"].shape[0]
    new_index = np.arange(npages)[::-1].copy()
    kc2 = np.empty_like(inp["k_cache"])
    vc2 = np.empty_like(inp["v_cache"])
    kc2[new_index] = inp["k_cache"]
    vc2[new_index] = inp["v_cache"]
    bt2 = np.where(bt >= 0, new_index[np.maximum(bt, 0)], -1).astype(np.int32)
    assert used.size > 0
    b, _ = orc.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], kc2, vc2, bt2,
                              inp["ctx_lens"], mask)
    np.testing.assert_array_equal(a, b)


def test_bad_page_is_flagged(orc):
    cfg = synth.config("tiny")
    inp = synth.draw_round_inputs(cfg)
    t = _tree(orc, cfg, inp)
    mask = orc.build_mask(t.parents, t.n_nodes)
    bt = inp["block_table"].copy()
    bt[0, 1] = 10 ** 6
    _, flags = orc.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"],
                                  inp["v_cache"], bt, inp["ctx_lens"], mask)
    assert flags & orc.BAD_PAGE
