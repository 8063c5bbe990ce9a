"""Shared plumbing for the GPU parity tests: host<->device copies and one
full round through the C ABI, with the oracle's stage results beside it.

Inputs come from the seeded generators only. The target logits are built
from the ORACLE's tree, never from the GPU's, and every oracle call gets
host arrays that the generators (or an earlier oracle step) produced --
except in the stage-wise comparisons, where the oracle is deliberately fed
the GPU's fp32 log-probs to check the next stage bit-exactly.
"""
import numpy as np
import torch

import oracle
from speculative_decoding_draft_depth_gb300 import ddt, synth


def dev(a, device="cuda"):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(device)


def host(t, dtype=None):
    a = t.detach().cpu()
    if a.dtype == torch.bfloat16:
        a = a.view(torch.int16)
    a = a.numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def make_ctx(cfg, inp, R_max=None):
    c = ddt.make_config(
        R_max=R_max or cfg.R, L=cfg.L, V=cfg.V, B=cfg.B, K=cfg.K, Hq=cfg.Hq, Hkv=cfg.Hkv, d=cfg.d,
        page_size=cfg.page, max_pages_per_req=inp["block_table"].shape[1],
        num_pages=inp["k_cache"].shape[0],
        draft_dtype=ddt.BF16 if cfg.logit_dtype == "bf16" else ddt.F32,
        target_dtype=ddt.BF16 if cfg.logit_dtype == "bf16" else ddt.F32,
        markov_dim=cfg.markov_dim, frontier=cfg.frontier, prefilter=cfg.prefilter)
    return ddt.Context(c)


class RoundCase:
    """One round on the GPU (ddt_round) and the oracle's view of it."""

    def __init__(self, cfg, seed=None):
        self.cfg = cfg
        self.inp = inp = synth.draw_round_inputs(cfg, seed)
        # oracle: fp64 log-probs and its own tree; the target follows that tree
        self.o_lp, self.o_ids, self.o_logz, _ = oracle.topk_logprobs(inp["draft_logits"], cfg.K)
        self.o_tree = oracle.build_tree(self.o_lp, self.o_ids, cfg.B)
        self.target = synth.GreedyTarget(cfg, inp["draft"], inp["agree"])
        self.target_logits = self.target.logits_for_tree(self.o_tree.tokens, self.o_tree.parents,
                                                         self.o_tree.n_nodes)
        self.ctx = make_ctx(cfg, inp)
        d = self.d = {k: dev(inp[k]) for k in ("draft_logits", "q", "k_tree", "v_tree", "k_cache",
                                                 "v_cache", "block_table", "ctx_lens")}
        d["target_logits"] = dev(self.target_logits)
        self.out = self.ctx.alloc_outputs(cfg.R)
        bufs = dict(self.out)
        bufs.update(d)
        self.ctx.ddt_round(cfg.R, bufs)
        torch.cuda.synchronize()
        self.status = self.ctx.ddt_device_status()
        self.g = {k: host(v) for k, v in self.out.items()}
        self.g_k_cache = host(d["k_cache"], np.uint16)
        self.g_v_cache = host(d["v_cache"], np.uint16)
        self.g_ctx_lens = host(d["ctx_lens"])

    # stage-wise oracle results (fed the GPU's own upstream outputs)
    def oracle_tree_from_gpu_lp(self):
        return oracle.build_tree(self.g["top_lp"].astype(np.float64), self.g["top_ids"],
                                 self.cfg.B)


# ------------------------------------------------------------------ tree checks
TIE_EPS = 1e-6


def prefix_scores(lp, ids, tokens, parents, depths, n):
    """S of each node of one tree, recomputed from its token paths (rank lookup)."""
    S = np.zeros(len(parents))
    for node in range(1, n + 1):
        d = depths[node] - 1
        rank = int(np.nonzero(ids[d] == tokens[node - 1])[0][0])
        S[node] = S[parents[node]] + lp[d, rank]
    return S


def tree_paths(tokens, parents, n):
    paths = {0: ()}
    for node in range(1, n + 1):
        paths[node] = paths[int(parents[node])] + (int(tokens[node - 1]),)
    return [paths[i] for i in range(1, n + 1)]


def check_tie_band(B, o_lp, o_ids, otree, g_tokens, g_parents, g_depths, g_n_nodes, rows):
    """End-to-end node set of the GPU tree (built from fp32 log-probs) against
    the oracle's (fp64): prefix scores within TIE_EPS nats of the B-th count as
    tied. Every prefix above the band must be present and none below it; the
    band is compared as a set: the GPU's tied nodes must all belong to the
    oracle's full band (every prefix within TIE_EPS of the B-th score, the ones
    the heap selected and the ones it left behind), and both trees take the
    same number of them."""
    for r in rows:
        n = int(otree.n_nodes[r])
        assert int(g_n_nodes[r]) == n
        So = otree.S[r, 1:n + 1]
        Sg = prefix_scores(o_lp[r], o_ids[r], g_tokens[r], g_parents[r], g_depths[r], n)[1:]
        if n < B:  # the whole prefix space: identical sets
            assert sorted(So) == sorted(Sg)
            continue
        SB = So.min()
        paths_o = tree_paths(otree.tokens[r], otree.parents[r], n)
        paths_g = tree_paths(g_tokens[r], g_parents[r], n)
        sure_o = {p for p, s in zip(paths_o, So) if s > SB + TIE_EPS}
        assert sure_o <= set(paths_g)
        assert all(s >= SB - TIE_EPS for s in Sg)
        band_o = {p for p, s in zip(paths_o, So) if abs(s - SB) <= TIE_EPS}
        band_g = {p for p, s in zip(paths_g, Sg) if abs(s - SB) <= TIE_EPS}
        band_all = {p for p, s in oracle.prefixes_at_least(o_lp[r], o_ids[r], SB - TIE_EPS)
                    if s <= SB + TIE_EPS}
        assert band_o <= band_all and band_g <= band_all
        assert len(band_o) == len(band_g)
