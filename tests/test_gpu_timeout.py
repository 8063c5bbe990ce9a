"""Failure detection on the GPU without a fault: the a4 kernel's bounded wait.

A test-only setting arms the next attention launch so that every CTA first
waits, with a short limit, on an on-chip barrier that nothing arrives at. The
wait must run out, the kernel must report DDT_DEV_TIMEOUT through the device
status word and wind down (no copy or MMA was issued), and the same context's
next launch must be normal and match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import RoundCase, dev
from speculative_decoding_draft_depth_gb300 import ddt, synth

pytestmark = pytest.mark.gpu

ATT_TOL = 1e-2
WAIT_CYCLES = 2_000_000  # about 1 ms at the SM clock


@pytest.mark.parametrize("name,overrides", [
    ("tiny", {}),                                                          # head dim 64
    ("batch64", dict(R=2, V=4096, ctx_args=(100, 700), seed=9)),           # head dim 128
])
def test_attention_wait_runs_out_and_context_recovers(name, overrides):
    cfg = synth.config(name, **overrides)
    rc = RoundCase(cfg)
    assert rc.status == 0
    inp = rc.inp
    gtree = rc.oracle_tree_from_gpu_lp()
    omask = oracle.build_mask(gtree.parents, gtree.n_nodes)
    d = {k: dev(inp[k]) for k in ("q", "k_tree", "v_tree", "k_cache", "v_cache", "block_table",
                                   "ctx_lens")}
    mask = dev(omask.view(np.int32))
    out = torch.empty_like(rc.out["attn_out"])
    ctx = rc.ctx

    def attend():
        ctx.ddt_tree_attention(d["q"], d["k_tree"], d["v_tree"], d["k_cache"], d["v_cache"],
                               d["block_table"], d["ctx_lens"], mask, cfg.R, out)

    ctx.ddt_debug_arm_attention_timeout(WAIT_CYCLES)
    attend()
    assert ctx.ddt_device_status() == ddt.DEV_TIMEOUT

    # the setting was one-shot: the next launch is normal and correct
    out.fill_(float("nan"))
    attend()
    assert ctx.ddt_device_status() == 0
    sel = np.array([(r, i, h) for r in range(cfg.R) for i in range(cfg.P) for h in range(cfg.Hq)],
                   np.int32)
    want, flags = oracle.tree_attention_rows(inp["q"], inp["k_tree"], inp["v_tree"],
                                             inp["k_cache"], inp["v_cache"], inp["block_table"],
                                             inp["ctx_lens"], omask, sel)
    assert flags == 0
    got = out.float().cpu().numpy()[sel[:, 0], sel[:, 1], sel[:, 2]]
    assert np.abs(got - want).max() <= ATT_TOL


def test_disarming_leaves_the_launch_normal():
    cfg = synth.config("tiny")
    rc = RoundCase(cfg)
    ctx = rc.ctx
    ctx.ddt_debug_arm_attention_timeout(WAIT_CYCLES)
    ctx.ddt_debug_arm_attention_timeout(0)  # disarm
    inp = rc.inp
    gtree = rc.oracle_tree_from_gpu_lp()
    omask = oracle.build_mask(gtree.parents, gtree.n_nodes)
    d = {k: dev(inp[k]) for k in ("q", "k_tree", "v_tree", "k_cache", "v_cache", "block_table",
                                   "ctx_lens")}
    out = torch.empty_like(rc.out["attn_out"])
    ctx.ddt_tree_attention(d["q"], d["k_tree"], d["v_tree"], d["k_cache"], d["v_cache"],
                           d["block_table"], d["ctx_lens"], dev(omask.view(np.int32)), cfg.R, out)
    assert ctx.ddt_device_status() == 0
