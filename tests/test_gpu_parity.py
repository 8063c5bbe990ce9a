"""GPU parity: every stage of the round, through the C ABI, against the fp64
CPU oracle on the same seeded inputs.

Tolerances: top-K ids, trees, masks, argmax, acceptance and compaction are
bit-exact; log-probs within 1e-5 absolute; attention within 1e-2 absolute
(bf16 inputs, fp32 accumulation and output). Tree construction is compared
stage-wise (the oracle's heap fed the GPU's fp32 log-probs, must match
bit-for-bit including order) and end to end (oracle fp64 log-probs: prefix
scores within 1e-6 nats count as tied and the tie band must agree).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import RoundCase, check_tie_band, dev, host, make_ctx
from speculative_decoding_draft_depth_gb300 import ddt, synth

pytestmark = pytest.mark.gpu

LP_TOL = 1e-5
ATT_TOL = 1e-2

CASES = {
    "tiny": dict(name="tiny"),
    "tiny_r3": dict(name="tiny", R=3, ctx_kind="uniform", ctx_args=(0, 300), seed=31),
    "single": dict(name="single"),
    "single_ctx0": dict(name="single", V=4096, ctx_args=(0,), seed=51),
    "single_ctx128": dict(name="single", V=4096, ctx_args=(128,), seed=52),
    "mid": dict(name="batch64", R=5, ctx_args=(1, 9000), seed=41),
    "wide_small": dict(name="wide256", R=6, rounds=1, ctx_args=(3000, 1.0, 9000), seed=43),
    # two row groups per KV head at head dim 64 (one run of tiles per row group)
    "wide_d64": dict(name="wide256", R=4, V=4096, d=64, rounds=1, ctx_args=(2000, 1.0, 6000),
                     seed=44),
    # three row groups (P * G = 388 rows): each row-group CTA loads its own K / V
    "rows3": dict(name="wide256", R=3, V=4096, B=96, rounds=1, ctx_args=(1500, 1.0, 4000),
                  seed=45),
}


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    kw = dict(CASES[request.param])
    cfg = synth.config(kw.pop("name"), **kw)
    return RoundCase(cfg)


@pytest.fixture(scope="module")
def full():
    """The 64-request metric workload at full size (R=64, L=15, V=151936, B=32)."""
    return RoundCase(synth.config("batch64"))


def _check_topk(rc):
    np.testing.assert_array_equal(rc.g["top_ids"], rc.o_ids)
    err = np.abs(rc.g["top_lp"].astype(np.float64) - rc.o_lp).max()
    assert err <= LP_TOL, err


def _check_tree_stagewise(rc):
    t = rc.oracle_tree_from_gpu_lp()
    np.testing.assert_array_equal(rc.g["n_nodes"], t.n_nodes)
    np.testing.assert_array_equal(rc.g["tree_tokens"], t.tokens)
    np.testing.assert_array_equal(rc.g["parents"], t.parents)
    np.testing.assert_array_equal(rc.g["depths"], t.depths)
    return t


def _check_tree_tie_band(rc):
    """End-to-end node set: GPU tree (from fp32 lp) vs oracle tree (fp64 lp)."""
    check_tie_band(rc.cfg.B, rc.o_lp, rc.o_ids, rc.o_tree, rc.g["tree_tokens"], rc.g["parents"],
                   rc.g["depths"], rc.g["n_nodes"], range(rc.cfg.R))


def _check_mask(rc, gtree):
    omask = oracle.build_mask(gtree.parents, gtree.n_nodes)
    np.testing.assert_array_equal(rc.g["mask"].view(np.uint32), omask)
    return omask


def _check_attention_rows(rc, mask, sel):
    inp = rc.inp
    want, flags = oracle.tree_attention_rows(inp["q"], inp["k_tree"], inp["v_tree"],
                                             inp["k_cache"], inp["v_cache"], inp["block_table"],
                                             inp["ctx_lens"], mask, sel)
    assert flags == 0
    got = rc.out["attn_out"].float().cpu().numpy()
    g = got[sel[:, 0], sel[:, 1], sel[:, 2]]
    err = np.abs(g - want).max()
    assert err <= ATT_TOL, err


def _check_accept(rc, gtree):
    a, _ = oracle.argmax(rc.target_logits)
    np.testing.assert_array_equal(rc.g["target_argmax"], a)
    acc_len, acc_nodes, acc_tokens, bonus = oracle.walk(a, gtree.tokens, gtree.parents,
                                                        gtree.n_nodes, rc.cfg.L)
    np.testing.assert_array_equal(rc.g["acc_len"], acc_len)
    np.testing.assert_array_equal(rc.g["acc_nodes"], acc_nodes)
    np.testing.assert_array_equal(rc.g["acc_tokens"], acc_tokens)
    np.testing.assert_array_equal(rc.g["bonus"], bonus)
    kc, vc, ctx = rc.inp["k_cache"].copy(), rc.inp["v_cache"].copy(), rc.inp["ctx_lens"].copy()
    flags = oracle.compact(kc, vc, rc.inp["block_table"], ctx, rc.inp["k_tree"], rc.inp["v_tree"],
                           acc_nodes, acc_len)
    assert flags == 0
    np.testing.assert_array_equal(rc.g_ctx_lens, ctx)
    assert np.array_equal(rc.g_k_cache, kc) and np.array_equal(rc.g_v_cache, vc)


# ------------------------------------------------------------------ cases
def test_round_status_clean(case):
    assert case.status == 0


def test_topk_logprobs(case):
    _check_topk(case)


def test_tree_stagewise_bit_exact(case):
    _check_tree_stagewise(case)


def test_tree_end_to_end_tie_band(case):
    _check_tree_tie_band(case)


def test_mask_fused_and_standalone(case):
    gtree = case.oracle_tree_from_gpu_lp()
    omask = _check_mask(case, gtree)
    m2 = torch.empty_like(case.out["mask"])
    case.ctx.ddt_build_mask(case.out["parents"], case.out["n_nodes"], case.cfg.R, m2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(m2).view(np.uint32), omask)


def test_attention_all_rows(case):
    cfg = case.cfg
    gtree = case.oracle_tree_from_gpu_lp()
    mask = oracle.build_mask(gtree.parents, gtree.n_nodes)
    rr, ii, hh = np.meshgrid(np.arange(cfg.R), np.arange(cfg.P), np.arange(cfg.Hq), indexing="ij")
    sel = np.stack([rr.ravel(), ii.ravel(), hh.ravel()], 1).astype(np.int32)
    _check_attention_rows(case, mask, sel)


def test_accept_walk_compaction(case):
    _check_accept(case, case.oracle_tree_from_gpu_lp())


# ------------------------------------------------------------------ full size
def test_full_topk(full):
    assert full.status == 0
    _check_topk(full)


def test_full_tree_and_mask(full):
    t = _check_tree_stagewise(full)
    _check_tree_tie_band(full)
    _check_mask(full, t)


def test_full_attention_sampled(full):
    cfg = full.cfg
    rng = np.random.default_rng(99)
    sel = []
    for r in range(cfg.R):
        for _ in range(3):
            sel.append((r, int(rng.integers(0, cfg.P)), int(rng.integers(0, cfg.Hq))))
        sel.append((r, cfg.P - 1, cfg.Hq - 1))
    gtree = full.oracle_tree_from_gpu_lp()
    mask = oracle.build_mask(gtree.parents, gtree.n_nodes)
    _check_attention_rows(full, mask, np.array(sel, np.int32))


def test_full_accept(full):
    _check_accept(full, full.oracle_tree_from_gpu_lp())


# ------------------------------------------------------------------ edge cases
def _topk_only(V, K, dtype, z, R=1, L=None):
    L = L or z.shape[1]
    c = ddt.make_config(R_max=R, L=L, V=V, B=max(K, 1), K=K, Hq=4, Hkv=1, d=64, page_size=16,
                        max_pages_per_req=4, num_pages=4,
                        draft_dtype=ddt.BF16 if dtype == "bf16" else ddt.F32)
    ctx = ddt.Context(c)
    lp = torch.empty((R, L, K), dtype=torch.float32, device="cuda")
    ids = torch.empty((R, L, K), dtype=torch.int32, device="cuda")
    ctx.ddt_topk_logprobs(dev(z), R, lp, ids)
    torch.cuda.synchronize()
    st = ctx.ddt_device_status()
    return host(lp), host(ids), st


@pytest.mark.parametrize("V,K,dtype,kind", [
    (1001, 32, "bf16", "normal"),      # ragged row length: unaligned rows, scalar path
    (4099, 17, "f32", "normal"),
    (151936, 64, "bf16", "quantized"),  # heavy ties: exact fallback
    (151936, 32, "bf16", "constant"),   # every logit equal
    (70000, 1, "bf16", "normal"),
    (64, 64, "f32", "normal"),          # K = V
    (16384 * 3, 32, "bf16", "normal"),  # exact multiple of the chunk
])
def test_topk_edge_cases(V, K, dtype, kind):
    rng = np.random.default_rng(V + K)
    R, L = 2, 3
    z = rng.standard_normal((R, L, V)).astype(np.float32) * 2
    if kind == "quantized":
        z = np.round(z * 2) / 2
    elif kind == "constant":
        z[:] = 1.5
    zin = synth.to_bf16_bits(z) if dtype == "bf16" else z
    lp, ids, st = _topk_only(V, K, dtype, zin, R=R, L=L)
    assert st == 0
    olp, oids, _, _ = oracle.topk_logprobs(zin, K)
    np.testing.assert_array_equal(ids, oids)
    assert np.abs(lp - olp).max() <= LP_TOL


def test_nan_logits_set_status_without_faulting():
    V, K = 4096, 8
    z = np.random.default_rng(1).standard_normal((1, 2, V)).astype(np.float32)
    z[0, 1, 77] = np.nan
    _, _, st = _topk_only(V, K, "f32", z, R=1, L=2)
    assert st & ddt.DEV_NAN_LOGITS


def test_argmax_edge_cases():
    cfg = synth.config("tiny", V=3001)
    inp = synth.draw_round_inputs(cfg)
    ctx = make_ctx(cfg, inp)
    rng = np.random.default_rng(3)
    t = rng.integers(-3, 4, size=(1, cfg.P, cfg.V)).astype(np.float32)  # many ties
    t[0, 0, :] = -0.0
    t[0, 0, 5] = 0.0
    t[0, 1, :] = -np.inf
    out = torch.empty((1, cfg.P), dtype=torch.int32, device="cuda")
    ctx.ddt_target_argmax(dev(t), 1, out)
    torch.cuda.synchronize()
    want, _ = oracle.argmax(t)
    np.testing.assert_array_equal(host(out), want)
    assert ctx.ddt_device_status() == 0


@pytest.mark.parametrize("name,overrides", [("tiny", dict(R=2)),
                                            ("batch64", dict(R=2, V=2048, ctx_args=(600, 900)))])
def test_bad_page_sets_status_without_faulting(name, overrides):
    cfg = synth.config(name, **overrides)
    inp = synth.draw_round_inputs(cfg)
    bt = inp["block_table"].copy()
    bt[1, 2] = 10 ** 7
    inp["block_table"] = bt
    ctx = make_ctx(cfg, inp)
    lp, ids, _, _ = oracle.topk_logprobs(inp["draft_logits"], cfg.K)
    t = oracle.build_tree(lp, ids, cfg.B)
    mask = oracle.build_mask(t.parents, t.n_nodes)
    out = torch.empty((cfg.R, cfg.P, cfg.Hq, cfg.d), dtype=torch.float32, device="cuda")
    ctx.ddt_tree_attention(dev(inp["q"]), dev(inp["k_tree"]), dev(inp["v_tree"]),
                           dev(inp["k_cache"]), dev(inp["v_cache"]), dev(bt), dev(inp["ctx_lens"]),
                           dev(mask), cfg.R, out)
    torch.cuda.synchronize()
    assert ctx.ddt_device_status() & ddt.DEV_BAD_PAGE
    # request 0 is untouched by the bad entry and still matches the oracle
    sel = np.array([(0, i, h) for i in range(cfg.P) for h in range(cfg.Hq)], np.int32)
    want, _ = oracle.tree_attention_rows(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"],
                                         inp["v_cache"], bt, inp["ctx_lens"], mask, sel)
    got = out.float().cpu().numpy()[0].reshape(-1, cfg.d)
    assert np.abs(got - want).max() <= ATT_TOL


def test_invalid_arguments_are_rejected_before_launch():
    cfg = synth.config("tiny")
    inp = synth.draw_round_inputs(cfg)
    ctx = make_ctx(cfg, inp)
    z = dev(inp["draft_logits"])
    lp = torch.empty((1, cfg.L, cfg.K), dtype=torch.float32, device="cuda")
    ids = torch.empty((1, cfg.L, cfg.K), dtype=torch.int32, device="cuda")
    with pytest.raises(ddt.DdtError) as e:
        ctx.ddt_topk_logprobs(z, 2, lp, ids)  # R > R_max
    assert e.value.status == ddt.EINVAL
    raw = torch.empty(z.numel() + 1, dtype=torch.float32, device="cuda")
    with pytest.raises(ddt.DdtError):
        ctx.ddt_topk_logprobs(raw[1:], 1, lp, ids)  # misaligned logits pointer
    ctx.ddt_topk_logprobs(z, 0, lp, ids)  # R = 0 is a no-op


def test_misaligned_element_pointers_are_rejected_before_launch():
    """An i32, f32 or f64 array off its element alignment is rejected with
    DDT_EINVAL before anything is enqueued. Every pointer lies inside one
    buffer owned by the test, far from its ends."""
    cfg = synth.config("tiny")  # R = 1, L = 4, V = 32
    inp = synth.draw_round_inputs(cfg)
    ctx = make_ctx(cfg, inp)
    lib = ddt.load()
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")

    def at(off):
        return ctypes.c_void_p(buf.data_ptr() + (1 << 16) + off)

    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # scheduler: conf two bytes off; then f64 stats four bytes off
    assert lib.ddt_schedule_prefix(ctx._h, at(2), 1, at(4096), at(8192), None, None, s) == ddt.EINVAL
    assert lib.ddt_schedule_prefix(ctx._h, at(0), 1, at(4096), at(8192), at(12288), at(16388),
                                   s) == ddt.EINVAL
    # stochastic verification: the guesses two bytes off
    assert lib.ddt_accept_stochastic(ctx._h, at(0), at(4096), at(8194), at(12288), at(16384), 1,
                                     at(20480), at(24576), None, s) == ddt.EINVAL
    # greedy walk: acc_len one byte off
    assert lib.ddt_walk(ctx._h, at(0), at(4096), at(8192), at(12288), 1, at(16385), at(20480),
                        at(24576), at(28672), s) == ddt.EINVAL
    assert ctx.ddt_device_status() == 0


def test_chain_tree_attention_is_causal_decode():
    """K=1, B=L: the chain's attention equals plain causal attention (torch SDPA)."""
    cfg = synth.config("batch64", R=2, K=1, B=15, V=4096, ctx_args=(100, 700), seed=8)
    rc = RoundCase(cfg)
    assert list(rc.g["parents"][0]) == list(range(-1, 15))
    inp = rc.inp
    got = rc.out["attn_out"].float()
    for r in range(cfg.R):
        ctx = int(inp["ctx_lens"][r])
        idx = np.arange(ctx)
        pg = inp["block_table"][r, idx // cfg.page]
        kc = np.concatenate([inp["k_cache"][pg, idx % cfg.page], inp["k_tree"][r]], 0)
        vc = np.concatenate([inp["v_cache"][pg, idx % cfg.page], inp["v_tree"][r]], 0)
        q = dev(inp["q"][r]).view(torch.bfloat16).float().permute(1, 0, 2)
        k = dev(kc).view(torch.bfloat16).float().permute(1, 0, 2).repeat_interleave(4, 0)
        v = dev(vc).view(torch.bfloat16).float().permute(1, 0, 2).repeat_interleave(4, 0)
        n = cfg.P
        allowed = torch.ones(n, ctx + n, dtype=torch.bool, device="cuda")
        allowed[:, ctx:] = torch.tril(torch.ones(n, n, dtype=torch.bool, device="cuda"))
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed)
        assert (got[r] - ref.permute(1, 0, 2)).abs().max().item() <= ATT_TOL
