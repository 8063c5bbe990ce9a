"""ddt_topk_logprobs_noalloc: the top-K entry point for callers that cannot
allocate device memory (its scratch is a fixed array inside libddt.so).

It must give the same result as the context-based ddt_topk_logprobs, call
after call, although every call reuses the same scratch, and the same ids
and log-probs as the oracle. The file's name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import dev, host
from speculative_decoding_draft_depth_gb300 import ddt, synth

pytestmark = pytest.mark.gpu

LP_TOL = 1e-5


def _noalloc():
    fn = ddt.load().ddt_topk_logprobs_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    return fn


def _call_noalloc(z, dtype, rows, V, K):
    lp = torch.full((rows, K), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((rows, K), -7, dtype=torch.int32, device="cuda")
    st = _noalloc()(ctypes.c_void_p(z.data_ptr()), dtype, rows, V, K,
                    ctypes.c_void_p(lp.data_ptr()), ctypes.c_void_p(ids.data_ptr()),
                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ddt.OK, st
    torch.cuda.synchronize()
    return host(lp), host(ids)


def _call_context(z, dtype, R, L, V, K):
    c = ddt.make_config(R_max=R, L=L, V=V, B=K, K=K, Hq=4, Hkv=1, d=64, page_size=16,
                        max_pages_per_req=1, num_pages=1, draft_dtype=dtype)
    ctx = ddt.Context(c)
    lp = torch.empty((R, L, K), dtype=torch.float32, device="cuda")
    ids = torch.empty((R, L, K), dtype=torch.int32, device="cuda")
    ctx.ddt_topk_logprobs(z, R, lp, ids)
    torch.cuda.synchronize()
    out = host(lp).reshape(R * L, K), host(ids).reshape(R * L, K)
    ctx.close()
    return out


@pytest.mark.parametrize("name,overrides,dtype", [
    ("batch64", dict(R=8, seed=71), ddt.BF16),
    ("tiny", dict(R=5, V=20000, seed=72), ddt.F32),
])
def test_noalloc_matches_context_entry_point_on_consecutive_calls(name, overrides, dtype):
    cfg = synth.config(name, **overrides)
    for call in range(2):
        inp = synth.draw_round_inputs(cfg, seed=cfg.seed + call)
        z = dev(inp["draft_logits"])
        rows = cfg.R * cfg.L
        lp, ids = _call_noalloc(z, dtype, rows, cfg.V, cfg.K)
        ref_lp, ref_ids = _call_context(z, dtype, cfg.R, cfg.L, cfg.V, cfg.K)
        np.testing.assert_array_equal(ids, ref_ids)
        assert np.abs(lp - ref_lp).max() <= LP_TOL


def test_noalloc_matches_oracle():
    cfg = synth.config("batch64", R=2, seed=73)
    inp = synth.draw_round_inputs(cfg)
    rows = cfg.R * cfg.L
    lp, ids = _call_noalloc(dev(inp["draft_logits"]), ddt.BF16, rows, cfg.V, cfg.K)
    o_lp, o_ids, _, _ = oracle.topk_logprobs(inp["draft_logits"], cfg.K)
    np.testing.assert_array_equal(ids, o_ids.reshape(rows, cfg.K))
    assert np.abs(lp - o_lp.reshape(rows, cfg.K)).max() <= LP_TOL


def test_noalloc_wide_list_merge():
    # K = 64: more candidates than one warp holds in the row selection
    cfg = synth.config("wide256", R=2, seed=74)
    assert cfg.K == 64
    inp = synth.draw_round_inputs(cfg)
    z = dev(inp["draft_logits"])
    rows = cfg.R * cfg.L
    lp, ids = _call_noalloc(z, ddt.BF16, rows, cfg.V, cfg.K)
    ref_lp, ref_ids = _call_context(z, ddt.BF16, cfg.R, cfg.L, cfg.V, cfg.K)
    np.testing.assert_array_equal(ids, ref_ids)
    assert np.abs(lp - ref_lp).max() <= LP_TOL


def test_noalloc_smaller_call_after_larger_one():
    # the second call must ignore the partial lists and counters the first left
    cfg = synth.config("batch64", R=8, seed=75)
    inp = synth.draw_round_inputs(cfg)
    z = dev(inp["draft_logits"])
    rows = cfg.R * cfg.L
    _call_noalloc(z, ddt.BF16, rows, cfg.V, cfg.K)
    small = dev(synth.draw_round_inputs(synth.config("batch64", R=1, seed=76))["draft_logits"])
    lp, ids = _call_noalloc(small, ddt.BF16, cfg.L, cfg.V, cfg.K)
    ref_lp, ref_ids = _call_context(small, ddt.BF16, 1, cfg.L, cfg.V, cfg.K)
    np.testing.assert_array_equal(ids, ref_ids)
    assert np.abs(lp - ref_lp).max() <= LP_TOL


def test_noalloc_at_its_scratch_limit():
    # rows * chunks exactly DDT_NOALLOC_MAX_ROW_CHUNKS: 4096 rows of 131072
    # bf16 logits (8 chunks) and K = 32; seeded N(0, 3^2) logits
    rows, V, K = 4096, 131072, 32
    g = torch.Generator(device="cuda").manual_seed(77)
    z = (torch.randn((rows, V), generator=g, device="cuda") * 3).to(torch.bfloat16)
    z16 = z.view(torch.int16)
    lp, ids = _call_noalloc(z16, ddt.BF16, rows, V, K)
    ref_lp, ref_ids = _call_context(z16, ddt.BF16, 2048, 2, V, K)
    np.testing.assert_array_equal(ids, ref_ids)
    assert np.abs(lp - ref_lp).max() <= LP_TOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    z = torch.zeros((16,), dtype=torch.int16, device="cuda")
    out = torch.zeros((16,), dtype=torch.int32, device="cuda")
    fn = _noalloc()
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    # more rows than the scratch holds
    assert fn(p(z), ddt.BF16, 4097, 8, 4, p(out), p(out), None) == ddt.EUNSUPPORTED
    # rows * chunks above the scratch: 4096 rows x 10 chunks, and 4096 x 9
    assert fn(p(z), ddt.BF16, 4096, 151936, 32, p(out), p(out), None) == ddt.EUNSUPPORTED
    assert fn(p(z), ddt.BF16, 4096, 131073, 32, p(out), p(out), None) == ddt.EUNSUPPORTED
    assert fn(p(z), ddt.BF16, 1, 8, 9, p(out), p(out), None) == ddt.EINVAL  # K > V
    assert fn(p(z), 5, 1, 8, 4, p(out), p(out), None) == ddt.EINVAL  # unknown dtype
