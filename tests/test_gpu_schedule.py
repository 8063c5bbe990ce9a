"""The hardware-aware prefix scheduler on the GPU ("DSpark Speculative
Decoding Explained: Block Drafting and Confidence Checks", "Survival
probability" and "Picking the budget") through the C ABI, against the
oracle.

The survivals and their ranking are the same bits on both sides; only the
running sums of the ranked survivals are added in another order. So the
kept guesses must match exactly, except when two budgets give tokens per ms
within 1e-12 of each other (an fp64 tie): then the GPU's choice must score
the oracle's best within that band."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_depth_gb300 import ddt, synth
from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu

TIE = 1e-12


def sched_ctx(R_max, L):
    c = ddt.make_config(R_max=R_max, L=L, V=64, B=8, K=8, Hq=4, Hkv=1, d=64, page_size=16,
                        max_pages_per_req=1, num_pages=1)
    return ddt.Context(c)


def costs(kind, R, N, rng):
    n = np.arange(N + 1, dtype=np.float64)
    if kind == "toy":  # the page's toy: 25 ms plus 0.1 ms per token checked
        c = 25.0 + 0.1 * (R + n)
    elif kind == "flat":
        c = np.full(N + 1, 3.0)
    elif kind == "steep":
        c = 1.0 + 2.0 * n
    elif kind == "convex":
        c = 5.0 + 0.05 * n + 0.004 * n ** 2
    elif kind == "random":
        c = rng.uniform(0.5, 2.0, size=N + 1)
    elif kind == "holes":
        c = np.where(rng.random(N + 1) < 0.3, -1.0, rng.uniform(1.0, 3.0, size=N + 1))
    else:
        raise ValueError(kind)
    return c.astype(np.float32)


def run_gpu(ctx, conf, cost, R=None):
    R = conf.shape[0] if R is None else R
    n_keep = torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda")
    n_total = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    stats = torch.zeros(2, dtype=torch.float64, device="cuda")
    ctx.ddt_schedule_prefix(dev(conf), R, dev(cost), n_keep, n_total, stats)
    torch.cuda.synchronize()
    return host(n_keep), int(host(n_total)[0]), host(stats), ctx.ddt_device_status()


def check(conf, cost, g_keep, g_n, g_stats):
    o_keep, o_n, o_theta, o_tok, _ = oracle.schedule_prefix(conf, cost)
    if g_n == o_n and np.array_equal(g_keep, o_keep):
        assert g_stats[0] == pytest.approx(o_theta, rel=TIE)
        assert g_stats[1] == pytest.approx(o_tok, rel=TIE)
        return "exact"
    # an fp64 tie between budgets: the GPU's set must score the best
    s = np.cumprod(np.clip(np.nan_to_num(conf.astype(np.float64), nan=0.0), 0, 1), axis=1)
    assert (g_keep >= 0).all() and (g_keep <= conf.shape[1]).all() and g_keep.sum() == g_n
    tokens = conf.shape[0] + sum(s[r, :g_keep[r]].sum() for r in range(conf.shape[0]))
    assert tokens / float(cost[g_n]) == pytest.approx(o_theta, rel=TIE)
    return "tie"


SHAPES = [(1, 1), (3, 5), (16, 5), (128, 5), (64, 15), (100, 7), (1500, 1), (1024, 3), (512, 16),
          (2048, 4)]  # both kernels: the rank-counting grid, and the bitonic sort (2048 x 4)
KINDS = ["toy", "flat", "steep", "convex", "random", "holes"]


@pytest.mark.parametrize("R,L", SHAPES)
def test_schedule_matches_oracle(R, L):
    rng = np.random.default_rng(R * 100 + L)
    conf = synth.draw_confidences(R, L, seed=R + L)
    ctx = sched_ctx(R, L)
    kinds = []
    for kind in KINDS:
        cost = costs(kind, R, R * L, rng)
        g_keep, g_n, g_stats, st = run_gpu(ctx, conf, cost)
        assert st == 0
        kinds.append(check(conf, cost, g_keep, g_n, g_stats))
    assert kinds.count("tie") <= 1, kinds


def test_level_survivals_and_exact_ties():
    """Many equal survivals (chances of 1 and repeated rows) and zero
    survivals: the ranking's tie order decides which requests keep a guess."""
    R, L = 40, 6
    rng = np.random.default_rng(5)
    conf = np.repeat(rng.choice([0.5, 1.0, 0.8], size=(4, L)).astype(np.float32), 10, axis=0)
    conf[::7, 3] = 0.0
    ctx = sched_ctx(R, L)
    for n_want in [1, 5, 17, 59, 120, 200]:
        cost = np.full(R * L + 1, 1e30, np.float32)
        cost[n_want] = 1.0
        g_keep, g_n, g_stats, st = run_gpu(ctx, conf, cost)
        o_keep, o_n, *_ = oracle.schedule_prefix(conf, cost)
        assert g_n == o_n == n_want
        np.testing.assert_array_equal(g_keep, o_keep)


def test_edge_cases():
    ctx = sched_ctx(8, 4)
    conf = synth.draw_confidences(8, 4, seed=3)
    # no valid cost: nothing is verified
    g_keep, g_n, g_stats, st = run_gpu(ctx, conf, np.full(33, -1.0, np.float32))
    assert g_n == 0 and (g_keep == 0).all() and g_stats[0] == 0.0 and g_stats[1] == 8.0
    # fewer requests than capacity
    g_keep, g_n, g_stats, st = run_gpu(ctx, conf[:5], costs("toy", 5, 20, None))
    check(conf[:5], costs("toy", 5, 20, None), g_keep[:5], g_n, g_stats)
    # R = 0 enqueues nothing
    g_keep, g_n, g_stats, st = run_gpu(ctx, conf, costs("toy", 8, 32, None), R=0)
    assert g_n == -7 and (g_keep == -7).all()
    # NaN and out-of-range confidences: clamped, NaN counted as 0 and reported
    bad = conf.copy()
    bad[1, 0] = np.nan
    bad[2, 1] = 1.5
    bad[3, 2] = -0.5
    cost = np.full(33, 2.0, np.float32)
    g_keep, g_n, g_stats, st = run_gpu(ctx, bad, cost)
    assert st & ddt.DEV_NAN_LOGITS
    o_keep, o_n, *_ = oracle.schedule_prefix(bad, cost)
    np.testing.assert_array_equal(g_keep, o_keep)
    assert g_keep[1] == 0


def test_optional_outputs_and_limits():
    ctx = sched_ctx(4, 3)
    conf = synth.draw_confidences(4, 3, seed=9)
    cost = costs("toy", 4, 12, None)
    n_keep = torch.empty(4, dtype=torch.int32, device="cuda")
    ctx.ddt_schedule_prefix(dev(conf), 4, dev(cost), n_keep)  # no n_total, no stats
    torch.cuda.synchronize()
    o_keep, *_ = oracle.schedule_prefix(conf, cost)
    np.testing.assert_array_equal(host(n_keep), o_keep)
    big = sched_ctx(2048, 5)  # 10240 slots > DDT_SCHED_MAX_SLOTS
    conf = synth.draw_confidences(2048, 5)
    with pytest.raises(ddt.DdtError) as e:
        big.ddt_schedule_prefix(dev(conf), 2048, dev(np.ones(10241, np.float32)),
                                torch.empty(2048, dtype=torch.int32, device="cuda"))
    assert e.value.status == ddt.EUNSUPPORTED
