"""Stochastic verification of drafted chains on the GPU ("DSpark Speculative
Decoding Explained: Block Drafting and Confidence Checks", the probability
rule) through the C ABI, against the oracle.

The kept prefix, the drawn token and the lengths must equal the oracle's.
The one exception is a decision or a draw whose fp64 boundary lies within a
tie band of the input uniform: there the GPU's fp32 arithmetic may take the
other side, and the test checks instead that the GPU's choice is valid with
the fp64 probabilities (the band is far above fp32 rounding of p/q and of
the running sums, and a random draw lands in it with probability ~1e-5).
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_depth_gb300 import ddt, synth
from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu

U_TIE = 1e-5    # |u - min(1, p/q)| within which either decision is right
CDF_TIE = 1e-5  # |running sum - r * total| within which either neighbour is right

BF16_NEG_INF = np.uint16(0xFF80)


def chain_ctx(R_max, L, V, draft_bf16, target_bf16):
    K = min(8, V)
    c = ddt.make_config(R_max=R_max, L=L, V=V, B=K, K=K, Hq=4, Hkv=1, d=64, page_size=16,
                        max_pages_per_req=1, num_pages=1,
                        draft_dtype=ddt.BF16 if draft_bf16 else ddt.F32,
                        target_dtype=ddt.BF16 if target_bf16 else ddt.F32)
    return ddt.Context(c)


def widen(z):
    return synth.bf16_bits_to_f32(z) if z.dtype == np.uint16 else z


def softmax64(z):
    z = widen(z).astype(np.float64)
    m = z.max(-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(-1, keepdims=True)


def run_gpu(ctx, draft, target, tokens, u, r, R=None, stream=None, n_guess=None):
    R = draft.shape[0] if R is None else R
    L = tokens.shape[1]
    acc_len = torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda")
    acc_tok = torch.full((max(R, 1), L + 1), -7, dtype=torch.int32, device="cuda")
    ng = None if n_guess is None else (n_guess if torch.is_tensor(n_guess) else dev(n_guess))
    ctx.ddt_accept_stochastic(dev(draft), dev(target), dev(tokens), dev(u), dev(r), R, acc_len,
                              acc_tok, n_guess=ng, stream=stream)
    torch.cuda.synchronize()
    return host(acc_len), host(acc_tok), ctx.ddt_device_status()


def run_oracle(draft, target, tokens, u, r, n_guess=None):
    # the oracle takes one logit dtype: widen bf16 (exactly) when the two differ
    if draft.dtype != target.dtype:
        draft, target = widen(draft), widen(target)
    return oracle.accept_stochastic(draft, target, tokens, u.astype(np.float64),
                                    r.astype(np.float64), n_guess=n_guess)


def check_request(i, g_len, g_tok, o_len, o_tok, draft, target, tokens, u, r, n_guess=None):
    """Exact agreement, or a disagreement explained by a tie (see above)."""
    L = tokens.shape[1]
    if g_len == o_len and np.array_equal(g_tok, o_tok):
        return "exact"
    n = L if n_guess is None else int(np.clip(n_guess[i], 0, L))  # guesses verified
    assert 1 <= g_len <= n + 1, (i, g_len)
    assert np.array_equal(g_tok[:g_len - 1], tokens[i, :g_len - 1]), i
    assert (g_tok[g_len:] == -1).all(), i
    p = softmax64(target[i])
    q = softmax64(draft[i])
    if g_len != o_len:
        k = min(g_len, o_len) - 1  # the first decision the two took differently
        x = tokens[i, k]
        a = 1.0 if q[k, x] == 0 else min(1.0, p[k, x] / q[k, x])
        assert abs(float(u[i, k]) - a) <= U_TIE, (i, k, float(u[i, k]), a)
    ks = g_len - 1
    w = np.maximum(p[ks] - q[ks], 0.0) if ks < n else p[n]
    W = w.sum()
    t = int(g_tok[ks])
    if W <= CDF_TIE:  # (almost) no weight: any in-range token or -1
        assert -1 <= t < w.size, (i, t)
        return "tie"
    assert 0 <= t < w.size, (i, t)
    cum = np.cumsum(w)
    x = float(r[i]) * W
    assert cum[t] - w[t] <= x + CDF_TIE and cum[t] > x - CDF_TIE, (i, t, x, cum[t], w[t])
    return "tie"


def compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u, r, n_guess=None):
    kinds = [check_request(i, g_len[i], g_tok[i], o_len[i], o_tok[i], draft, target, tokens, u,
                           r, n_guess) for i in range(len(o_len))]
    # ties are rare: a run where most requests need the band has a real bug
    assert kinds.count("tie") <= max(1, len(kinds) // 16), kinds
    return kinds


def draw(R, L, V, dtype="bf16", seed=0, boost=False):
    cfg = synth.config("tiny", R=R, L=L, V=V, logit_dtype=dtype, seed=seed, boost=boost)
    return synth.draw_chain_inputs(cfg)


CASES = {
    # name: (R, L, V, draft dtype, target dtype, seed)
    "tiny_f32": (3, 4, 50, "f32", "f32", 61),
    "aligned_bf16": (4, 7, 40000, "bf16", "bf16", 62),
    "ragged_bf16": (5, 6, 40001, "bf16", "bf16", 63),
    "bf16_draft_f32_target": (3, 5, 20000, "bf16", "f32", 64),
    "f32_draft_bf16_target": (3, 5, 9999, "f32", "bf16", 65),
    "one_chunk_f32": (6, 3, 8192, "f32", "f32", 66),
    "max_L": (2, 18, 151936, "bf16", "bf16", 67),
}


def case_inputs(name):
    R, L, V, dd, dt, seed = CASES[name]
    d = draw(R, L, V, "f32", seed)
    draft = synth.to_bf16_bits(d["draft"]) if dd == "bf16" else d["draft"]
    target = synth.to_bf16_bits(d["target"]) if dt == "bf16" else d["target"]
    return draft, target, d["tokens"], d["u"], d["r"]


@pytest.mark.parametrize("name", sorted(CASES))
def test_chain_matches_oracle(name):
    draft, target, tokens, u, r = case_inputs(name)
    R, L = tokens.shape
    V = draft.shape[-1]
    ctx = chain_ctx(R, L, V, draft.dtype == np.uint16, target.dtype == np.uint16)
    g_len, g_tok, st = run_gpu(ctx, draft, target, tokens, u, r)
    assert st == 0
    o_len, o_tok = run_oracle(draft, target, tokens, u, r)
    compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u, r)


def test_batch64_chains_match_oracle():
    """The full workload (64 chains of 15 guesses, V = 151936, bf16), every
    request against the oracle, twice through one context (the arrival
    counters reset themselves)."""
    cfg = synth.config("batch64")
    d = synth.draw_chain_inputs(cfg)
    ctx = chain_ctx(cfg.R, cfg.L, cfg.V, True, True)
    o_len, o_tok = run_oracle(d["draft"], d["target"], d["tokens"], d["u"], d["r"])
    for _ in range(2):
        g_len, g_tok, st = run_gpu(ctx, d["draft"], d["target"], d["tokens"], d["u"], d["r"])
        assert st == 0
        compare(g_len, g_tok, o_len, o_tok, d["draft"], d["target"], d["tokens"], d["u"], d["r"])
    # the workload keeps a spread of lengths (not all rejected, not all kept)
    assert 1.5 < o_len.mean() < cfg.L


# ------------------------------------------------------------------ edge cases
def base_case(R=4, L=5, V=3000, seed=70):
    d = draw(R, L, V, "bf16", seed)
    return d["draft"], d["target"], d["tokens"], d["u"], d["r"]


def run_both(draft, target, tokens, u, r):
    R, L = tokens.shape
    ctx = chain_ctx(R, L, draft.shape[-1], True, True)
    g_len, g_tok, st = run_gpu(ctx, draft, target, tokens, u, r)
    o_len, o_tok = run_oracle(draft, target, tokens, u, r)
    return g_len, g_tok, st, o_len, o_tok


def test_identical_models_keep_every_guess():
    draft, target, tokens, u, r = base_case()
    target[:, :-1] = draft  # p = q on every guessed row: ratio exactly 1
    g_len, g_tok, st, o_len, o_tok = run_both(draft, target, tokens, u, r)
    assert st == 0
    L = tokens.shape[1]
    assert (o_len == L + 1).all() and (g_len == L + 1).all()
    np.testing.assert_array_equal(g_tok, o_tok)


def test_u_zero_keeps_and_u_near_one_rejects():
    draft, target, tokens, u, r = base_case(seed=71)
    u0 = np.zeros_like(u)
    g_len, g_tok, st, o_len, o_tok = run_both(draft, target, tokens, u0, r)
    assert st == 0 and (g_len == tokens.shape[1] + 1).all()
    np.testing.assert_array_equal(g_tok, o_tok)
    u1 = np.full_like(u, np.nextafter(np.float32(1), np.float32(0)))
    g_len, g_tok, st, o_len, o_tok = run_both(draft, target, tokens, u1, r)
    assert st == 0
    compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u1, r)


def test_zero_target_probability_rejects():
    draft, target, tokens, u, r = base_case(seed=72)
    R = tokens.shape[0]
    for i in range(R):  # p(x_2) = 0: guess 2 is never kept, nor drawn again
        target[i, 2, tokens[i, 2]] = BF16_NEG_INF
    u0 = np.zeros_like(u)
    g_len, g_tok, st, o_len, o_tok = run_both(draft, target, tokens, u0, r)
    assert st == 0
    assert (o_len == 3).all() and (g_len == 3).all()
    np.testing.assert_array_equal(g_tok, o_tok)
    assert (g_tok[:, 2] != tokens[:, 2]).all()


@pytest.mark.parametrize("rv", [0.0, float(np.nextafter(np.float32(1), np.float32(0)))])
def test_draw_at_the_ends_of_the_cdf(rv):
    draft, target, tokens, u, r = base_case(seed=73)
    rr = np.full_like(r, rv)
    g_len, g_tok, st, o_len, o_tok = run_both(draft, target, tokens, u, rr)
    assert st == 0
    compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u, rr)


def test_fewer_requests_than_capacity_and_empty_batch():
    draft, target, tokens, u, r = base_case(R=5, seed=74)
    ctx = chain_ctx(8, tokens.shape[1], draft.shape[-1], True, True)
    g_len, g_tok, st = run_gpu(ctx, draft, target, tokens, u, r)
    assert st == 0
    o_len, o_tok = run_oracle(draft, target, tokens, u, r)
    compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u, r)
    # R = 0 enqueues nothing: the outputs keep their fill
    g_len0, g_tok0, st = run_gpu(ctx, draft, target, tokens, u, r, R=0)
    assert st == 0 and (g_len0 == -7).all() and (g_tok0 == -7).all()
    # and the context still answers the same afterwards
    g_len2, g_tok2, _ = run_gpu(ctx, draft, target, tokens, u, r)
    np.testing.assert_array_equal(g_len2, g_len)
    np.testing.assert_array_equal(g_tok2, g_tok)


def test_out_of_range_guess_sets_status():
    draft, target, tokens, u, r = base_case(seed=75)
    V = draft.shape[-1]
    bad = tokens.copy()
    bad[0, 1] = V
    u0 = np.zeros_like(u)
    ctx = chain_ctx(tokens.shape[0], tokens.shape[1], V, True, True)
    g_len, g_tok, st = run_gpu(ctx, draft, target, bad, u0, r)
    assert st & ddt.DEV_BAD_TREE
    assert g_len[0] <= 2
    # the other requests are untouched by request 0's bad guess
    o_len, o_tok = run_oracle(draft, target, tokens, u0, r)
    np.testing.assert_array_equal(g_len[1:], o_len[1:])
    np.testing.assert_array_equal(g_tok[1:], o_tok[1:])


def test_nan_logits_set_status():
    draft, target, tokens, u, r = base_case(seed=76)
    draft[1, 3, 17] = np.uint16(0x7FC0)  # a bf16 NaN
    ctx = chain_ctx(tokens.shape[0], tokens.shape[1], draft.shape[-1], True, True)
    _, _, st = run_gpu(ctx, draft, target, tokens, u, r)
    assert st & ddt.DEV_NAN_LOGITS


def test_side_stream():
    draft, target, tokens, u, r = base_case(seed=77)
    ctx = chain_ctx(tokens.shape[0], tokens.shape[1], draft.shape[-1], True, True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g_len, g_tok, st = run_gpu(ctx, draft, target, tokens, u, r, stream=s)
    assert st == 0
    o_len, o_tok = run_oracle(draft, target, tokens, u, r)
    compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u, r)


# ------------------------------------------ a scheduled prefix (guesses per request)
def test_random_guess_counts_match_oracle():
    """Request i verifies only its first n_i guesses, n_i drawn from [0, L]
    (0 and L both present): kept prefixes, draws and bonus rows (target row
    n_i) against the oracle, on a ragged vocabulary."""
    draft, target, tokens, u, r = case_inputs("ragged_bf16")
    R, L = tokens.shape
    ng = np.array([0, L, 2, 1, 4], dtype=np.int32)[:R]
    ctx = chain_ctx(R, L, draft.shape[-1], True, True)
    g_len, g_tok, st = run_gpu(ctx, draft, target, tokens, u, r, n_guess=ng)
    assert st == 0
    o_len, o_tok = run_oracle(draft, target, tokens, u, r, n_guess=ng)
    compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u, r, ng)
    assert (g_len <= ng + 1).all()
    assert g_len[0] == 1  # nothing verified: only the bonus from target row 0


def test_guess_counts_with_every_guess_kept_take_the_bonus_from_row_n():
    draft, target, tokens, u, r = base_case(R=6, L=5, seed=78)
    target[:, :-1] = draft  # ratio exactly 1 on every guessed row
    ng = np.arange(6, dtype=np.int32) % 6  # 0..5
    u0 = np.zeros_like(u)
    ctx = chain_ctx(6, 5, draft.shape[-1], True, True)
    g_len, g_tok, st = run_gpu(ctx, draft, target, tokens, u0, r, n_guess=ng)
    assert st == 0
    o_len, o_tok = run_oracle(draft, target, tokens, u0, r, n_guess=ng)
    np.testing.assert_array_equal(o_len, ng + 1)
    compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u0, r, ng)


def test_rows_past_the_guess_count_are_not_read():
    """NaNs planted in draft rows k >= n_i and target rows k > n_i are never
    seen: no NaN status, and the result is that of clean rows."""
    draft, target, tokens, u, r = base_case(R=4, L=6, seed=79)
    ng = np.array([2, 0, 6, 3], dtype=np.int32)
    o_len, o_tok = run_oracle(draft, target, tokens, u, r, n_guess=ng)
    d2, t2 = draft.copy(), target.copy()
    for i, n in enumerate(ng):
        d2[i, n:, :] = np.uint16(0x7FC0)
        t2[i, n + 1:, :] = np.uint16(0x7FC0)
    ctx = chain_ctx(4, 6, draft.shape[-1], True, True)
    g_len, g_tok, st = run_gpu(ctx, d2, t2, tokens, u, r, n_guess=ng)
    assert st == 0
    compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u, r, ng)


def test_out_of_range_guess_count_is_clamped_and_sets_status():
    draft, target, tokens, u, r = base_case(R=3, L=5, seed=80)
    ng = np.array([-1, 7, 3], dtype=np.int32)
    ctx = chain_ctx(3, 5, draft.shape[-1], True, True)
    g_len, g_tok, st = run_gpu(ctx, draft, target, tokens, u, r, n_guess=ng)
    assert st & ddt.DEV_BAD_TREE
    o_len, o_tok = run_oracle(draft, target, tokens, u, r, n_guess=np.clip(ng, 0, 5))
    compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u, r, np.clip(ng, 0, 5))


def test_scheduler_output_feeds_verification_on_the_device():
    """ddt_schedule_prefix's n_keep, left on the device, is the guess count
    of ddt_accept_stochastic: the two calls chained against the oracle's
    schedule_prefix then accept_stochastic, on the 64-chain workload."""
    cfg = synth.config("batch64")
    d = synth.draw_chain_inputs(cfg)
    R, L = cfg.R, cfg.L
    conf = synth.draw_confidences(R, L, seed=81)
    cost = (25.0 + 0.1 * (R + np.arange(R * L + 1))).astype(np.float32)
    ctx = chain_ctx(R, L, cfg.V, True, True)
    keep = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    ctx.ddt_schedule_prefix(dev(conf), R, dev(cost), keep)
    g_len, g_tok, st = run_gpu(ctx, d["draft"], d["target"], d["tokens"], d["u"], d["r"],
                               n_guess=keep)
    assert st == 0
    o_keep = oracle.schedule_prefix(conf, cost.astype(np.float64))[0]
    np.testing.assert_array_equal(host(keep), o_keep)
    assert 0 < o_keep.sum() < R * L  # the budget cuts some chains, not all
    o_len, o_tok = run_oracle(d["draft"], d["target"], d["tokens"], d["u"], d["r"],
                              n_guess=o_keep)
    compare(g_len, g_tok, o_len, o_tok, d["draft"], d["target"], d["tokens"], d["u"], d["r"],
            o_keep)


def test_guess_counts_at_the_most_requests():
    """2048 requests (the context's limit): the row pass's scan of the
    counts runs 8 requests per thread."""
    R, L, V = 2048, 3, 64
    d = draw(R, L, V, "f32", seed=82)
    rng = np.random.default_rng(83)
    ng = rng.integers(0, L + 1, size=R).astype(np.int32)
    ctx = chain_ctx(R, L, V, False, False)
    g_len, g_tok, st = run_gpu(ctx, d["draft"], d["target"], d["tokens"], d["u"], d["r"],
                               n_guess=ng)
    assert st == 0
    o_len, o_tok = run_oracle(d["draft"], d["target"], d["tokens"], d["u"], d["r"], n_guess=ng)
    compare(g_len, g_tok, o_len, o_tok, d["draft"], d["target"], d["tokens"], d["u"], d["r"], ng)


@pytest.mark.parametrize("name", sorted(CASES))
def test_case_with_guess_counts(name):
    """Every shape and dtype pair of the chain cases, with random counts:
    each variant of the counted row pass and of the draw."""
    draft, target, tokens, u, r = case_inputs(name)
    R, L = tokens.shape
    ng = np.random.default_rng(85).integers(0, L + 1, size=R).astype(np.int32)
    ctx = chain_ctx(R, L, draft.shape[-1], draft.dtype == np.uint16, target.dtype == np.uint16)
    g_len, g_tok, st = run_gpu(ctx, draft, target, tokens, u, r, n_guess=ng)
    assert st == 0
    o_len, o_tok = run_oracle(draft, target, tokens, u, r, n_guess=ng)
    compare(g_len, g_tok, o_len, o_tok, draft, target, tokens, u, r, ng)


# ------------------------------------- a vocabulary past the staged decision
@pytest.mark.parametrize("counts", [False, True])
def test_wide_vocabulary_decides_per_warp(counts):
    """V = 600000 at L = 18: the 2L + 1 rows of 37 chunks each hold more
    pairs than a decision stages in shared memory (1024), so a warp merges
    each row's pairs from global memory. With counts, only the rows a
    request verifies."""
    R, L, V = 2, 18, 600000
    d = draw(R, L, V, "bf16", seed=85, boost=True)  # request 0 keeps 13 guesses
    ng = np.array([9, L], np.int32) if counts else None  # request 0's bonus: row 9
    ctx = chain_ctx(R, L, V, True, True)
    g_len, g_tok, st = run_gpu(ctx, d["draft"], d["target"], d["tokens"], d["u"], d["r"],
                               n_guess=ng)
    assert st == 0
    o_len, o_tok = run_oracle(d["draft"], d["target"], d["tokens"], d["u"], d["r"], n_guess=ng)
    compare(g_len, g_tok, o_len, o_tok, d["draft"], d["target"], d["tokens"], d["u"], d["r"], ng)
