"""Pins of the oracle's stochastic chain verification ("DSpark Speculative
Decoding Explained: Block Drafting and Confidence Checks", the probability
rule: keep guess x_k with probability min(1, p/q), replace the first rejected
guess by a draw from max(0, p - q), a bonus draw from p when all survive).

  * the page's toy: its tables, Python's random.Random(42) and the oracle's
    rule reproduce the five printed passes and their 13 tokens;
  * the committed token's distribution is the target's (integrated over a
    grid of the uniforms) and the toy's 20,000-step frequencies agree with
    the target within Monte-Carlo error;
  * with a constant acceptance rate a and g guesses, the mean tokens per
    pass is the page's (1 - a^(g+1)) / (1 - a);
  * the logits form equals the probability form after a softmax, also for
    logits far from zero;
  * the rule's edges: p(x) = 0 is never kept, a zero weight is never drawn,
    q(x) = 0 counts as ratio 1.
"""
import os
import random

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _toy():
    vocab, big, mix, rows = None, {}, None, {"pass": []}
    for line in open(os.path.join(HERE, "golden", "dspark_toy.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "vocab":
            vocab = rest
        elif key == "big":
            big[rest[0]] = {t.split(":")[0]: float(t.split(":")[1]) for t in rest[1:]}
        elif key == "draft_mix":
            mix = (float(rest[0]), float(rest[1]))
        elif key == "pass":
            rows["pass"].append(rest)
        else:
            rows[key] = rest
    return vocab, big, mix, rows


def test_toy_printed_passes():
    vocab, big, (keep, spread), rows = _toy()
    V = len(vocab)

    def p_of(prev):
        return [big[prev].get(t, 0.0) for t in vocab]

    def q_of(prev):
        return [keep * x + spread / V for x in p_of(prev)]

    rng = random.Random(int(rows["seed"][0]))
    k, prev, total = int(rows["guesses"][0]), rows["start"][0], 0
    for want in rows["pass"]:
        # the drafter's k guesses (cumulative-weight draws, one uniform each)
        guesses, qs, ctx = [], [], prev
        for _ in range(k):
            q = q_of(ctx)
            t = rng.choices(vocab, weights=q)[0]
            guesses.append(vocab.index(t))
            qs.append(q)
            ctx = t
        # the target rows along the guessed path, and the verifier's uniforms
        ps, ctx = [], prev
        for g in guesses:
            ps.append(p_of(ctx))
            ctx = vocab[g]
        ps.append(p_of(ctx))
        state = rng.getstate()
        stream = [rng.random() for _ in range(k + 1)]
        n = len(oracle.verify_chain(np.array(ps), np.array(qs), guesses, stream[:k], 0.0))
        used = min(n, k)  # uniforms the accept tests consumed
        out = oracle.verify_chain(np.array(ps), np.array(qs), guesses, stream[:k], stream[used])
        rng.setstate(state)
        for _ in range(used + 1):
            rng.random()
        words = [vocab[t] for t in out]
        assert words == want, (words, want)
        total += len(out)
        prev = words[-1]
    assert total == int(rows["total"][0])


def test_output_distribution_is_the_target():
    rng = np.random.default_rng(5)
    V, N = 6, 300
    for _ in range(3):
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V))
        bonus = rng.dirichlet(np.ones(V))
        grid = (np.arange(N) + 0.5) / N
        dist = np.zeros(V)
        for x in range(V):
            for u in grid:
                # r's grid in one call per u: the accept decision ignores r
                first = oracle.verify_chain(np.stack([p, bonus]), q[None], [x], [u], 0.5)
                if len(first) == 2:  # kept: the committed token is x
                    dist[x] += q[x] / N
                    continue
                for r in grid:
                    out = oracle.verify_chain(np.stack([p, bonus]), q[None], [x], [u], r)
                    dist[out[0]] += q[x] / (N * N)
        assert np.abs(dist - p).max() < 3.0 / N, (dist, p)


def test_scheduled_prefix_output_follows_the_target():
    """The rule's guarantee on a cut chain: with L = 3 guesses drafted but a
    count of n = 1, the committed first token is distributed as target row 0,
    and after a kept guess the bonus follows target row 1 (row n, not row L).
    Every (guess, u, r) of a grid is one request; each weighs q_0(x) / N^2."""
    rng = np.random.default_rng(6)
    V, N, L = 6, 60, 3
    p = rng.dirichlet(np.ones(V), size=L + 1)   # target rows 0..L
    q = rng.dirichlet(np.ones(V), size=L)       # draft rows 0..L-1
    grid = (np.arange(N) + 0.5) / N
    x, ui, ri = np.meshgrid(np.arange(V), np.arange(N), np.arange(N), indexing="ij")
    x, ui, ri = x.ravel(), ui.ravel(), ri.ravel()
    R = x.size
    draft = np.broadcast_to(np.log(q), (R, L, V)).astype(np.float64).copy()
    target = np.broadcast_to(np.log(p), (R, L + 1, V)).astype(np.float64).copy()
    tokens = np.zeros((R, L), np.int32)
    tokens[:, 0] = x
    u = np.zeros((R, L))
    u[:, 0] = grid[ui]
    acc_len, acc_tokens = oracle.accept_stochastic(draft, target, tokens, u, grid[ri],
                                                   n_guess=np.ones(R, np.int32))
    assert acc_len.max() == 2  # one guess verified, then the bonus
    w = q[0][x] / (N * N)
    first = np.bincount(acc_tokens[:, 0], weights=w, minlength=V)
    assert np.abs(first - p[0]).max() < 3.0 / N, (first, p[0])
    kept = acc_len == 2
    bonus = np.bincount(acc_tokens[kept, 1], weights=w[kept], minlength=V) / w[kept].sum()
    assert np.abs(bonus - p[1]).max() < 3.0 / N, (bonus, p[1])
    assert np.abs(bonus - p[L]).max() > 6.0 / N  # row L would be told apart


def test_toy_lossless_frequencies():
    vocab, big, (keep, spread), rows = _toy()
    V = len(vocab)
    p = np.array([big["to"].get(t, 0.0) for t in vocab])
    q = keep * p + spread / V
    rng = np.random.default_rng(20000)
    n = 20000
    counts = np.zeros(V)
    xs = rng.choice(V, size=n, p=q / q.sum())
    us, rs = rng.random(n), rng.random(n)
    for x, u, r in zip(xs, us, rs):
        out = oracle.verify_chain(np.stack([p, p]), q[None], [x], [u], r)
        counts[out[0]] += 1
    freq = counts / n
    for t, want in (t.split(":") for t in rows["after_to_target"]):
        i = vocab.index(t)
        sd = np.sqrt(float(want) * (1 - float(want)) / n)
        assert abs(freq[i] - float(want)) < 4 * sd, (t, freq[i], want)
    # the page's own measured frequencies sit within the same error bars
    for t, got in (t.split(":") for t in rows["after_to_measured"]):
        want = float(dict(x.split(":") for x in rows["after_to_target"])[t])
        assert abs(float(got) - want) < 4 * np.sqrt(want * (1 - want) / n)


def test_constant_acceptance_mean_tokens():
    # every guess survives with probability a: p(x) = a q(x) at the guess
    rng = np.random.default_rng(7)
    V, trials = 5, 40000
    for a, g in ((0.5, 4), (0.5, 8), (0.8, 6)):
        q = np.full((g, V), 1.0 / V)
        p = np.full((g + 1, V), 0.0)
        p[:g, 0] = a / V
        p[:g, 1:] = (1 - a / V) / (V - 1)
        p[g] = 1.0 / V
        total = 0
        for _ in range(trials // 10):
            u = rng.random(g)
            total += len(oracle.verify_chain(p, q, [0] * g, u, rng.random()))
        mean = total / (trials // 10)
        want = (1 - a ** (g + 1)) / (1 - a)
        assert abs(mean - want) < 0.05 * want, (a, g, mean, want)


def test_logits_form_matches_probabilities():
    rng = np.random.default_rng(3)
    R, L, V = 3, 4, 50
    draft = (rng.standard_normal((R, L, V)) * 2).astype(np.float32)
    target = (rng.standard_normal((R, L + 1, V)) * 2).astype(np.float32)
    tokens = rng.integers(0, V, size=(R, L)).astype(np.int32)
    u, r = rng.random((R, L)), rng.random(R)
    acc_len, acc_tokens = oracle.accept_stochastic(draft, target, tokens, u, r)

    def sm(z):
        e = np.exp(z.astype(np.float64) - z.max(-1, keepdims=True))
        return e / e.sum(-1, keepdims=True)

    for i in range(R):
        want = oracle.verify_chain(sm(target[i]), sm(draft[i]), tokens[i], u[i], r[i])
        assert acc_len[i] == len(want)
        assert list(acc_tokens[i, :acc_len[i]]) == want
        assert (acc_tokens[i, acc_len[i]:] == -1).all()
    # equal distributions keep every guess
    acc_len, acc_tokens = oracle.accept_stochastic(draft, np.concatenate(
        [draft, draft[:, :1]], 1), tokens, np.full((R, L), 0.999999), r)
    assert (acc_len == L + 1).all()
    assert (acc_tokens[:, :L] == tokens).all()


def test_boundaries_the_rule_fixes():
    """Cases the rule decides at its edges: a guess the target gives
    probability 0 is kept with probability 0 (so never, even at u = 0); a
    token whose weight is 0 is never drawn (even at r = 0); a guess the draft
    gives probability 0 counts as ratio 1 (the stated reading: such a guess
    cannot come from the draft, and the rule would divide by zero)."""
    p = np.array([[0.0, 0.5, 0.5], [0.2, 0.3, 0.5]])
    q = np.array([[0.5, 0.25, 0.25]])
    # p(x) = 0: rejected at u = 0; the leftover max(0, p - q) = (0, .25, .25)
    # gives token 0 no weight, so r = 0 draws token 1
    assert oracle.verify_chain(p, q, [0], [0.0], 0.0) == [1]
    # q(x) = 0 with p(x) > 0: kept whatever u, then the bonus from p's last row
    q0 = np.array([[0.0, 0.5, 0.5]])
    p0 = np.array([[0.4, 0.3, 0.3], [0.2, 0.3, 0.5]])
    assert oracle.verify_chain(p0, q0, [0], [0.999], 0.0) == [0, 0]
    # bonus at r = 0 skips a zero-weight first token
    pz = np.array([[0.5, 0.5, 0.0], [0.0, 0.4, 0.6]])
    qz = np.array([[0.5, 0.5, 0.0]])
    assert oracle.verify_chain(pz, qz, [1], [0.0], 0.0) == [1, 1]


def test_large_logits():
    """Logits far from zero (+900 on the draft, -900 on the target: a softmax
    must shift by the row max, or exp overflows or underflows) give the same
    answers as the probability form of the same logits."""
    rng = np.random.default_rng(5)
    R, L, V = 2, 3, 40
    dfar = ((rng.standard_normal((R, L, V)) * 2) + 900.0).astype(np.float32)
    tfar = ((rng.standard_normal((R, L + 1, V)) * 2) - 900.0).astype(np.float32)
    tokens = rng.integers(0, V, size=(R, L)).astype(np.int32)
    u, r = rng.random((R, L)), rng.random(R)
    acc_len, acc_tokens = oracle.accept_stochastic(dfar, tfar, tokens, u, r)

    def sm(z):
        z = z.astype(np.float64)
        e = np.exp(z - z.max(-1, keepdims=True))
        return e / e.sum(-1, keepdims=True)

    for i in range(R):
        want = oracle.verify_chain(sm(tfar[i]), sm(dfar[i]), tokens[i], u[i], r[i])
        assert acc_len[i] == len(want) and list(acc_tokens[i, :acc_len[i]]) == want


def test_scheduled_prefix_lengths():
    """Verifying only the first n guesses of a request (the prefix a
    scheduler kept) is the rule on the chain cut to n guesses: the bonus then
    comes from target row n. n = 0 draws the bonus from row 0 at once."""
    rng = np.random.default_rng(9)
    R, L, V = 7, 5, 30
    draft = (rng.standard_normal((R, L, V)) * 2).astype(np.float32)
    target = (rng.standard_normal((R, L + 1, V)) * 2).astype(np.float32)
    target[:, :L] = draft + (0.3 * rng.standard_normal((R, L, V))).astype(np.float32)
    tokens = rng.integers(0, V, size=(R, L)).astype(np.int32)
    u, r = rng.random((R, L)), rng.random(R)
    n = np.array([0, 1, 2, 3, 5, 9, -1], np.int32)  # 9 is clamped to L, -1 to 0
    u[5:] = 0.0  # the clamped requests keep every guess they verify
    acc_len, acc_tokens = oracle.accept_stochastic(draft, target, tokens, u, r, n_guess=n)
    assert acc_len[5] == L + 1 and acc_len[6] == 1
    for i in range(R):
        m = min(max(int(n[i]), 0), L)
        cut_len, cut_tok = oracle.accept_stochastic(
            draft[i:i + 1, :m] if m > 0 else np.zeros((1, 0, V), np.float32),
            np.concatenate([target[i:i + 1, :m], target[i:i + 1, m:m + 1]], axis=1),
            tokens[i:i + 1, :m], u[i:i + 1, :m], r[i:i + 1])
        assert acc_len[i] == cut_len[0] and acc_len[i] <= m + 1
        np.testing.assert_array_equal(acc_tokens[i, :acc_len[i]], cut_tok[0, :cut_len[0]])
        assert (acc_tokens[i, acc_len[i]:] == -1).all()
    # no n_guess is n = L everywhere
    full = oracle.accept_stochastic(draft, target, tokens, u, r)
    same = oracle.accept_stochastic(draft, target, tokens, u, r, n_guess=np.full(R, L, np.int32))
    np.testing.assert_array_equal(full[0], same[0])
    np.testing.assert_array_equal(full[1], same[1])
