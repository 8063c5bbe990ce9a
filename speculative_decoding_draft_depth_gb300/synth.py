"""Seeded synthetic inputs for one batched draft-tree round.

This module is the only code shared by the CUDA path's tests/bench and the
CPU oracle. It draws random data and arranges it in the round's layouts; it
holds none of the round's arithmetic (no log-softmax, top-K, heap, mask,
attention or acceptance). Everything comes from numpy's PCG64 with the
seeds given below. bf16 tensors are produced as raw bit patterns (uint16,
round-to-nearest-even from float32).

Workloads (shapes of the pages' DFlash/DDTree/TreeSpark settings; the pages'
benchmark prompts and trained drafters are not available, so these seeded
draws stand in for them):

  tiny     R=1,  L=4,  V=32,     B=8,  K=8,  fp32 logits N(0,1)*3, Hq=4,
           Hkv=1, d=64, ctx 64, agreement 0.7                       (seed 0)
  single   R=1,  L=15, V=151936, B=32, K=32, bf16 logits N(0,1) plus a Zipf
           boost 8*r^-1.1 on 20 random tokens per depth, agreement
           0.8-0.03*depth, Qwen3-8B attention (32/8/128), ctx 4096  (seed 1)
  batch64  R=64, as 'single' with ctx ~ U[512,16384], per-request agreement
           a_r ~ U[0.5,0.9] decaying 0.03/depth, pages permuted     (seed 3)
  wide256  R=256, B=K=64, ctx lognormal(ln 4096, 1) capped at 32768, logits
           of 'single' divided by T ~ U[0.3,1.5] per (request, depth),
           agreement 0.75, Qwen3-4B attention (32/8/128)            (seed 4)
  treespark R=8, 7 depths, V=151936, parent-conditioned tree with k=4
           children per parent, frontier F=4, N=32 nodes; backbone logits
           bf16 N(0,1)*3, Markov head W and embeddings E bf16 N(0, 0.02)
           [V, 256], anchors uniform; Qwen3-4B attention, ctx 2048  (seed 2)
  sparkling R=64, L=15, V=151936, the SparklingTree table tree: top-C=128
           prefilter per depth, Markov head W, E bf16 N(0, 0.02) [V, 256],
           budget B=64; logits, contexts and agreement as batch64  (seed 5)

Chains for stochastic verification (draw_chain_inputs): the draft logits of
the chosen workload; target rows 0..L-1 are the draft row plus N(0, s_r^2)
noise with s_r ~ U[0.2, 1.0] per request, row L is a fresh draw like a draft
row; the guesses are sampled from the draft rows at temperature 1 (Gumbel-max
on the stored logits, a data-construction step); u [R, L] and r [R] are
float32 uniforms in [0, 1).

Confidences for the prefix scheduler (draw_confidences): per request a base
chance b_r ~ U[0.5, 0.95]; guess k survives its predecessors with chance
sigmoid(logit(b_r) - 0.15 k + 0.5 e), e ~ N(0, 1), stored as float32.
"""
from dataclasses import dataclass, field, replace

import numpy as np

VOCAB_QWEN3 = 151936


@dataclass(frozen=True)
class RoundConfig:
    name: str
    R: int
    L: int
    V: int
    B: int
    K: int
    Hq: int
    Hkv: int
    d: int
    page: int
    logit_dtype: str  # "bf16" or "f32"
    ctx_kind: str  # "fixed", "uniform", "lognormal"
    ctx_args: tuple
    seed: int
    boost: bool = True
    temp_range: tuple = None  # per (request, depth) temperature on logits
    agree_kind: str = "decay"  # "const", "decay", "per_request"
    agree_args: tuple = (0.8, 0.03)
    rounds: int = 1
    spare_pages: int = 8
    markov_dim: int = 0  # H of the parent-conditioned tree's Markov head
    frontier: int = 0  # F of the parent-conditioned tree
    prefilter: int = 0  # C of the SparklingTree table tree (kept tokens per depth)

    @property
    def P(self):
        return self.B + 1

    @property
    def W(self):
        return (self.P + 31) // 32


CONFIGS = {
    "tiny": RoundConfig("tiny", R=1, L=4, V=32, B=8, K=8, Hq=4, Hkv=1, d=64, page=16,
                        logit_dtype="f32", ctx_kind="fixed", ctx_args=(64,), seed=0,
                        boost=False, agree_kind="const", agree_args=(0.7,)),
    "single": RoundConfig("single", R=1, L=15, V=VOCAB_QWEN3, B=32, K=32, Hq=32, Hkv=8, d=128,
                          page=16, logit_dtype="bf16", ctx_kind="fixed", ctx_args=(4096,), seed=1,
                          agree_kind="decay", agree_args=(0.8, 0.03)),
    "batch64": RoundConfig("batch64", R=64, L=15, V=VOCAB_QWEN3, B=32, K=32, Hq=32, Hkv=8, d=128,
                           page=16, logit_dtype="bf16", ctx_kind="uniform",
                           ctx_args=(512, 16384), seed=3, agree_kind="per_request",
                           agree_args=(0.5, 0.9, 0.03)),
    "wide256": RoundConfig("wide256", R=256, L=15, V=VOCAB_QWEN3, B=64, K=64, Hq=32, Hkv=8,
                           d=128, page=16, logit_dtype="bf16", ctx_kind="lognormal",
                           ctx_args=(4096, 1.0, 32768), seed=4, temp_range=(0.3, 1.5),
                           agree_kind="const", agree_args=(0.75,), rounds=8),
    "treespark": RoundConfig("treespark", R=8, L=7, V=VOCAB_QWEN3, B=32, K=4, Hq=32, Hkv=8,
                             d=128, page=16, logit_dtype="bf16", ctx_kind="fixed",
                             ctx_args=(2048,), seed=2, boost=False, agree_kind="const",
                             agree_args=(0.75,), markov_dim=256, frontier=4),
    "sparkling": RoundConfig("sparkling", R=64, L=15, V=VOCAB_QWEN3, B=64, K=64, Hq=32, Hkv=8,
                             d=128, page=16, logit_dtype="bf16", ctx_kind="uniform",
                             ctx_args=(512, 16384), seed=5, agree_kind="per_request",
                             agree_args=(0.5, 0.9, 0.03), markov_dim=256, prefilter=128),
}


def config(name, **overrides):
    """A named workload, optionally with fields replaced (e.g. a smaller R)."""
    return replace(CONFIGS[name], **overrides)


# ---------------------------------------------------------------- bf16 bits
def to_bf16_bits(x):
    """float32 -> bf16 bit patterns, round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, np.uint16)
    flat_u, flat_o = u.reshape(-1), out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_u.size, step):
        c = flat_u[s:s + step]
        flat_o[s:s + step] = ((c + (((c >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)
    return out


def bf16_bits_to_f32(b):
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng, shape, scale=1.0):
    """N(0, scale^2) drawn in float32 chunks and stored as bf16 bits."""
    out = np.empty(shape, np.uint16)
    flat = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat.size, step):
        n = min(step, flat.size - s)
        x = rng.standard_normal(n, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        flat[s:s + n] = to_bf16_bits(x)
    return out


# ---------------------------------------------------------------- contexts
def draw_ctx_lens(cfg, rng):
    if cfg.ctx_kind == "fixed":
        return np.full((cfg.R,), cfg.ctx_args[0], np.int32)
    if cfg.ctx_kind == "uniform":
        lo, hi = cfg.ctx_args
        return rng.integers(lo, hi + 1, size=cfg.R).astype(np.int32)
    if cfg.ctx_kind == "lognormal":
        median, sigma, cap = cfg.ctx_args
        x = rng.lognormal(np.log(median), sigma, size=cfg.R)
        return np.clip(np.rint(x), 1, cap).astype(np.int32)
    raise ValueError(cfg.ctx_kind)


def draw_paged_cache(cfg, rng, ctx_lens):
    """Random-permuted page pool big enough for every round's growth.

    Returns k_cache, v_cache [num_pages, page, Hkv, d] (bf16 bits),
    block_table [R, max_pages] int32 (-1 past each request's pages).
    """
    grow = cfg.rounds * (cfg.L + 1)
    need = [(int(c) + grow + cfg.page - 1) // cfg.page for c in ctx_lens]
    max_pages = max(need)
    num_pages = sum(need) + cfg.spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    block_table = np.full((cfg.R, max_pages), -1, np.int32)
    pos = 0
    for r, n in enumerate(need):
        block_table[r, :n] = perm[pos:pos + n]
        pos += n
    shape = (num_pages, cfg.page, cfg.Hkv, cfg.d)
    k_cache = _normal_bf16(rng, shape)
    v_cache = _normal_bf16(rng, shape)
    return k_cache, v_cache, block_table


# ---------------------------------------------------------------- drafter
@dataclass
class DraftLogits:
    z: np.ndarray  # [R, L, V] bf16 bits (uint16) or float32
    boosted: np.ndarray = field(default=None)  # [R, L, 20] boosted token ids, Zipf rank order
    boost_val: np.ndarray = field(default=None)  # [20] boost added per Zipf rank


def draw_draft_logits(cfg, rng):
    R, L, V = cfg.R, cfg.L, cfg.V
    if not cfg.boost:
        z = (rng.standard_normal((R, L, V), dtype=np.float32) * np.float32(3.0))
        if cfg.logit_dtype == "bf16":
            z = to_bf16_bits(z)
        return DraftLogits(z=z)
    nb = 20
    ranks = np.arange(1, nb + 1, dtype=np.float64)
    boost_val = (8.0 * ranks ** -1.1).astype(np.float32)
    boosted = np.empty((R, L, nb), np.int64)
    temps = None
    if cfg.temp_range is not None:
        lo, hi = cfg.temp_range
        temps = rng.uniform(lo, hi, size=(R, L)).astype(np.float32)
    out = np.empty((R, L, V), np.uint16 if cfg.logit_dtype == "bf16" else np.float32)
    for r in range(R):
        row = rng.standard_normal((L, V), dtype=np.float32)
        for d in range(L):
            toks = rng.choice(V, size=nb, replace=False)
            boosted[r, d] = toks
            row[d, toks] += boost_val
            if temps is not None:
                row[d] /= temps[r, d]
        out[r] = to_bf16_bits(row) if cfg.logit_dtype == "bf16" else row
    return DraftLogits(z=out, boosted=boosted, boost_val=boost_val)


def draw_round_inputs(cfg, seed=None):
    """Everything one round consumes except the target logits."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    draft = draw_draft_logits(cfg, rng)
    ctx_lens = draw_ctx_lens(cfg, rng)
    k_cache, v_cache, block_table = draw_paged_cache(cfg, rng, ctx_lens)
    P = cfg.P
    q = _normal_bf16(rng, (cfg.R, P, cfg.Hq, cfg.d))
    k_tree = _normal_bf16(rng, (cfg.R, P, cfg.Hkv, cfg.d))
    v_tree = _normal_bf16(rng, (cfg.R, P, cfg.Hkv, cfg.d))
    agree = draw_agreement(cfg, rng)
    return dict(draft=draft, draft_logits=draft.z, ctx_lens=ctx_lens, k_cache=k_cache,
                v_cache=v_cache, block_table=block_table, q=q, k_tree=k_tree, v_tree=v_tree,
                agree=agree)


def draw_markov_head(cfg, seed=None, scale=0.02):
    """The parent-conditioned tree's Markov head: W, E [V, H] bf16 N(0, scale)
    (0.02 by default), and one anchor (root) token per request."""
    rng = np.random.default_rng([cfg.seed if seed is None else seed, 17])
    H = cfg.markov_dim
    W = _normal_bf16(rng, (cfg.V, H), scale=scale)
    E = _normal_bf16(rng, (cfg.V, H), scale=scale)
    anchors = rng.integers(0, cfg.V, size=cfg.R).astype(np.int32)
    return W, E, anchors


def draw_next_round(cfg, k, seed=None):
    """Round k >= 1 of a multi-round workload: new draft logits, queries and
    tree K/V (the cache and the context lengths carry over from round k - 1,
    as compaction left them). Seeded by (seed, k)."""
    base = cfg.seed if seed is None else seed
    rng = np.random.default_rng([base, k])
    draft = draw_draft_logits(cfg, rng)
    P = cfg.P
    q = _normal_bf16(rng, (cfg.R, P, cfg.Hq, cfg.d))
    k_tree = _normal_bf16(rng, (cfg.R, P, cfg.Hkv, cfg.d))
    v_tree = _normal_bf16(rng, (cfg.R, P, cfg.Hkv, cfg.d))
    agree = draw_agreement(cfg, rng)
    return dict(draft=draft, draft_logits=draft.z, q=q, k_tree=k_tree, v_tree=v_tree,
                agree=agree)


def draw_chain_inputs(cfg, seed=None, noise=(0.2, 1.0)):
    """One batch of drafted chains for stochastic verification: draft
    [R, L, V] and target [R, L+1, V] logits (cfg.logit_dtype), guesses
    tokens [R, L] int32, u [R, L] and r [R] float32 in [0, 1), and the
    per-request noise scale s [R]."""
    rng = np.random.default_rng([cfg.seed if seed is None else seed, 23])
    R, L, V = cfg.R, cfg.L, cfg.V
    draft = draw_draft_logits(cfg, rng).z
    bf16 = cfg.logit_dtype == "bf16"
    target = np.empty((R, L + 1, V), np.uint16 if bf16 else np.float32)
    tokens = np.empty((R, L), np.int32)
    sig = rng.uniform(noise[0], noise[1], size=R).astype(np.float32)
    one = replace(cfg, R=1, L=1)
    for i in range(R):
        zd = bf16_bits_to_f32(draft[i]) if bf16 else draft[i]
        zt = zd + sig[i] * rng.standard_normal((L, V), dtype=np.float32)
        last = draw_draft_logits(one, rng).z[0]
        target[i, :L] = to_bf16_bits(zt) if bf16 else zt
        target[i, L] = last[0]
        # Gumbel-max: -log of a unit exponential is a standard Gumbel draw
        e = rng.standard_exponential((L, V), dtype=np.float32)
        np.maximum(e, np.float32(1e-30), out=e)
        np.log(e, out=e)
        tokens[i] = np.argmax(zd - e, axis=-1)
    u = rng.random((R, L), dtype=np.float32)
    r = rng.random(R, dtype=np.float32)
    return dict(draft=draft, target=target, tokens=tokens, u=u, r=r, noise=sig)


def draw_confidences(R, L, seed=0):
    """[R, L] float32 chances that each drafted guess survives given that
    the ones before it did (see the module docstring)."""
    rng = np.random.default_rng([seed, 29])
    b = rng.uniform(0.5, 0.95, size=(R, 1))
    z = np.log(b / (1.0 - b)) - 0.15 * np.arange(L) + 0.5 * rng.standard_normal((R, L))
    return (1.0 / (1.0 + np.exp(-z))).astype(np.float32)


# ---------------------------------------------------------------- target
def draw_agreement(cfg, rng):
    """Per request: (base, decay) of the target's agreement with draft top-1."""
    if cfg.agree_kind == "const":
        return np.stack([np.full(cfg.R, cfg.agree_args[0]), np.zeros(cfg.R)], 1)
    if cfg.agree_kind == "decay":
        base, dec = cfg.agree_args
        return np.stack([np.full(cfg.R, base), np.full(cfg.R, dec)], 1)
    if cfg.agree_kind == "per_request":
        lo, hi, dec = cfg.agree_args
        return np.stack([rng.uniform(lo, hi, size=cfg.R), np.full(cfg.R, dec)], 1)
    raise ValueError(cfg.agree_kind)


def _path_seed(seed, r, path):
    """FNV-1a over (seed, request, token path): a stable per-prefix seed."""
    h = 0xCBF29CE484222325
    for v in (seed, r, len(path), *path):
        for byte in int(v & 0xFFFFFFFFFFFFFFFF).to_bytes(8, "little"):
            h ^= byte
            h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


class GreedyTarget:
    """A synthetic target model whose greedy next token depends only on the
    token path (the prefix drafted after the bonus token).

    At depth delta (number of drafted tokens on the path) it agrees with the
    drafter's top-1 token of draft row delta with probability
    a = base - decay * delta (clipped to [0, 1]); otherwise it picks another
    token: for boosted workloads one of the other 19 boosted tokens with
    weight exp(boost), for unboosted ones a token drawn from the softmax of
    that draft row with the top-1 excluded. Past the last draft row the token
    is uniform over the vocabulary. All choices are seeded by the path.
    """

    def __init__(self, cfg, draft, agree, seed=None):
        self.cfg = cfg
        self.draft = draft
        self.agree = agree
        self.seed = cfg.seed if seed is None else seed
        z = draft.z
        zf = bf16_bits_to_f32(z) if z.dtype == np.uint16 else z
        self._top1 = np.argmax(zf, axis=-1)  # [R, L] (data construction only)
        if draft.boosted is None:
            self._zrows = zf.astype(np.float64)
        else:
            self._zrows = None

    def next_token(self, r, path):
        cfg = self.cfg
        delta = len(path)
        rng = np.random.default_rng(_path_seed(self.seed, r, path))
        if delta >= cfg.L:
            return int(rng.integers(0, cfg.V))
        base, dec = self.agree[r]
        a = min(1.0, max(0.0, base - dec * delta))
        top1 = int(self._top1[r, delta])
        if rng.random() < a:
            return top1
        if self.draft.boosted is not None:
            toks = [int(t) for t in self.draft.boosted[r, delta] if int(t) != top1]
            w = np.exp(self.draft.boost_val[: len(toks)].astype(np.float64))
            return toks[int(rng.choice(len(toks), p=w / w.sum()))]
        row = self._zrows[r, delta]
        w = np.exp(row - row.max())
        w[top1] = 0.0
        return int(rng.choice(cfg.V, p=w / w.sum()))

    def logits_for_tree(self, tree_tokens, parents, n_nodes, dtype=None):
        """Target logits [R, P, V]: N(0,1) base, +20 on the greedy token of
        each node's path. Positions past n_nodes get base noise plus a
        uniform token. dtype follows the drafter's logits unless given."""
        cfg = self.cfg
        R, P, V = cfg.R, cfg.P, cfg.V
        dtype = dtype or cfg.logit_dtype
        rng = np.random.default_rng(self.seed + 7919)
        out = np.empty((R, P, V), np.uint16 if dtype == "bf16" else np.float32)
        for r in range(R):
            paths = {0: ()}
            row = rng.standard_normal((P, V), dtype=np.float32)
            for i in range(P):
                if i == 0 or i <= n_nodes[r]:
                    if i > 0:
                        paths[i] = paths[int(parents[r, i])] + (int(tree_tokens[r, i - 1]),)
                    t = self.next_token(r, paths[i])
                else:
                    t = int(rng.integers(0, V))
                row[i, t] += np.float32(20.0)
            out[r] = to_bf16_bits(row) if dtype == "bf16" else row
        return out

    def greedy_decode(self, r, n):
        """Plain autoregressive greedy decoding of n tokens under this target."""
        path = ()
        for _ in range(n):
            path = path + (self.next_token(r, path),)
        return list(path)
