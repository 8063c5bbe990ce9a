"""Plain fp64 CPU oracle for one batched DDTree draft-tree round.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The
product path (the CUDA library and its binding) never imports it, and the two
share no code; only the seeded input generators feed both.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double). This module
marshals numpy arrays into it; bf16 tensors travel as their raw 16-bit
patterns (``numpy.uint16``) and are widened exactly inside the C code. One
small helper is plain Python: ``prefixes_at_least`` enumerates the prefixes
near a score cut (the tie band of the tree tests), a handful per request,
with fp64 sums.

Pages cited (by title and section):
  "SparklingTree: 30-40% faster speculative decoding over DSpark",
      "How is the tree actually created?", Steps 1-4.
  "DDTree Explained: From Block Diffusion to Optimal Diffusion Draft Trees
      for Speculative Decoding", sections 3-5 (Prop. 1, Prop. 2, Lemma 1,
      Algorithm 1, implementation highlights).
  "Robot2050/TreeSpark", items 1, 2 and 4, and the batched engine
      description.
  "SparklingTree ...", "Building SparklingTree" and "Solving the candidate
      tree construction" (the prefilter and the Markov table: NEXT row 2).
  "DSpark Speculative Decoding Explained: Block Drafting and Confidence
      Checks", the probability rule and its toy (stochastic verification:
      NEXT row 3), and "Survival probability" / "Picking the budget" with the
      DSpark post's "Hardware aware prefix scheduler" (NEXT row 4).

Parity status: every function here is pinned by a ``-m "not gpu"`` test
against something other than itself (closed forms, brute force, library
routines for special cases, the pages' printed numbers).
"""
import ctypes
import os

import numpy as np

from . import build as _build

NAN_SEEN = 1
BAD_ARG = 2
BAD_PAGE = 4

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.orc_topk_logprobs.argtypes = [p, i32, i64, i64, i32, p, p, p]
        L.orc_topk_logprobs.restype = i32
        L.orc_build_tree.argtypes = [p, p, i32, i32, i32, i32, p, p, p, p, p, p]
        L.orc_build_tree.restype = i32
        L.orc_build_tree_bruteforce.argtypes = [p, p, i32, i32, i32, i64, p, p, p, p, p, p]
        L.orc_build_tree_bruteforce.restype = i64
        L.orc_build_mask.argtypes = [p, p, i32, i32, p]
        L.orc_build_mask.restype = None
        L.orc_tree_attention_rows.argtypes = [p, p, p, p, p, p, i32, i64, p, p, i32, i32,
                                              i32, i32, i32, i32, dbl, p, i64, p]
        L.orc_tree_attention_rows.restype = i32
        L.orc_argmax.argtypes = [p, i32, i64, i64, p]
        L.orc_argmax.restype = i32
        L.orc_walk.argtypes = [p, p, p, p, i32, i32, i32, p, p, p, p]
        L.orc_walk.restype = None
        L.orc_cond_tree.argtypes = [p, i32, p, p, i32, p, i32, i32, i64, i32, i32, i32, i32,
                                    p, p, p, p, p, p, p, p, p, p]
        L.orc_cond_tree.restype = i32
        L.orc_cond_parent_lists.argtypes = [p, i32, p, p, i32, i32, i32, i64, i32, i32, i64,
                                            p, p, p, p, p]
        L.orc_cond_parent_lists.restype = i32
        L.orc_compact.argtypes = [p, p, p, i32, i64, p, p, p, p, p, i32, i32, i32, i32, i32, i32]
        L.orc_compact.restype = i32
        L.orc_markov_table.argtypes = [p, i32, p, p, i32, p, i32, i32, i64, i32, i32, p, p]
        L.orc_markov_table.restype = i32
        L.orc_markov_tree.argtypes = [p, p, i32, i32, i32, i32, p, p, p, p, p, p]
        L.orc_markov_tree.restype = i32
        L.orc_markov_tree_bruteforce.argtypes = [p, p, i32, i32, i32, i64, p, p, p, p, p]
        L.orc_markov_tree_bruteforce.restype = i64
        L.orc_verify_chain.argtypes = [p, p, p, p, ctypes.c_double, i32, i64, p]
        L.orc_verify_chain.restype = i32
        L.orc_accept_stochastic.argtypes = [p, p, i32, p, p, p, i32, i32, i64, p, p, p]
        L.orc_accept_stochastic.restype = i32
        L.orc_schedule_prefix.argtypes = [p, i32, i32, p, p, p, p]
        L.orc_schedule_prefix.restype = i32
        L.orc_schedule_bruteforce.argtypes = [p, i32, i32, p]
        L.orc_schedule_bruteforce.restype = ctypes.c_double
        L.orc_num_threads.argtypes = []
        L.orc_num_threads.restype = i32
        _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().orc_num_threads())


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _logit_dtype(a):
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float64:
        return 2
    raise TypeError("logits must be float32, float64 or bf16 bits (uint16), got %s" % a.dtype)


def topk_logprobs(z, K):
    """Per row of z [..., V]: (lp [..., K] fp64, ids [..., K] int32, logZ [...], flags).

    lp = z - logsumexp(z); ids are the K largest logits, value descending,
    equal values by lower id.
    """
    z = np.ascontiguousarray(z)
    V = z.shape[-1]
    rows = int(np.prod(z.shape[:-1]))
    lp = np.empty(z.shape[:-1] + (K,), np.float64)
    ids = np.empty(z.shape[:-1] + (K,), np.int32)
    logz = np.empty(z.shape[:-1], np.float64)
    flags = lib().orc_topk_logprobs(_ptr(z), _logit_dtype(z), rows, V, K, _ptr(lp), _ptr(ids), _ptr(logz))
    if flags & BAD_ARG:
        raise ValueError("bad arguments to topk_logprobs")
    return lp, ids, logz, flags


class Tree:
    """Per-request tree arrays (R leading)."""

    def __init__(self, R, L, B):
        P = B + 1
        self.tokens = np.empty((R, B), np.int32)
        self.parents = np.empty((R, P), np.int32)
        self.depths = np.empty((R, P), np.int32)
        self.S = np.empty((R, P), np.float64)
        self.ranks = np.empty((R, P, L), np.int32)
        self.n_nodes = np.empty((R,), np.int32)


def build_tree(lp, ids, B):
    """Algorithm 1 (heap) on lp/ids [R, L, K] (lp widened to fp64)."""
    lp = np.ascontiguousarray(lp, dtype=np.float64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    R, L, K = lp.shape
    t = Tree(R, L, B)
    rc = lib().orc_build_tree(_ptr(lp), _ptr(ids), R, L, K, B, _ptr(t.tokens), _ptr(t.parents),
                              _ptr(t.depths), _ptr(t.S), _ptr(t.ranks), _ptr(t.n_nodes))
    if rc:
        raise ValueError("bad arguments to build_tree")
    return t


def prefixes_at_least(lp, ids, smin):
    """Every prefix of one request's token space whose score is at least smin.

    The DDTree prefix space ("DDTree Explained ...", section 4 and Algorithm
    1): a prefix is a path of tokens, one per depth, depth d's token drawn
    from the K candidates of that depth; its score is the fp64 sum of the
    chosen candidates' log-probs. lp/ids [L, K] with each depth's lp in
    descending order (the top-K order). Returns [(token path, score)].
    A depth-first walk visits a node's children in rank order and stops at
    the first one below smin: lp <= 0, so a prefix scores no more than its
    parent, and a later rank scores no more than an earlier one."""
    lp = np.ascontiguousarray(lp, dtype=np.float64)
    L, K = lp.shape
    out = []
    stack = [((), 0.0, 0)]
    while stack:
        path, S, d = stack.pop()
        if d == L:
            continue
        for j in range(K):
            s = S + lp[d, j]
            if s < smin:
                break
            p = path + (int(ids[d, j]),)
            out.append((p, s))
            stack.append((p, s, d + 1))
    return out


def build_tree_bruteforce(lp, ids, B, max_prefixes=5_000_000):
    """Sort-every-prefix construction for one request: lp/ids [L, K]."""
    lp = np.ascontiguousarray(lp, dtype=np.float64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    L, K = lp.shape
    t = Tree(1, L, B)
    n = lib().orc_build_tree_bruteforce(_ptr(lp), _ptr(ids), L, K, B, max_prefixes, _ptr(t.tokens),
                                        _ptr(t.parents), _ptr(t.depths), _ptr(t.S), _ptr(t.ranks),
                                        _ptr(t.n_nodes))
    if n < 0:
        raise ValueError("prefix space too large for brute force")
    return t


def build_mask(parents, n_nodes):
    """Ancestor bitmask [R, P, ceil(P/32)] uint32 from parents [R, P]."""
    parents = np.ascontiguousarray(parents, dtype=np.int32)
    n_nodes = np.ascontiguousarray(n_nodes, dtype=np.int32)
    R, P = parents.shape
    W = (P + 31) // 32
    mask = np.empty((R, P, W), np.uint32)
    lib().orc_build_mask(_ptr(parents), _ptr(n_nodes), R, P, _ptr(mask))
    return mask


def tree_attention_rows(q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_lens, mask, sel,
                        scale=None):
    """fp64 tree attention for the query rows sel [n, 3] = (r, i, h).

    q [R,P,Hq,d], k_tree/v_tree [R,P,Hkv,d], k_cache/v_cache [pages,page,Hkv,d]
    (all bf16 bit patterns, uint16); block_table [R, max_pages] int32;
    ctx_lens [R] int32; mask [R, P, W] uint32. Returns [n, d] fp64.
    """
    arrs = [np.ascontiguousarray(x) for x in (q, k_tree, v_tree, k_cache, v_cache)]
    for a in arrs:
        if a.dtype != np.uint16:
            raise TypeError("attention tensors are bf16 bit patterns (uint16)")
    q, k_tree, v_tree, k_cache, v_cache = arrs
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    ctx_lens = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    sel = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 3)
    R, P, Hq, d = q.shape
    Hkv = k_tree.shape[2]
    pages, page = k_cache.shape[0], k_cache.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.empty((sel.shape[0], d), np.float64)
    flags = lib().orc_tree_attention_rows(
        _ptr(q), _ptr(k_tree), _ptr(v_tree), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], pages, _ptr(ctx_lens), _ptr(mask), R, P, Hq, Hkv, d, page,
        float(scale), _ptr(sel), sel.shape[0], _ptr(out))
    if flags & BAD_ARG:
        raise ValueError("bad arguments to tree_attention_rows")
    return out, flags


def tree_attention(q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_lens, mask, scale=None):
    """All query rows: returns [R, P, Hq, d] fp64."""
    R, P, Hq, d = q.shape
    rr, ii, hh = np.meshgrid(np.arange(R), np.arange(P), np.arange(Hq), indexing="ij")
    sel = np.stack([rr.ravel(), ii.ravel(), hh.ravel()], axis=1)
    out, flags = tree_attention_rows(q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_lens,
                                     mask, sel, scale)
    return out.reshape(R, P, Hq, d), flags


def argmax(t):
    """First index of the row maximum over the last axis."""
    t = np.ascontiguousarray(t)
    V = t.shape[-1]
    rows = int(np.prod(t.shape[:-1]))
    out = np.empty(t.shape[:-1], np.int32)
    flags = lib().orc_argmax(_ptr(t), _logit_dtype(t), rows, V, _ptr(out))
    return out, flags


def walk(a, tree_tokens, parents, n_nodes, L):
    """Greedy verifier walk. Returns (acc_len, acc_nodes, acc_tokens, bonus)."""
    a = np.ascontiguousarray(a, dtype=np.int32)
    tree_tokens = np.ascontiguousarray(tree_tokens, dtype=np.int32)
    parents = np.ascontiguousarray(parents, dtype=np.int32)
    n_nodes = np.ascontiguousarray(n_nodes, dtype=np.int32)
    R, B = tree_tokens.shape
    acc_len = np.empty((R,), np.int32)
    acc_nodes = np.empty((R, L), np.int32)
    acc_tokens = np.empty((R, L + 1), np.int32)
    bonus = np.empty((R,), np.int32)
    lib().orc_walk(_ptr(a), _ptr(tree_tokens), _ptr(parents), _ptr(n_nodes), R, B, L,
                   _ptr(acc_len), _ptr(acc_nodes), _ptr(acc_tokens), _ptr(bonus))
    return acc_len, acc_nodes, acc_tokens, bonus


def compact(k_cache, v_cache, block_table, ctx_lens, k_tree, v_tree, acc_nodes, acc_len):
    """KV compaction in place on k_cache / v_cache / ctx_lens (numpy arrays)."""
    for a in (k_cache, v_cache, ctx_lens):
        if not a.flags.c_contiguous:
            raise ValueError("in-place arrays must be contiguous")
    k_tree = np.ascontiguousarray(k_tree)
    v_tree = np.ascontiguousarray(v_tree)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    acc_nodes = np.ascontiguousarray(acc_nodes, dtype=np.int32)
    acc_len = np.ascontiguousarray(acc_len, dtype=np.int32)
    R, P, Hkv, d = k_tree.shape
    L = acc_nodes.shape[1]
    pages, page = k_cache.shape[0], k_cache.shape[1]
    return lib().orc_compact(_ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
                             pages, _ptr(ctx_lens), _ptr(k_tree), _ptr(v_tree), _ptr(acc_nodes),
                             _ptr(acc_len), R, P, L, Hkv, d, page)


def round_(inputs, target_logits_fn=None, target_logits=None, B=None, K=None):
    """One whole round a1..a7 on host arrays (used for the CPU baseline).

    inputs: dict with draft_logits, q, k_tree, v_tree, k_cache, v_cache,
    block_table, ctx_lens (copied before compaction). Returns a dict.
    """
    z = inputs["draft_logits"]
    lp, ids, _, f1 = topk_logprobs(z, K)
    tree = build_tree(lp, ids, B)
    mask = build_mask(tree.parents, tree.n_nodes)
    attn, f2 = tree_attention(inputs["q"], inputs["k_tree"], inputs["v_tree"], inputs["k_cache"],
                              inputs["v_cache"], inputs["block_table"], inputs["ctx_lens"], mask)
    if target_logits is None:
        target_logits = target_logits_fn(tree)
    a, f3 = argmax(target_logits)
    L = z.shape[1]
    acc_len, acc_nodes, acc_tokens, bonus = walk(a, tree.tokens, tree.parents, tree.n_nodes, L)
    ctx = inputs["ctx_lens"].copy()
    f4 = compact(inputs["k_cache"], inputs["v_cache"], inputs["block_table"], ctx, inputs["k_tree"],
                 inputs["v_tree"], acc_nodes, acc_len)
    return dict(lp=lp, ids=ids, tree=tree, mask=mask, attn=attn, a=a, acc_len=acc_len,
                acc_nodes=acc_nodes, acc_tokens=acc_tokens, bonus=bonus, ctx_lens=ctx,
                flags=f1 | f2 | f3 | f4)


class CondTree:
    """Outputs of the parent-conditioned tree for R requests."""

    def __init__(self, R, D, k, F, N):
        P = N + 1
        self.tokens = np.full((R, N), -1, np.int32)
        self.parents = np.full((R, P), -1, np.int32)
        self.depths = np.full((R, P), -1, np.int32)
        self.S = np.zeros((R, P), np.float64)
        self.n_nodes = np.zeros(R, np.int32)
        self.cand_lp = np.zeros((R, D, F, k), np.float64)
        self.cand_ids = np.zeros((R, D, F, k), np.int32)
        self.frontier_tok = np.zeros((R, D, F), np.int32)


def cond_tree(ell, W, E, anchors, k, F, N, replay_lp=None, replay_ids=None):
    """Parent-conditioned tree ("Robot2050/TreeSpark", items 1-2): per-depth
    logits ell [R, D, V] plus the Markov bias W e(t_u) (W, E [V, H], same
    dtype), per-parent top-k, frontier of F by path score, top-N packing.
    With replay_lp / replay_ids [R, D, F, k] the per-parent lists are taken
    as given (the frontier and packing logic runs on them)."""
    ell = np.ascontiguousarray(ell)
    W = np.ascontiguousarray(W)
    E = np.ascontiguousarray(E)
    anchors = np.ascontiguousarray(anchors, dtype=np.int32)
    R, D, V = ell.shape
    H = W.shape[1]
    t = CondTree(R, D, k, F, N)
    rl = ri = None
    if replay_lp is not None:
        rl = np.ascontiguousarray(replay_lp, dtype=np.float64)
        ri = np.ascontiguousarray(replay_ids, dtype=np.int32)
    rc = lib().orc_cond_tree(_ptr(ell), _logit_dtype(ell), _ptr(W), _ptr(E), _logit_dtype(W),
                             _ptr(anchors), R, D, V, H, k, F, N,
                             _ptr(rl) if rl is not None else None,
                             _ptr(ri) if ri is not None else None,
                             _ptr(t.tokens), _ptr(t.parents), _ptr(t.depths), _ptr(t.S),
                             _ptr(t.n_nodes), _ptr(t.cand_lp), _ptr(t.cand_ids),
                             _ptr(t.frontier_tok))
    if rc:
        raise ValueError("bad arguments to cond_tree")
    return t


def cond_parent_lists(ell, W, E, req, depth, tok, k):
    """Children lists (lp [n, k] fp64, ids [n, k]) of given parents: request
    req[i], depth row depth[i] (0-based), parent token tok[i]."""
    ell = np.ascontiguousarray(ell)
    W = np.ascontiguousarray(W)
    E = np.ascontiguousarray(E)
    req = np.ascontiguousarray(req, dtype=np.int32)
    depth = np.ascontiguousarray(depth, dtype=np.int32)
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    R, D, V = ell.shape
    n = len(req)
    lp = np.empty((n, k), np.float64)
    ids = np.empty((n, k), np.int32)
    rc = lib().orc_cond_parent_lists(_ptr(ell), _logit_dtype(ell), _ptr(W), _ptr(E),
                                     _logit_dtype(W), R, D, V, W.shape[1], k, n, _ptr(req),
                                     _ptr(depth), _ptr(tok), _ptr(lp), _ptr(ids))
    if rc:
        raise ValueError("bad arguments to cond_parent_lists")
    return lp, ids


# ---------------------------------------------------------------- NEXT row 2
def markov_table(ell, W, E, anchors, C):
    """The SparklingTree prefilter and Markov table ("SparklingTree ...",
    "Solving the candidate tree construction"): cand [R, L, C] the C best
    tokens of every depth's logits (value desc, lower id first) and
    tab [R, L, C, C] fp64 with tab[r, d, a, b] = lp_d(b | a), the log-softmax
    over the kept tokens b of l_d[b] + W[b] . E[parent a] (parent a: the
    anchor at d = 0, else the a-th kept token of depth d - 1; rows a >= 1 of
    depth 0 are -inf)."""
    ell = np.ascontiguousarray(ell)
    W = np.ascontiguousarray(W)
    E = np.ascontiguousarray(E)
    anchors = np.ascontiguousarray(anchors, dtype=np.int32)
    R, L, V = ell.shape
    cand = np.empty((R, L, C), np.int32)
    tab = np.empty((R, L, C, C), np.float64)
    rc = lib().orc_markov_table(_ptr(ell), _logit_dtype(ell), _ptr(W), _ptr(E), _logit_dtype(W),
                                _ptr(anchors), R, L, V, W.shape[1], C, _ptr(cand), _ptr(tab))
    if rc:
        raise ValueError("bad arguments to markov_table")
    return cand, tab


class MarkovTree:
    """Outputs of the table heap for R requests (P = B + 1 positions)."""

    def __init__(self, R, B):
        P = B + 1
        self.tokens = np.full((R, B), -1, np.int32)
        self.parents = np.full((R, P), -1, np.int32)
        self.depths = np.full((R, P), -1, np.int32)
        self.S = np.zeros((R, P), np.float64)
        self.cand = np.full((R, P), -1, np.int32)
        self.n_nodes = np.zeros(R, np.int32)


def markov_tree(cand, tab, B):
    """Best-first tree over the table ("SparklingTree ...", "Building
    SparklingTree", Steps 2-6, with each parent's list read from the table):
    Algorithm 1 where a node's children are its table row ordered by
    (lp desc, token asc). tab may be the GPU's fp32 table (widened exactly)."""
    cand = np.ascontiguousarray(cand, dtype=np.int32)
    tab = np.ascontiguousarray(tab, dtype=np.float64)
    R, L, C = cand.shape
    t = MarkovTree(R, B)
    rc = lib().orc_markov_tree(_ptr(cand), _ptr(tab), R, L, C, B, _ptr(t.tokens), _ptr(t.parents),
                               _ptr(t.depths), _ptr(t.S), _ptr(t.cand), _ptr(t.n_nodes))
    if rc:
        raise ValueError("bad arguments to markov_tree")
    return t


def markov_tree_bruteforce(cand, tab, B, max_prefixes=2_000_000):
    """The same tree for one request by listing and sorting every prefix."""
    cand = np.ascontiguousarray(cand, dtype=np.int32)
    tab = np.ascontiguousarray(tab, dtype=np.float64)
    R, L, C = cand.shape
    assert R == 1
    t = MarkovTree(1, B)
    n = lib().orc_markov_tree_bruteforce(_ptr(cand), _ptr(tab), L, C, B, max_prefixes,
                                         _ptr(t.tokens), _ptr(t.parents), _ptr(t.depths),
                                         _ptr(t.S), _ptr(t.n_nodes))
    if n < 0:
        raise ValueError("too many prefixes for the brute force")
    return t


# ---------------------------------------------------------------- NEXT row 3
def verify_chain(p, q, tokens, u, r):
    """Stochastic verification of one drafted chain ("DSpark Speculative
    Decoding Explained ...", the probability rule): p [L+1, V] target and
    q [L, V] draft weights, tokens [L], uniforms u [L] (guess k kept iff
    u[k] < min(1, p/q)) and r (the replacement or bonus draw by inverse CDF
    in index order). Returns the committed tokens."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    L1, V = p.shape
    L = L1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    u = np.ascontiguousarray(u, dtype=np.float64)
    out = np.full(L + 1, -1, np.int32)
    n = lib().orc_verify_chain(_ptr(p), _ptr(q), _ptr(tokens), _ptr(u), float(r), L, V, _ptr(out))
    if n < 0:
        raise ValueError("bad arguments to verify_chain")
    return [int(t) for t in out[:n]]


def accept_stochastic(draft, target, tokens, u, r, n_guess=None):
    """The same rule on logits at temperature 1 for R requests: draft
    [R, L, V], target [R, L+1, V] (same dtype), tokens [R, L], u [R, L],
    r [R]. n_guess [R] (optional): request i verifies only its first
    n_guess[i] guesses. Returns acc_len [R] and acc_tokens [R, L+1] (-1
    padded)."""
    draft = np.ascontiguousarray(draft)
    target = np.ascontiguousarray(target)
    R, L, V = draft.shape
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    u = np.ascontiguousarray(u, dtype=np.float64)
    r = np.ascontiguousarray(r, dtype=np.float64)
    ng = None if n_guess is None else np.ascontiguousarray(n_guess, dtype=np.int32)
    acc_len = np.empty(R, np.int32)
    acc_tokens = np.empty((R, L + 1), np.int32)
    rc = lib().orc_accept_stochastic(_ptr(draft), _ptr(target), _logit_dtype(draft), _ptr(tokens),
                                     _ptr(u), _ptr(r), R, L, V,
                                     None if ng is None else _ptr(ng), _ptr(acc_len),
                                     _ptr(acc_tokens))
    if rc:
        raise ValueError("bad arguments to accept_stochastic")
    return acc_len, acc_tokens


def schedule_prefix(conf, cost):
    """The hardware-aware prefix scheduler ("DSpark Speculative Decoding
    Explained ...", "Survival probability" and "Picking the budget"):
    conf [R, L] conditional survival chances, cost [R*L + 1] step costs in
    ms indexed by the number of verified guesses. Returns n_keep [R],
    n_total, tokens per ms, expected tokens and the status bits."""
    conf = np.ascontiguousarray(conf, dtype=np.float64)
    R, L = conf.shape
    cost = np.ascontiguousarray(cost, dtype=np.float64)
    if cost.shape != (R * L + 1,):
        raise ValueError("cost must have R*L + 1 entries")
    n_keep = np.empty(R, np.int32)
    n_total = np.zeros(1, np.int32)
    stats = np.zeros(2, np.float64)
    rc = lib().orc_schedule_prefix(_ptr(conf), R, L, _ptr(cost), _ptr(n_keep), _ptr(n_total),
                                   _ptr(stats))
    if rc & BAD_ARG:
        raise ValueError("bad arguments to schedule_prefix")
    return n_keep, int(n_total[0]), float(stats[0]), float(stats[1]), int(rc)


def schedule_bruteforce(conf, cost):
    """Best tokens per ms over every subset of the slots (R*L <= 20)."""
    conf = np.ascontiguousarray(conf, dtype=np.float64)
    R, L = conf.shape
    cost = np.ascontiguousarray(cost, dtype=np.float64)
    return float(lib().orc_schedule_bruteforce(_ptr(conf), R, L, _ptr(cost)))
