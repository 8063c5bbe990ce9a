"""Thin ctypes binding over libddt.so (include/ddt.h).

Argument marshalling only: every step of the round runs in the library's
sm_103a kernels. Tensors are torch CUDA tensors (torch supplies device
memory and streams); bf16 tensors may be torch.bfloat16 or int16/uint16
views of the same bits. There is no fallback: if the library is missing or
fails to load, loading raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libddt.so")

OK, EINVAL, EUNSUPPORTED, ECUDA, ENOMEM = 0, 1, 2, 3, 4
BF16, F32 = 0, 1
DEV_NAN_LOGITS, DEV_BAD_PAGE, DEV_BAD_TREE, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8

EXPORTS = ("ddt_create", "ddt_destroy", "ddt_workspace_bytes", "ddt_topk_logprobs",
           "ddt_build_tree", "ddt_build_tree_conditioned", "ddt_build_mask", "ddt_tree_attention", "ddt_target_argmax",
           "ddt_walk", "ddt_compact", "ddt_accept", "ddt_round", "ddt_round_conditioned",
           "ddt_markov_table", "ddt_build_tree_markov", "ddt_round_markov",
           "ddt_accept_stochastic", "ddt_schedule_prefix", "ddt_device_status", "ddt_strerror",
           "ddt_last_cuda_error", "ddt_debug_arm_attention_timeout")


class DdtError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _lib.ddt_strerror(status).decode() if _lib is not None else str(status)
        extra = ""
        if status == ECUDA and _lib is not None:
            extra = " (cudaError %d)" % _lib.ddt_last_cuda_error()
        super().__init__("%s: %s%s" % (where, msg, extra))


class Config(ctypes.Structure):
    _fields_ = [("R_max", ctypes.c_int32), ("L", ctypes.c_int32), ("V", ctypes.c_int32),
                ("B", ctypes.c_int32), ("K", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages_per_req", ctypes.c_int32), ("num_pages", ctypes.c_int64),
                ("draft_dtype", ctypes.c_int32), ("target_dtype", ctypes.c_int32),
                ("markov_dim", ctypes.c_int32), ("frontier", ctypes.c_int32),
                ("prefilter", ctypes.c_int32)]


_P = ctypes.c_void_p


class RoundArgs(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32)] + [(n, _P) for n in (
        "draft_logits", "target_logits", "q", "k_tree", "v_tree", "k_cache", "v_cache",
        "block_table", "ctx_lens", "top_lp", "top_ids", "tree_tokens", "parents", "depths",
        "n_nodes", "mask", "attn_out", "target_argmax", "acc_len", "acc_nodes", "acc_tokens",
        "bonus", "att_event_begin", "att_event_end")]


_lib = None


def load(path=LIB_PATH):
    """Load libddt.so and declare its signatures; raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libddt.so not built at %s (run __graft_entry__.build())" % path)
    L = ctypes.CDLL(path)
    i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "ddt_create": ([ctypes.POINTER(Config), ctypes.POINTER(_P)], i32),
        "ddt_destroy": ([_P], None),
        "ddt_workspace_bytes": ([ctypes.POINTER(Config)], sz),
        "ddt_topk_logprobs": ([_P, _P, i32, _P, _P, _P], i32),
        "ddt_build_tree": ([_P, _P, _P, i32, _P, _P, _P, _P, _P, _P], i32),
        "ddt_build_mask": ([_P, _P, _P, i32, _P, _P], i32),
        "ddt_build_tree_conditioned": ([_P, _P, _P, _P, _P, i32, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _P], i32),
        "ddt_tree_attention": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, i32, _P, _P], i32),
        "ddt_target_argmax": ([_P, _P, i32, _P, _P], i32),
        "ddt_walk": ([_P, _P, _P, _P, _P, i32, _P, _P, _P, _P, _P], i32),
        "ddt_compact": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, i32, _P], i32),
        "ddt_accept": ([_P, _P, _P, _P, _P, i32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
                       i32),
        "ddt_round": ([_P, ctypes.POINTER(RoundArgs), _P], i32),
        "ddt_round_conditioned": ([_P, ctypes.POINTER(RoundArgs), _P, _P, _P, _P], i32),
        "ddt_markov_table": ([_P, _P, _P, _P, _P, i32, _P, _P, _P], i32),
        "ddt_build_tree_markov": ([_P, _P, _P, i32, _P, _P, _P, _P, _P, _P], i32),
        "ddt_round_markov": ([_P, ctypes.POINTER(RoundArgs), _P, _P, _P, _P], i32),
        "ddt_accept_stochastic": ([_P, _P, _P, _P, _P, _P, i32, _P, _P, _P, _P], i32),
        "ddt_schedule_prefix": ([_P, _P, i32, _P, _P, _P, _P, _P], i32),
        "ddt_device_status": ([_P, ctypes.POINTER(i32)], i32),
        "ddt_debug_arm_attention_timeout": ([_P, i64], i32),
        "ddt_strerror": ([i32], ctypes.c_char_p),
        "ddt_last_cuda_error": ([], i32),
    }
    for name, (argt, rest) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = argt
        fn.restype = rest
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, where):
    if status != OK:
        raise DdtError(status, where)


def make_config(R_max, L, V, B, Hq, Hkv, d, page_size, max_pages_per_req, num_pages, K=0,
                draft_dtype=BF16, target_dtype=BF16, markov_dim=0, frontier=0, prefilter=0):
    return Config(R_max, L, V, B, K, Hq, Hkv, d, page_size, max_pages_per_req, num_pages,
                  draft_dtype, target_dtype, markov_dim, frontier, prefilter)


def workspace_bytes(cfg):
    return int(load().ddt_workspace_bytes(ctypes.byref(cfg)))


class Context:
    """One ddt_ctx (and its device workspace) on the current CUDA device."""

    def __init__(self, cfg):
        lib = load()
        self.cfg = cfg
        h = _P()
        _check(lib.ddt_create(ctypes.byref(cfg), ctypes.byref(h)), "ddt_create")
        self._h = h
        self.K = cfg.K if cfg.K else min(cfg.B, cfg.V)
        self.P = cfg.B + 1
        self.W = (self.P + 31) // 32

    def close(self):
        if getattr(self, "_h", None):
            _lib.ddt_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- one call per C entry point -----------------------------------------
    def ddt_topk_logprobs(self, draft_logits, R, top_lp, top_ids, stream=None):
        _check(_lib.ddt_topk_logprobs(self._h, _ptr(draft_logits), R, _ptr(top_lp), _ptr(top_ids),
                                      _stream(stream)), "ddt_topk_logprobs")

    def ddt_build_tree(self, top_lp, top_ids, R, tree_tokens, parents, depths, n_nodes, mask=None,
                       stream=None):
        _check(_lib.ddt_build_tree(self._h, _ptr(top_lp), _ptr(top_ids), R, _ptr(tree_tokens),
                                   _ptr(parents), _ptr(depths), _ptr(n_nodes), _ptr(mask),
                                   _stream(stream)), "ddt_build_tree")

    def ddt_build_tree_conditioned(self, draft_logits, W, E, anchors, R, tree_tokens, parents,
                                   depths, n_nodes, mask=None, cand_lp=None, cand_ids=None,
                                   frontier_tok=None, stream=None):
        _check(_lib.ddt_build_tree_conditioned(
            self._h, _ptr(draft_logits), _ptr(W), _ptr(E), _ptr(anchors), R, _ptr(cand_lp),
            _ptr(cand_ids), _ptr(frontier_tok), _ptr(tree_tokens), _ptr(parents), _ptr(depths),
            _ptr(n_nodes), _ptr(mask), _stream(stream)), "ddt_build_tree_conditioned")

    def ddt_build_mask(self, parents, n_nodes, R, mask, stream=None):
        _check(_lib.ddt_build_mask(self._h, _ptr(parents), _ptr(n_nodes), R, _ptr(mask),
                                   _stream(stream)), "ddt_build_mask")

    def ddt_tree_attention(self, q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_lens, mask,
                           R, out, stream=None):
        _check(_lib.ddt_tree_attention(self._h, _ptr(q), _ptr(k_tree), _ptr(v_tree), _ptr(k_cache),
                                       _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), _ptr(mask),
                                       R, _ptr(out), _stream(stream)), "ddt_tree_attention")

    def ddt_target_argmax(self, target_logits, R, argmax_out, stream=None):
        _check(_lib.ddt_target_argmax(self._h, _ptr(target_logits), R, _ptr(argmax_out),
                                      _stream(stream)), "ddt_target_argmax")

    def ddt_walk(self, argmax, tree_tokens, parents, n_nodes, R, acc_len, acc_nodes, acc_tokens,
                 bonus, stream=None):
        _check(_lib.ddt_walk(self._h, _ptr(argmax), _ptr(tree_tokens), _ptr(parents),
                             _ptr(n_nodes), R, _ptr(acc_len), _ptr(acc_nodes), _ptr(acc_tokens),
                             _ptr(bonus), _stream(stream)), "ddt_walk")

    def ddt_compact(self, k_cache, v_cache, block_table, ctx_lens, k_tree, v_tree, acc_nodes,
                    acc_len, R, stream=None):
        _check(_lib.ddt_compact(self._h, _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                _ptr(ctx_lens), _ptr(k_tree), _ptr(v_tree), _ptr(acc_nodes),
                                _ptr(acc_len), R, _stream(stream)), "ddt_compact")

    def ddt_accept(self, target_logits, tree_tokens, parents, n_nodes, R, argmax_out, acc_len,
                   acc_nodes, acc_tokens, bonus, k_cache, v_cache, block_table, k_tree, v_tree,
                   ctx_lens, stream=None):
        _check(_lib.ddt_accept(self._h, _ptr(target_logits), _ptr(tree_tokens), _ptr(parents),
                               _ptr(n_nodes), R, _ptr(argmax_out), _ptr(acc_len), _ptr(acc_nodes),
                               _ptr(acc_tokens), _ptr(bonus), _ptr(k_cache), _ptr(v_cache),
                               _ptr(block_table), _ptr(k_tree), _ptr(v_tree), _ptr(ctx_lens),
                               _stream(stream)), "ddt_accept")

    def ddt_accept_stochastic(self, draft_logits, target_logits, draft_tokens, u, r, R, acc_len,
                              acc_tokens, n_guess=None, stream=None):
        """Temperature-1 verification of R drafted chains of L guesses.
        n_guess: None (every guess), or an int32 [R] CUDA tensor of the
        guesses each request verifies, e.g. ddt_schedule_prefix's n_keep."""
        _check(_lib.ddt_accept_stochastic(self._h, _ptr(draft_logits), _ptr(target_logits),
                                          _ptr(draft_tokens), _ptr(u), _ptr(r), R, _ptr(acc_len),
                                          _ptr(acc_tokens), _ptr(n_guess), _stream(stream)),
               "ddt_accept_stochastic")

    def ddt_schedule_prefix(self, conf, R, cost_ms, n_keep, n_total=None, stats=None,
                            stream=None):
        """The guesses each of R requests verifies: conf [R, L] f32,
        cost_ms [R*L + 1] f32, n_keep [R] i32 out; n_total [1] i32 and
        stats [2] f64 (tokens per ms, expected tokens) optional."""
        _check(_lib.ddt_schedule_prefix(self._h, _ptr(conf), R, _ptr(cost_ms), _ptr(n_keep),
                                        _ptr(n_total), _ptr(stats), _stream(stream)),
               "ddt_schedule_prefix")

    def ddt_round(self, R, bufs, stream=None, att_events=None):
        """bufs: dict of tensors named like the fields of ddt_round_args.
        att_events: optional (begin, end) torch.cuda.Event pair, recorded by
        the library around the attention launch (each already created, e.g.
        by one earlier record())."""
        a = self._round_args(R, bufs, att_events)
        _check(_lib.ddt_round(self._h, ctypes.byref(a), _stream(stream)), "ddt_round")

    def ddt_markov_table(self, draft_logits, W, E, anchors, R, cand_ids, tab_lp, stream=None):
        _check(_lib.ddt_markov_table(self._h, _ptr(draft_logits), _ptr(W), _ptr(E), _ptr(anchors),
                                     R, _ptr(cand_ids), _ptr(tab_lp), _stream(stream)),
               "ddt_markov_table")

    def ddt_build_tree_markov(self, cand_ids, tab_lp, R, tree_tokens, parents, depths, n_nodes,
                              mask=None, stream=None):
        _check(_lib.ddt_build_tree_markov(self._h, _ptr(cand_ids), _ptr(tab_lp), R,
                                          _ptr(tree_tokens), _ptr(parents), _ptr(depths),
                                          _ptr(n_nodes), _ptr(mask), _stream(stream)),
               "ddt_build_tree_markov")

    def ddt_round_markov(self, R, bufs, W, E, anchors, stream=None, att_events=None):
        """The SparklingTree round: bufs as for ddt_round (top_lp / top_ids
        unused), W, E [V, H] bf16 and anchors [R] int32."""
        a = self._round_args(R, bufs, att_events)
        _check(_lib.ddt_round_markov(self._h, ctypes.byref(a), _ptr(W), _ptr(E), _ptr(anchors),
                                     _stream(stream)), "ddt_round_markov")

    def _round_args(self, R, bufs, att_events):
        """ddt_round_args from a dict of tensors named like its fields (absent
        ones are NULL) and the optional attention event pair."""
        a = RoundArgs()
        a.R = R
        for name, _ in RoundArgs._fields_[1:]:
            if name.startswith("att_event"):
                continue
            setattr(a, name, _ptr(bufs.get(name)))
        if att_events is not None:
            a.att_event_begin = ctypes.c_void_p(att_events[0].cuda_event)
            a.att_event_end = ctypes.c_void_p(att_events[1].cuda_event)
        return a

    def ddt_round_conditioned(self, R, bufs, W, E, anchors, stream=None, att_events=None):
        """The parent-conditioned round: bufs as for ddt_round (draft_logits are
        the backbone's per-depth logits; top_lp / top_ids unused), W, E [V, H]
        bf16 and anchors [R] int32."""
        a = self._round_args(R, bufs, att_events)
        _check(_lib.ddt_round_conditioned(self._h, ctypes.byref(a), _ptr(W), _ptr(E), _ptr(anchors),
                                          _stream(stream)), "ddt_round_conditioned")

    def ddt_device_status(self):
        out = ctypes.c_int32(0)
        _check(_lib.ddt_device_status(self._h, ctypes.byref(out)), "ddt_device_status")
        return out.value

    def ddt_debug_arm_attention_timeout(self, wait_cycles):
        """Test only: the next a4 launch starts with a bounded wait that runs
        out after wait_cycles SM cycles (see include/ddt.h)."""
        _check(_lib.ddt_debug_arm_attention_timeout(self._h, int(wait_cycles)),
               "ddt_debug_arm_attention_timeout")

    # -- allocation helper (plumbing) ----------------------------------------
    def alloc_outputs(self, R, device="cuda"):
        """Output buffers of one round for R requests, named as in ddt_round_args."""
        c, K, P, W = self.cfg, self.K, self.P, self.W
        i32 = dict(dtype=torch.int32, device=device)
        return dict(
            top_lp=torch.empty((R, c.L, K), dtype=torch.float32, device=device),
            top_ids=torch.empty((R, c.L, K), **i32),
            tree_tokens=torch.empty((R, c.B), **i32),
            parents=torch.empty((R, P), **i32),
            depths=torch.empty((R, P), **i32),
            n_nodes=torch.empty((R,), **i32),
            mask=torch.empty((R, P, W), **i32),
            attn_out=torch.empty((R, P, c.Hq, c.d), dtype=torch.float32, device=device),
            target_argmax=torch.empty((R, P), **i32),
            acc_len=torch.empty((R,), **i32),
            acc_nodes=torch.empty((R, c.L), **i32),
            acc_tokens=torch.empty((R, c.L + 1), **i32),
            bonus=torch.empty((R,), **i32),
        )
