"""The C ABI: the library builds, loads and exports every function that
include/ddt.h declares; host-side validation rejects bad configurations
before touching the GPU. No compute call runs here (no GPU needed)."""
import ctypes
import os
import re

import pytest

from speculative_decoding_draft_depth_gb300 import build as ddt_build
from speculative_decoding_draft_depth_gb300 import ddt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ddt_build.build()
    return ddt.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "ddt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ddt_[a-z_]+)\s*\(", src)))


def test_header_declares_the_round(lib):
    names = _declared()
    for n in ("ddt_topk_logprobs", "ddt_build_tree", "ddt_build_mask", "ddt_tree_attention",
              "ddt_target_argmax", "ddt_walk", "ddt_compact", "ddt_accept", "ddt_round"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(ddt.EXPORTS) <= set(_declared())


def _declarations():
    """name -> parameter count of every function include/ddt.h declares."""
    src = open(os.path.join(ROOT, "include", "ddt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(ddt_[a-z_]+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header(lib):
    """The ctypes binding passes as many arguments as each declaration takes
    (a parameter added on one side only fails here, not on a GPU)."""
    decl = _declarations()
    assert set(ddt.EXPORTS) <= set(decl)
    for name in ddt.EXPORTS:
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == decl[name], (name, len(fn.argtypes), decl[name])


def _cfg(**kw):
    base = dict(R_max=64, L=15, V=151936, B=32, Hq=32, Hkv=8, d=128, page_size=16,
                max_pages_per_req=1040, num_pages=40000)
    base.update(kw)
    return ddt.make_config(**base)


def test_workspace_bytes_and_validation(lib):
    ws = ddt.workspace_bytes(_cfg())
    assert ws > 0
    # larger R_max never needs less workspace
    assert ddt.workspace_bytes(_cfg(R_max=128)) > ws
    for bad in (dict(R_max=0), dict(L=0), dict(B=0), dict(K=200, V=100), dict(Hq=30, Hkv=8),
                dict(page_size=0), dict(num_pages=0), dict(draft_dtype=7)):
        assert ddt.workspace_bytes(_cfg(**bad)) == 0, bad
    # a pool of 2^31 token rows or more: a4's row coordinates are 32-bit
    assert ddt.workspace_bytes(_cfg(num_pages=(2**31 - 1) // 16)) > 0
    for unsupported in (dict(L=19), dict(B=128), dict(d=96), dict(num_pages=2**27)):
        assert ddt.workspace_bytes(_cfg(**unsupported)) == 0, unsupported
    # the Markov-head trees: the head's width is required, and the table's
    # workspace grows with the prefilter width
    assert ddt.workspace_bytes(_cfg(prefilter=128)) == 0
    assert ddt.workspace_bytes(_cfg(markov_dim=256)) == 0
    assert ddt.workspace_bytes(_cfg(markov_dim=96, prefilter=128)) == 0
    assert ddt.workspace_bytes(_cfg(markov_dim=256, prefilter=129)) == 0
    mk = ddt.workspace_bytes(_cfg(markov_dim=256, prefilter=128))
    assert mk > ws + 64 * 15 * 128 * 128 * 4


def test_create_rejects_bad_config_without_a_gpu(lib):
    h = ctypes.c_void_p()
    assert lib.ddt_create(ctypes.byref(_cfg(B=0)), ctypes.byref(h)) == ddt.EINVAL
    assert lib.ddt_create(ctypes.byref(_cfg(d=96)), ctypes.byref(h)) == ddt.EUNSUPPORTED
    assert not h.value
    assert lib.ddt_create(None, ctypes.byref(h)) == ddt.EINVAL


def test_calls_reject_null_context(lib):
    assert lib.ddt_topk_logprobs(None, None, 1, None, None, None) == ddt.EINVAL
    assert lib.ddt_round(None, None, None) == ddt.EINVAL
    assert lib.ddt_round_conditioned(None, None, None, None, None, None) == ddt.EINVAL
    assert lib.ddt_round_markov(None, None, None, None, None, None) == ddt.EINVAL
    assert lib.ddt_markov_table(None, None, None, None, None, 1, None, None, None) == ddt.EINVAL
    assert lib.ddt_build_tree_markov(None, None, None, 1, None, None, None, None, None,
                                     None) == ddt.EINVAL
    assert lib.ddt_accept_stochastic(None, None, None, None, None, None, 1, None, None, None,
                                     None) == ddt.EINVAL
    assert lib.ddt_schedule_prefix(None, None, 1, None, None, None, None, None) == ddt.EINVAL
    assert lib.ddt_device_status(None, None) == ddt.EINVAL


def test_strerror(lib):
    assert lib.ddt_strerror(ddt.OK) == b"ok"
    assert lib.ddt_strerror(ddt.EINVAL) == b"invalid argument"
    assert lib.ddt_strerror(99) == b"unknown status"


def test_library_missing_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        ddt.load(str(tmp_path / "nope.so")) if ddt._lib is None else ddt_missing(tmp_path)


def ddt_missing(tmp_path):
    # once loaded, a second load path is not consulted; emulate a fresh import
    saved = ddt._lib
    ddt._lib = None
    try:
        ddt.load(str(tmp_path / "nope.so"))
    finally:
        ddt._lib = saved
