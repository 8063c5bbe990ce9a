"""Pins for the oracle's per-depth log-softmax + top-K (step a1).

Pinned against closed forms, scipy's logsumexp, a full numpy sort and
torch's bf16 widening -- never against the oracle itself.
"""
import numpy as np
import pytest
import scipy.special
import torch

from speculative_decoding_draft_depth_gb300 import synth


def test_uniform_row_closed_form(orc):
    # every logit equal: lp = -log V exactly, ids are the K lowest ids
    V, K = 1000, 16
    z = np.full((3, V), 2.75, np.float32)
    lp, ids, logz, flags = orc.topk_logprobs(z, K)
    assert flags == 0
    np.testing.assert_allclose(lp, -np.log(V), rtol=0, atol=1e-13)
    np.testing.assert_array_equal(ids, np.tile(np.arange(K), (3, 1)))
    np.testing.assert_allclose(logz, 2.75 + np.log(V), atol=1e-13)


def test_one_hot_row_closed_form(orc):
    # one logit a, the rest 0: logZ = log(e^a + V - 1)
    V, K, a, hot = 500, 4, 6.5, 123
    z = np.zeros((1, V), np.float32)
    z[0, hot] = a
    lp, ids, _, _ = orc.topk_logprobs(z, K)
    logz = np.log(np.exp(a) + V - 1)
    assert ids[0, 0] == hot
    np.testing.assert_allclose(lp[0, 0], a - logz, atol=1e-13)
    np.testing.assert_array_equal(ids[0, 1:], [0, 1, 2])  # ties at 0 by lowest id
    np.testing.assert_allclose(lp[0, 1:], -logz, atol=1e-13)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_random_rows_against_scipy_and_full_sort(orc, dtype):
    rng = np.random.default_rng(11)
    rows, V, K = 40, 3001, 32
    zf = (rng.standard_normal((rows, V)) * 3).astype(np.float32)
    # plant exact duplicates so ties are exercised
    zf[:, 100] = zf[:, 2000]
    zf[:, 7] = zf[:, 5]
    if dtype == "bf16":
        z = synth.to_bf16_bits(zf)
        zw = torch.from_numpy(z.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    else:
        z = zf
        zw = zf.astype(np.float64)
    lp, ids, logz, _ = orc.topk_logprobs(z, K)
    ref_logz = scipy.special.logsumexp(zw, axis=1)
    np.testing.assert_allclose(logz, ref_logz, rtol=0, atol=1e-12)
    for r in range(rows):
        order = np.lexsort((np.arange(V), -zw[r]))  # value desc, id asc
        np.testing.assert_array_equal(ids[r], order[:K])
        np.testing.assert_allclose(lp[r], zw[r, order[:K]] - ref_logz[r], atol=1e-12)


def test_k_equals_v_and_probabilities_sum_to_one(orc):
    rng = np.random.default_rng(5)
    z = rng.standard_normal((4, 64)).astype(np.float32) * 4
    lp, ids, _, _ = orc.topk_logprobs(z, 64)
    np.testing.assert_allclose(np.exp(lp).sum(axis=1), 1.0, atol=1e-12)
    for r in range(4):
        assert sorted(ids[r].tolist()) == list(range(64))
        assert np.all(np.diff(lp[r]) <= 0)


def test_bad_k_rejected(orc):
    with pytest.raises(ValueError):
        orc.topk_logprobs(np.zeros((1, 8), np.float32), 9)


def test_nan_flagged(orc):
    z = np.zeros((2, 16), np.float32)
    z[1, 3] = np.nan
    _, _, _, flags = orc.topk_logprobs(z, 4)
    assert flags & orc.NAN_SEEN
