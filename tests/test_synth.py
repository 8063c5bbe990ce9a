"""The seeded input generators of the chain and scheduler workloads hold the
recipe they state: the same seed gives the same batch, shapes and dtypes
follow the configuration, uniforms lie in [0, 1), guesses are sampled from
the draft rows, the target rows are the draft plus the request's noise, and
survival confidences fall along a block. No method arithmetic is checked
here (the generators hold none)."""
import numpy as np

from speculative_decoding_draft_depth_gb300 import synth


def _chains(R=8, L=3, V=4096, dtype="f32", seed=3):
    cfg = synth.config("tiny", R=R, L=L, V=V, logit_dtype=dtype, seed=seed)
    return cfg, synth.draw_chain_inputs(cfg)


def test_chain_inputs_are_seeded_and_shaped():
    cfg, a = _chains()
    _, b = _chains()
    _, c = _chains(seed=4)
    for k in ("draft", "target", "tokens", "u", "r", "noise"):
        np.testing.assert_array_equal(a[k], b[k])
    assert not np.array_equal(a["draft"], c["draft"])
    R, L, V = cfg.R, cfg.L, cfg.V
    assert a["draft"].shape == (R, L, V) and a["draft"].dtype == np.float32
    assert a["target"].shape == (R, L + 1, V) and a["target"].dtype == np.float32
    assert a["tokens"].shape == (R, L) and a["tokens"].dtype == np.int32
    assert ((a["tokens"] >= 0) & (a["tokens"] < V)).all()
    for k, shape in (("u", (R, L)), ("r", (R,))):
        assert a[k].shape == shape and a[k].dtype == np.float32
        assert ((a[k] >= 0) & (a[k] < 1)).all()
    _, h = _chains(dtype="bf16")
    assert h["draft"].dtype == np.uint16 and h["target"].dtype == np.uint16


def test_target_rows_are_the_draft_plus_the_request_noise():
    _, a = _chains(R=6, L=3, V=8192)
    d = a["target"][:, :-1] - a["draft"]
    sd = d.reshape(d.shape[0], -1).std(axis=1)
    np.testing.assert_allclose(sd, a["noise"], rtol=0.03)
    assert ((a["noise"] >= 0.2) & (a["noise"] <= 1.0)).all()


def test_guesses_are_sampled_from_the_draft_rows():
    """E over sampled guesses of log q(x) equals minus the entropy of q when
    x ~ q; the argmax or a uniform pick would miss it by far."""
    _, a = _chains(R=400, L=4, V=64, seed=9)
    z = a["draft"].astype(np.float64)
    m = z.max(-1, keepdims=True)
    logq = z - m - np.log(np.exp(z - m).sum(-1, keepdims=True))
    got = np.take_along_axis(logq, a["tokens"][..., None].astype(np.int64), -1).mean()
    want = (np.exp(logq) * logq).sum(-1).mean()
    assert abs(got - want) < 0.05, (got, want)
    top = logq.max(-1).mean()
    uniform = logq.mean()
    assert top - want > 0.5 and want - uniform > 0.5


def test_confidences_are_seeded_and_fall_along_a_block():
    c = synth.draw_confidences(2000, 8, seed=1)
    np.testing.assert_array_equal(c, synth.draw_confidences(2000, 8, seed=1))
    assert c.shape == (2000, 8) and c.dtype == np.float32
    assert ((c > 0) & (c < 1)).all()
    m = c.mean(axis=0)
    assert m[0] > m[-1] + 0.1
    assert (np.diff(m) < 0.01).all()
