"""Pins of the token-mixer block oracle (oracle/block.py) against what the
pages and the mathematics fix: the order of the block's steps (slides, frame
"The memory sits inside a familiar language-model block"; reading notes 2.9),
causality, sequence independence of packed batches, the convolution's tap
order, RMSNorm's normalisation, and linearity in the output projection.
Planted mistakes (a convolution that does not restart at a sequence start,
SiLU before the convolution, RMSNorm over the whole row instead of each
head) each fail one of them."""
import numpy as np
import pytest

from oracle import block, gates, recurrence

GP = dict(a=1.0, b=0.5, s=1.2, tau=4.0, log_mu_min=-2.0, comba_d=0.3)


def _params(rng, d_model, H, d, width=4):
    n_in = 4 * H * d + 4 * H
    return dict(W_in=rng.standard_normal((d_model, n_in)) / np.sqrt(d_model),
                conv_w=rng.standard_normal((3 * H * d, width)) * 0.5,
                rms_w=1.0 + 0.1 * rng.standard_normal(d),
                W_o=rng.standard_normal((H * d, d_model)) / np.sqrt(H * d))


def _run(x, p, H, d, cu=None, **kw):
    return block.block_forward(x, p["W_in"], p["conv_w"], p["rms_w"], p["W_o"], H, d, GP,
                               cu_seqlens=cu, **kw)


def test_short_conv_worked_example():
    # width 2, taps (0.5 on the previous token, 2 on the current one)
    P = np.array([[1.0], [-2.0], [3.0]])
    w = np.array([[0.5, 2.0]])
    out = block.short_conv(P, w, [0, 3])
    assert np.allclose(out[:, 0], [2.0, -4.0 + 0.5, 6.0 - 1.0])
    # a second sequence starting at token 1 restarts the window there
    out2 = block.short_conv(P, w, [0, 1, 3])
    assert np.allclose(out2[:, 0], [2.0, -4.0, 6.0 - 1.0])


def test_short_conv_is_a_causal_convolution():
    rng = np.random.default_rng(0)
    P = rng.standard_normal((9, 3))
    w = rng.standard_normal((3, 4))
    out = block.short_conv(P, w, [0, 9])
    for c in range(3):
        # full convolution with the kernel reversed (tap j is width-1-j back)
        ref = np.convolve(P[:, c], w[c, ::-1])[:9]
        assert np.allclose(out[:, c], ref)


def test_silu_and_rms_norm_closed_forms():
    x = np.array([-3.0, 0.0, 2.0])
    assert np.allclose(block.silu(x), x / (1 + np.exp(-x)))
    assert block.silu(np.array([0.0]))[0] == 0.0
    rng = np.random.default_rng(1)
    o = rng.standard_normal((5, 2, 8))
    r = block.rms_norm(o, np.ones(8), 0.0)
    assert np.allclose(np.sqrt(np.mean(r * r, axis=-1)), 1.0)
    assert np.allclose(block.rms_norm(3.7 * o, np.ones(8), 0.0), r)     # scale invariant


def test_block_is_causal():
    rng = np.random.default_rng(2)
    H, d, dm, T = 2, 4, 6, 10
    p = _params(rng, dm, H, d)
    x = rng.standard_normal((T, dm))
    y, _, _ = _run(x, p, H, d)
    x2 = x.copy()
    x2[6] += 1.0
    y2, _, _ = _run(x2, p, H, d)
    assert np.allclose(y[:6], y2[:6])
    assert not np.allclose(y[6:], y2[6:])


def test_packed_sequences_are_independent():
    rng = np.random.default_rng(3)
    H, d, dm = 2, 4, 6
    p = _params(rng, dm, H, d)
    xa, xb = rng.standard_normal((5, dm)), rng.standard_normal((7, dm))
    ya, SA, MA = _run(xa, p, H, d)
    yb, SB, MB = _run(xb, p, H, d)
    y, S, M = _run(np.concatenate([xa, xb]), p, H, d, cu=[0, 5, 12])
    assert np.allclose(y[:5], ya) and np.allclose(y[5:], yb)
    assert np.allclose(S[0], SA[0]) and np.allclose(S[1], SB[0])
    assert np.allclose(M[1], MB[0])


def test_block_steps_in_the_pages_order():
    """The core sees exactly the normalised, corrected q, k and the gates of
    the projections, and y is W_o applied to the gated, normalised output."""
    rng = np.random.default_rng(4)
    H, d, dm, T = 2, 4, 6, 9
    p = _params(rng, dm, H, d)
    x = rng.standard_normal((T, dm))
    y, S, M, parts = _run(x, p, H, d, return_parts=True)
    Hd = H * d
    P = x @ p["W_in"]
    conv = block.silu(block.short_conv(P[:, :3 * Hd], p["conv_w"], [0, T]))
    qh, kh = gates.prepare_qk(conv[:, :Hd].reshape(T, H, d), conv[:, Hd:2 * Hd].reshape(T, H, d),
                              GP["comba_d"])
    assert np.allclose(parts["q_hat"], qh) and np.allclose(parts["k_hat"], kh)
    assert np.allclose(np.linalg.norm(parts["k_hat"], axis=-1), 1.0)
    o, _, _ = recurrence.forward(qh, kh, conv[:, 2 * Hd:].reshape(T, H, d), parts["alpha"],
                                 parts["mu"], parts["eta"], parts["beta"])
    assert np.allclose(parts["o"], o)
    assert np.all(parts["alpha"] + parts["beta"] <= 1.0 + 1e-12)


def test_linear_in_the_output_projection():
    rng = np.random.default_rng(5)
    H, d, dm, T = 2, 4, 6, 8
    p = _params(rng, dm, H, d)
    x = rng.standard_normal((T, dm))
    W1, W2 = rng.standard_normal((H * d, dm)), rng.standard_normal((H * d, dm))
    y1, _, _ = _run(x, dict(p, W_o=W1), H, d)
    y2, _, _ = _run(x, dict(p, W_o=W2), H, d)
    y12, _, _ = _run(x, dict(p, W_o=W1 + W2), H, d)
    assert np.allclose(y12, y1 + y2)


# ---- planted mistakes, each caught by a pin above


_orig_conv = block.short_conv


@pytest.mark.parametrize("mistake", ["no_restart", "silu_first", "rms_whole_row"])
def test_planted_mistakes_are_caught(monkeypatch, mistake):
    rng = np.random.default_rng(6)
    H, d, dm = 2, 4, 6
    p = _params(rng, dm, H, d)
    xa, xb = rng.standard_normal((5, dm)), rng.standard_normal((7, dm))
    if mistake == "no_restart":
        monkeypatch.setattr(block, "short_conv", lambda P, w, cu: _orig_conv(P, w, [0, len(P)]))
        ya, _, _ = _run(xa, p, H, d)
        yb, _, _ = _run(xb, p, H, d)
        y, _, _ = _run(np.concatenate([xa, xb]), p, H, d, cu=[0, 5, 12])
        assert not (np.allclose(y[:5], ya) and np.allclose(y[5:], yb))
    elif mistake == "silu_first":
        T = 9
        x = rng.standard_normal((T, dm))
        _, _, _, parts = _run(x, p, H, d, return_parts=True)
        orig_silu = block.silu
        monkeypatch.setattr(block, "short_conv",
                            lambda P, w, cu: _orig_conv(orig_silu(P), w, cu))
        monkeypatch.setattr(block, "silu", lambda z: np.asarray(z, np.float64))
        _, _, _, bad = _run(x, p, H, d, return_parts=True)
        assert not np.allclose(bad["q_hat"], parts["q_hat"])
    else:
        rng2 = np.random.default_rng(7)
        o = rng2.standard_normal((5, H, d)) * np.array([1.0, 10.0])[None, :, None]
        good = block.rms_norm(o, np.ones(d), 0.0)
        flat = o.reshape(5, H * d)
        bad = (flat / np.sqrt(np.mean(flat * flat, axis=-1, keepdims=True))).reshape(5, H, d)
        # per-head RMS is 1 for the right form only
        assert np.allclose(np.sqrt(np.mean(good * good, axis=-1)), 1.0)
        assert not np.allclose(np.sqrt(np.mean(bad * bad, axis=-1)), 1.0)
