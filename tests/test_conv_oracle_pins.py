"""Pins of the causal conv1d oracle (oracle/conv.py) to facts outside it:
the width-1 closed form, the impulse response (the kernel read off in
reverse), numpy's full convolution on one sequence, sequence independence
in a packed batch, the SiLU closed form, and hand-derived
pre_num_conv_tokens for the article's cut patterns ([FLA-CP] §3.3, §5.1:
"flash-linear-attention 上下文并行CP ...")."""
import numpy as np
import pytest

from oracle import conv


def test_width_one_is_elementwise():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 9, 8))
    w = rng.standard_normal((8, 1))
    b = rng.standard_normal(8)
    y = conv.causal_conv1d(x, w, b, activation=None)
    np.testing.assert_allclose(y, x * w[:, 0] + b, rtol=1e-15)


def test_impulse_response_reads_the_kernel_backwards():
    W, T, p = 4, 12, 5
    w = np.arange(1.0, 1.0 + 8 * W).reshape(8, W)
    x = np.zeros((1, T, 8))
    x[0, p, 3] = 1.0
    y = conv.causal_conv1d(x, w, None, activation=None)
    expect = np.zeros(T)
    for t in range(p, p + W):
        expect[t] = w[3, W - 1 - (t - p)]
    np.testing.assert_array_equal(y[0, :, 3], expect)
    assert not np.delete(y[0], 3, axis=1).any()


@pytest.mark.parametrize("W", [1, 2, 4, 7])
def test_single_sequence_equals_numpy_convolve(W):
    rng = np.random.default_rng(2 + W)
    T, C = 50, 16
    x = rng.standard_normal((1, T, C))
    w = rng.standard_normal((C, W))
    b = rng.standard_normal(C)
    y = conv.causal_conv1d(x, w, b, activation=None)
    for c in range(C):
        ref = np.convolve(x[0, :, c], w[c, ::-1])[:T] + b[c]
        np.testing.assert_allclose(y[0, :, c], ref, rtol=1e-12, atol=1e-12)


def test_packed_sequences_are_independent():
    rng = np.random.default_rng(3)
    lengths = [5, 1, 0, 17, 3]
    cu = np.cumsum([0] + lengths)
    x = rng.standard_normal((1, cu[-1], 8))
    w = rng.standard_normal((8, 4))
    b = rng.standard_normal(8)
    y = conv.causal_conv1d(x, w, b, cu_seqlens=cu)
    for n in range(len(lengths)):
        s, e = cu[n], cu[n + 1]
        if e > s:
            np.testing.assert_array_equal(y[:, s:e], conv.causal_conv1d(x[:, s:e], w, b))


def test_silu_closed_form():
    x = np.array([[[0.0] * 8, [1.0] * 8, [-2.0] * 8, [30.0] * 8]])
    y = conv.causal_conv1d(x, np.ones((8, 1)), None, activation="silu")
    np.testing.assert_allclose(y[0, :, 0], [0.0, 1 / (1 + np.exp(-1.0)), -2 / (1 + np.exp(2.0)), 30.0],
                               rtol=1e-13)


@pytest.mark.parametrize("lengths,R,W,zigzag,expect", [
    ([3000, 4000, 3240], 2, 4, False, [0, 3]),       # cut inside the second sequence
    ([5120, 5120], 2, 4, False, [0, 0]),             # cut on a sequence start
    ([5118, 5122], 2, 4, False, [0, 2]),             # the sequence began 2 tokens before the cut
    ([5119, 5121], 2, 8, False, [0, 1]),
    ([7000, 3240], 4, 4, False, [0, 3, 3, 3]),       # the first sequence spans three segments
    ([8], 2, 4, True, [0, 2, 3, 3]),                 # zigzag parts of 2 tokens: halo capped by the start
    ([3, 5], 2, 3, True, [0, 2, 1, 2]),
])
def test_pre_num_conv_tokens_hand_derived(lengths, R, W, zigzag, expect):
    cu = np.cumsum([0] + lengths)
    assert conv.pre_num_conv_tokens(cu, cu[-1], R, W, zigzag=zigzag) == expect
