"""Pins for the causal Conv1D + SiLU oracle (the short convolution in front of
the selective SSM, "Mambaとは？Transformer以外の系列モデル", section Mamba block
のarchitecture, steps 2-3; its decode state: section training、prefill、decode
では計算の姿が違う).

Each pin is a function of an oracle callable ``fn(x, w, bias=None, state0=None)
-> (out, stateT)``.  The C loop and the NumPy restatement both pass every pin;
every planted mistake (a mutated copy built here on the CPU) fails one.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from oracle import numpy_oracle


def c_conv(x, w, bias=None, state0=None):
    return oracle.conv1d(x, w, bias=bias, state0=state0, threads=2)


def np_conv(x, w, bias=None, state0=None):
    return numpy_oracle.conv1d(x, w, bias=bias, state0=state0)


def silu(v):
    return v * expit(v)


def rand_conv(rng, batch=2, d=3, L=19, W=4, state=True):
    return dict(x=rng.standard_normal((batch, d, L)), w=rng.standard_normal((d, W)),
                bias=rng.standard_normal(d), state0=rng.standard_normal((batch, d, W - 1)) if state else None)


def pin_library_convolution(fn):
    """From a zero state the pre-activation is numpy's full convolution of the row
    with the reversed taps, truncated to the first L outputs (causal)."""
    rng = np.random.default_rng(1)
    for W in (1, 2, 4, 7):
        p = rand_conv(rng, W=W, state=False)
        out, _ = fn(**p)
        for b in range(p["x"].shape[0]):
            for c in range(p["x"].shape[1]):
                pre = np.convolve(p["x"][b, c], p["w"][c, ::-1])[: p["x"].shape[2]] + p["bias"][c]
                np.testing.assert_allclose(out[b, c], silu(pre), rtol=1e-12, atol=1e-14)


def pin_identity_tap(fn):
    """Only the last tap set: the output is silu(x + bias), whatever the state."""
    rng = np.random.default_rng(2)
    p = rand_conv(rng, W=4)
    p["w"] = np.zeros_like(p["w"])
    p["w"][:, -1] = 1.0
    out, _ = fn(**p)
    np.testing.assert_allclose(out, silu(p["x"] + p["bias"][None, :, None]), rtol=1e-13, atol=1e-15)


def pin_impulse_response(fn):
    """An impulse at t = 0 from a zero state: silu(w[W-1-t]) for t < W, then silu(0) = 0."""
    W, L = 4, 9
    w = np.array([[0.5, -1.25, 2.0, 0.75]])
    x = np.zeros((1, 1, L))
    x[0, 0, 0] = 1.0
    out, _ = fn(x, w)
    want = np.zeros(L)
    want[:W] = silu(w[0, ::-1])
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-14, atol=1e-15)


def pin_causality(fn):
    """Changing inputs at t >= k leaves every output before k unchanged."""
    rng = np.random.default_rng(3)
    p = rand_conv(rng, L=25)
    out, _ = fn(**p)
    q = dict(p, x=p["x"].copy())
    q["x"][:, :, 12:] += 5.0
    out2, _ = fn(**q)
    np.testing.assert_array_equal(out[:, :, :12], out2[:, :, :12])
    assert np.all(np.abs(out[:, :, 12] - out2[:, :, 12]) > 0)


def pin_state_is_the_last_inputs(fn):
    """The state after a sequence is its last W-1 inputs (shorter sequences keep
    the tail of the incoming state in front of them)."""
    rng = np.random.default_rng(4)
    p = rand_conv(rng, L=10, W=4)
    _, sT = fn(**p)
    np.testing.assert_array_equal(sT, p["x"][:, :, -3:])
    p = rand_conv(rng, L=2, W=5)
    _, sT = fn(**p)
    np.testing.assert_array_equal(sT, np.concatenate([p["state0"][:, :, 2:], p["x"]], axis=2))


def pin_split_continue(fn):
    """Convolving [0, L) equals convolving [0, k), then [k, L) from the first part's state."""
    rng = np.random.default_rng(5)
    for W in (2, 4, 6):
        p = rand_conv(rng, L=23, W=W)
        out, sT = fn(**p)
        for k in (1, W - 1, 11):
            o1, s1 = fn(p["x"][:, :, :k], p["w"], p["bias"], p["state0"])
            o2, s2 = fn(p["x"][:, :, k:], p["w"], p["bias"], s1)
            np.testing.assert_allclose(np.concatenate([o1, o2], axis=2), out, rtol=1e-13, atol=1e-15)
            np.testing.assert_array_equal(s2, sT)


PINS = [pin_library_convolution, pin_identity_tap, pin_impulse_response, pin_causality,
        pin_state_is_the_last_inputs, pin_split_continue]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
@pytest.mark.parametrize("impl", [c_conv, np_conv], ids=["c", "numpy"])
def test_pin(impl, pin):
    pin(impl)


def test_two_conv_oracles_agree():
    rng = np.random.default_rng(6)
    for shape in [(2, 5, 33, 4), (1, 3, 2, 5), (3, 2, 40, 1)]:
        b, d, L, W = shape
        p = rand_conv(rng, b, d, L, W)
        oc, sc = c_conv(**p)
        on, sn = np_conv(**p)
        np.testing.assert_allclose(oc, on, rtol=1e-13, atol=1e-15)
        np.testing.assert_array_equal(sc, sn)


def test_conv_step_equals_conv():
    """Tokens fed one by one through the decode step reproduce the sequence conv."""
    rng = np.random.default_rng(7)
    p = rand_conv(rng, 2, 3, 12, 4)
    out, sT = oracle.conv1d(**p)
    state = p["state0"]
    for t in range(12):
        y, state = oracle.conv1d_step(state, p["x"][:, :, t], p["w"], p["bias"])
        np.testing.assert_array_equal(y, out[:, :, t])
    np.testing.assert_array_equal(state, sT)


# ---------------------------------------------------- planted mistakes ----

def _mutant(kind):
    def fn(x, w, bias=None, state0=None):
        x, w = np.asarray(x, np.float64), np.asarray(w, np.float64)
        batch, d, L = x.shape
        W = w.shape[1]
        if kind == "reversed_taps":
            w = w[:, ::-1]
        s0 = np.zeros((batch, d, W - 1)) if (state0 is None or kind == "state_ignored") else state0
        xt = np.concatenate([np.zeros((batch, d, 1)), s0, x], axis=2)  # one extra zero in front
        shift = 0 if kind == "window_one_early" else 1
        pre = np.zeros((batch, d, L))
        if bias is not None and kind != "bias_ignored":
            pre += bias[None, :, None]
        for k in range(W):
            pre += w[None, :, k, None] * xt[:, :, shift + k:shift + k + L]
        out = pre if kind == "no_silu" else pre * expit(pre)
        full = xt[:, :, 1:]
        sT = full[:, :, : W - 1] if kind == "state_first_inputs" else full[:, :, L:]
        return out, sT.copy()
    return fn


MUTANTS = ["reversed_taps", "state_ignored", "window_one_early", "bias_ignored", "no_silu", "state_first_inputs"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistake(kind):
    fn = _mutant(kind)
    failed = []
    for pin in PINS:
        try:
            pin(fn)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {kind}"


def test_unmutated_copy_passes():
    fn = _mutant("none")
    for pin in PINS:
        pin(fn)
