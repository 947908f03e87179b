"""Pins of the block-step oracles (causal conv1d + SiLU, gated RMSNorm) to things other than
themselves: library routines in float64, closed forms and invariants.  No GPU."""
import numpy as np
import pytest
import torch

from oracle import block


def rng(seed):
    return np.random.default_rng(seed)


# ---- causal conv1d ---------------------------------------------------------------------------

def torch_conv(x, w, bias, state=None, silu=True):
    """The library routine: torch's grouped conv1d in float64, left padding K - 1, trimmed."""
    xt = torch.from_numpy(x).double()                     # [b, L, C]
    if state is not None:
        xt = torch.cat([torch.from_numpy(state).double(), xt], dim=1)
    b, Lp, C = xt.shape
    K = w.shape[1]
    inp = xt.transpose(1, 2)                              # [b, C, L']
    pad = 0 if state is not None else K - 1
    out = torch.nn.functional.conv1d(inp, torch.from_numpy(w).double().unsqueeze(1),
                                     None if bias is None else torch.from_numpy(bias).double(),
                                     padding=pad, groups=C)
    L = x.shape[1]
    out = out[:, :, :L] if state is None else out[:, :, :L]
    out = out.transpose(1, 2)
    return (torch.nn.functional.silu(out) if silu else out).numpy()


@pytest.mark.parametrize("b,L,C,K", [(2, 37, 5, 4), (1, 9, 3, 2), (3, 64, 16, 4), (1, 5, 2, 1),
                                     (2, 3, 4, 4)])
def test_conv_matches_library_conv1d(b, L, C, K):
    r = rng(L * C + K)
    x = r.normal(size=(b, L, C))
    w = r.normal(size=(C, K))
    bias = r.normal(size=C)
    got, _ = block.causal_conv1d(x, w, bias)
    np.testing.assert_allclose(got, torch_conv(x, w, bias), rtol=1e-12, atol=1e-12)
    got_ns, _ = block.causal_conv1d(x, w, None, apply_silu=False)
    np.testing.assert_allclose(got_ns, torch_conv(x, w, None, silu=False), rtol=1e-12, atol=1e-12)


def test_conv_with_state_matches_library_on_the_concatenation():
    r = rng(3)
    b, L, C, K = 2, 20, 6, 4
    x = r.normal(size=(b, L, C))
    st = r.normal(size=(b, K - 1, C))
    w = r.normal(size=(C, K))
    bias = r.normal(size=C)
    got, _ = block.causal_conv1d(x, w, bias, state=st)
    np.testing.assert_allclose(got, torch_conv(x, w, bias, state=st), rtol=1e-12, atol=1e-12)


def test_conv_impulse_response_is_the_kernel_in_causal_order():
    """An impulse at t0 in channel c gives out[t0 + j] = w[c, K - 1 - j] (no bias, no SiLU)."""
    C, K, L, t0 = 3, 4, 12, 5
    w = np.arange(1.0, C * K + 1).reshape(C, K)
    x = np.zeros((1, L, C))
    x[0, t0, 1] = 1.0
    got, _ = block.causal_conv1d(x, w, None, apply_silu=False)
    for j in range(K):
        assert got[0, t0 + j, 1] == w[1, K - 1 - j]
    assert np.all(got[0, :t0] == 0) and np.all(got[0, :, 0] == 0) and np.all(got[0, :, 2] == 0)


def test_conv_width_one_is_pointwise():
    r = rng(5)
    x = r.normal(size=(2, 7, 4))
    w = r.normal(size=(4, 1))
    got, st = block.causal_conv1d(x, w, None, apply_silu=False)
    np.testing.assert_allclose(got, x * w[:, 0], rtol=0, atol=0)
    assert st.shape == (2, 0, 4)


def test_conv_split_sequence_equals_one_call():
    r = rng(9)
    b, L, C, K = 2, 30, 5, 4
    x = r.normal(size=(b, L, C))
    w = r.normal(size=(C, K))
    bias = r.normal(size=C)
    full, fin = block.causal_conv1d(x, w, bias)
    for cut in (1, 2, 3, 17):
        a, st = block.causal_conv1d(x[:, :cut], w, bias)
        c, st2 = block.causal_conv1d(x[:, cut:], w, bias, state=st)
        np.testing.assert_allclose(np.concatenate([a, c], axis=1), full, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(st2, fin, rtol=0, atol=0)
    np.testing.assert_array_equal(fin, x[:, L - (K - 1):])


def test_conv_pin_catches_a_flipped_kernel(monkeypatch):
    """A plausible mistake (the kernel applied in reverse) fails the impulse pin."""
    real = block.causal_conv1d

    def flipped(x, w, bias=None, state=None, apply_silu=True):
        return real(x, np.asarray(w)[:, ::-1], bias, state, apply_silu)

    monkeypatch.setattr(block, "causal_conv1d", flipped)
    with pytest.raises(AssertionError):
        test_conv_impulse_response_is_the_kernel_in_causal_order()


# ---- gated RMSNorm -----------------------------------------------------------------------------

def torch_norm(y, z, w, eps, g):
    yt = torch.from_numpy(y).double()
    D = yt.shape[-1]
    yr = yt.reshape(-1, D // g, g)
    out = torch.nn.functional.rms_norm(yr, (g,), eps=eps).reshape(yt.shape)
    if w is not None:
        out = out * torch.from_numpy(w).double()
    if z is not None:
        out = out * torch.nn.functional.silu(torch.from_numpy(z).double())
    return out.numpy()


@pytest.mark.parametrize("rows,D,g", [(7, 64, 64), (3, 5120, 5120), (4, 96, 32), (1, 1, 1),
                                      (5, 40, 8)])
def test_norm_matches_library_rms_norm(rows, D, g):
    r = rng(rows * D + g)
    y = r.normal(size=(rows, D)) * 3.0
    z = r.normal(size=(rows, D))
    w = r.normal(size=D)
    np.testing.assert_allclose(block.gated_rmsnorm(y, z, w, 1e-5, g), torch_norm(y, z, w, 1e-5, g),
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(block.gated_rmsnorm(y, None, None, 1e-3, g),
                               torch_norm(y, None, None, 1e-3, g), rtol=1e-12, atol=1e-12)


def test_norm_scale_invariance_and_unit_rms():
    r = rng(1)
    y = r.normal(size=(6, 48))
    a = block.gated_rmsnorm(y, eps=0.0)
    np.testing.assert_allclose(block.gated_rmsnorm(17.5 * y, eps=0.0), a, rtol=1e-13)
    np.testing.assert_allclose(np.sqrt(np.mean(a * a, axis=-1)), 1.0, rtol=1e-13)
    # groups are normalised independently of each other
    g = block.gated_rmsnorm(y, eps=0.0, group_size=16)
    for k in range(3):
        np.testing.assert_allclose(g[:, 16 * k:16 * (k + 1)],
                                   block.gated_rmsnorm(y[:, 16 * k:16 * (k + 1)], eps=0.0),
                                   rtol=1e-13)


def test_silu_matches_library():
    v = np.array([-30.0, -1.0, 0.0, 1.0, 2.5, 40.0])
    np.testing.assert_allclose(block.silu(v), torch.nn.functional.silu(torch.from_numpy(v)).numpy(),
                               rtol=1e-15, atol=0)
