"""Parity of the recurrent step (ssd_step_fwd, through the C ABI) with the CPU oracle.

The oracle of one step is the oracle's sequential scan over a single token, with the step's
entering state as initial state: the same recurrence, written once in plain C.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, assert_close, dtype_name, sample_heads, to_device
from mamba_ssd_scan_05_b300 import (SSDError, ssd_scan_fwd, ssd_step_fwd, workloads)

pytestmark = pytest.mark.gpu


def step_inputs(b, H, P, N, G, dtype, seed, state=True, L=1):
    return workloads.make_shape_inputs(b, L, H, P, N, G, dtype, seed=seed, d_mode="normal",
                                       h0_mode="normal" if state else "none")


def check_step(inp, y, s_out, use_D=True, heads=None, what=""):
    dn = dtype_name(inp["x"].dtype)
    y_ref, h_ref = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                               inp["D"] if use_D else None, inp["h0"], heads=heads)
    if heads is None:
        got_y, got_h = y.float().cpu(), s_out.cpu()
    else:
        got_y = torch.stack([y[b, :, h, :].float().cpu() for b, h in heads])
        got_h = torch.stack([s_out[b, h].cpu() for b, h in heads])
    assert_close(got_y, y_ref, dn, f"{what} y")
    assert_close(got_h, h_ref, dn, f"{what} state")
    # the state is float32 arithmetic on float32 storage: hold it to the float32 bar
    mx, mean = oracle.error_metrics(got_h, h_ref)
    assert mx <= 1e-5 and mean <= 1e-5, f"{what} state: {mx:.2e} / {mean:.2e}"


# b, H, P, N, G, dtype: the 16-byte vector form (N = 128, 256) and the any-shape form
CASES = [
    (3, 8, 64, 128, 2, "bf16"),
    (2, 4, 128, 256, 1, "bf16"),
    (2, 6, 64, 128, 3, "f32"),
    (1, 4, 72, 256, 4, "f32"),
    (2, 3, 5, 7, 1, "f32"),
    (2, 4, 40, 48, 2, "bf16"),
    (1, 2, 1, 1, 1, "f32"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}H{}P{}N{}G{}{}".format(*c))
def test_step_matches_oracle(case):
    b, H, P, N, G, dt = case
    inp = step_inputs(b, H, P, N, G, dt, seed=P * N + b)
    dev = to_device(inp)
    state = dev["h0"].clone()
    y, s_out = ssd_step_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], state)
    torch.cuda.synchronize()
    assert s_out.data_ptr() == state.data_ptr(), "default is an in-place update"
    check_step(inp, y, s_out, what=str(case))


def test_step_zero_state_no_skip_and_three_dim_form():
    inp = step_inputs(2, 4, 64, 128, 1, "bf16", seed=7, state=False)
    dev = to_device(inp)
    y, s_out = ssd_step_fwd(dev["x"][:, 0], dev["dt"][:, 0], dev["A"], dev["B"][:, 0],
                            dev["C"][:, 0], None, None)
    torch.cuda.synchronize()
    assert y.shape == dev["x"][:, 0].shape
    check_step(inp, y.unsqueeze(1), s_out, use_D=False, what="zero state")


def test_step_in_place_equals_out_of_place():
    inp = step_inputs(2, 8, 64, 256, 2, "bf16", seed=11)
    dev = to_device(inp)
    s_a = dev["h0"].clone()
    s_b = torch.full_like(dev["h0"], float("nan"))
    y_a, _ = ssd_step_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], s_a)
    y_b, _ = ssd_step_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                          dev["h0"], state_out=s_b)
    torch.cuda.synchronize()
    assert torch.equal(s_a, s_b) and torch.equal(y_a, y_b)


@pytest.mark.parametrize("N,dt", [(128, "bf16"), (256, "f32"), (24, "bf16")])
def test_repeated_steps_match_the_scan(N, dt):
    """L single steps, state carried on the device, equal one scan over the L tokens."""
    b, L, H, P, G = 2, 40, 4, 64, 2
    inp = step_inputs(b, H, P, N, G, dt, seed=N + L, L=L)
    dev = to_device(inp)
    state = dev["h0"].clone()
    ys = []
    for t in range(L):
        tok = {k: dev[k][:, t:t + 1].contiguous() for k in ("x", "dt", "B", "C")}
        y, state = ssd_step_fwd(tok["x"], tok["dt"], dev["A"], tok["B"], tok["C"], dev["D"],
                                state)
        ys.append(y)
    y_steps = torch.cat(ys, dim=1)
    torch.cuda.synchronize()
    # against the oracle over all L tokens ...
    dn = dtype_name(inp["x"].dtype)
    y_ref, h_ref = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                               inp["h0"])
    assert_close(y_steps.float().cpu(), y_ref, dn, "steps y")
    assert_close(state.cpu(), h_ref, dn, "steps state")
    # ... and against the scan kernels on the same tokens
    y_scan, h_scan = ssd_scan_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                                  dev["h0"], chunk_size=64)
    torch.cuda.synchronize()
    assert_close(y_steps.float().cpu(), y_scan.float().cpu().double().numpy(), dn, "steps vs scan y")
    # (the tensor-core scan rounds w o X to bf16 for its state GEMM: the dtype's bar applies)
    assert_close(state.cpu(), h_scan.cpu().double().numpy(), dn, "steps vs scan state")


def test_decode_workload_full_size_sampled_heads():
    w = workloads.DECODE[0]
    inp = workloads.make_inputs(w)
    dev = to_device(inp)
    state = dev["h0"].clone()
    y, s_out = ssd_step_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], state)
    torch.cuda.synchronize()
    heads = sample_heads(w.batch, w.nheads, k=8, seed=5)
    check_step(inp, y, s_out, heads=heads, what=w.name)


def test_step_dt_zero_keeps_state_and_huge_dt_resets_it():
    inp = step_inputs(1, 4, 64, 128, 1, "f32", seed=3)
    inp["dt"][:, :, :2] = 0.0          # heads 0, 1: state unchanged
    inp["dt"][:, :, 2:] = 1.0e4        # heads 2, 3: exp(dt A) underflows, state = dt x B^T
    dev = to_device(inp)
    y, s = ssd_step_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                        dev["h0"].clone())
    torch.cuda.synchronize()
    check_step(inp, y, s, what="dt extremes")
    assert torch.equal(s[:, :2].cpu(), inp["h0"][:, :2])


def test_step_argument_errors_raise():
    inp = step_inputs(1, 2, 64, 128, 1, "bf16", seed=1)
    dev = to_device(inp)
    n = dev["h0"].numel()
    buf = torch.zeros(n + 64, dtype=torch.float32, device="cuda")
    s_in = buf[:n].view(dev["h0"].shape)
    s_out = buf[64:].view(dev["h0"].shape)     # overlaps s_in without being s_in
    with pytest.raises(SSDError):
        ssd_step_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], s_in,
                     state_out=s_out)
    with pytest.raises(ValueError):            # more than one token
        two = step_inputs(1, 2, 64, 128, 1, "bf16", seed=1, L=2)
        d2 = to_device(two)
        ssd_step_fwd(d2["x"], d2["dt"], d2["A"], d2["B"], d2["C"], d2["D"], d2["h0"])
