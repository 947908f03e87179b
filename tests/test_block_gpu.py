"""Parity of the block steps around the scan (causal conv1d + SiLU, gated RMSNorm), through the
C ABI, with their float64 CPU oracles."""
import numpy as np
import pytest
import torch

import oracle
from oracle import block
from mamba_ssd_scan_05_b300 import (SSDError, ssd_block_get_status, ssd_causal_conv1d_fwd,
                                    ssd_gated_rmsnorm_fwd, ssd_scan_set_wait_cycles, workloads)

pytestmark = pytest.mark.gpu

# float32 outputs: float32 arithmetic, a few ulp; bf16 outputs: one rounding of the result
TOL = {"f32": (1e-5, 1e-5), "bf16": (8e-3, 4e-3)}


def close(got, ref, dtype, what):
    mx, mean = oracle.error_metrics(got, ref)
    tmax, tmean = TOL[dtype]
    assert np.all(np.isfinite(oracle._f64(got))), f"{what}: non-finite"
    assert mx <= tmax and mean <= tmean, f"{what}: max {mx:.2e} mean {mean:.2e}"


def cuda(d):
    return {k: (None if v is None else v.cuda()) for k, v in d.items()}


# ---- causal conv1d -----------------------------------------------------------------------------

# b, L, C, K, dtype, state, bias, silu: vector paths (C % 8 / C % 4), scalar path (odd C),
# every width, sequences shorter than the window, several token blocks with a ragged end
CONV = [
    (2, 100, 64, 4, "bf16", False, True, True),
    (1, 257, 40, 4, "bf16", True, True, True),
    (2, 33, 12, 3, "f32", True, False, True),
    (1, 70, 7, 4, "f32", False, True, False),
    (2, 5, 24, 8, "bf16", True, True, True),
    (1, 2, 16, 4, "f32", True, True, True),
    (3, 64, 5, 1, "bf16", False, True, True),
    (1, 96, 16, 2, "f32", False, False, False),
    (1, 40, 8, 5, "bf16", True, False, True),
    (1, 31, 20, 6, "f32", True, True, True),
    (1, 65, 32, 7, "bf16", False, True, True),
    # several 64-token blocks with a ragged end; 96- and 128-thread blocks over the channels
    (1, 300, 768, 4, "bf16", True, True, True),
    (2, 129, 1024, 4, "f32", False, True, True),
    # streaming kernel: channel tails inside a 256-byte tile column, token tails, every width
    (2, 200, 200, 4, "bf16", True, True, True),
    (1, 1000, 1000, 4, "f32", True, True, True),
    (3, 64, 136, 8, "bf16", True, True, True),
    (1, 65, 520, 2, "bf16", False, True, True),
    (2, 130, 8, 6, "bf16", True, False, True),
    (1, 3, 4, 5, "f32", True, True, True),
]


@pytest.mark.parametrize("case", CONV, ids=lambda c: "b{}L{}C{}K{}{}{}{}{}".format(
    *c[:5], "st" if c[5] else "", "bias" if c[6] else "", "silu" if c[7] else ""))
def test_conv_matches_oracle(case):
    b, L, C, K, dt, with_state, with_bias, silu = case
    inp = workloads.make_conv_inputs(b, L, C, K, dt, seed=L * C + K, state=with_state)
    dev = cuda(inp)
    bias = dev["bias"] if with_bias else None
    out, st = ssd_causal_conv1d_fwd(dev["x"], dev["weight"], bias, dev["state"], silu=silu,
                                    return_state=True)
    torch.cuda.synchronize()
    ref, ref_st = block.causal_conv1d(inp["x"], inp["weight"], inp["bias"] if with_bias else None,
                                      inp["state"], apply_silu=silu)
    close(out.float().cpu(), ref, dt, f"{case} out")
    # the new state is the last K - 1 inputs: exact copies
    if K > 1:
        assert np.array_equal(st.float().cpu().double().numpy(), ref_st), f"{case} state"


def _misaligned(t):
    """A copy of t whose data starts one element past a 16-byte boundary (the register kernel
    then runs instead of the streaming one)."""
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = flat[1:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("K", [1, 4, 8])
def test_conv_streaming_and_register_kernels_agree_bitwise(dt, K):
    """Both kernels evaluate bias + sum_k w x in the same order and the same SiLU, so the two
    outputs and states must be equal bit for bit."""
    inp = cuda(workloads.make_conv_inputs(2, 333, 264, K, dt, seed=K, state=True))
    out, st = ssd_causal_conv1d_fwd(inp["x"], inp["weight"], inp["bias"], inp["state"],
                                    return_state=True)
    xm = _misaligned(inp["x"])
    sm = _misaligned(inp["state"]) if K > 1 else None
    out2, st2 = ssd_causal_conv1d_fwd(xm, inp["weight"], inp["bias"], sm, return_state=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    if K > 1:
        assert torch.equal(st, st2)


def test_conv_split_sequence_equals_one_call_bitwise():
    inp = cuda(workloads.make_conv_inputs(2, 150, 64, 4, "bf16", seed=4))
    full, fin = ssd_causal_conv1d_fwd(inp["x"], inp["weight"], inp["bias"], return_state=True)
    for cut in (1, 2, 3, 33, 100):
        a, st = ssd_causal_conv1d_fwd(inp["x"][:, :cut].contiguous(), inp["weight"], inp["bias"],
                                      return_state=True)
        c, st2 = ssd_causal_conv1d_fwd(inp["x"][:, cut:].contiguous(), inp["weight"], inp["bias"],
                                       st, return_state=True)
        torch.cuda.synchronize()
        assert torch.equal(torch.cat([a, c], dim=1), full) and torch.equal(st2, fin), cut


def test_conv_empty_sequence_passes_the_state_through():
    inp = cuda(workloads.make_conv_inputs(2, 0, 16, 4, "bf16", seed=2, state=True))
    out, st = ssd_causal_conv1d_fwd(inp["x"], inp["weight"], inp["bias"], inp["state"],
                                    return_state=True)
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(st, inp["state"])
    out, st = ssd_causal_conv1d_fwd(inp["x"], inp["weight"], inp["bias"], None, return_state=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st) == 0


def test_conv_workload_full_size_sampled_channels():
    c = workloads.CONV
    inp = workloads.make_conv_inputs(c["batch"], c["seqlen"], c["channels"], c["width"],
                                     c["dtype"], seed=c["seed"])
    dev = cuda(inp)
    out = ssd_causal_conv1d_fwd(dev["x"], dev["weight"], dev["bias"])
    torch.cuda.synchronize()
    ch = np.random.default_rng(0).choice(c["channels"], size=24, replace=False)
    ch.sort()
    ref, _ = block.causal_conv1d(inp["x"][:, :, ch], inp["weight"][ch], inp["bias"][ch])
    close(out[:, :, ch].float().cpu(), ref, c["dtype"], "conv workload")


def test_conv_rejects_overlap_and_bad_width():
    inp = cuda(workloads.make_conv_inputs(1, 64, 16, 4, "bf16", seed=1))
    with pytest.raises(SSDError):
        ssd_causal_conv1d_fwd(inp["x"], inp["weight"], out=inp["x"])          # in place
    with pytest.raises(SSDError):
        ssd_causal_conv1d_fwd(inp["x"], torch.ones((16, 9), device="cuda"))   # width 9


# ---- gated RMSNorm ---------------------------------------------------------------------------

# rows, D, group, dtype, gate, weight
NORM = [
    (16, 5120, 5120, "bf16", True, True),
    (7, 64, 16, "bf16", True, True),
    (5, 40, 8, "f32", True, False),
    (9, 48, 48, "f32", False, True),
    (3, 7, 7, "bf16", True, True),
    (4, 12, 3, "f32", True, True),
    (2, 1, 1, "f32", True, True),
    (3, 16384, 1024, "bf16", True, True),
    (2, 12288, 1, "f32", False, False),
]


@pytest.mark.parametrize("case", NORM, ids=lambda c: "r{}D{}g{}{}{}{}".format(
    *c[:4], "z" if c[4] else "", "w" if c[5] else ""))
def test_norm_matches_oracle(case):
    rows, D, g, dt, gate, weight = case
    inp = workloads.make_norm_inputs(rows, D, dt, seed=rows * D + g)
    dev = cuda(inp)
    out = ssd_gated_rmsnorm_fwd(dev["y"], dev["z"] if gate else None,
                                dev["weight"] if weight else None, eps=1e-5, group_size=g)
    torch.cuda.synchronize()
    ref = block.gated_rmsnorm(inp["y"], inp["z"] if gate else None,
                              inp["weight"] if weight else None, 1e-5, g)
    close(out.float().cpu(), ref, dt, f"{case}")


def test_norm_in_place_and_scan_shaped_input():
    """The scan's y [b, L, H, P] viewed as [b, L, H * P]: one group per token; out may be y."""
    inp = workloads.make_norm_inputs(2 * 33, 4 * 64, "bf16", seed=8)
    dev = cuda(inp)
    yd = dev["y"].view(2, 33, 4, 64).clone()
    zd = dev["z"].view(2, 33, 4, 64)
    ref = ssd_gated_rmsnorm_fwd(yd.view(2, 33, 256), zd.view(2, 33, 256), dev["weight"])
    ssd_gated_rmsnorm_fwd(yd.view(2, 33, 256), zd.view(2, 33, 256), dev["weight"],
                          out=yd.view(2, 33, 256))
    torch.cuda.synchronize()
    assert torch.equal(yd.view(2, 33, 256), ref)
    close(ref.float().cpu().reshape(66, 256),
          block.gated_rmsnorm(inp["y"], inp["z"], inp["weight"]), "bf16", "scan-shaped")


def test_norm_workload_full_size_sampled_rows():
    n = workloads.NORM
    inp = workloads.make_norm_inputs(n["rows"], n["dim"], n["dtype"], seed=n["seed"])
    dev = cuda(inp)
    out = ssd_gated_rmsnorm_fwd(dev["y"], dev["z"], dev["weight"], group_size=n["group_size"])
    torch.cuda.synchronize()
    rows = np.random.default_rng(1).choice(n["rows"], size=64, replace=False)
    ref = block.gated_rmsnorm(inp["y"][rows], inp["z"][rows], inp["weight"], 1e-5,
                              n["group_size"])
    close(out[rows].float().cpu(), ref, n["dtype"], "norm workload")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_norm_streaming_and_register_kernels_both_match_oracle(dt):
    """The same rows through the streaming kernel (aligned) and the register kernel (one
    element off a 16-byte boundary); several groups per row, more rows than the grid holds."""
    inp = workloads.make_norm_inputs(3000, 768, dt, seed=77)
    dev = cuda(inp)
    ref = block.gated_rmsnorm(inp["y"], inp["z"], inp["weight"], 1e-5, 64)
    a = ssd_gated_rmsnorm_fwd(dev["y"], dev["z"], dev["weight"], group_size=64)
    b = ssd_gated_rmsnorm_fwd(_misaligned(dev["y"]), _misaligned(dev["z"]), dev["weight"],
                              group_size=64)
    torch.cuda.synchronize()
    close(a.float().cpu(), ref, dt, "streaming")
    close(b.float().cpu(), ref, dt, "register")


def test_block_kernels_wait_limit_runs_out_then_next_call_is_clean():
    """With a wait limit of one cycle, any wait of the streaming kernels that is not satisfied
    at its first poll gives up (over thousands of HBM-bound tiles some always are): the kernels
    stop and report SSD_ERR_TIMEOUT through ssd_block_get_status.  With the default limit the
    next calls match the oracle and report SSD_OK."""
    cin = workloads.make_conv_inputs(4, 2048, 2048, 4, "bf16", seed=5)
    nin = workloads.make_norm_inputs(8192, 2048, "bf16", seed=6)
    cd, nd = cuda(cin), cuda(nin)
    assert ssd_block_get_status() == 0
    for run in ("conv", "norm"):
        ssd_scan_set_wait_cycles(1)
        try:
            if run == "conv":
                ssd_causal_conv1d_fwd(cd["x"], cd["weight"], cd["bias"])
            else:
                ssd_gated_rmsnorm_fwd(nd["y"], nd["z"], nd["weight"])
            status = ssd_block_get_status()
        finally:
            ssd_scan_set_wait_cycles(0)
        assert status == 4, f"{run}: expected SSD_ERR_TIMEOUT, got {status}"
        assert ssd_block_get_status() == 0, "the status word is cleared by the read"
    out = ssd_causal_conv1d_fwd(cd["x"], cd["weight"], cd["bias"])
    nout = ssd_gated_rmsnorm_fwd(nd["y"], nd["z"], nd["weight"])
    assert ssd_block_get_status() == 0
    ref, _ = block.causal_conv1d(cin["x"], cin["weight"], cin["bias"], None)
    close(out.float().cpu(), ref, "bf16", "conv after timeout")
    close(nout.float().cpu(), block.gated_rmsnorm(nin["y"], nin["z"], nin["weight"]), "bf16",
          "norm after timeout")


def test_norm_rejects_bad_groups():
    inp = cuda(workloads.make_norm_inputs(2, 12, "f32", seed=1))
    with pytest.raises(SSDError):
        ssd_gated_rmsnorm_fwd(inp["y"], group_size=5)
    with pytest.raises(SSDError):
        ssd_gated_rmsnorm_fwd(inp["y"], eps=-1.0)
