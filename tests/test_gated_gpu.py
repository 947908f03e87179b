"""The scan with the gated RMSNorm of its output (ssd_scan_fwd_gated), against the oracle.

out = rmsnorm(y) * w * silu(z) over groups of features (Qiita "Mamba-2 / SSD" article, section
4.2, step 4), with y the scan.  The reference composes the two float64 oracles.  Where the
norm is fused into the tensor-core kernel (d_state 128, groups of 8 to 64 features) no y
scratch is needed; the other problems run the scan into workspace scratch and then the norm.
"""
import pytest
import torch

import oracle
from gpu_helpers import assert_close, to_device
from mamba_ssd_scan_05_b300 import (make_dims, ssd_scan_fwd, ssd_scan_fwd_gated,
                                    ssd_scan_gated_workspace_bytes, ssd_scan_workspace_bytes,
                                    workloads)
from oracle import block

pytestmark = pytest.mark.gpu


def gated_reference(inp, z, w, eps, g):
    y, hT = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
    b, L, H, P = y.shape
    out = block.gated_rmsnorm(y.reshape(b, L, H * P), z.reshape(b, L, H * P), w, eps, g)
    return out.reshape(b, L, H, P), hT


# b, L, H, P, N, G, Q, dtype, group: fused (tensor core, d_state 128), then unfused forms
CASES = [
    (2, 300, 4, 64, 128, 1, 256, "bf16", 64),
    (1, 520, 4, 64, 128, 2, 128, "bf16", 32),
    (1, 384, 2, 128, 128, 1, 128, "bf16", 16),
    (2, 130, 4, 64, 128, 1, 64, "bf16", 8),
    (2, 4096, 16, 64, 128, 1, 256, "bf16", 64),      # ranges cut chains: the look-back runs
    (1, 300, 4, 64, 128, 1, 256, "bf16", 256),       # a group across heads: unfused
    (2, 200, 4, 128, 256, 2, 128, "bf16", 64),       # d_state 256: unfused
    (1, 200, 4, 32, 16, 1, 64, "f32", 32),           # float32: unfused
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}L{}H{}P{}N{}G{}Q{}{}g{}".format(*c))
@pytest.mark.parametrize("with_w", [True, False], ids=["w", "now"])
def test_gated_scan_matches_oracle(case, with_w):
    b, L, H, P, N, G, Q, dt, g = case
    inp = workloads.make_shape_inputs(b, L, H, P, N, G, dt, seed=L + g, h0_mode="normal",
                                      d_mode="normal")
    gen = torch.Generator().manual_seed(L * 7 + g)
    tdtype = torch.bfloat16 if dt == "bf16" else torch.float32
    z = torch.randn(b, L, H, P, generator=gen).to(tdtype)
    w = (1.0 + 0.1 * torch.randn(H * P, generator=gen)).float() if with_w else None
    eps = 1e-5
    dev = to_device(inp)
    zd, wd = z.cuda(), (None if w is None else w.cuda())
    dims = make_dims(dev["x"], dev["B"])
    fused = ssd_scan_gated_workspace_bytes(dims, Q, g) == ssd_scan_workspace_bytes(dims, Q)
    assert fused == (N == 128 and dt == "bf16" and g <= 64), "fused form where it applies"
    out, hT = ssd_scan_fwd_gated(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], zd,
                                 dev["D"], dev["h0"], wd, eps=eps, group_size=g, chunk_size=Q)
    torch.cuda.synchronize()
    ref, h_ref = gated_reference(inp, z, w, eps, g)
    assert_close(out.float().cpu(), ref, dt, f"gated out ({'fused' if fused else 'unfused'})")
    assert_close(hT.cpu(), h_ref, dt, "gated final state")


def test_fused_and_plain_scan_share_the_state_and_agree_on_the_output():
    """The fused form's final state is the plain scan's, bit for bit, and its output equals the
    norm applied to the plain scan's (bf16-rounded) y within rounding."""
    inp = workloads.make_shape_inputs(2, 1000, 8, 64, 128, 2, "bf16", seed=41, h0_mode="normal",
                                      d_mode="normal")
    dev = to_device(inp)
    z = torch.randn(2, 1000, 8, 64, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    out, h1 = ssd_scan_fwd_gated(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], z.cuda(),
                                 dev["D"], dev["h0"], group_size=64, chunk_size=128)
    y, h2 = ssd_scan_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                         chunk_size=128)
    torch.cuda.synchronize()
    assert torch.equal(h1, h2)
    ref = block.gated_rmsnorm(y.float().cpu().reshape(2, 1000, 512),
                              z.reshape(2, 1000, 512), None, 1e-5, 64).reshape(2, 1000, 8, 64)
    assert_close(out.float().cpu(), ref, "bf16", "fused vs norm(plain scan)")
