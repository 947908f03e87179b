"""Closed forms of the scan, checked on the tensor-core path (bf16, fp32 accumulation).

Each case fixes the answer by mathematics, not only by the oracle:
  reset      dt so large that exp(dt A) underflows: the state forgets everything before the
             token, h_t = dt_t x_t B_t^T and y_t = dt_t (C_t . B_t) x_t + D x_t
             (youngju.dev Mamba article, "LTIからSelectionへの切り替え": a large step size
             resets the state to the current input)
  b_zero     B = 0: no input reaches the state, y = D x + exp(A cum_t) C_t h0 and the final
             state is exp(A sum dt) h0
  homogeneity  y(2 x, 2 h0) = 2 y(x, h0), exactly (a power-of-two scale is exact in bf16 and
             in every float32 step)
  superposition  y(x1 + x2, h01 + h02) = y(x1, h01) + y(x2, h02)
  groups     G = H with each group's B/C copied to its heads equals G < H, bit for bit
The sizes span several 128-token tiles and enough work units that the persistent grid cuts
chains between CTAs (so the cross-CTA state hand-off runs), with and without the state-only
pre-pass, and both d_state values the kernel takes.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, check_all_heads, run_gpu, to_device
from mamba_ssd_scan_05_b300 import SSD_PATH_TC, make_dims, ssd_scan_resolve_path, workloads

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634

# b, L, H, P, N, G, Q: the first takes the state-only pre-pass (ranges shorter than chains),
# the second does not (ranges longer than chains); the third is the large-state tile
SHAPES = [
    (2, 4096, 16, 64, 128, 1, 256),
    (1, 640, 512, 64, 128, 4, 128),
    (2, 1000, 8, 128, 256, 2, 128),
]
IDS = ["N128-prepass", "N128-longranges", "N256"]


def tc_inputs(shape, seed, h0=True):
    b, L, H, P, N, G, Q = shape
    inp = workloads.make_shape_inputs(b, L, H, P, N, G, "bf16", seed=seed,
                                      h0_mode="normal" if h0 else "none", d_mode="normal")
    assert ssd_scan_resolve_path(make_dims(inp["x"], inp["B"]), Q, SSD_PATH_TC) == SSD_PATH_TC
    return inp, Q


def block_log2_ranges(dt, A, tile=128, block=32):
    """Decay range, in log2 units, of every 32-token block of every 128-token tile: the sum of
    -dt_t A log2(e) over the block's tokens after its first (how far the decay factor falls
    between the block's first and last row)."""
    dt = dt.float().double().numpy()                       # [b, L, H]
    b, L, H = dt.shape
    a2 = -dt * A.double().numpy()[None, None, :] * LOG2E
    out = []
    for t0 in range(0, L, block):
        t1 = min(t0 + block, L)
        out.append(a2[:, t0 + 1:t1, :].sum(axis=1))
    return np.stack(out, axis=1)                             # [b, blocks, H]


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_reset_large_dt(shape):
    """dt = 1000 on every token: the state holds only the current token's input."""
    inp, Q = tc_inputs(shape, seed=11)
    inp["dt"] = torch.full_like(inp["dt"], 1000.0)
    # every 32-token block's decay range is far beyond what the kernel's factored form of the
    # diagonal blocks covers (2^100), so each diagonal block takes the per-element exponential
    assert block_log2_ranges(inp["dt"], inp["A"]).min() >= 100.0
    dev = to_device(inp)
    y, hT = run_gpu(dev, Q, path=SSD_PATH_TC)
    check_all_heads(inp, y, hT, what="reset")
    # the closed form, from the stored inputs
    x = inp["x"].double()
    dt = inp["dt"].double()
    H, G = x.shape[2], inp["B"].shape[2]
    Bh = inp["B"].double().repeat_interleave(H // G, dim=2)     # [b, L, H, N]
    Ch = inp["C"].double().repeat_interleave(H // G, dim=2)
    cb = (Ch * Bh).sum(-1)                                       # [b, L, H]
    y_ref = (dt * cb)[..., None] * x + inp["D"].double()[None, None, :, None] * x
    assert_close(y.float().cpu(), y_ref.numpy(), "bf16", "reset y (closed form)")
    h_ref = (dt[:, -1, :, None, None] * x[:, -1, :, :, None] * Bh[:, -1, :, None, :])
    assert_close(hT.cpu(), h_ref.numpy(), "bf16", "reset final state (closed form)")


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_sparse_resets_mix_both_diagonal_forms(shape):
    """A huge dt on scattered tokens: some 32-token blocks keep a small decay range (factored
    diagonal form), the blocks holding a reset token exceed it (per-element form)."""
    inp, Q = tc_inputs(shape, seed=12)
    g = torch.Generator().manual_seed(5)
    mask = torch.rand(inp["dt"].shape, generator=g) < 0.01
    inp["dt"] = torch.where(mask, torch.full_like(inp["dt"], 300.0), inp["dt"])
    r = block_log2_ranges(inp["dt"], inp["A"])
    assert (r >= 100.0).any() and (r < 100.0).any()
    dev = to_device(inp)
    y, hT = run_gpu(dev, Q, path=SSD_PATH_TC)
    check_all_heads(inp, y, hT, what="sparse resets")


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_b_zero_only_initial_state_and_skip(shape):
    inp, Q = tc_inputs(shape, seed=13)
    inp["B"] = torch.zeros_like(inp["B"])
    dev = to_device(inp)
    y, hT = run_gpu(dev, Q, path=SSD_PATH_TC)
    check_all_heads(inp, y, hT, what="B=0")
    x = inp["x"].double()
    H, G = x.shape[2], inp["C"].shape[2]
    Ch = inp["C"].double().repeat_interleave(H // G, dim=2)      # [b, L, H, N]
    cum = torch.cumsum(inp["dt"].double() * inp["A"].double()[None, None, :], dim=1)
    h0 = inp["h0"].double()                                       # [b, H, P, N]
    ch0 = torch.einsum("blhn,bhpn->blhp", Ch, h0)
    y_ref = torch.exp(cum)[..., None] * ch0 + inp["D"].double()[None, None, :, None] * x
    assert_close(y.float().cpu(), y_ref.numpy(), "bf16", "B=0 y (closed form)")
    h_ref = torch.exp(cum[:, -1])[:, :, None, None] * h0
    assert_close(hT.cpu(), h_ref.numpy(), "bf16", "B=0 final state (closed form)")


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_homogeneity_exact(shape):
    inp, Q = tc_inputs(shape, seed=14)
    dev = to_device(inp)
    y1, h1 = run_gpu(dev, Q, path=SSD_PATH_TC)
    dev2 = dict(dev)
    dev2["x"] = dev["x"] * 2
    dev2["h0"] = dev["h0"] * 2
    y2, h2 = run_gpu(dev2, Q, path=SSD_PATH_TC)
    assert torch.equal(y2, y1 * 2)
    assert torch.equal(h2, h1 * 2)
    dev3 = dict(dev)
    dev3["x"] = -dev["x"]
    dev3["h0"] = -dev["h0"]
    y3, h3 = run_gpu(dev3, Q, path=SSD_PATH_TC)
    assert torch.equal(y3, -y1)
    assert torch.equal(h3, -h1)


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_superposition(shape):
    inp, Q = tc_inputs(shape, seed=15)
    other, _ = tc_inputs(shape, seed=16)
    dev = to_device(inp)
    y1, h1 = run_gpu(dev, Q, path=SSD_PATH_TC)
    dev2 = dict(dev)
    dev2["x"] = other["x"].cuda()
    dev2["h0"] = other["h0"].cuda()
    y2, h2 = run_gpu(dev2, Q, path=SSD_PATH_TC)
    both = dict(inp)
    both["x"] = (inp["x"].float() + other["x"].float()).to(torch.bfloat16)
    both["h0"] = inp["h0"] + other["h0"]
    dev3 = to_device(both)
    y3, h3 = run_gpu(dev3, Q, path=SSD_PATH_TC)
    check_all_heads(both, y3, h3, what="sum input")
    # superposition itself: y(x1 + x2) against y(x1) + y(x2), both from the GPU
    assert_close(y3.float().cpu(), (y1.double() + y2.double()).cpu().numpy(), "bf16",
                 "y(x1 + x2) vs y(x1) + y(x2)")
    assert_close(h3.cpu(), (h1.double() + h2.double()).cpu().numpy(), "bf16",
                 "final(x1 + x2) vs final(x1) + final(x2)")
    # and the sum of the two GPU outputs against the sum of the oracle's two outputs
    ref_y, ref_h = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                               inp["h0"])
    oth_y, oth_h = oracle.scan(other["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                               other["h0"])
    assert_close((y1.double() + y2.double()).cpu().numpy(), ref_y + oth_y, "bf16",
                 "superposition y")
    assert_close((h1.double() + h2.double()).cpu().numpy(), ref_h + oth_h, "bf16",
                 "superposition final state")


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_replicated_groups_equal_shared_groups(shape):
    inp, Q = tc_inputs(shape, seed=17)
    H, G = inp["x"].shape[2], inp["B"].shape[2]
    dev = to_device(inp)
    y1, h1 = run_gpu(dev, Q, path=SSD_PATH_TC)
    rep = dict(dev)
    rep["B"] = dev["B"].repeat_interleave(H // G, dim=2).contiguous()
    rep["C"] = dev["C"].repeat_interleave(H // G, dim=2).contiguous()
    y2, h2 = run_gpu(rep, Q, path=SSD_PATH_TC)
    assert torch.equal(y1, y2)
    assert torch.equal(h1, h2)


def test_decay_range_around_the_factored_limit():
    """Tiles whose whole-tile log2 decay is just below and just above 160 (the limit of the
    factored evaluation on the d_state 128 kernel), mixed in one sequence, with growing
    (A > 0) heads too: every tile must match the oracle whichever way it is evaluated."""
    b, L, H, P, N, G, Q = 2, 128 * 12, 6, 64, 128, 1, 256
    inp = workloads.make_shape_inputs(b, L, H, P, N, G, "bf16", seed=31, h0_mode="normal",
                                      d_mode="normal")
    A = torch.tensor([-1.0, -2.0, -4.0, -8.0, -16.0, 0.05], dtype=torch.float32)
    inp["A"] = A
    # per tile a target log2 decay: 150, 159, 161, 170, ... cycling; dt constant in the tile
    targets = torch.tensor([150.0, 159.0, 161.0, 170.0, 40.0, 300.0])
    dt = torch.empty(b, L, H)
    for k in range(L // 128):
        tgt = targets[k % len(targets)]
        for h in range(H):
            a = float(A[h])
            # a growing head (A > 0) gets a small step, so that its state stays finite
            dt[:, k * 128:(k + 1) * 128, h] = tgt / (128 * -a * LOG2E) if a < 0 else 0.01
    inp["dt"] = dt.to(torch.bfloat16)
    dev = to_device(inp)
    y, hT = run_gpu(dev, Q, path=SSD_PATH_TC)
    check_all_heads(inp, y, hT, what="decay around the factored limit")
