"""Packed variable-length batches (ssd_scan_fwd_varlen): every sequence starts from its own
state, so each must match the oracle run on that sequence alone."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, assert_close, dtype_name
from mamba_ssd_scan_05_b300 import (SSD_PATH_AUTO, SSD_PATH_CHUNKED, SSD_PATH_TC, SSDError,
                                    ssd_scan_fwd, ssd_scan_fwd_varlen, workloads)

pytestmark = pytest.mark.gpu


def cuda(inp):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}


def check_each_sequence(inp, y, hT, use_h0=True):
    dn = dtype_name(inp["x"].dtype)
    cu = inp["cu_seqlens"]
    for i in range(len(cu) - 1):
        a, b = cu[i], cu[i + 1]
        h0 = inp["h0"][i:i + 1] if use_h0 else None
        if b == a:
            want = h0[0].double().numpy() if use_h0 else np.zeros(hT[i].shape)
            assert np.array_equal(hT[i].cpu().double().numpy(), want), f"seq {i} (empty)"
            continue
        y_ref, h_ref = oracle.scan(inp["x"][:, a:b], inp["dt"][:, a:b], inp["A"], inp["B"][:, a:b],
                                   inp["C"][:, a:b], inp["D"], h0)
        assert_close(y[:, a:b].float().cpu(), y_ref, dn, f"seq {i} y")
        assert_close(hT[i:i + 1].cpu(), h_ref, dn, f"seq {i} state")


@pytest.mark.parametrize("path", [SSD_PATH_AUTO, SSD_PATH_CHUNKED])
def test_mixed_lengths_match_the_oracle_per_sequence(path):
    lengths = [300, 0, 1, 127, 128, 129, 1000, 64]
    inp = workloads.make_varlen_inputs(lengths, 8, 64, 128, 2, "bf16", seed=5)
    dev = cuda(inp)
    y, hT = ssd_scan_fwd_varlen(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"],
                                inp["cu_seqlens"], dev["D"], dev["h0"], chunk_size=128, path=path)
    torch.cuda.synchronize()
    check_each_sequence(inp, y, hT)


def test_packed_matches_separate_calls_and_repeats_bitwise():
    """The packed call (sequences on concurrent streams, capped grids) agrees with one call per
    sequence within rounding, matches the oracle per sequence, and gives the same bits when
    repeated: the work plan and the lane assignment are fixed, not timing-dependent."""
    lengths = [513, 77, 256, 1200, 3000, 5, 640]
    inp = workloads.make_varlen_inputs(lengths, 4, 64, 128, 1, "bf16", seed=6)
    dev = cuda(inp)
    args = (dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], inp["cu_seqlens"], dev["D"],
            dev["h0"])
    y, hT = ssd_scan_fwd_varlen(*args, chunk_size=256)
    y2, hT2 = ssd_scan_fwd_varlen(*args, chunk_size=256)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(hT, hT2)
    check_each_sequence(inp, y, hT)
    cu = inp["cu_seqlens"]
    for i in range(len(lengths)):
        a, b = cu[i], cu[i + 1]
        sl = {k: dev[k][:, a:b].contiguous() for k in ("x", "dt", "B", "C")}
        yi, hi = ssd_scan_fwd(sl["x"], sl["dt"], dev["A"], sl["B"], sl["C"], dev["D"],
                              dev["h0"][i:i + 1].contiguous(), chunk_size=256)
        torch.cuda.synchronize()
        assert_close(y[:, a:b].float().cpu(), yi.float().cpu(), "bf16", f"seq {i} y")
        assert_close(hT[i:i + 1].cpu(), hi.cpu(), "bf16", f"seq {i} state")


def test_float32_and_no_initial_states():
    lengths = [40, 200, 3]
    inp = workloads.make_varlen_inputs(lengths, 4, 32, 16, 1, "f32", seed=7)
    dev = cuda(inp)
    y, hT = ssd_scan_fwd_varlen(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"],
                                inp["cu_seqlens"], dev["D"], None, chunk_size=64)
    torch.cuda.synchronize()
    check_each_sequence(inp, y, hT, use_h0=False)


def test_workload_sampled_sequences():
    v = workloads.VARLEN
    lengths = workloads.varlen_lengths(v["nseq"], v["min_len"], v["max_len"], v["seed"])
    inp = workloads.make_varlen_inputs(lengths, v["nheads"], v["headdim"], v["dstate"],
                                       v["ngroups"], v["dtype"], seed=v["seed"])
    dev = cuda(inp)
    y, hT = ssd_scan_fwd_varlen(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"],
                                inp["cu_seqlens"], dev["D"], dev["h0"], chunk_size=v["chunk"])
    torch.cuda.synchronize()
    cu = inp["cu_seqlens"]
    dn = dtype_name(inp["x"].dtype)
    for i in (0, len(lengths) // 2, len(lengths) - 1):
        a, b = cu[i], cu[i + 1]
        heads = [(0, 0), (0, v["nheads"] - 1), (0, 37)]
        y_ref, h_ref = oracle.scan(inp["x"][:, a:b], inp["dt"][:, a:b], inp["A"], inp["B"][:, a:b],
                                   inp["C"][:, a:b], inp["D"], inp["h0"][i:i + 1], heads=heads)
        got_y = torch.stack([y[0, a:b, h, :].float().cpu() for _, h in heads])
        got_h = torch.stack([hT[i, h].cpu() for _, h in heads])
        assert_close(got_y, y_ref, dn, f"seq {i} y")
        assert_close(got_h, h_ref, dn, f"seq {i} state")


def test_bad_offsets_raise():
    inp = workloads.make_varlen_inputs([10, 20], 4, 64, 128, 1, "bf16", seed=1)
    dev = cuda(inp)
    for cu in ([0, 10, 29], [0, 20, 10, 30][:3], [1, 10, 30]):
        with pytest.raises(SSDError):
            ssd_scan_fwd_varlen(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], cu, dev["D"],
                                None)
