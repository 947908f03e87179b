"""The no-allocation entry point (ssd_scan_fwd_noalloc) through the C ABI.

It serves callers that cannot allocate device memory: they pass inputs and outputs only and the
library uses its own fixed device buffer.  On two calls in a row -- the second one a smaller
problem, so that it runs over what the first left in the shared buffer -- its results must
match the CPU oracle and the regular entry point's, and an oversized problem must be refused
before anything runs.  This file is named so pytest collects it last.
"""
import ctypes

import pytest
import torch

from gpu_helpers import TOL, assert_close, check_against_oracle, to_device
from mamba_ssd_scan_05_b300 import SSD_PATH_CHUNKED, make_dims, ssd_scan_fwd, workloads
from mamba_ssd_scan_05_b300._binding import load_library

SSD_OK, SSD_ERR_WORKSPACE = 0, 5
NOALLOC_BYTES = 64 << 20


def _noalloc_fn():
    lib = load_library()
    fn = lib.ssd_scan_fwd_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.c_void_p, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(fn, dev, chunk):
    dims = make_dims(dev["x"], dev["B"])
    b, L, H, P = dev["x"].shape
    N = dev["B"].shape[3]
    y = torch.full_like(dev["x"], float("nan"))
    hT = torch.full((b, H, P, N), float("nan"), dtype=torch.float32, device=dev["x"].device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(ctypes.addressof(dims), _p(dev["x"]), _p(dev["dt"]), _p(dev["A"]), _p(dev["B"]),
            _p(dev["C"]), _p(dev["D"]), _p(dev["h0"]), int(chunk), _p(y), _p(hT), stream)
    torch.cuda.synchronize()
    return rc, y, hT


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_oracle_and_regular_entry_point_twice(dtype):
    fn = _noalloc_fn()
    # two input sets scanned back to back, the second smaller than the first
    shapes = [(2, 700, 4, 64, 128, 2), (1, 333, 2, 64, 128, 1)]
    for call, (seed, shape) in enumerate(zip((11, 12), shapes)):
        inp = workloads.make_shape_inputs(*shape, dtype, seed=seed, h0_mode="normal",
                                          d_mode="normal")
        dev = to_device(inp)
        rc, y, hT = _call(fn, dev, 128)
        assert rc == SSD_OK, f"call {call}: return code {rc}"
        check_against_oracle(inp, y, hT, what=f"no-alloc call {call}")
        y_ref, h_ref = ssd_scan_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"],
                                    dev["D"], dev["h0"], chunk_size=128)
        torch.cuda.synchronize()
        assert_close(y.float().cpu(), y_ref.float().cpu(), dtype, f"call {call} y")
        assert_close(hT.cpu(), h_ref.cpu(), dtype, f"call {call} final_state")


@pytest.mark.gpu
def test_noalloc_rejects_problem_beyond_static_scratch():
    fn = _noalloc_fn()
    # 1 x 8192 tokens x 64 heads x 64 x 256 fp32 chunk states at chunk 64 is ~1 GiB of scratch
    inp = workloads.make_shape_inputs(1, 8192, 64, 64, 256, 1, "bf16", seed=3)
    dev = to_device(inp)
    dims = make_dims(dev["x"], dev["B"])
    lib = load_library()
    assert lib.ssd_scan_workspace_bytes(ctypes.byref(dims), 64, SSD_PATH_CHUNKED) > NOALLOC_BYTES
    rc, y, _ = _call(fn, dev, 64)
    assert rc == SSD_ERR_WORKSPACE
    assert torch.isnan(y).all(), "an oversized call must not run"
