"""ssd_scan_kernels_per_call against the kernels a profiler sees one call launch.

The d_state 128 scan adds a state-only pass kernel when the sequence is cut into pieces no
longer than its 128-token tiles per CTA (few heads, long sequence); many heads keep one kernel.
The chunked path always runs its three kernels.
"""
import pytest
import torch
from torch.profiler import ProfilerActivity, profile

from gpu_helpers import to_device
from mamba_ssd_scan_05_b300 import (SSD_PATH_CHUNKED, SSD_PATH_TC, make_dims, ssd_scan_fwd,
                                    ssd_scan_get_status, ssd_scan_kernels_per_call,
                                    ssd_scan_workspace_bytes, workloads)

pytestmark = pytest.mark.gpu

CASES = [
    # (b, L, H, P, N, G, Q, dtype, path, expected kernels)
    ((1, 4096, 8, 64, 128, 1, 256, "bf16"), SSD_PATH_TC, 2),     # 8 units: pieces cut chains
    ((4, 256, 80, 64, 128, 1, 256, "bf16"), SSD_PATH_TC, 1),     # 320 units, 2 tiles each
    ((2, 1000, 4, 128, 256, 2, 128, "bf16"), SSD_PATH_TC, 1),    # d_state 256: one kernel
    ((1, 300, 4, 64, 64, 1, 64, "f32"), SSD_PATH_CHUNKED, 3),
]


def _kernel_events(fn):
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    names = [e.name for e in prof.events()
             if e.device_type == torch.autograd.DeviceType.CUDA]
    return [n for n in names if "memset" not in n.lower() and "memcpy" not in n.lower()]


def _aligned_case():
    # as many heads as SMs: every CTA's range is one whole chain, so nothing is published and
    # the state-only pass does not run although the plan is in its mode
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    return ((1, 1024, nsm, 64, 128, 1, 256, "bf16"), SSD_PATH_TC, 1)


@pytest.mark.parametrize("case", CASES + ["aligned"],
                         ids=["tc128-pieces", "tc128-many-heads", "tc256", "chunked",
                              "tc128-ranges-are-chains"])
def test_kernels_per_call_matches_profiler(case):
    if case == "aligned":
        case = _aligned_case()
    (b, L, H, P, N, G, Q, dt), path, expected = case
    inp = workloads.make_shape_inputs(b, L, H, P, N, G, dt, seed=5, h0_mode="normal",
                                      d_mode="normal")
    dev = to_device(inp)
    dims = make_dims(dev["x"], dev["B"])
    assert ssd_scan_kernels_per_call(dims, Q, path) == expected
    ws = torch.empty(ssd_scan_workspace_bytes(dims, Q, path), dtype=torch.uint8, device="cuda")
    args = (dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"])

    def call():
        ssd_scan_fwd(*args, chunk_size=Q, path=path, workspace=ws)

    call()                                   # first call: attributes, tensor maps, warm-up
    torch.cuda.synchronize()
    kernels = _kernel_events(call)
    assert len(kernels) == expected, kernels
    assert ssd_scan_get_status(ws) == 0
