"""Device-side failure reporting of the tensor-core path, without faulting the GPU.

Every wait inside the tensor-core kernels is bounded.  With the limit set far below the time a
wait normally takes (ssd_scan_set_wait_cycles), a normal problem must end with
SSD_ERR_TIMEOUT in the workspace status word, and the context must stay usable: the next call
on the same workspace, with the default limit, returns SSD_OK and matches the oracle.  Also:
a workspace smaller than the problem needs is refused before anything runs.
"""
import pytest
import torch

from gpu_helpers import check_against_oracle, to_device
from mamba_ssd_scan_05_b300 import (SSD_PATH_TC, SSDError, make_dims, ssd_scan_fwd,
                                    ssd_scan_get_status, ssd_scan_set_wait_cycles,
                                    ssd_scan_workspace_bytes, workloads)

pytestmark = pytest.mark.gpu

SSD_OK, SSD_ERR_TIMEOUT, SSD_ERR_WORKSPACE = 0, 4, 5


@pytest.mark.parametrize("shape", [(2, 2048, 8, 64, 128, 1, 256), (2, 1000, 4, 128, 256, 2, 128)],
                         ids=["N128", "N256"])
def test_wait_limit_runs_out_then_next_call_is_clean(shape):
    b, L, H, P, N, G, Q = shape
    inp = workloads.make_shape_inputs(b, L, H, P, N, G, "bf16", seed=21, h0_mode="normal",
                                      d_mode="normal")
    dev = to_device(inp)
    dims = make_dims(dev["x"], dev["B"])
    ws = torch.empty(ssd_scan_workspace_bytes(dims, Q, SSD_PATH_TC), dtype=torch.uint8,
                     device="cuda")
    args = (dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"])
    # a limit of 200 cycles: shorter than a TMA load from HBM or one tile's GEMMs.  Both shapes
    # cut chains across CTAs: for N = 128 the separate state-only pass gives up at its first
    # copy and publishes nothing, and the scan's look-back then gives up too; for N = 256 the
    # scan's own waits do.
    ssd_scan_set_wait_cycles(200)
    try:
        ssd_scan_fwd(*args, chunk_size=Q, path=SSD_PATH_TC, workspace=ws)
        status = ssd_scan_get_status(ws)
    finally:
        ssd_scan_set_wait_cycles(0)
    assert status == SSD_ERR_TIMEOUT
    y, hT = ssd_scan_fwd(*args, chunk_size=Q, path=SSD_PATH_TC, workspace=ws)
    assert ssd_scan_get_status(ws) == SSD_OK
    check_against_oracle(inp, y, hT, what="after a timed-out call")


def test_undersized_workspace_is_refused():
    inp = workloads.make_shape_inputs(1, 512, 4, 64, 128, 1, "bf16", seed=22)
    dev = to_device(inp)
    dims = make_dims(dev["x"], dev["B"])
    need = ssd_scan_workspace_bytes(dims, 256)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    y = torch.full_like(dev["x"], float("nan"))
    with pytest.raises(SSDError) as err:
        ssd_scan_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], None,
                     chunk_size=256, y=y, workspace=small)
    assert err.value.code == SSD_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(y).all(), "a refused call must not run"
