"""Helpers for the GPU parity tests: run the CUDA path through the C ABI, compare to the oracle."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from mamba_ssd_scan_05_b300 import workloads

# Tolerances: max|dy| / max|y_ref| and sum|dy| / sum|y_ref| (float32 storage: 1e-4 on the max;
# bf16 storage with float32 accumulation: 2e-2 on the max, 5e-3 on the mean); final_state to
# the same bounds.
TOL = {"f32": (1e-4, 1e-4), "bf16": (2e-2, 5e-3)}


def dtype_name(t: torch.dtype) -> str:
    return "f32" if t == torch.float32 else "bf16"


def to_device(inp: dict, device="cuda") -> dict:
    return {k: (None if v is None else v.to(device, non_blocking=False).contiguous())
            for k, v in inp.items()}


def run_gpu(inp_dev: dict, chunk: int, path: int = -1, use_D: bool = True, use_h0: bool = True):
    """One ssd_scan_fwd call; also checks the call's device status word."""
    from mamba_ssd_scan_05_b300 import (make_dims, ssd_scan_fwd, ssd_scan_get_status,
                                        ssd_scan_workspace_bytes)
    dims = make_dims(inp_dev["x"], inp_dev["B"])
    need = ssd_scan_workspace_bytes(dims, chunk, path)
    assert need > 0, "problem rejected"
    ws = torch.empty(need, dtype=torch.uint8, device=inp_dev["x"].device)
    y, hT = ssd_scan_fwd(inp_dev["x"], inp_dev["dt"], inp_dev["A"], inp_dev["B"], inp_dev["C"],
                         inp_dev["D"] if use_D else None,
                         inp_dev["h0"] if use_h0 else None, chunk_size=chunk, path=path,
                         workspace=ws)
    assert ssd_scan_get_status(ws) == 0, "device status word reports an error"
    return y, hT


def assert_close(got, ref, dtype: str, what: str):
    mx, mean = oracle.error_metrics(got, ref)
    tmax, tmean = TOL[dtype]
    assert np.all(np.isfinite(oracle._f64(got))), f"{what}: non-finite values"
    assert mx <= tmax, f"{what}: max rel err {mx:.3e} > {tmax:.0e}"
    assert mean <= tmean, f"{what}: mean rel err {mean:.3e} > {tmean:.0e}"
    return mx, mean


def check_against_oracle(inp_cpu: dict, y_dev, hT_dev, heads=None, use_D=True, use_h0=True,
                         what=""):
    """Compare GPU outputs with the oracle on all heads, or on the sampled (b, h) heads."""
    dt_name = dtype_name(inp_cpu["x"].dtype)
    D = inp_cpu["D"] if use_D else None
    h0 = inp_cpu["h0"] if use_h0 else None
    if heads is None:
        y_ref, h_ref = oracle.scan(inp_cpu["x"], inp_cpu["dt"], inp_cpu["A"], inp_cpu["B"],
                                   inp_cpu["C"], D, h0)
        got_y = y_dev.float().cpu()
        got_h = None if hT_dev is None else hT_dev.cpu()
    else:
        y_ref, h_ref = oracle.scan(inp_cpu["x"], inp_cpu["dt"], inp_cpu["A"], inp_cpu["B"],
                                   inp_cpu["C"], D, h0, heads=heads)
        got_y = torch.stack([y_dev[b, :, h, :].float().cpu() for b, h in heads])
        got_h = None if hT_dev is None else torch.stack([hT_dev[b, h].cpu() for b, h in heads])
    r = {"y": assert_close(got_y, y_ref, dt_name, f"{what} y")}
    if got_h is not None:
        r["final_state"] = assert_close(got_h, h_ref, dt_name, f"{what} final_state")
    return r


def check_all_heads(inp_cpu: dict, y_dev, hT_dev, what="", heads_per_batch: int = 16,
                    use_D=True, use_h0=True):
    """Compare every (b, h) head with the oracle, a batch of heads at a time.

    The metrics are the global ones of ``assert_close`` (max|dy| / max|y_ref| and
    sum|dy| / sum|y_ref| over all heads), accumulated batch by batch so that the float64
    copies of a large workload never sit in host memory all at once.  Returns the two metrics
    for y and for the final state.
    """
    dt_name = dtype_name(inp_cpu["x"].dtype)
    bsz, _, H, _ = inp_cpu["x"].shape
    D = inp_cpu["D"] if use_D else None
    h0 = inp_cpu["h0"] if use_h0 else None
    heads = [(b, h) for b in range(bsz) for h in range(H)]
    acc = {"y": [0.0, 0.0, 0.0, 0.0], "final_state": [0.0, 0.0, 0.0, 0.0]}
    for i in range(0, len(heads), heads_per_batch):
        part = heads[i:i + heads_per_batch]
        y_ref, h_ref = oracle.scan(inp_cpu["x"], inp_cpu["dt"], inp_cpu["A"], inp_cpu["B"],
                                   inp_cpu["C"], D, h0, heads=part)
        got_y = torch.stack([y_dev[b, :, h, :] for b, h in part]).double().cpu().numpy()
        pairs = [("y", got_y, y_ref)]
        if hT_dev is not None:
            got_h = torch.stack([hT_dev[b, h] for b, h in part]).double().cpu().numpy()
            pairs.append(("final_state", got_h, h_ref))
        for name, got, ref in pairs:
            assert np.all(np.isfinite(got)), f"{what} {name}: non-finite values"
            d = np.abs(got - ref)
            a = acc[name]
            a[0] = max(a[0], float(d.max(initial=0.0)))
            a[1] = max(a[1], float(np.abs(ref).max(initial=0.0)))
            a[2] += float(d.sum())
            a[3] += float(np.abs(ref).sum())
    tmax, tmean = TOL[dt_name]
    out = {}
    for name, (dmax, rmax, dsum, rsum) in acc.items():
        if name == "final_state" and hT_dev is None:
            continue
        mx = dmax / rmax if rmax > 0 else dmax
        mean = dsum / rsum if rsum > 0 else dsum
        assert mx <= tmax, f"{what} {name}: max rel err {mx:.3e} > {tmax:.0e}"
        assert mean <= tmean, f"{what} {name}: mean rel err {mean:.3e} > {tmean:.0e}"
        out[name] = (mx, mean)
    return out


@functools.lru_cache(maxsize=2)
def workload_inputs(idx: int) -> dict:
    return workloads.make_inputs(workloads.WORKLOADS[idx])


def sample_heads(b: int, H: int, k: int = 4, seed: int = 0):
    rng = np.random.default_rng(seed)
    heads = {(0, 0), (b - 1, H - 1)}
    while len(heads) < min(k, b * H):
        heads.add((int(rng.integers(b)), int(rng.integers(H))))
    return sorted(heads)
