"""The C-ABI library loads, exports every declared symbol, and checks arguments (no GPU)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER_DIR = os.path.join(ROOT, "include")


def declared_symbols():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(ssd_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from mamba_ssd_scan_05_b300 import build
    build.build()
    from mamba_ssd_scan_05_b300 import load_library
    return load_library()


def test_header_declares_entry_points():
    names = declared_symbols()
    for must in ("ssd_scan_fwd", "ssd_scan_workspace_bytes", "ssd_scan_get_status",
                 "ssd_scan_fwd_host", "ssd_scan_strerror"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_version_and_strerror(lib):
    import mamba_ssd_scan_05_b300 as m
    assert m.ssd_scan_version() >= 200
    for code in range(6):
        assert m.ssd_scan_strerror(code)
    assert "unknown" in m.ssd_scan_strerror(99)


def dims(b=1, L=256, H=4, P=64, N=128, G=1, dtype=1):
    from mamba_ssd_scan_05_b300 import ssd_dims
    return ssd_dims(b, L, H, P, N, G, dtype)


def test_resolve_path_rules(lib):
    import mamba_ssd_scan_05_b300 as m
    assert m.ssd_scan_resolve_path(dims(dtype=0, P=32, N=16), 64) == m.SSD_PATH_CHUNKED
    assert m.ssd_scan_resolve_path(dims(dtype=1, P=40, N=16), 64) == m.SSD_PATH_CHUNKED
    assert m.ssd_scan_resolve_path(dims(dtype=1), 256, m.SSD_PATH_CHUNKED) == m.SSD_PATH_CHUNKED
    # invalid problems come back as negative error codes
    assert m.ssd_scan_resolve_path(dims(H=6, G=4), 64) == -1
    assert m.ssd_scan_resolve_path(dims(), 0) == -1
    assert m.ssd_scan_resolve_path(dims(), 257) == -1
    assert m.ssd_scan_resolve_path(dims(dtype=7), 64) == -1
    assert m.ssd_scan_resolve_path(dims(N=300), 64) == -2
    assert m.ssd_scan_resolve_path(dims(), 64, 5) == -1


def test_kernels_per_call_without_a_device(lib):
    """The chunked path's three kernels are fixed; the tensor-core count needs the device's SM
    count, so without a device it is an error code, as is an invalid problem."""
    import mamba_ssd_scan_05_b300 as m
    assert m.ssd_scan_kernels_per_call(dims(dtype=0, P=32, N=16), 64) == 3
    assert m.ssd_scan_kernels_per_call(dims(dtype=1), 256, m.SSD_PATH_CHUNKED) == 3
    assert m.ssd_scan_kernels_per_call(dims(H=6, G=4), 64) == -1
    assert m.ssd_scan_kernels_per_call(dims(N=300), 64) == -2


def test_workspace_bytes(lib):
    import mamba_ssd_scan_05_b300 as m
    d = dims(b=2, L=300, H=3, P=5, N=7)
    got = m.ssd_scan_workspace_bytes(d, 64, m.SSD_PATH_CHUNKED)
    nc = (300 + 63) // 64
    states = 2 * 3 * nc * 5 * 7 * 4
    assert got >= 256 + states
    assert got % 256 == 0
    assert m.ssd_scan_workspace_bytes(dims(H=6, G=4), 64) == 0


def test_fwd_rejects_bad_arguments_before_any_launch(lib):
    """Argument errors return synchronously, before any CUDA call (safe without a GPU)."""
    import mamba_ssd_scan_05_b300 as m
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: checks fail first
    ws = ctypes.c_void_p(0x20000)
    d = dims()
    args = [fake, fake, fake, fake, fake, None, None, 64, fake, None]
    # bad shape
    assert lib.ssd_scan_fwd(ctypes.byref(dims(H=6, G=4)), *args, ws, 1 << 30, None) == 1
    # bad chunk
    bad = list(args); bad[7] = 0
    assert lib.ssd_scan_fwd(ctypes.byref(d), *bad, ws, 1 << 30, None) == 1
    # missing x
    bad = list(args); bad[0] = None
    assert lib.ssd_scan_fwd(ctypes.byref(d), *bad, ws, 1 << 30, None) == 1
    # misaligned x
    bad = list(args); bad[0] = ctypes.c_void_p(0x10002)
    assert lib.ssd_scan_fwd(ctypes.byref(d), *bad, ws, 1 << 30, None) == 1
    # workspace missing / too small / misaligned
    assert lib.ssd_scan_fwd(ctypes.byref(d), *args, None, 1 << 30, None) == 5
    assert lib.ssd_scan_fwd(ctypes.byref(d), *args, ws, 16, None) == 5
    assert lib.ssd_scan_fwd(ctypes.byref(d), *args, ctypes.c_void_p(0x20010), 1 << 30, None) == 5
    # explicit AUTO is not a valid explicit path
    assert lib.ssd_scan_fwd_path(ctypes.byref(d), *args, ws, 1 << 30, None, -1) == 1
    # null dims
    assert lib.ssd_scan_fwd(None, *args, ws, 1 << 30, None) == 1
    assert lib.ssd_scan_get_status(None, None) == 1


def test_host_arena_bytes(lib):
    import mamba_ssd_scan_05_b300 as m
    d = dims(b=1, L=64, H=2, P=32, N=16, dtype=0)
    need = m.ssd_scan_host_arena_bytes(d, 64)
    assert need > 2 * (64 * 2 * 32 * 4)
    assert m.ssd_scan_host_arena_bytes(dims(H=6, G=4), 64) == 0


def test_step_argument_checks_need_no_gpu(lib):
    """ssd_step_fwd rejects bad arguments before it touches the GPU."""
    import ctypes
    import mamba_ssd_scan_05_b300 as m
    p = ctypes.c_void_p(1 << 20)            # never dereferenced: the checks return first
    q = ctypes.c_void_p((1 << 20) + 4096)
    def call(d, x=p, dt=p, A=p, B=p, C=p, D=None, s_in=None, s_out=q, y=p):
        return lib.ssd_step_fwd(ctypes.byref(d), x, dt, A, B, C, D, s_in, s_out, y, None)
    assert call(dims(L=2)) == 1
    assert call(dims(L=0)) == 1
    assert call(dims(L=1), x=None) == 1
    assert call(dims(L=1), s_out=None) == 1
    assert call(dims(L=1, H=6, G=4)) == 1
    assert call(dims(L=1, dtype=5)) == 1
    assert call(dims(L=1), x=ctypes.c_void_p((1 << 20) + 8)) == 1          # misaligned
    # states overlapping without being the same buffer
    assert call(dims(L=1, b=1, H=1, P=4, N=4), s_in=ctypes.c_void_p(1 << 20),
                s_out=ctypes.c_void_p((1 << 20) + 16)) == 1


def test_varlen_workspace_checks_offsets(lib):
    import mamba_ssd_scan_05_b300 as m
    d = dims(b=1, L=300, H=8, P=64, N=128)
    # two non-empty tensor-core sequences run concurrently: a workspace slice per lane, each
    # with hand-off slots for 64 CTAs (2 x 64 x 64 x 128 floats)
    good = m.ssd_scan_varlen_workspace_bytes(d, [0, 100, 100, 300], 128)
    assert good >= 2 * (2 * 64 * 64 * 128 * 4)
    # one non-empty sequence runs as a plain scan: the whole scan workspace
    one = m.ssd_scan_varlen_workspace_bytes(dims(b=1, L=200, H=8, P=64, N=128), [0, 0, 200], 128)
    assert one >= m.ssd_scan_workspace_bytes(dims(b=1, L=200, H=8, P=64, N=128), 128)
    assert m.ssd_scan_varlen_workspace_bytes(d, [0, 100, 299], 128) == 0      # wrong total
    assert m.ssd_scan_varlen_workspace_bytes(d, [0, 200, 100, 300], 128) == 0  # decreasing
    assert m.ssd_scan_varlen_workspace_bytes(dims(b=2, L=300), [0, 300], 128) == 0  # batch != 1


def test_wait_limit_setter_round_trip(lib):
    import mamba_ssd_scan_05_b300 as m
    m.ssd_scan_set_wait_cycles(0)
    # the call returns the previous limit; <= 0 restores the default (2^32 cycles)
    assert m.ssd_scan_set_wait_cycles(0) == 1 << 32
    assert m.ssd_scan_set_wait_cycles(500) == 1 << 32
    assert m.ssd_scan_set_wait_cycles(-1) == 500
    assert m.ssd_scan_set_wait_cycles(0) == 1 << 32
