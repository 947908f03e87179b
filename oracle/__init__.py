"""CPU oracle for the Mamba-2 SSD forward scan.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference leg of ``bench.py`` import this package.  The product (``mamba_ssd_scan_05_b300``)
never imports it, and this package imports nothing from the product.

Three independent float64 forms of the same method, each written from the pages:

``scan``       the sequential recurrence (plain C, ``ssd_oracle.c``).  This is THE oracle: the
               definition of what the path computes.
               youngju.dev "Mamba / selective SSM" article, section "LTIからSelectionへの切り替え"
               (Abar_t = exp(dt_t A), Bbar_t = dt_t B_t, h_t = Abar_t h_{t-1} + Bbar_t x_t,
               y_t = C_t h_t), plus the skip term D x of the SelectiveSSM listing in the same
               article, with A one scalar per head (Qiita "Mamba-2 / SSD" article, section 4.2).

``quadratic``  the materialised semiseparable matrix y = M x with
               M_ij = C_i^T Abar_{i:j} Bbar_j for i >= j, 0 otherwise, and
               Abar_{i:j} = Abar_i ... Abar_{j+1}
               (youngju.dev article, section "State Space Dualityの発見", the M_ij display).
               Brute force, for tiny inputs only; used to pin ``scan``.

``chunked``    the chunk algorithm: split the sequence into chunks of Q tokens; inside a chunk
               the attention-like dual form with the decay mask exp(cum_i - cum_j); between
               chunks the state recurrence (Qiita article section 4.2, "chunk内は行列積、chunk間は
               スキャン"; youngju.dev article, section "SSDアルゴリズムとチャンク分割", the
               ``_chunk_scan`` listing).  That listing is incomplete: it omits dt_j on the key
               side, has no inter-chunk pass and exponentiates before masking.  This form
               multiplies by dt_j (Bbar = dt B), adds the state pass between chunks and masks
               before the exponential.  Exposes the per-stage intermediates.

Layouts (row-major, any float dtype in, float64 out):
    x  [b, L, H, P]   dt [b, L, H]   A [H]   B, C [b, L, G, N]   D [H]   h0 [b, H, P, N]
Head h uses group g = h // (H // G).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssd_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile an oracle C source (default ``ssd_oracle.c``) into a shared library (gcc, OpenMP)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC", "-std=c11",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class OracleLib:
    """A loaded oracle shared library (the real one, or a test's deliberately broken copy)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        d = ctypes.POINTER(ctypes.c_double)
        lib.ssd_oracle_scan.restype = ctypes.c_int
        lib.ssd_oracle_scan.argtypes = [ctypes.c_int64] * 4 + [d] * 9 + [ctypes.c_int]
        lib.ssd_oracle_version.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def scan_problems(self, x, dt, A, B, C, D=None, h0=None, n_threads: int = 0):
        """Run independent (batch, head) problems already gathered per problem.

        x [n, L, P], dt [n, L], A [n], B, C [n, L, N], D [n] or None, h0 [n, P, N] or None.
        Returns (y [n, L, P], hT [n, P, N], threads_used), all float64.
        """
        x, dt, A, B, C = (_f64(v) for v in (x, dt, A, B, C))
        D = _f64(D)
        h0 = _f64(h0)
        n, L, P = x.shape
        N = B.shape[-1]
        if dt.shape != (n, L) or A.shape != (n,) or B.shape != (n, L, N) or C.shape != (n, L, N):
            raise ValueError("oracle: inconsistent problem shapes")
        if D is not None and D.shape != (n,):
            raise ValueError("oracle: D must be [n]")
        if h0 is not None and h0.shape != (n, P, N):
            raise ValueError("oracle: h0 must be [n, P, N]")
        y = np.empty((n, L, P), dtype=np.float64)
        hT = np.empty((n, P, N), dtype=np.float64)
        used = self.lib.ssd_oracle_scan(n, L, P, N, _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                        _ptr(C), _ptr(D), _ptr(h0), _ptr(y), _ptr(hT),
                                        int(n_threads))
        if used < 1:
            raise RuntimeError("oracle: ssd_oracle_scan failed")
        return y, hT, used


def default_lib() -> OracleLib:
    """The oracle library built from ``ssd_oracle.c`` (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = OracleLib(_LIB_PATH)
    return _lib


def _f64(a):
    """Any CPU array-like (numpy, torch incl. bf16) -> contiguous float64 numpy array."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        import torch
        a = a.detach().to("cpu")
        if a.dtype != torch.float64:
            a = a.float().double()
        return np.ascontiguousarray(a.numpy())
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def group_of_head(h: int, H: int, G: int) -> int:
    """Reading used throughout: contiguous blocks of H // G heads share one B/C group."""
    return h // (H // G)


def scan_problems(x, dt, A, B, C, D=None, h0=None, n_threads: int = 0, lib: OracleLib = None):
    """``OracleLib.scan_problems`` on the default library (or ``lib``)."""
    return (lib or default_lib()).scan_problems(x, dt, A, B, C, D, h0, n_threads)


def gather_problems(x, dt, A, B, C, D=None, h0=None, heads=None):
    """Gather per-(b, h) float64 problems from the full layouts.

    heads: iterable of (b, h) pairs, or None for all of them in (b, h) order.
    """
    bsz, L, H, P = x.shape
    G = B.shape[2]
    if H % G != 0:
        raise ValueError("oracle: nheads must be a multiple of ngroups")
    if heads is None:
        heads = [(b, h) for b in range(bsz) for h in range(H)]
    heads = list(heads)
    xs = np.stack([_f64(x[b, :, h, :]) for b, h in heads]) if heads else np.zeros((0, L, P))
    dts = np.stack([_f64(dt[b, :, h]) for b, h in heads]) if heads else np.zeros((0, L))
    As = np.array([float(A[h]) for _, h in heads], dtype=np.float64)
    Bs = np.stack([_f64(B[b, :, group_of_head(h, H, G), :]) for b, h in heads]) if heads else None
    Cs = np.stack([_f64(C[b, :, group_of_head(h, H, G), :]) for b, h in heads]) if heads else None
    Ds = None if D is None else np.array([float(D[h]) for _, h in heads], dtype=np.float64)
    h0s = None if h0 is None else np.stack([_f64(h0[b, h]) for b, h in heads])
    return heads, xs, dts, As, Bs, Cs, Ds, h0s


def scan(x, dt, A, B, C, D=None, h0=None, heads=None, n_threads: int = 0, lib=None):
    """The oracle on the full layouts.

    Without ``heads``: returns y [b, L, H, P] and hT [b, H, P, N] (float64).
    With ``heads`` (list of (b, h)): returns y [k, L, P] and hT [k, P, N] in that order.
    """
    full = heads is None
    heads, xs, dts, As, Bs, Cs, Ds, h0s = gather_problems(x, dt, A, B, C, D, h0, heads)
    if len(heads) == 0:
        bsz, L, H, P = x.shape
        N = B.shape[-1]
        if full:
            return np.zeros((bsz, L, H, P)), np.zeros((bsz, H, P, N))
        return np.zeros((0, L, P)), np.zeros((0, P, N))
    y, hT, _ = scan_problems(xs, dts, As, Bs, Cs, Ds, h0s, n_threads, lib=lib)
    if not full:
        return y, hT
    bsz, L, H, P = x.shape
    N = B.shape[-1]
    yf = np.empty((bsz, L, H, P), dtype=np.float64)
    hf = np.empty((bsz, H, P, N), dtype=np.float64)
    for i, (b, h) in enumerate(heads):
        yf[b, :, h, :] = y[i]
        hf[b, h] = hT[i]
    return yf, hf


def quadratic(x, dt, A, B, C, D=None, h0=None):
    """Materialised semiseparable form y = M x (+ initial-state and skip terms), float64.

    For each (b, h): M_ij = (C_i . B_j) * dt_j * prod_{k=j+1..i} exp(dt_k A) for i >= j, else 0.
    The initial state h0 (the state before token 0) enters as
    C_i^T (prod_{k=0..i} exp(dt_k A)) h0, the unrolled recurrence's first term.
    Tiny inputs only (O(L^2) per head).  Returns y [b, L, H, P], hT [b, H, P, N].
    """
    x, dt, B, C = (_f64(v) for v in (x, dt, B, C))
    A = _f64(A)
    D = _f64(D)
    h0 = _f64(h0)
    bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros((bsz, L, H, P))
    hT = np.zeros((bsz, H, P, N))
    for b in range(bsz):
        for h in range(H):
            g = group_of_head(h, H, G)
            abar = np.exp(dt[b, :, h] * A[h])            # Abar_k
            Bg, Cg, xh, dth = B[b, :, g, :], C[b, :, g, :], x[b, :, h, :], dt[b, :, h]
            M = np.zeros((L, L))
            for i in range(L):
                # decay[j] = Abar_i * Abar_{i-1} * ... * Abar_{j+1}  (empty product = 1 at j = i)
                decay = np.ones(i + 1)
                for j in range(i - 1, -1, -1):
                    decay[j] = decay[j + 1] * abar[j + 1]
                M[i, : i + 1] = (Cg[i] @ Bg[: i + 1].T) * dth[: i + 1] * decay
            yh = M @ xh
            if h0 is not None:
                carry = np.cumprod(abar)                 # prod_{k=0..i} Abar_k
                yh += carry[:, None] * (Cg @ h0[b, h].T)  # C_i^T h0, scaled
            if D is not None:
                yh += D[h] * xh
            y[b, :, h, :] = yh
            # final state: h_{L-1} = sum_j Abar_{L-1:j} Bbar_j x_j^T + Abar_{L-1:-1} h0
            if L > 0:
                decay_end = np.ones(L)
                for j in range(L - 2, -1, -1):
                    decay_end[j] = decay_end[j + 1] * abar[j + 1]
                hT[b, h] = (xh * (dth * decay_end)[:, None]).T @ Bg
                if h0 is not None:
                    hT[b, h] += np.prod(abar) * h0[b, h]
            elif h0 is not None:
                hT[b, h] = h0[b, h]
    return y, hT


def chunked(x, dt, A, B, C, D=None, h0=None, chunk_size: int = 256, keep_stages: bool = False):
    """The chunk algorithm in float64, steps in the pages' order.

    Per (b, h) and chunk c of Q = chunk_size tokens (the sequence is padded to a multiple of Q
    with dt = 0, x = 0, B = C = 0; padded rows are cropped):
      S1  a_t = dt_t A; cum = inclusive cumsum of a inside the chunk;
          Lmask_ij = exp(cum_i - cum_j) for i >= j (masked before exp), 0 otherwise
      S2  G = C_c B_c^T;  Y_diag = (Lmask o G o dt_j) X_c;
          chunk state S_c = X_c^T diag(exp(cum_last - cum) * dt) B_c      [P x N]
      S3  h_c = exp(cum_last) h_{c-1} + S_c, with h_{-1} = h0 (or 0); final state = h_last
      S4  Y = Y_diag + diag(exp(cum)) C_c h_{c-1}^T + D X_c
    Returns (y [b, L, H, P], hT [b, H, P, N]) and, with keep_stages, a dict of per-(b, h, c)
    intermediates: cum, G, Ydiag, S, h_in (state entering the chunk), Yoff.
    """
    x, dt, B, C = (_f64(v) for v in (x, dt, B, C))
    A = _f64(A)
    D = _f64(D)
    h0 = _f64(h0)
    bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    Q = int(chunk_size)
    if Q <= 0:
        raise ValueError("chunk_size must be positive")
    nc = (L + Q - 1) // Q
    pad = nc * Q - L
    y = np.zeros((bsz, L, H, P))
    hT = np.zeros((bsz, H, P, N))
    stages = {} if keep_stages else None
    tril = np.tril(np.ones((Q, Q), dtype=bool))
    for b in range(bsz):
        for h in range(H):
            g = group_of_head(h, H, G)
            xh = np.pad(x[b, :, h, :], ((0, pad), (0, 0)))
            dth = np.pad(dt[b, :, h], (0, pad))
            Bg = np.pad(B[b, :, g, :], ((0, pad), (0, 0)))
            Cg = np.pad(C[b, :, g, :], ((0, pad), (0, 0)))
            hstate = np.zeros((P, N)) if h0 is None else h0[b, h].copy()
            yh = np.zeros((nc * Q, P))
            for c in range(nc):
                sl = slice(c * Q, (c + 1) * Q)
                Xc, dtc, Bc, Cc = xh[sl], dth[sl], Bg[sl], Cg[sl]
                cum = np.cumsum(dtc * A[h])                                   # S1
                diff = cum[:, None] - cum[None, :]
                Lmask = np.where(tril, np.exp(np.where(tril, diff, 0.0)), 0.0)
                Gm = Cc @ Bc.T                                                # S2
                Ydiag = (Lmask * Gm * dtc[None, :]) @ Xc
                r = np.exp(cum[-1] - cum)
                S = (Xc * (r * dtc)[:, None]).T @ Bc
                Yoff = np.exp(cum)[:, None] * (Cc @ hstate.T)                 # S4
                Yc = Ydiag + Yoff
                if D is not None:
                    Yc = Yc + D[h] * Xc
                yh[sl] = Yc
                if keep_stages:
                    stages[(b, h, c)] = dict(cum=cum, G=Gm, Ydiag=Ydiag, S=S,
                                             h_in=hstate.copy(), Yoff=Yoff)
                hstate = np.exp(cum[-1]) * hstate + S                         # S3
            y[b, :, h, :] = yh[:L]
            hT[b, h] = hstate
    if keep_stages:
        return y, hT, stages
    return y, hT


def error_metrics(y, y_ref):
    """The two parity metrics: max|dy| / max|y_ref| and sum|dy| / sum|y_ref| (float64)."""
    y = _f64(y)
    y_ref = _f64(y_ref)
    d = np.abs(y - y_ref)
    den_max = float(np.max(np.abs(y_ref))) if y_ref.size else 0.0
    den_sum = float(np.sum(np.abs(y_ref))) if y_ref.size else 0.0
    max_rel = float(np.max(d)) / den_max if den_max > 0 else float(np.max(d, initial=0.0))
    mean_rel = float(np.sum(d)) / den_sum if den_sum > 0 else float(np.sum(d))
    return max_rel, mean_rel
