// ssd_scan.cu -- the C ABI of libssd_scan.so: argument checks, kernel-family dispatch, the
// host-buffer variant and status reporting.  Every declaration is in include/ssd_scan.h.
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"

using namespace ssd;

namespace {

constexpr int kMaxChunk = 256;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t elem_bytes(int32_t dtype) { return dtype == SSD_F32 ? 4 : 2; }

// Shape checks shared by every entry point.  Returns SSD_OK or SSD_ERR_INVALID.
int check_dims(const ssd_dims* d, int chunk_size) {
    if (!d) return SSD_ERR_INVALID;
    if (d->batch < 1 || d->seqlen < 0 || d->nheads < 1 || d->headdim < 1 || d->dstate < 1 ||
        d->ngroups < 1)
        return SSD_ERR_INVALID;
    if (d->nheads % d->ngroups != 0) return SSD_ERR_INVALID;
    if (d->dtype != SSD_F32 && d->dtype != SSD_BF16) return SSD_ERR_INVALID;
    if (chunk_size < 1 || chunk_size > kMaxChunk) return SSD_ERR_INVALID;
    // keep every element count comfortably inside int64 arithmetic
    const double elems = (double)d->batch * (double)d->seqlen * (double)d->nheads *
                         (double)d->headdim;
    const double states = (double)d->batch * (double)d->nheads * (double)d->headdim *
                          (double)d->dstate;
    if (elems > 4.0e15 || states > 4.0e15) return SSD_ERR_INVALID;
    return SSD_OK;
}

int resolve(const ssd_dims* d, int chunk_size, int path) {
    const int rc = check_dims(d, chunk_size);
    if (rc != SSD_OK) return -rc;
    const bool tc_ok = tc_supports(d->dtype, d->headdim, d->dstate, chunk_size);
    const bool ch_ok = chunked_supports(d->headdim, d->dstate, chunk_size);
    switch (path) {
        case SSD_PATH_AUTO:
            if (tc_ok) return SSD_PATH_TC;
            if (ch_ok) return SSD_PATH_CHUNKED;
            return -SSD_ERR_UNSUPPORTED;
        case SSD_PATH_TC: return tc_ok ? SSD_PATH_TC : -SSD_ERR_UNSUPPORTED;
        case SSD_PATH_CHUNKED: return ch_ok ? SSD_PATH_CHUNKED : -SSD_ERR_UNSUPPORTED;
        default: return -SSD_ERR_INVALID;
    }
}

size_t workspace_for(const ssd_dims* d, int chunk_size, int resolved) {
    if (resolved == SSD_PATH_TC)
        return tc_workspace_bytes(d->batch, d->seqlen, d->nheads, d->headdim, d->dstate,
                                  chunk_size);
    return chunked_workspace_bytes(d->batch, d->seqlen, d->nheads, d->headdim, d->dstate,
                                   chunk_size);
}

// The gated RMSNorm to fuse into a tensor-core scan's output (ssd_scan_fwd_gated).
struct Gate {
    const void* z;
    const float* w;
    float eps;
    int group;
};

int run(const ssd_dims* d, const void* x, const void* dt, const float* A, const void* B,
        const void* C, const float* D, const float* h0, int chunk_size, void* y, float* hT,
        void* workspace, size_t workspace_bytes, void* stream, int path,
        bool clear_status = true, const Gate* gate = nullptr, int max_ctas = 0,
        uint8_t* status = nullptr) {
    const int r = resolve(d, chunk_size, path);
    if (r < 0) return -r;
    if (!A || (d->seqlen > 0 && (!x || !dt || !B || !C || !y))) return SSD_ERR_INVALID;
    // x, B, C and y are moved in 16-byte vectors (and by TMA); dt is read element-wise
    if (!aligned(x, 16) || !aligned(dt, elem_bytes(d->dtype)) || !aligned(B, 16) ||
        !aligned(C, 16) || !aligned(y, 16) || !aligned(A, 4) || !aligned(D, 4) ||
        !aligned(h0, 4) || !aligned(hT, 4))
        return SSD_ERR_INVALID;
    if (!workspace || !aligned(workspace, 256)) return SSD_ERR_WORKSPACE;
    const size_t need = (r == SSD_PATH_TC && max_ctas > 0)
                            ? tc_workspace_bytes_ctas(d->dstate, max_ctas)
                            : workspace_for(d, chunk_size, r);
    if (workspace_bytes < need) return SSD_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the status word reports on this call only
    if (clear_status && cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (d->seqlen == 0) {
        if (!hT) return SSD_OK;
        const size_t sb = sizeof(float) * (size_t)(d->batch * d->nheads * d->headdim * d->dstate);
        const cudaError_t e = h0 ? cudaMemcpyAsync(hT, h0, sb, cudaMemcpyDeviceToDevice, st)
                                 : cudaMemsetAsync(hT, 0, sb, st);
        return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    }
    ScanArgs a;
    a.batch = d->batch; a.seqlen = d->seqlen; a.nheads = d->nheads; a.headdim = d->headdim;
    a.dstate = d->dstate; a.ngroups = d->ngroups; a.dtype = d->dtype; a.chunk = chunk_size;
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.h0 = h0; a.y = y; a.hT = hT;
    a.ws = static_cast<uint8_t*>(workspace); a.ws_bytes = workspace_bytes; a.stream = st;
    a.max_ctas = max_ctas;
    a.status = status;
    if (gate) {
        a.gated = 1;
        a.z = gate->z;
        a.norm_w = gate->w;
        a.eps = gate->eps;
        a.group = gate->group;
    }
    return r == SSD_PATH_TC ? tc_launch(a) : chunked_launch(a);
}

// Whether ssd_scan_fwd_gated fuses the norm into the scan kernel for this problem.
bool gated_fused(const ssd_dims* d, int chunk_size, int64_t group) {
    return resolve(d, chunk_size, SSD_PATH_AUTO) == SSD_PATH_TC && d->dstate == 128 &&
           group <= 64 && tc128_gated_supports(d->headdim, (int)group);
}

// y scratch of the unfused form of ssd_scan_fwd_gated, after the scan's own workspace.
size_t gated_scratch_offset(const ssd_dims* d, int chunk_size) {
    return align_up(workspace_for(d, chunk_size, resolve(d, chunk_size, SSD_PATH_AUTO)), 256);
}

// Byte sizes of every tensor of a problem, in the host-arena order.
struct Sizes {
    size_t x, dt, A, bc, D, st;
};
Sizes sizes_of(const ssd_dims* d) {
    Sizes s;
    const size_t eb = elem_bytes(d->dtype);
    s.x = eb * (size_t)(d->batch * d->seqlen * d->nheads * d->headdim);
    s.dt = eb * (size_t)(d->batch * d->seqlen * d->nheads);
    s.A = sizeof(float) * (size_t)d->nheads;
    s.bc = eb * (size_t)(d->batch * d->seqlen * d->ngroups * d->dstate);
    s.D = sizeof(float) * (size_t)d->nheads;
    s.st = sizeof(float) * (size_t)(d->batch * d->nheads * d->headdim * d->dstate);
    return s;
}

// ---- the host-buffer entry point's copy pipeline ----------------------------------------------

constexpr int kHostPieces = 8;          // at most this many pieces per call

// Per device: a copy-in and a copy-out stream and the events that order them against the
// caller's stream, created on first use and kept for the life of the process.  Calls enqueue
// under the mutex, so an event is never re-recorded before the previous call's waits on it
// have been enqueued.
constexpr int kVarlenLanes = 4;         // concurrent sequences of a packed batch
constexpr int64_t kTileTokens = 128;    // the tensor-core kernels' tile (work estimate)
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    cudaEvent_t in_done[kHostPieces] = {}, scan_done[kHostPieces] = {};
    cudaStream_t lane[kVarlenLanes] = {};
    cudaEvent_t lane_done[kVarlenLanes] = {};
    bool ready = false;
};
std::mutex g_pipe_mutex;
HostPipe g_pipe[64];

int host_pipe(HostPipe** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSD_ERR_CUDA;
    HostPipe& hp = g_pipe[dev];
    if (!hp.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.fork, ef) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.join, ef) != cudaSuccess)
            return SSD_ERR_CUDA;
        for (int i = 0; i < kHostPieces; ++i)
            if (cudaEventCreateWithFlags(&hp.in_done[i], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.scan_done[i], ef) != cudaSuccess)
                return SSD_ERR_CUDA;
        for (int i = 0; i < kVarlenLanes; ++i)
            if (cudaStreamCreateWithFlags(&hp.lane[i], cudaStreamNonBlocking) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.lane_done[i], ef) != cudaSuccess)
                return SSD_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return SSD_OK;
}

}  // namespace

extern "C" {

int ssd_scan_resolve_path(const ssd_dims* dims, int chunk_size, int path) {
    return resolve(dims, chunk_size, path);
}

size_t ssd_scan_workspace_bytes(const ssd_dims* dims, int chunk_size, int path) {
    const int r = resolve(dims, chunk_size, path);
    if (r < 0) return 0;
    return workspace_for(dims, chunk_size, r);
}

int ssd_scan_kernels_per_call(const ssd_dims* dims, int chunk_size, int path) {
    const int r = resolve(dims, chunk_size, path);
    if (r < 0) return r;
    if (r == SSD_PATH_CHUNKED) return 3;   // chunk states, state passing, chunk outputs
    if (dims->dstate == 128)
        return tc128_kernels_per_call(dims->batch, dims->seqlen, dims->nheads, dims->headdim);
    return 1;
}

int ssd_scan_fwd(const ssd_dims* dims, const void* x, const void* dt, const float* A,
                 const void* B, const void* C, const float* D, const float* initial_state,
                 int chunk_size, void* y, float* final_state, void* workspace,
                 size_t workspace_bytes, void* stream) {
    return run(dims, x, dt, A, B, C, D, initial_state, chunk_size, y, final_state, workspace,
               workspace_bytes, stream, SSD_PATH_AUTO);
}

int ssd_scan_fwd_path(const ssd_dims* dims, const void* x, const void* dt, const float* A,
                      const void* B, const void* C, const float* D, const float* initial_state,
                      int chunk_size, void* y, float* final_state, void* workspace,
                      size_t workspace_bytes, void* stream, int path) {
    if (path == SSD_PATH_AUTO) return SSD_ERR_INVALID;
    return run(dims, x, dt, A, B, C, D, initial_state, chunk_size, y, final_state, workspace,
               workspace_bytes, stream, path);
}

size_t ssd_scan_host_arena_bytes(const ssd_dims* dims, int chunk_size) {
    const int r = resolve(dims, chunk_size, SSD_PATH_AUTO);
    if (r < 0) return 0;
    const Sizes s = sizes_of(dims);
    return align_up(s.x, 256) * 2 + align_up(s.dt, 256) + align_up(s.A, 256) +
           align_up(s.bc, 256) * 2 + align_up(s.D, 256) + align_up(s.st, 256) * 2 +
           workspace_for(dims, chunk_size, r);
}

int ssd_scan_fwd_host(const ssd_dims* dims, const void* x, const void* dt, const float* A,
                      const void* B, const void* C, const float* D, const float* initial_state,
                      int chunk_size, void* y, float* final_state, void* device_arena,
                      size_t arena_bytes, void* stream) {
    const int r = resolve(dims, chunk_size, SSD_PATH_AUTO);
    if (r < 0) return -r;
    if (!A || (dims->seqlen > 0 && (!x || !dt || !B || !C || !y))) return SSD_ERR_INVALID;
    if (!device_arena || !aligned(device_arena, 256)) return SSD_ERR_INVALID;
    if (arena_bytes < ssd_scan_host_arena_bytes(dims, chunk_size)) return SSD_ERR_WORKSPACE;
    const Sizes s = sizes_of(dims);
    uint8_t* p = static_cast<uint8_t*>(device_arena);
    auto take = [&p](size_t n) { uint8_t* q = p; p += align_up(n, 256); return q; };
    uint8_t* dx = take(s.x);
    uint8_t* ddt = take(s.dt);
    float* dA = reinterpret_cast<float*>(take(s.A));
    uint8_t* dB = take(s.bc);
    uint8_t* dC = take(s.bc);
    float* dD = reinterpret_cast<float*>(take(s.D));
    float* dh0 = reinterpret_cast<float*>(take(s.st));
    uint8_t* dy = take(s.x);
    float* dhT = reinterpret_cast<float*>(take(s.st));
    uint8_t* dws = p;
    const size_t ws_bytes = arena_bytes - (size_t)(p - static_cast<uint8_t*>(device_arena));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;

    // Pieces: with at least kHostPieces rows, groups of batch rows (independent problems); with
    // fewer, each row cut into kHostPieces / b stretches of the sequence whose state is carried
    // on the device (multiples of 256 tokens, so each piece boundary is also a chunk and tile
    // boundary).  Piece p's copies in run on the copy-in stream while piece p - 1 scans on
    // `stream` and earlier pieces' outputs go back on the copy-out stream; more pieces leave
    // less of the first copy in and the last copy out without overlap.
    const int64_t b = dims->batch, L = dims->seqlen;
    const int64_t blocks = (L + 255) / 256;                           // 256-token blocks
    const int ns = (int)std::max<int64_t>(1, std::min<int64_t>(kHostPieces / std::max<int64_t>(b, 1), blocks));
    const bool by_rows = ns == 1;
    const int ngr = by_rows ? (int)std::max<int64_t>(1, std::min<int64_t>(kHostPieces, b)) : (int)b;
    const int np = ngr * ns;
    auto row_lo = [&](int g) { return b * g / ngr; };                // row group g's first row
    auto tok_lo = [&](int j) { return std::min<int64_t>(256 * (blocks * j / ns), L); };
    // per-token / per-row byte strides of each tensor
    const size_t eb = elem_bytes(dims->dtype);
    const size_t x_tok = eb * (size_t)(dims->nheads * dims->headdim);
    const size_t dt_tok = eb * (size_t)dims->nheads;
    const size_t bc_tok = eb * (size_t)(dims->ngroups * dims->dstate);
    const size_t st_row = sizeof(float) * (size_t)(dims->nheads * dims->headdim * dims->dstate);

    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe* hp = nullptr;
    int rc = host_pipe(&hp);
    if (rc != SSD_OK) return rc;
    bool ok = true;
    auto chk = [&ok](cudaError_t e) { ok = ok && e == cudaSuccess; };
    // the copy streams start after everything already on `stream` (which may still be using
    // the arena from an earlier call)
    chk(cudaEventRecord(hp->fork, st));
    chk(cudaStreamWaitEvent(hp->in, hp->fork, 0));
    chk(cudaStreamWaitEvent(hp->out, hp->fork, 0));
    // A and D once, with the first piece
    chk(cudaMemcpyAsync(dA, A, s.A, h2d, hp->in));
    if (D) chk(cudaMemcpyAsync(dD, D, s.D, h2d, hp->in));
    if (initial_state) chk(cudaMemcpyAsync(dh0, initial_state, s.st, h2d, hp->in));
    for (int i = 0; i < np && ok && rc == SSD_OK; ++i) {
        // rows lo .. hi - 1, tokens t0 .. t1 - 1 (one row when the rows are cut into stretches)
        const int g = i / ns, j = i % ns;
        const int64_t lo = by_rows ? row_lo(g) : g, hi = by_rows ? row_lo(g + 1) : g + 1;
        const int64_t t0 = tok_lo(j), t1 = tok_lo(j + 1);
        ssd_dims pd = *dims;
        pd.batch = hi - lo;
        pd.seqlen = t1 - t0;
        const int64_t tok0 = lo * L + t0, ntok = pd.batch * pd.seqlen;   // contiguous tokens
        const size_t ox = x_tok * (size_t)tok0, n_x = x_tok * (size_t)ntok;
        const size_t odt = dt_tok * (size_t)tok0, n_dt = dt_tok * (size_t)ntok;
        const size_t obc = bc_tok * (size_t)tok0, n_bc = bc_tok * (size_t)ntok;
        const auto* cx = static_cast<const uint8_t*>(x);
        const auto* cdt = static_cast<const uint8_t*>(dt);
        const auto* cB = static_cast<const uint8_t*>(B);
        const auto* cC = static_cast<const uint8_t*>(C);
        if (n_x) chk(cudaMemcpyAsync(dx + ox, cx + ox, n_x, h2d, hp->in));
        if (n_dt) chk(cudaMemcpyAsync(ddt + odt, cdt + odt, n_dt, h2d, hp->in));
        if (n_bc) chk(cudaMemcpyAsync(dB + obc, cB + obc, n_bc, h2d, hp->in));
        if (n_bc) chk(cudaMemcpyAsync(dC + obc, cC + obc, n_bc, h2d, hp->in));
        chk(cudaEventRecord(hp->in_done[i], hp->in));
        chk(cudaStreamWaitEvent(st, hp->in_done[i], 0));
        if (!ok) break;
        // the piece's entering and final state: its rows of h0 / hT, or (stretches of a row)
        // the row's running state, which alternates between its slices of the two buffers
        const size_t so = st_row / sizeof(float) * (size_t)lo;
        const float* h_in;
        float* h_out;
        if (by_rows) {
            h_in = initial_state ? dh0 + so : nullptr;
            h_out = final_state ? dhT + so : nullptr;
        } else {
            h_in = j == 0 ? (initial_state ? dh0 + so : nullptr) : ((j & 1) ? dhT : dh0) + so;
            h_out = j == ns - 1 ? (final_state ? ((j & 1) ? dh0 : dhT) + so : nullptr)
                                : ((j & 1) ? dh0 : dhT) + so;
        }
        rc = run(&pd, dx + ox, ddt + odt, dA, dB + obc, dC + obc, D ? dD : nullptr, h_in,
                 chunk_size, dy + ox, h_out, dws, ws_bytes, stream, SSD_PATH_AUTO,
                 /*clear_status=*/i == 0);
        if (rc != SSD_OK) break;
        chk(cudaEventRecord(hp->scan_done[i], st));
        chk(cudaStreamWaitEvent(hp->out, hp->scan_done[i], 0));
        if (n_x) chk(cudaMemcpyAsync(static_cast<uint8_t*>(y) + ox, dy + ox, n_x, d2h, hp->out));
        if (by_rows && final_state)
            chk(cudaMemcpyAsync(final_state + so, dhT + so, st_row * (size_t)pd.batch, d2h,
                                hp->out));
        if (!by_rows && final_state && j == ns - 1)
            chk(cudaMemcpyAsync(final_state + so, ((j & 1) ? dh0 : dhT) + so, st_row, d2h,
                                hp->out));
    }
    // `stream` ends after both copy streams: the caller's synchronisation covers every copy
    chk(cudaEventRecord(hp->join, hp->in));
    chk(cudaStreamWaitEvent(st, hp->join, 0));
    chk(cudaEventRecord(hp->join, hp->out));
    chk(cudaStreamWaitEvent(st, hp->join, 0));
    if (rc != SSD_OK) return rc;
    return ok ? SSD_OK : SSD_ERR_CUDA;
}

// Sequence i of a packed batch as a one-row problem: tokens cu[i] .. cu[i+1] - 1.
static bool varlen_dims(const ssd_dims* dims, const int64_t* cu, int64_t i, ssd_dims* out) {
    *out = *dims;
    out->batch = 1;
    out->seqlen = cu[i + 1] - cu[i];
    return true;
}

static int check_varlen(const ssd_dims* dims, const int64_t* cu, int64_t nseq) {
    if (!dims || !cu || nseq < 1 || dims->batch != 1) return SSD_ERR_INVALID;
    if (cu[0] != 0 || cu[nseq] != dims->seqlen) return SSD_ERR_INVALID;
    for (int64_t i = 0; i < nseq; ++i)
        if (cu[i + 1] < cu[i]) return SSD_ERR_INVALID;
    return SSD_OK;
}

// A packed batch whose non-empty sequences all take the tensor-core path, and more than one,
// runs them concurrently: on up to kVarlenLanes streams, each with its own workspace slice
// (hand-off slots for kVarlenCtas CTAs) and a grid of a quarter of the SMs.  With fewer CTAs
// per sequence a short sequence's chains are not cut into look-back pieces, and the lanes
// overlap each other's pipeline fill and drain.  Returns the number of lanes, or 0 for the
// sequential form (one launch after another on the caller's stream, one shared workspace).
constexpr int kVarlenCtas = 64;
static int varlen_lanes(const ssd_dims* dims, const int64_t* cu, int64_t nseq, int chunk_size,
                        int path) {
    int64_t busy = 0;
    for (int64_t i = 0; i < nseq; ++i) {
        ssd_dims di;
        varlen_dims(dims, cu, i, &di);
        if (di.seqlen == 0) continue;
        if (resolve(&di, chunk_size, path) != SSD_PATH_TC) return 0;
        ++busy;
    }
    return busy < 2 ? 0 : (int)std::min<int64_t>(kVarlenLanes, busy);
}
static size_t varlen_slice_bytes(const ssd_dims* dims) {
    return align_up(tc_workspace_bytes_ctas(dims->dstate, kVarlenCtas), 256);
}

size_t ssd_scan_varlen_workspace_bytes(const ssd_dims* dims, const int64_t* cu_seqlens,
                                       int64_t nseq, int chunk_size, int path) {
    if (check_varlen(dims, cu_seqlens, nseq) != SSD_OK) return 0;
    size_t need = 0;
    for (int64_t i = 0; i < nseq; ++i) {
        ssd_dims di;
        varlen_dims(dims, cu_seqlens, i, &di);
        if (di.seqlen == 0) continue;
        const int r = resolve(&di, chunk_size, path);
        if (r < 0) return 0;
        need = std::max(need, workspace_for(&di, chunk_size, r));
    }
    const int lanes = varlen_lanes(dims, cu_seqlens, nseq, chunk_size, path);
    if (lanes > 0) need = (size_t)lanes * varlen_slice_bytes(dims);
    return std::max(need, (size_t)kWsHeaderBytes);
}

int ssd_scan_fwd_varlen(const ssd_dims* dims, const int64_t* cu_seqlens, int64_t nseq,
                        const void* x, const void* dt, const float* A, const void* B,
                        const void* C, const float* D, const float* initial_state,
                        int chunk_size, void* y, float* final_state, void* workspace,
                        size_t workspace_bytes, void* stream, int path) {
    int rc = check_varlen(dims, cu_seqlens, nseq);
    if (rc != SSD_OK) return rc;
    rc = check_dims(dims, chunk_size);
    if (rc != SSD_OK) return rc;
    // every sequence must resolve and fit the workspace before anything is enqueued
    const size_t need = ssd_scan_varlen_workspace_bytes(dims, cu_seqlens, nseq, chunk_size, path);
    if (need == 0) return SSD_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256)) return SSD_ERR_WORKSPACE;
    if (workspace_bytes < need) return SSD_ERR_WORKSPACE;
    const size_t eb = elem_bytes(dims->dtype);
    const int64_t H = dims->nheads, P = dims->headdim, N = dims->dstate, G = dims->ngroups;
    // the x, y, B and C slices of every sequence start on 16-byte boundaries
    if ((H * P * eb) % 16 || (G * N * eb) % 16) return SSD_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return SSD_ERR_CUDA;
    const size_t state_elems = (size_t)(H * P * N);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    // sequence i on `lane_st` with the workspace `wsp` of `wsb` bytes
    auto scan_one = [&](int64_t i, cudaStream_t lane_st, uint8_t* wsp, size_t wsb,
                        int max_ctas) -> int {
        ssd_dims di;
        varlen_dims(dims, cu_seqlens, i, &di);
        const int64_t t0 = cu_seqlens[i];
        const float* h0 = initial_state ? initial_state + i * state_elems : nullptr;
        float* hT = final_state ? final_state + i * state_elems : nullptr;
        if (di.seqlen == 0) {   // an empty sequence: its final state is its initial state
            if (!hT) return SSD_OK;
            const size_t sb = sizeof(float) * state_elems;
            const cudaError_t e = h0 ? cudaMemcpyAsync(hT, h0, sb, cudaMemcpyDeviceToDevice, lane_st)
                                     : cudaMemsetAsync(hT, 0, sb, lane_st);
            return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
        }
        return run(&di, static_cast<const uint8_t*>(x) + eb * (size_t)(t0 * H * P),
                   static_cast<const uint8_t*>(dt) + eb * (size_t)(t0 * H), A,
                   static_cast<const uint8_t*>(B) + eb * (size_t)(t0 * G * N),
                   static_cast<const uint8_t*>(C) + eb * (size_t)(t0 * G * N), D, h0,
                   chunk_size, static_cast<uint8_t*>(y) + eb * (size_t)(t0 * H * P), hT, wsp,
                   wsb, lane_st, path, /*clear_status=*/false, nullptr, max_ctas, ws);
    };
    const int lanes = varlen_lanes(dims, cu_seqlens, nseq, chunk_size, path);
    if (lanes == 0) {
        for (int64_t i = 0; i < nseq; ++i) {
            rc = scan_one(i, st, ws, workspace_bytes, 0);
            if (rc != SSD_OK) return rc;
        }
        return SSD_OK;
    }
    // concurrent form: longest sequences first, each to the lane with the least work so far
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SSD_ERR_CUDA;
    const int ctas = std::max(1, std::min(kVarlenCtas, nsm / lanes));
    const size_t slice = varlen_slice_bytes(dims);
    std::vector<int64_t> order((size_t)nseq);
    for (int64_t i = 0; i < nseq; ++i) order[(size_t)i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
        return cu_seqlens[a + 1] - cu_seqlens[a] > cu_seqlens[b + 1] - cu_seqlens[b];
    });
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe* hp = nullptr;
    rc = host_pipe(&hp);
    if (rc != SSD_OK) return rc;
    bool ok = cudaEventRecord(hp->fork, st) == cudaSuccess;
    for (int l = 0; l < lanes && ok; ++l) ok = cudaStreamWaitEvent(hp->lane[l], hp->fork, 0) == cudaSuccess;
    int64_t load[kVarlenLanes] = {};
    for (size_t k = 0; k < order.size() && ok && rc == SSD_OK; ++k) {
        const int64_t i = order[k];
        int l = 0;
        for (int m = 1; m < lanes; ++m)
            if (load[m] < load[l]) l = m;
        load[l] += (cu_seqlens[i + 1] - cu_seqlens[i] + kTileTokens - 1) / kTileTokens + 1;
        rc = scan_one(i, hp->lane[l], ws + (size_t)l * slice, slice, ctas);
    }
    // `stream` continues after every lane, also on an error (nothing is left unordered)
    for (int l = 0; l < lanes; ++l) {
        ok = cudaEventRecord(hp->lane_done[l], hp->lane[l]) == cudaSuccess && ok;
        ok = cudaStreamWaitEvent(st, hp->lane_done[l], 0) == cudaSuccess && ok;
    }
    if (rc != SSD_OK) return rc;
    return ok ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_step_fwd(const ssd_dims* dims, const void* x, const void* dt, const float* A,
                 const void* B, const void* C, const float* D, const float* state_in,
                 float* state_out, void* y, void* stream) {
    if (!dims || dims->seqlen != 1) return SSD_ERR_INVALID;
    const int rc = check_dims(dims, 1);
    if (rc != SSD_OK) return rc;
    if (!x || !dt || !A || !B || !C || !y || !state_out) return SSD_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(dt, elem_bytes(dims->dtype)) || !aligned(B, 16) ||
        !aligned(C, 16) || !aligned(y, 16) || !aligned(A, 4) || !aligned(D, 4) ||
        !aligned(state_in, 4) || !aligned(state_out, 4))
        return SSD_ERR_INVALID;
    // the state is updated in place or copied to a separate buffer, never a partial overlap
    const size_t sb = sizeof(float) * (size_t)(dims->batch * dims->nheads * dims->headdim *
                                               dims->dstate);
    if (state_in && state_in != state_out) {
        const uintptr_t i0 = reinterpret_cast<uintptr_t>(state_in);
        const uintptr_t o0 = reinterpret_cast<uintptr_t>(state_out);
        if (i0 < o0 + sb && o0 < i0 + sb) return SSD_ERR_INVALID;
    }
    if (dims->batch * dims->nheads > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
    StepArgs a;
    a.batch = dims->batch; a.nheads = dims->nheads; a.headdim = dims->headdim;
    a.dstate = dims->dstate; a.ngroups = dims->ngroups; a.dtype = dims->dtype;
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D;
    a.s_in = state_in; a.s_out = state_out; a.y = y;
    a.stream = static_cast<cudaStream_t>(stream);
    return step_launch(a);
}

int ssd_causal_conv1d_fwd(int64_t batch, int64_t seqlen, int64_t channels, int width,
                          int32_t dtype, const void* x, const float* weight, const float* bias,
                          const void* state_in, void* state_out, int silu, void* out,
                          void* stream) {
    if (batch < 1 || batch > 65535 || seqlen < 0 || channels < 1 || width < 1 || width > 8)
        return SSD_ERR_INVALID;
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_INVALID;
    if ((double)batch * (double)seqlen * (double)channels > 4.0e15) return SSD_ERR_INVALID;
    if (!weight || (seqlen > 0 && (!x || !out))) return SSD_ERR_INVALID;
    const size_t eb = elem_bytes(dtype);
    if (!aligned(x, eb) || !aligned(out, eb) || !aligned(state_in, eb) ||
        !aligned(state_out, eb) || !aligned(weight, 4) || !aligned(bias, 4))
        return SSD_ERR_INVALID;
    // no buffer the kernel writes may overlap one it reads
    auto overlap = [](const void* a, size_t na, const void* b, size_t nb) {
        if (!a || !b || !na || !nb) return false;
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
        return a0 < b0 + nb && b0 < a0 + na;
    };
    const size_t xs = eb * (size_t)(batch * seqlen * channels);
    const size_t ss = eb * (size_t)(batch * (width - 1) * channels);
    if (overlap(out, xs, x, xs) || overlap(out, xs, state_in, ss) ||
        overlap(state_out, ss, x, xs) || overlap(state_out, ss, state_in, ss) ||
        overlap(state_out, ss, out, xs))
        return SSD_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (seqlen == 0) {   // nothing to convolve: the state passes through
        if (!state_out || ss == 0) return SSD_OK;
        const cudaError_t e = state_in
                                  ? cudaMemcpyAsync(state_out, state_in, ss,
                                                    cudaMemcpyDeviceToDevice, st)
                                  : cudaMemsetAsync(state_out, 0, ss, st);
        return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    }
    ConvArgs a;
    a.batch = batch; a.seqlen = seqlen; a.channels = channels; a.width = width; a.dtype = dtype;
    a.x = x; a.weight = weight; a.bias = bias; a.s_in = state_in; a.s_out = state_out;
    a.silu = silu ? 1 : 0; a.out = out; a.stream = st;
    return conv_launch(a);
}

int ssd_gated_rmsnorm_fwd(int64_t rows, int64_t dim, int64_t group_size, int32_t dtype,
                          const void* y, const void* z, const float* weight, float eps,
                          void* out, void* stream) {
    if (rows < 0 || dim < 1 || group_size < 1 || dim % group_size != 0) return SSD_ERR_INVALID;
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_INVALID;
    if (!(eps >= 0.f) || eps > 1.0e30f) return SSD_ERR_INVALID;
    if (rows > 0 && (!y || !out)) return SSD_ERR_INVALID;
    const size_t eb = elem_bytes(dtype);
    if (!aligned(y, eb) || !aligned(z, eb) || !aligned(out, eb) || !aligned(weight, 4))
        return SSD_ERR_INVALID;
    if (rows > 0x7fffffffLL || dim / group_size > 12288) return SSD_ERR_UNSUPPORTED;
    if (rows == 0) return SSD_OK;
    NormArgs a;
    a.rows = rows; a.dim = dim; a.group_size = group_size; a.dtype = dtype;
    a.y = y; a.z = z; a.weight = weight; a.eps = eps; a.out = out;
    a.stream = static_cast<cudaStream_t>(stream);
    return norm_launch(a);
}

size_t ssd_scan_gated_workspace_bytes(const ssd_dims* dims, int chunk_size, int64_t group_size) {
    const int r = resolve(dims, chunk_size, SSD_PATH_AUTO);
    if (r < 0 || group_size < 1 || (dims->nheads * dims->headdim) % group_size != 0) return 0;
    if (gated_fused(dims, chunk_size, group_size)) return workspace_for(dims, chunk_size, r);
    return gated_scratch_offset(dims, chunk_size) +
           align_up(elem_bytes(dims->dtype) *
                        (size_t)(dims->batch * dims->seqlen * dims->nheads * dims->headdim),
                    256);
}

int ssd_scan_fwd_gated(const ssd_dims* dims, const void* x, const void* dt, const float* A,
                       const void* B, const void* C, const float* D, const float* initial_state,
                       int chunk_size, const void* z, const float* norm_weight, float eps,
                       int64_t group_size, void* out, float* final_state, void* workspace,
                       size_t workspace_bytes, void* stream) {
    const int r = resolve(dims, chunk_size, SSD_PATH_AUTO);
    if (r < 0) return -r;
    const int64_t dim = dims->nheads * dims->headdim;
    if (group_size < 1 || dim % group_size != 0) return SSD_ERR_INVALID;
    if (!(eps >= 0.f) || eps > 1.0e30f) return SSD_ERR_INVALID;
    if (dims->seqlen > 0 && (!z || !out)) return SSD_ERR_INVALID;
    const bool fused = gated_fused(dims, chunk_size, group_size);
    // z is read like y (16-byte vectors); the fused form reads the weight as float4
    if (!aligned(z, 16) || !aligned(norm_weight, fused ? 16 : 4)) return SSD_ERR_INVALID;
    if (!workspace || !aligned(workspace, 256)) return SSD_ERR_WORKSPACE;
    if (workspace_bytes < ssd_scan_gated_workspace_bytes(dims, chunk_size, group_size))
        return SSD_ERR_WORKSPACE;
    if (fused) {
        const Gate g{z, norm_weight, eps, (int)group_size};
        return run(dims, x, dt, A, B, C, D, initial_state, chunk_size, out, final_state,
                   workspace, workspace_bytes, stream, SSD_PATH_AUTO, true, &g);
    }
    // unfused: the scan into the workspace's y scratch, then the gated RMSNorm kernel
    const size_t off = gated_scratch_offset(dims, chunk_size);
    void* ys = static_cast<uint8_t*>(workspace) + off;
    int rc = run(dims, x, dt, A, B, C, D, initial_state, chunk_size, ys, final_state, workspace,
                 off, stream, SSD_PATH_AUTO);
    if (rc != SSD_OK) return rc;
    return ssd_gated_rmsnorm_fwd(dims->batch * dims->seqlen, dim, group_size, dims->dtype, ys, z,
                                 norm_weight, eps, out, stream);
}

int ssd_scan_get_status(void* workspace, void* stream) {
    if (!workspace) return SSD_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SSD_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return SSD_ERR_CUDA;
    return v == 0 ? SSD_OK : v;
}

const char* ssd_scan_strerror(int code) {
    switch (code) {
        case SSD_OK: return "ok";
        case SSD_ERR_INVALID: return "invalid argument (pointer, alignment, size or shape)";
        case SSD_ERR_UNSUPPORTED: return "problem not supported by the selected kernel family";
        case SSD_ERR_CUDA: return "CUDA runtime error";
        case SSD_ERR_TIMEOUT: return "a bounded device-side wait gave up";
        case SSD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        default: return "unknown error code";
    }
}

int ssd_scan_version(void) { return 300; }   // 0.3.0: + fused gated scan, wait-limit setter

}  // extern "C"
