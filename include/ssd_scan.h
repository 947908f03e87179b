/*
 * ssd_scan.h -- C ABI of libssd_scan.so, the B300 (sm_103a) Mamba-2 SSD forward scan.
 *
 * The operation (per batch row b and head h, tokens t = 0..L-1, state h_t a P x N matrix):
 *
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * x_t B_t^T
 *     y_t = C_t^T h_t + D_h * x_t                     (y_t[p] = sum_n C_t[n] h_t[p][n] + D_h x_t[p])
 *
 * with h_{-1} = initial_state (or zeros) and final_state = h_{L-1}.  Sources:
 *   - youngju.dev "Mamba / selective SSM" article, section "LTIからSelectionへの切り替え":
 *     Abar_t = exp(Delta_t A), Bbar_t = Delta_t B_t, h_t = Abar_t h_{t-1} + Bbar_t x_t, y_t = C_t h_t;
 *     the SelectiveSSM listing of the same article adds the skip term D * x.
 *   - Qiita "Mamba-2 / SSD" article, section 4.2: A = -exp(A_log) is one scalar per head, and the
 *     scan is computed by the SSD chunk algorithm (matmuls inside a chunk, a scan between chunks)
 *     with a chunk_size argument; section 4.1: heads as in attention, B/C shared by head groups.
 *   - youngju.dev article, section "State Space Dualityの発見": the same y as y = M x with the
 *     semiseparable M_ij = C_i^T Abar_{i:j} Bbar_j (i >= j); section "SSDアルゴリズムとチャンク分割":
 *     the chunk split, the cumulative-sum decay mask and the intra-chunk dual form.
 *
 * Conventions for every entry point:
 *   - All tensors are dense, row-major, contiguous, and live in DEVICE memory unless a function
 *     says otherwise.  The library never allocates device memory except inside the functions
 *     whose comment says so (none here do); the caller owns every buffer.
 *   - Layouts (T = the element type named by ssd_dims.dtype):
 *       x              [batch, seqlen, nheads, headdim]   T
 *       dt             [batch, seqlen, nheads]            T   (already positive: post-softplus)
 *       A              [nheads]                           float32 (normally < 0)
 *       B, C           [batch, seqlen, ngroups, dstate]   T
 *       D              [nheads]                           float32, or NULL for no skip term
 *       initial_state  [batch, nheads, headdim, dstate]   float32, or NULL for zeros
 *       y              [batch, seqlen, nheads, headdim]   T   (written)
 *       final_state    [batch, nheads, headdim, dstate]   float32 (written), or NULL
 *     Head h reads B/C group h / (nheads / ngroups).
 *   - Base pointers of x, B, C, y must be 16-byte aligned; dt aligned to its element size;
 *     initial_state and final_state 4-byte aligned; workspace 256-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every
 *     launch and copy is enqueued on it; the functions return without synchronising, except
 *     ssd_scan_get_status, which synchronises `stream`.
 *   - Errors: argument and shape errors are returned synchronously, before anything is
 *     enqueued.  No C++ exception crosses this boundary.  A device-side bounded wait that runs
 *     out sets an error word in the workspace; read it with ssd_scan_get_status.
 *   - Calls on different streams may run concurrently if each has its own workspace.
 */
#ifndef SSD_SCAN_H_
#define SSD_SCAN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of x, dt, B, C and y.  Arithmetic is float32 on the device in both cases. */
typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* Problem shape.  All sizes are element counts. */
typedef struct {
    int64_t batch;    /* b  >= 1 */
    int64_t seqlen;   /* L  >= 0 (0: nothing to scan; final_state = initial_state) */
    int64_t nheads;   /* H  >= 1 */
    int64_t headdim;  /* P  >= 1 */
    int64_t dstate;   /* N  >= 1 */
    int64_t ngroups;  /* G  >= 1, H % G == 0 */
    int32_t dtype;    /* ssd_dtype */
} ssd_dims;

/* Return codes. */
enum {
    SSD_OK = 0,
    SSD_ERR_INVALID = 1,      /* bad pointer, alignment, size or shape */
    SSD_ERR_UNSUPPORTED = 2,  /* valid problem that no kernel of this build handles */
    SSD_ERR_CUDA = 3,         /* a CUDA runtime call failed (launch, copy, attribute) */
    SSD_ERR_TIMEOUT = 4,      /* a device-side bounded wait gave up (see ssd_scan_get_status) */
    SSD_ERR_WORKSPACE = 5     /* workspace NULL or smaller than ssd_scan_workspace_bytes */
};

/* Kernel family.  SSD_PATH_AUTO picks: bf16 with headdim % 64 == 0 and dstate in {128, 256}
 * -> SSD_PATH_TC (tcgen05 tensor cores, TMA, TMEM); everything else -> SSD_PATH_CHUNKED
 * (float32 CUDA-core kernels that follow the chunk algorithm with the caller's chunk_size). */
enum { SSD_PATH_AUTO = -1, SSD_PATH_CHUNKED = 0, SSD_PATH_TC = 1 };

/* Which kernel family `path` (SSD_PATH_AUTO or explicit) resolves to for this problem, or a
 * negative SSD_ERR_* code if the problem is invalid or the explicit path cannot run it. */
int ssd_scan_resolve_path(const ssd_dims* dims, int chunk_size, int path);

/* Device workspace bytes ssd_scan_fwd needs for this problem and path (0 on invalid input).
 * The workspace holds a status word, per-chunk float32 states for the chunked path, and the
 * cross-block state hand-off slots of the tensor-core path; for d_state 128 also the segment
 * records of its state-only pass (long sequences over few heads: ranges of tiles shorter than
 * the chains), which balance that pass over the SMs.  Its contents need no initialisation;
 * calls sharing one workspace must be ordered on one stream. */
size_t ssd_scan_workspace_bytes(const ssd_dims* dims, int chunk_size, int path);

/* How many kernels one ssd_scan_fwd (or ssd_scan_fwd_gated) call enqueues for this problem on
 * the current device, or a negative SSD_ERR_* code.  Chunked path: 3.  Tensor-core path: 1,
 * or 2 for d_state 128 when the CTAs' ranges of 128-token tiles are no longer than the (batch,
 * head) chains and some range ends inside a chain: a state-only pass kernel then runs first
 * (long sequences over few heads).  Memsets of the status word and hand-off flags come on top. */
int ssd_scan_kernels_per_call(const ssd_dims* dims, int chunk_size, int path);

/*
 * ssd_scan_fwd -- y and final_state of the scan defined above, enqueued on `stream`.
 *
 * chunk_size: the chunk length Q of the SSD chunk algorithm, 1 <= Q <= 256.  The result does
 * not depend on Q beyond rounding (the chunk algorithm is exact); the chunked path cuts the
 * sequence at multiples of Q, the tensor-core path evaluates each Q-chunk in 128-token tiles.
 * A sequence length that is not a multiple of Q ends in a partial chunk (treated as padding
 * tokens with dt = 0; no y is written for them).
 *
 * Returns SSD_OK once all work is enqueued, or an SSD_ERR_* code (nothing enqueued).
 */
int ssd_scan_fwd(const ssd_dims* dims,
                 const void* x, const void* dt, const float* A,
                 const void* B, const void* C, const float* D,
                 const float* initial_state, int chunk_size,
                 void* y, float* final_state,
                 void* workspace, size_t workspace_bytes, void* stream);

/* ssd_scan_fwd with an explicit kernel family (SSD_PATH_*).  Returns SSD_ERR_UNSUPPORTED if
 * that family cannot run the problem. */
int ssd_scan_fwd_path(const ssd_dims* dims,
                      const void* x, const void* dt, const float* A,
                      const void* B, const void* C, const float* D,
                      const float* initial_state, int chunk_size,
                      void* y, float* final_state,
                      void* workspace, size_t workspace_bytes, void* stream, int path);

/*
 * Host-buffer variant: every tensor argument is a HOST pointer (page-locked memory makes the
 * copies asynchronous), and `device_arena` is a caller-owned device buffer of at least
 * ssd_scan_host_arena_bytes(dims, chunk_size) bytes (256-byte aligned).  The problem is cut
 * into up to 8 pieces -- groups of batch rows when there are 8 rows or more, else each row cut
 * into 8 / batch stretches of multiples of 256 tokens with the row's state carried on the
 * device -- and each piece's copies in, scan and copies out form a pipeline: the copies run on
 * two library-owned streams of the current device (created on first use), ordered against
 * `stream` with events, so piece p's inputs travel while piece p - 1 is scanned and earlier
 * pieces' outputs come back.  `stream` itself waits
 * for every copy: the host outputs are valid after the caller synchronises `stream`.  Calls
 * enqueue under a process-wide lock.  The status word (ssd_scan_get_status on the arena's
 * workspace part) covers the whole call.  Same errors as ssd_scan_fwd.
 */
size_t ssd_scan_host_arena_bytes(const ssd_dims* dims, int chunk_size);
int ssd_scan_fwd_host(const ssd_dims* dims,
                      const void* x, const void* dt, const float* A,
                      const void* B, const void* C, const float* D,
                      const float* initial_state, int chunk_size,
                      void* y, float* final_state,
                      void* device_arena, size_t arena_bytes, void* stream);

/*
 * No-allocation variant.  The pages have no counterpart: this entry point exists for callers
 * that cannot allocate device memory when they run the scan -- code that must not call
 * cudaMalloc (or any allocator) because a framework owns all device memory through its own
 * pool, because allocation is forbidden after start-up in the host process, or because a CUDA
 * graph is being captured.  The caller passes only inputs and outputs (device pointers, as for
 * ssd_scan_fwd); the scratch comes from a fixed SSD_NOALLOC_SCRATCH_BYTES buffer compiled into
 * the library's device image, which every GPU that loads the library holds until the process
 * exits.
 *
 *   - Runs the chunked kernel family (SSD_PATH_CHUNKED) for any dtype the ABI accepts.
 *   - Problems whose scratch (ssd_scan_workspace_bytes(dims, chunk_size, SSD_PATH_CHUNKED))
 *     exceeds SSD_NOALLOC_SCRATCH_BYTES are rejected with SSD_ERR_WORKSPACE before anything is
 *     enqueued.  Other errors as ssd_scan_fwd.
 *   - The scratch is the one of the CURRENT device: `stream` must belong to it (a stream of
 *     another device is rejected with SSD_ERR_INVALID).
 *   - The first call on each device looks up the buffer's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make that first call
 *     before any stream capture.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 *   - Every call shares the one buffer per device, and the buffer keeps the last call's
 *     contents (the status word is cleared at the start of each call).  Calls whose work
 *     overlaps on the GPU (different streams without ordering, or other host threads) race on
 *     the buffer; order them on one stream.
 *   - ssd_scan_get_status is not available for this variant (the caller holds no workspace);
 *     a device-side failure surfaces as a CUDA error on `stream`.
 */
#define SSD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int ssd_scan_fwd_noalloc(const ssd_dims* dims,
                         const void* x, const void* dt, const float* A,
                         const void* B, const void* C, const float* D,
                         const float* initial_state, int chunk_size,
                         void* y, float* final_state, void* stream);

/*
 * ssd_scan_fwd_varlen -- the scan over a packed batch of variable-length sequences: batch row
 * 0 of `dims` holds nseq sequences back to back, sequence i being tokens cu_seqlens[i] ..
 * cu_seqlens[i+1] - 1.  Each sequence starts from its own initial state (the state resets at
 * every sequence start: youngju.dev article, section "状態初期化とシーケンス境界") and
 * ends in its own final state; y is written for every token.
 *
 *   - dims.batch == 1, dims.seqlen = total tokens; cu_seqlens is a HOST array of nseq + 1
 *     non-decreasing offsets with cu_seqlens[0] = 0 and cu_seqlens[nseq] = dims.seqlen.
 *     Empty sequences are allowed (final state = initial state).
 *   - x, dt, B, C, y as for ssd_scan_fwd with batch 1; initial_state / final_state are
 *     [nseq, nheads, headdim, dstate] float32 (each nullable as for ssd_scan_fwd).
 *   - nheads * headdim and ngroups * dstate elements must each be a multiple of 16 bytes, so
 *     that every sequence's x, y, B and C slices start on a 16-byte boundary
 *     (else SSD_ERR_UNSUPPORTED).
 *   - workspace: at least ssd_scan_varlen_workspace_bytes.  `path` as for ssd_scan_fwd_path,
 *     or SSD_PATH_AUTO.
 *   - When every non-empty sequence takes the tensor-core path and there are at least two,
 *     the sequences run concurrently on up to four library-owned streams of the current device
 *     (longest first, each to the least loaded stream), each stream with its own slice of the
 *     workspace and a grid of a quarter of the SMs; `stream` waits for all of them (events).
 *     Otherwise one scan per non-empty sequence is enqueued on `stream`, in order, sharing the
 *     workspace.
 *   - The status word is cleared once and every scan reports into it, so ssd_scan_get_status
 *     covers all of them.  Returns as ssd_scan_fwd; every sequence is checked before anything
 *     is enqueued.
 */
size_t ssd_scan_varlen_workspace_bytes(const ssd_dims* dims, const int64_t* cu_seqlens,
                                       int64_t nseq, int chunk_size, int path);
int ssd_scan_fwd_varlen(const ssd_dims* dims, const int64_t* cu_seqlens, int64_t nseq,
                        const void* x, const void* dt, const float* A,
                        const void* B, const void* C, const float* D,
                        const float* initial_state, int chunk_size,
                        void* y, float* final_state,
                        void* workspace, size_t workspace_bytes, void* stream, int path);

/*
 * ssd_step_fwd -- one recurrent step per (batch row, head): the scan above for a single token,
 * for decoding, where tokens arrive one at a time and the state lives between calls.
 *
 *     state[b,h] <- exp(dt[b,h] * A[h]) * state[b,h] + dt[b,h] * x[b,h] B[b,g]^T
 *     y[b,h,p]    = sum_n C[b,g,n] * state[b,h][p][n] + D[h] * x[b,h,p]     (g = h / (H / G))
 *
 * i.e. ssd_scan_fwd with seqlen 1, initial_state = state_in and final_state = state_out (the
 * recurrent mode: waylandz.com chapter 32, section 32.2.4; the recurrence: youngju.dev article,
 * section "LTIからSelectionへの切り替え").
 *
 *   - dims.seqlen must be 1; the layouts are those above with L = 1: x [batch, 1, nheads,
 *     headdim], dt [batch, 1, nheads], B, C [batch, 1, ngroups, dstate] (dtype T), y [batch, 1,
 *     nheads, headdim] (T, written).  Any headdim and dstate.
 *   - state_in, state_out: [batch, nheads, headdim, dstate] float32, device memory.  state_in
 *     NULL means a zero state; state_out is required and is written completely.  state_out may
 *     equal state_in (update in place); otherwise the two must not overlap.
 *   - D may be NULL (no skip term).  Alignment as for ssd_scan_fwd (x, B, C, y 16 bytes; dt
 *     its element size; A, D and the states 4 bytes).
 *   - Needs no workspace and allocates nothing.  Enqueued on `stream`.
 *   - Returns SSD_OK once enqueued; SSD_ERR_INVALID for bad arguments (including seqlen != 1 or
 *     partially overlapping states), SSD_ERR_UNSUPPORTED if batch * nheads exceeds 2^31 - 1,
 *     SSD_ERR_CUDA if the launch fails.  Nothing is enqueued on an error.
 */
int ssd_step_fwd(const ssd_dims* dims,
                 const void* x, const void* dt, const float* A,
                 const void* B, const void* C, const float* D,
                 const float* state_in, float* state_out, void* y, void* stream);

/*
 * ssd_causal_conv1d_fwd -- the depthwise causal convolution and SiLU that produce the scan's
 * inputs in a Mamba block (youngju.dev "Mamba / selective SSM" article, the Mamba block listing:
 * a depthwise Conv1d of width d_conv with padding d_conv - 1, cut to the first L outputs, then
 * SiLU; Qiita "Mamba-2 / SSD" article, section 5.1: the causal-conv1d step before the scan).
 * Per batch row b, token t and channel c, with K = width:
 *
 *     out[b,t,c] = silu(bias[c] + sum_{k<K} weight[c,k] * x[b, t-(K-1)+k, c])
 *
 * where inputs before t = 0 come from state_in (zeros when NULL).  silu = 0 skips the SiLU.
 *
 *   - x, out:       [batch, seqlen, channels]  T (dtype)     device memory
 *   - weight:       [channels, width]          float32
 *   - bias:         [channels]                 float32, or NULL (no bias)
 *   - state_in:     [batch, width - 1, channels] T, or NULL: the width - 1 inputs before x
 *   - state_out:    [batch, width - 1, channels] T, or NULL (not written): the last width - 1
 *                   inputs of state_in ++ x, so the next call continues the sequence
 *   - 1 <= width <= 8, batch <= 65535.  Element alignment suffices.  16-byte aligned x, out
 *     and states with channels % (16 / sizeof(T)) == 0 take the streaming kernel (tiles of 64
 *     tokens through shared memory by TMA; seqlen < 2^31 - 2^16); other buffers the register
 *     kernel (seqlen <= 1048560 = 65535 blocks of 16 tokens, else SSD_ERR_UNSUPPORTED: split
 *     the sequence and carry the state).
 *   - No output may overlap an input, and state_out may not overlap out (SSD_ERR_INVALID).
 *   - Needs no workspace; enqueued on `stream`.  Returns SSD_OK, SSD_ERR_INVALID,
 *     SSD_ERR_UNSUPPORTED (sizes beyond the grid limits) or SSD_ERR_CUDA.  A bounded device
 *     wait of the streaming kernel that gives up is reported by ssd_block_get_status.
 */
int ssd_causal_conv1d_fwd(int64_t batch, int64_t seqlen, int64_t channels, int width,
                          int32_t dtype, const void* x, const float* weight, const float* bias,
                          const void* state_in, void* state_out, int silu, void* out,
                          void* stream);

/*
 * ssd_gated_rmsnorm_fwd -- the step after the scan, y = rmsnorm(y) * silu(z) (Qiita "Mamba-2 /
 * SSD" article, section 4.2, step 4), per row over groups of group_size features:
 *
 *     out[r,i] = y[r,i] / sqrt(mean_{j in group(i)} y[r,j]^2 + eps) * weight[i] * silu(z[r,i])
 *
 *   - y, z, out: [rows, dim] T (for the scan's y: rows = batch * seqlen, dim = nheads * headdim)
 *   - z NULL: no gate.  weight: [dim] float32, or NULL (ones).  eps >= 0 (the pages give no
 *     value; 1e-5 is the binding's default).  group_size divides dim (dim: one group per row).
 *   - dim / group_size <= 12288, rows <= 2^31 - 1 (else SSD_ERR_UNSUPPORTED).
 *   - out may equal y or z (a row is read completely before any of it is written); element
 *     alignment suffices.  16-byte aligned buffers with group_size % (16 / sizeof(T)) == 0 and
 *     rows of y (and z) up to 48 KB take the streaming kernel (whole rows through shared memory
 *     by bulk copies); others the register kernel.
 *   - Needs no workspace; enqueued on `stream`.  Returns SSD_OK, SSD_ERR_INVALID,
 *     SSD_ERR_UNSUPPORTED or SSD_ERR_CUDA.  A bounded device wait of the streaming kernel that
 *     gives up is reported by ssd_block_get_status.
 */
int ssd_gated_rmsnorm_fwd(int64_t rows, int64_t dim, int64_t group_size, int32_t dtype,
                          const void* y, const void* z, const float* weight, float eps,
                          void* out, void* stream);

/*
 * ssd_block_get_status -- the device-side status of the streaming conv1d and RMSNorm kernels
 * (which take no workspace): synchronises `stream`, then returns SSD_OK, or SSD_ERR_TIMEOUT if
 * a bounded wait of one of those kernels gave up (ssd_scan_set_wait_cycles sets the limit; the
 * kernel then stops early and its output is incomplete) since the last call, and clears it.
 * The word is per device and shared by all streams of the process.  SSD_ERR_CUDA if the
 * synchronisation or the read failed.
 */
int ssd_block_get_status(void* stream);

/*
 * ssd_scan_fwd_gated -- the scan followed by the gated RMSNorm of its output, the block's next
 * step (Qiita "Mamba-2 / SSD" article, section 4.2, step 4: y = rmsnorm(y) * silu(z)):
 *
 *     out[b,t,f] = y[b,t,f] / sqrt(mean_{f' in group(f)} y[b,t,f']^2 + eps) * w[f] * silu(z[b,t,f])
 *
 * with y the scan of ssd_scan_fwd, f = h * headdim + p the feature index of a token, and groups
 * of group_size consecutive features.
 *
 *   - z: [batch, seqlen, nheads, headdim] of the element type (16-byte aligned); out: the same
 *     (written; y itself is not).  norm_weight: [nheads * headdim] float32 (or NULL for ones);
 *     eps >= 0.  group_size divides nheads * headdim.  Everything else as ssd_scan_fwd.
 *   - When the problem runs on the tensor-core kernel for d_state 128 and group_size is 8, 16,
 *     32 or 64 (a group then lies inside one head's 64-feature slice), the norm is applied in
 *     the scan kernel's epilogue from the float32 y, and y never goes to memory (norm_weight
 *     must then be 16-byte aligned).  Otherwise the scan writes y into the workspace and the
 *     gated RMSNorm kernel (ssd_gated_rmsnorm_fwd) reads it.
 *   - workspace: at least ssd_scan_gated_workspace_bytes (0 on invalid input).  Errors and
 *     status word as ssd_scan_fwd.
 */
size_t ssd_scan_gated_workspace_bytes(const ssd_dims* dims, int chunk_size, int64_t group_size);
int ssd_scan_fwd_gated(const ssd_dims* dims,
                       const void* x, const void* dt, const float* A,
                       const void* B, const void* C, const float* D,
                       const float* initial_state, int chunk_size,
                       const void* z, const float* norm_weight, float eps, int64_t group_size,
                       void* out, float* final_state,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Synchronise `stream`, then read and clear the device status word of `workspace` (the first
 * 4 bytes).  Returns SSD_OK, SSD_ERR_TIMEOUT if a bounded device wait gave up in a call that
 * used this workspace, or SSD_ERR_CUDA if synchronisation or the read failed. */
int ssd_scan_get_status(void* workspace, void* stream);

/* Limit, in SM clock cycles, of every device-side wait of the tensor-core kernels (a barrier
 * between warp roles, or the hand-off of a running state between thread blocks) and of the
 * streaming conv1d / RMSNorm kernels (a copy into shared memory).  A wait that reaches it makes
 * the kernel stop, record SSD_ERR_TIMEOUT in the workspace status word (ssd_scan_get_status;
 * ssd_block_get_status for the conv1d and RMSNorm) and return; the context stays usable.  cycles <= 0 restores the
 * default, 2^32 cycles (about 2 s at the B300's maximum SM clock).  The setting is process-wide
 * and applies to launches enqueued after the call; a limit far below a wait's normal length
 * makes calls fail with SSD_ERR_TIMEOUT, which is what tests of the timeout path use it for.
 * Returns the previous limit. */
int64_t ssd_scan_set_wait_cycles(int64_t cycles);

/* Static description of a return code. */
const char* ssd_scan_strerror(int code);

/* Library version (major * 10000 + minor * 100 + patch). */
int ssd_scan_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SSD_SCAN_H_ */
