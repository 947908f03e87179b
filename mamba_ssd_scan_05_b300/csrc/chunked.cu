// chunked.cu -- the SSD chunk algorithm on CUDA cores, float32 arithmetic (any shape, fp32 or
// bf16 storage).  This is the path for float32 problems (whose 1e-4 accuracy bar rules out
// bf16/tf32 tensor-core operands) and for shapes the tensor-core kernel does not tile.
//
// It follows the chunk algorithm step by step (Qiita "Mamba-2 / SSD" article section 4.2:
// matmuls inside a chunk, a scan between chunks; youngju.dev Mamba article, section
// "SSDアルゴリズムとチャンク分割": cumulative sum of dt*A inside the chunk, decay mask
// exp(cum_i - cum_j) on the causal lower triangle, attention-like product), with the caller's
// chunk length Q:
//   kernel 1  chunk_state   per (b, h, chunk):  cum = cumsum(dt*A) inside the chunk,
//                            S_c = X_c^T diag(exp(cum_last - cum) * dt) B_c   (P x N, fp32)
//   kernel 2  state_pass    per (b, h):         h_c = exp(cum_last,c) h_{c-1} + S_c, storing
//                            the state ENTERING each chunk in place of S_c; final_state
//   kernel 3  chunk_output  per (b, h, chunk):  y = (L o C B^T o dt_j) X + diag(exp(cum)) C h_in^T
//                            + D x, with L_ij = exp(cum_i - cum_j) masked to i >= j before exp
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kQMax = 256;   // largest chunk this path stages in shared memory
constexpr int kPB = 32;      // headdim rows per block
constexpr int kTT = 32;      // tokens per staged sub-tile (kernel 1) / tile edge (kernel 3)
constexpr int kNMax = 256;   // largest d_state (8 accumulators of 32 lanes in kernel 1)

struct ChunkParams {
    int64_t batch, L, H, P, N, G;
    int Q, nc, npb;
    const void* x;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const float* h0;
    void* y;
    float* hT;
    float* clast;    // [b, H, nc]      cum at the chunk's last token
    float* states;   // [b, H, nc, P, N] chunk states, then the state entering each chunk
};

// Inclusive prefix sum over the block's 256 threads (thread order).
__device__ __forceinline__ float block_inclusive_scan(float v, float* warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float s = lane < kThreads / 32 ? warp_sums[lane] : 0.f;
#pragma unroll
        for (int o = 1; o < kThreads / 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += n;
        }
        if (lane < kThreads / 32) warp_sums[lane] = s;
    }
    __syncthreads();
    if (warp > 0) v += warp_sums[warp - 1];
    return v;
}

// cum[t] = sum_{k<=t} dt_k A_h inside the chunk (t < Q; tokens past the sequence end are
// padding with dt = 0), and dts[t] = dt_t.  Ends with a block barrier.
template <typename T>
__device__ __forceinline__ void chunk_cumsum(const ChunkParams& p, int64_t b, int64_t h, int c,
                                             float* cum, float* dts, float* warp_sums) {
    const int t = threadIdx.x;
    const int64_t tok = (int64_t)c * p.Q + t;
    float d = 0.f;
    if (t < p.Q && tok < p.L)
        d = to_f32<T>(static_cast<const T*>(p.dt)[(b * p.L + tok) * p.H + h]);
    const float s = block_inclusive_scan(d * p.A[h], warp_sums);
    if (t < p.Q) {
        cum[t] = s;
        dts[t] = d;
    }
    __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_state_kernel(ChunkParams p) {
    extern __shared__ float sm[];
    __shared__ float warp_sums[kThreads / 32];
    float* cum = sm;                    // [kQMax]
    float* w = cum + kQMax;             // [kQMax]
    float* xs = w + kQMax;              // [kTT][kPB]
    float* Bs = xs + kTT * kPB;         // [kTT][N]
    const int c = blockIdx.x;
    const int64_t h = blockIdx.y / p.npb;
    const int pb = blockIdx.y % p.npb;
    const int64_t b = blockIdx.z;
    const int64_t g = h / (p.H / p.G);
    const int tid = threadIdx.x;

    chunk_cumsum<T>(p, b, h, c, cum, w, warp_sums);     // w temporarily holds dt
    const float cl = cum[p.Q - 1];
    if (tid < p.Q) w[tid] = expf(cl - cum[tid]) * w[tid];   // exp(cum_last - cum_t) * dt_t
    if (pb == 0 && tid == 0) p.clast[(b * p.H + h) * p.nc + c] = cl;
    __syncthreads();

    const int pi = tid >> 5, ni = tid & 31;
    float acc[kPB / 8][kNMax / 32];
#pragma unroll
    for (int m = 0; m < kPB / 8; ++m)
#pragma unroll
        for (int k = 0; k < kNMax / 32; ++k) acc[m][k] = 0.f;

    const T* X = static_cast<const T*>(p.x);
    const T* Bg = static_cast<const T*>(p.B);
    const int p0 = pb * kPB;
    for (int s0 = 0; s0 < p.Q; s0 += kTT) {
        for (int e = tid; e < kTT * kPB; e += kThreads) {
            const int tt = e / kPB, pp = e % kPB;
            const int64_t tok = (int64_t)c * p.Q + s0 + tt;
            float v = 0.f;
            if (s0 + tt < p.Q && tok < p.L && p0 + pp < p.P)
                v = w[s0 + tt] * to_f32<T>(X[((b * p.L + tok) * p.H + h) * p.P + p0 + pp]);
            xs[e] = v;
        }
        for (int e = tid; e < kTT * p.N; e += kThreads) {
            const int tt = e / p.N, n = e % p.N;
            const int64_t tok = (int64_t)c * p.Q + s0 + tt;
            float v = 0.f;
            if (s0 + tt < p.Q && tok < p.L)
                v = to_f32<T>(Bg[((b * p.L + tok) * p.G + g) * p.N + n]);
            Bs[e] = v;
        }
        __syncthreads();
        for (int tt = 0; tt < kTT; ++tt) {
#pragma unroll
            for (int m = 0; m < kPB / 8; ++m) {
                const float xv = xs[tt * kPB + pi + 8 * m];
#pragma unroll
                for (int k = 0; k < kNMax / 32; ++k)
                    if (ni + 32 * k < p.N) acc[m][k] += xv * Bs[tt * p.N + ni + 32 * k];
            }
        }
        __syncthreads();
    }
    float* S = p.states + ((b * p.H + h) * p.nc + c) * p.P * p.N;
#pragma unroll
    for (int m = 0; m < kPB / 8; ++m) {
        const int pp = p0 + pi + 8 * m;
        if (pp >= p.P) continue;
#pragma unroll
        for (int k = 0; k < kNMax / 32; ++k) {
            const int n = ni + 32 * k;
            if (n < p.N) S[(int64_t)pp * p.N + n] = acc[m][k];
        }
    }
}

__global__ void __launch_bounds__(kThreads) state_pass_kernel(ChunkParams p) {
    const int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t h = blockIdx.y, b = blockIdx.z;
    const int64_t PN = p.P * p.N;
    if (e >= PN) return;
    const int64_t bh = b * p.H + h;
    float s = p.h0 ? p.h0[bh * PN + e] : 0.f;
    for (int c = 0; c < p.nc; ++c) {
        float* slot = p.states + (bh * p.nc + c) * PN + e;
        const float chunk_state = *slot;
        *slot = s;                                             // state entering chunk c
        s = expf(p.clast[bh * p.nc + c]) * s + chunk_state;    // h_c = exp(cum_last) h_{c-1} + S_c
    }
    if (p.hT) p.hT[bh * PN + e] = s;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_output_kernel(ChunkParams p) {
    extern __shared__ float sm[];
    __shared__ float warp_sums[kThreads / 32];
    const int N = (int)p.N, NP = N + 1;   // padded row stride
    float* cum = sm;                      // [kQMax]
    float* dts = cum + kQMax;             // [kQMax]
    float* Cs = dts + kQMax;              // [kTT][NP]
    float* Bs = Cs + kTT * NP;            // [kTT][NP]
    float* hs = Bs + kTT * NP;            // [kPB][NP]
    float* xs = hs + kPB * NP;            // [kTT][kPB]
    float* W = xs + kTT * kPB;            // [kTT][kTT + 1]
    const int c = blockIdx.x;
    const int64_t h = blockIdx.y / p.npb;
    const int pb = blockIdx.y % p.npb;
    const int64_t b = blockIdx.z;
    const int64_t g = h / (p.H / p.G);
    const int tid = threadIdx.x;
    const int p0 = pb * kPB;
    const int64_t tok0 = (int64_t)c * p.Q;
    const int64_t rem = p.L - tok0;
    const int len = rem < p.Q ? (int)rem : p.Q;

    chunk_cumsum<T>(p, b, h, c, cum, dts, warp_sums);
    const float* hin = p.states + ((b * p.H + h) * p.nc + c) * p.P * p.N;
    for (int e = tid; e < kPB * N; e += kThreads) {
        const int pp = e / N, n = e % N;
        hs[pp * NP + n] = (p0 + pp < p.P) ? hin[(int64_t)(p0 + pp) * N + n] : 0.f;
    }
    const T* X = static_cast<const T*>(p.x);
    const T* Bg = static_cast<const T*>(p.B);
    const T* Cg = static_cast<const T*>(p.C);
    T* Y = static_cast<T*>(p.y);
    const float Dh = p.D ? p.D[h] : 0.f;
    const int ii = tid >> 3, pc = tid & 7;

    for (int i0 = 0; i0 < len; i0 += kTT) {
        for (int e = tid; e < kTT * N; e += kThreads) {
            const int r = e / N, n = e % N;
            Cs[r * NP + n] = (i0 + r < len)
                ? to_f32<T>(Cg[((b * p.L + tok0 + i0 + r) * p.G + g) * p.N + n]) : 0.f;
        }
        __syncthreads();
        // off-diagonal term: exp(cum_i) * C_i . h_in[p]
        float acc[kPB / 8];
        const int i = i0 + ii;
        const float ei = (i < len) ? expf(cum[i]) : 0.f;
#pragma unroll
        for (int m = 0; m < kPB / 8; ++m) {
            const int pp = pc + 8 * m;
            float s = 0.f;
            for (int n = 0; n < N; ++n) s += Cs[ii * NP + n] * hs[pp * NP + n];
            acc[m] = ei * s;
        }
        // diagonal block: sum_{j<=i} exp(cum_i - cum_j) dt_j (C_i . B_j) x_j
        for (int j0 = 0; j0 <= i0; j0 += kTT) {
            for (int e = tid; e < kTT * N; e += kThreads) {
                const int r = e / N, n = e % N;
                Bs[r * NP + n] = (j0 + r < len)
                    ? to_f32<T>(Bg[((b * p.L + tok0 + j0 + r) * p.G + g) * p.N + n]) : 0.f;
            }
            for (int e = tid; e < kTT * kPB; e += kThreads) {
                const int r = e / kPB, pp = e % kPB;
                xs[e] = (j0 + r < len && p0 + pp < p.P)
                    ? to_f32<T>(X[((b * p.L + tok0 + j0 + r) * p.H + h) * p.P + p0 + pp]) : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int m = 0; m < kTT / 8; ++m) {
                const int jj = pc + 8 * m;
                const int j = j0 + jj;
                float v = 0.f;
                if (j <= i && i < len && j < len) {   // mask before exp
                    float s = 0.f;
                    for (int n = 0; n < N; ++n) s += Cs[ii * NP + n] * Bs[jj * NP + n];
                    v = expf(cum[i] - cum[j]) * dts[j] * s;
                }
                W[ii * (kTT + 1) + jj] = v;
            }
            __syncthreads();
#pragma unroll
            for (int m = 0; m < kPB / 8; ++m) {
                const int pp = pc + 8 * m;
                float s = 0.f;
#pragma unroll 8
                for (int jj = 0; jj < kTT; ++jj) s += W[ii * (kTT + 1) + jj] * xs[jj * kPB + pp];
                acc[m] += s;
            }
            __syncthreads();
        }
        if (i < len) {
#pragma unroll
            for (int m = 0; m < kPB / 8; ++m) {
                const int pp = p0 + pc + 8 * m;
                if (pp >= p.P) continue;
                const int64_t idx = ((b * p.L + tok0 + i) * p.H + h) * p.P + pp;
                Y[idx] = from_f32<T>(acc[m] + Dh * to_f32<T>(X[idx]));
            }
        }
        __syncthreads();
    }
}

size_t state_smem(int64_t N) { return sizeof(float) * (2 * kQMax + kTT * kPB + kTT * N); }
size_t output_smem(int64_t N) {
    return sizeof(float) * (2 * kQMax + 2 * kTT * (N + 1) + kPB * (N + 1) + kTT * kPB +
                            kTT * (kTT + 1));
}

template <typename T>
int launch_typed(const ChunkParams& p, cudaStream_t st) {
    const size_t s1 = state_smem(p.N), s3 = output_smem(p.N);
    if (cudaFuncSetAttribute(chunk_state_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)s1) != cudaSuccess ||
        cudaFuncSetAttribute(chunk_output_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)s3) != cudaSuccess)
        return SSD_ERR_CUDA;
    const dim3 g13((unsigned)p.nc, (unsigned)(p.H * p.npb), (unsigned)p.batch);
    chunk_state_kernel<T><<<g13, kThreads, s1, st>>>(p);
    const dim3 g2((unsigned)((p.P * p.N + kThreads - 1) / kThreads), (unsigned)p.H,
                  (unsigned)p.batch);
    state_pass_kernel<<<g2, kThreads, 0, st>>>(p);
    chunk_output_kernel<T><<<g13, kThreads, s3, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

bool chunked_supports(int64_t P, int64_t N, int Q) {
    return P >= 1 && N >= 1 && N <= kNMax && Q >= 1 && Q <= kQMax && P <= 4096;
}

size_t chunked_workspace_bytes(int64_t b, int64_t L, int64_t H, int64_t P, int64_t N, int Q) {
    const int64_t nc = (L + Q - 1) / Q;
    size_t bytes = kWsHeaderBytes;
    bytes += align_up(sizeof(float) * (size_t)(b * H * nc), 256);
    bytes += align_up(sizeof(float) * (size_t)(b * H * nc) * (size_t)(P * N), 256);
    return bytes;
}

int chunked_launch(const ScanArgs& a) {
    ChunkParams p;
    p.batch = a.batch; p.L = a.seqlen; p.H = a.nheads; p.P = a.headdim; p.N = a.dstate;
    p.G = a.ngroups; p.Q = a.chunk;
    p.nc = (int)((a.seqlen + a.chunk - 1) / a.chunk);
    p.npb = (int)((a.headdim + kPB - 1) / kPB);
    p.x = a.x; p.dt = a.dt; p.A = a.A; p.B = a.B; p.C = a.C; p.D = a.D; p.h0 = a.h0;
    p.y = a.y; p.hT = a.hT;
    uint8_t* base = a.ws + kWsHeaderBytes;
    p.clast = reinterpret_cast<float*>(base);
    base += align_up(sizeof(float) * (size_t)(a.batch * a.nheads * p.nc), 256);
    p.states = reinterpret_cast<float*>(base);
    if (p.nc > 0x7fffffff || p.H * p.npb > 65535 || p.batch > 65535) return SSD_ERR_UNSUPPORTED;
    if (a.dtype == SSD_F32) return launch_typed<float>(p, a.stream);
    return launch_typed<__nv_bfloat16>(p, a.stream);
}

}  // namespace ssd
