// block.cu -- the two steps around the scan in a Mamba-2 block, as HBM-bound CUDA kernels.
//
// ssd_causal_conv1d_fwd: the depthwise causal convolution (width K <= 8) of the input branch,
// then SiLU (youngju.dev "Mamba / selective SSM" article, the Mamba block listing: a depthwise
// Conv1d with padding K - 1 cut to the first L outputs, then F.silu):
//     out[b, t, c] = silu(bias[c] + sum_{k<K} w[c, k] x[b, t - (K-1) + k, c]),
// with the K - 1 inputs before t = 0 taken from a carried state (zeros by default); the last
// K - 1 inputs become the new state.
//
// ssd_gated_rmsnorm_fwd: the step after the scan, y = rmsnorm(y) * silu(z) (Qiita "Mamba-2 /
// SSD" article, section 4.2, step 4), per row over groups of group_size features:
//     out[r, i] = y[r, i] * rsqrt(mean_{j in group(i)} y[r, j]^2 + eps) * w[i] * silu(z[r, i]).
//
// Both read every input element once and write every output element once; the layouts are
// channel-last (the scan's own [batch, seqlen, heads * headdim]), so a thread moves 16-byte
// vectors of consecutive channels and a warp 512 contiguous bytes.
#include "block_math.cuh"
#include "common.cuh"

namespace ssd {
namespace {

// silu(v) = v / (1 + exp(-v)): the shared form of block_math.cuh (the streaming kernels of
// block_staged.cu compute the same bits)
__device__ __forceinline__ float silu_f(float v) { return bm::silu1(v); }

// VEC consecutive elements of T <-> float, at a 16-byte aligned address when VEC > 1.
template <typename T, int VEC> struct Vec;
// The raw bits of VEC elements (what a load brings in), converted when used.
template <typename T, int VEC> struct Raw {
    static constexpr int kWords = (int)(VEC * sizeof(T) + 3) / 4;
    uint32_t w[kWords];
    __device__ __forceinline__ void load(const T* p) {
        if constexpr (kWords == 4) {
            const uint4 q = *reinterpret_cast<const uint4*>(p);
            w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
        } else if constexpr (sizeof(T) == 4) {
            w[0] = __float_as_uint(*reinterpret_cast<const float*>(p));
        } else {
            w[0] = (uint32_t)(*reinterpret_cast<const unsigned short*>(p)) << 16;
        }
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < kWords; ++i) w[i] = 0u;
    }
    __device__ __forceinline__ void get(float (&v)[VEC]) const {
        if constexpr (sizeof(T) == 4) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[e] = __uint_as_float(w[e]);
        } else if constexpr (VEC == 1) {
            v[0] = __uint_as_float(w[0]);
        } else {
#pragma unroll
            for (int i = 0; i < VEC / 2; ++i) {
                v[2 * i] = __uint_as_float(w[i] << 16);
                v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        }
    }
};

template <> struct Vec<float, 1> {
    static __device__ __forceinline__ void load(const float* p, float (&v)[1]) { v[0] = *p; }
    static __device__ __forceinline__ void store(float* p, const float (&v)[1]) { *p = v[0]; }
};
template <> struct Vec<__nv_bfloat16, 1> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[1]) {
        v[0] = __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[1]) {
        *p = __float2bfloat16_rn(v[0]);
    }
};
template <> struct Vec<float, 4> {
    static __device__ __forceinline__ void load(const float* p, float (&v)[4]) {
        const float4 q = *reinterpret_cast<const float4*>(p);
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    }
    static __device__ __forceinline__ void store(float* p, const float (&v)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <> struct Vec<__nv_bfloat16, 8> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
        const uint4 q = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// ---- causal depthwise conv1d + SiLU ----------------------------------------------------------

constexpr int kConvThreads = 128;
constexpr int kConvTokens = 16;     // tokens per thread (a sliding window in registers)
constexpr int kConvAhead = 8;       // tokens whose inputs a thread loads before it uses any

struct ConvParams {
    int64_t L, C;
    const void* x;
    const float* w;       // [C, K]
    const float* bias;    // [C] or null
    const void* s_in;     // [b, K-1, C] or null
    void* s_out;          // [b, K-1, C] or null
    void* out;
    int silu;
};

// Thread: VEC consecutive channels, tokens t0 .. t0 + kConvTokens - 1 of one batch row.
template <typename T, int VEC, int K>
__global__ void __launch_bounds__(kConvThreads, 4) conv_kernel(const ConvParams p) {
    const int64_t c0 = ((int64_t)blockIdx.x * kConvThreads + threadIdx.x) * VEC;
    if (c0 >= p.C) return;
    const int64_t b = blockIdx.z;
    const int64_t t0 = (int64_t)blockIdx.y * kConvTokens;
    const T* x = static_cast<const T*>(p.x) + b * p.L * p.C + c0;
    const T* sin = p.s_in ? static_cast<const T*>(p.s_in) + b * (K - 1) * p.C + c0 : nullptr;
    T* out = static_cast<T*>(p.out) + b * p.L * p.C + c0;
    float w[K][VEC], bias[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        bias[e] = p.bias ? p.bias[c0 + e] : 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) w[k][e] = p.w[(c0 + e) * K + k];
    }
    // win[k] holds input t - (K-1) + k for the next output t (k < K - 1)
    float win[K > 1 ? K - 1 : 1][VEC];
#pragma unroll
    for (int k = 0; k < K - 1; ++k) {
        const int64_t t = t0 - (K - 1) + k;
        if (t >= 0) {
            Vec<T, VEC>::load(x + t * p.C, win[k]);
        } else if (sin) {
            Vec<T, VEC>::load(sin + (t + K - 1) * p.C, win[k]);   // state row K - 1 + t
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) win[k][e] = 0.f;
        }
    }
    const int64_t t_end = min(t0 + kConvTokens, p.L);
    for (int64_t tg = t0; tg < t_end; tg += kConvAhead) {
        // the next kConvAhead tokens' inputs are all in flight before the first is used
        Raw<T, VEC> ahead[kConvAhead];
#pragma unroll
        for (int g = 0; g < kConvAhead; ++g) {
            if (tg + g < t_end) ahead[g].load(x + (tg + g) * p.C);
            else ahead[g].zero();
        }
#pragma unroll
        for (int g = 0; g < kConvAhead; ++g) {
            const int64_t t = tg + g;
            if (t >= t_end) break;
            float cur[VEC], o[VEC];
            ahead[g].get(cur);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float a = fmaf(w[K - 1][e], cur[e], bias[e]);
#pragma unroll
                for (int k = 0; k < K - 1; ++k) a = fmaf(w[k][e], win[k][e], a);
                o[e] = p.silu ? silu_f(a) : a;
            }
            Vec<T, VEC>::store(out + t * p.C, o);
#pragma unroll
            for (int k = 0; k + 1 < K - 1; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) win[k][e] = win[k + 1][e];
            if (K > 1) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) win[K - 2][e] = cur[e];
            }
        }
    }
    // the last block of the row writes the new state: the last K - 1 inputs, which are in the
    // window once the row's final token has been processed
    if (p.s_out && t_end == p.L) {
        T* so = static_cast<T*>(p.s_out) + b * (K - 1) * p.C + c0;
#pragma unroll
        for (int k = 0; k < K - 1; ++k) Vec<T, VEC>::store(so + k * p.C, win[k]);
    }
}

template <typename T, int VEC>
int conv_launch_k(int K, dim3 grid, cudaStream_t st, const ConvParams& p) {
    switch (K) {
        case 1: conv_kernel<T, VEC, 1><<<grid, kConvThreads, 0, st>>>(p); break;
        case 2: conv_kernel<T, VEC, 2><<<grid, kConvThreads, 0, st>>>(p); break;
        case 3: conv_kernel<T, VEC, 3><<<grid, kConvThreads, 0, st>>>(p); break;
        case 4: conv_kernel<T, VEC, 4><<<grid, kConvThreads, 0, st>>>(p); break;
        case 5: conv_kernel<T, VEC, 5><<<grid, kConvThreads, 0, st>>>(p); break;
        case 6: conv_kernel<T, VEC, 6><<<grid, kConvThreads, 0, st>>>(p); break;
        case 7: conv_kernel<T, VEC, 7><<<grid, kConvThreads, 0, st>>>(p); break;
        case 8: conv_kernel<T, VEC, 8><<<grid, kConvThreads, 0, st>>>(p); break;
        default: return SSD_ERR_UNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

template <typename T, int VEC>
int conv_launch_t(const ConvArgs& a, const ConvParams& p) {
    // grid y counts token blocks (at most 65535), grid z batch rows (checked by the caller)
    if ((a.seqlen + kConvTokens - 1) / kConvTokens > 65535) return SSD_ERR_UNSUPPORTED;
    const int64_t threads_c = (a.channels + VEC - 1) / VEC;
    const dim3 grid((unsigned)((threads_c + kConvThreads - 1) / kConvThreads),
                    (unsigned)((a.seqlen + kConvTokens - 1) / kConvTokens), (unsigned)a.batch);
    return conv_launch_k<T, VEC>(a.width, grid, a.stream, p);
}

bool vec_ok(const void* p) { return !p || reinterpret_cast<uintptr_t>(p) % 16 == 0; }

// ---- gated RMSNorm ---------------------------------------------------------------------------

constexpr int kNormThreads = 128;
constexpr int kNormCache = 5;       // vectors of y and z a thread keeps in registers (raw)

struct NormParams {
    int64_t D, g;
    const void* y;
    const void* z;        // or null
    const float* w;       // or null
    float eps;
    void* out;
};

// One CTA per row.  Every lane of a warp runs the same iterations (the loop bounds are per
// warp; vectors past the row end contribute nothing).  The first kNormCache vectors of y and z
// of a thread are loaded up front and kept as raw words; later ones are loaded when needed.
// Pass 1: sums of squares per group (one warp sum and one shared atomic when the warp's 32
// consecutive vectors share a group); pass 2: scale, weight, gate, store.
template <typename T, int VEC>
__global__ void __launch_bounds__(kNormThreads) norm_kernel(const NormParams p) {
    extern __shared__ float gsum[];                   // [D / g]
    const int64_t row = blockIdx.x;
    const T* y = static_cast<const T*>(p.y) + row * p.D;
    const T* z = p.z ? static_cast<const T*>(p.z) + row * p.D : nullptr;
    T* out = static_cast<T*>(p.out) + row * p.D;
    const int64_t nv = p.D / VEC, ng = p.D / p.g;
    const int lane = threadIdx.x & 31;
    Raw<T, VEC> yc[kNormCache], zc[kNormCache];
#pragma unroll
    for (int ci = 0; ci < kNormCache; ++ci) {
        const int64_t i = threadIdx.x + (int64_t)ci * kNormThreads;
        if (i < nv) {
            yc[ci].load(y + i * VEC);
            if (z) zc[ci].load(z + i * VEC);
        }
    }
    for (int64_t i = threadIdx.x; i < ng; i += kNormThreads) gsum[i] = 0.f;
    __syncthreads();
    auto sumsq_warp = [&](int64_t i, const float (&v)[VEC], bool valid) {
        const int64_t i0 = i - lane;                          // the warp's first vector
        const int64_t i1 = min(i0 + 31, nv - 1);              // its last valid vector
        float ss = 0.f;
        if (valid) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) ss = fmaf(v[e], v[e], ss);
        }
        if (i0 * VEC / p.g == i1 * VEC / p.g) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) atomicAdd(&gsum[i0 * VEC / p.g], ss);
        } else if (valid) {
            atomicAdd(&gsum[i * VEC / p.g], ss);
        }
    };
#pragma unroll
    for (int ci = 0; ci < kNormCache; ++ci) {
        const int64_t i = threadIdx.x + (int64_t)ci * kNormThreads;
        if (i - lane < nv) {
            float v[VEC];
            yc[ci].get(v);
            sumsq_warp(i, v, i < nv);
        }
    }
    for (int64_t i = threadIdx.x + (int64_t)kNormCache * kNormThreads; i - lane < nv;
         i += kNormThreads) {
        float v[VEC];
        const bool valid = i < nv;
        if (valid) Vec<T, VEC>::load(y + i * VEC, v);
        sumsq_warp(i, v, valid);
    }
    __syncthreads();
    const float inv_g = 1.f / (float)p.g;
    // pass 2: y * rsqrt(mean square + eps) * w * silu(z)
    auto emit = [&](int64_t i, const float (&v)[VEC], const float (&zz)[VEC]) {
        float o[VEC], wv[VEC];
        const float r = rsqrtf(fmaf(gsum[i * VEC / p.g], inv_g, p.eps));
        if (p.w) {
            if constexpr (VEC % 4 == 0) {      // 16-byte weight loads (the vector path)
#pragma unroll
                for (int q = 0; q < VEC / 4; ++q) {
                    const float4 f = *reinterpret_cast<const float4*>(p.w + i * VEC + 4 * q);
                    wv[4 * q] = f.x; wv[4 * q + 1] = f.y; wv[4 * q + 2] = f.z; wv[4 * q + 3] = f.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) wv[e] = p.w[i * VEC + e];
            }
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            float a = v[e] * r;
            if (p.w) a *= wv[e];
            if (z) a *= silu_f(zz[e]);
            o[e] = a;
        }
        Vec<T, VEC>::store(out + i * VEC, o);
    };
#pragma unroll
    for (int ci = 0; ci < kNormCache; ++ci) {
        const int64_t i = threadIdx.x + (int64_t)ci * kNormThreads;
        if (i < nv) {
            float v[VEC], zz[VEC];
            yc[ci].get(v);
            if (z) zc[ci].get(zz);
            emit(i, v, zz);
        }
    }
    for (int64_t i = threadIdx.x + (int64_t)kNormCache * kNormThreads; i < nv; i += kNormThreads) {
        float v[VEC], zz[VEC];
        Vec<T, VEC>::load(y + i * VEC, v);
        if (z) Vec<T, VEC>::load(z + i * VEC, zz);
        emit(i, v, zz);
    }
}

template <typename T, int VEC>
int norm_launch_t(const NormArgs& a, const NormParams& p) {
    const size_t smem = sizeof(float) * (size_t)(a.dim / a.group_size);
    norm_kernel<T, VEC><<<(unsigned)a.rows, kNormThreads, smem, a.stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

int norm_launch(const NormArgs& a) {
    // the streaming kernel (block_staged.cu) for aligned rows that fit two ring stages
    const int st = norm_staged_launch(a);
    if (st != SSD_ERR_UNSUPPORTED) return st;
    NormParams p;
    p.D = a.dim; p.g = a.group_size; p.y = a.y; p.z = a.z; p.w = a.weight; p.eps = a.eps;
    p.out = a.out;
    const bool v = vec_ok(a.y) && vec_ok(a.z) && vec_ok(a.out) && vec_ok(a.weight);
    if (a.dtype == SSD_BF16)
        return (v && a.group_size % 8 == 0) ? norm_launch_t<__nv_bfloat16, 8>(a, p)
                                            : norm_launch_t<__nv_bfloat16, 1>(a, p);
    return (v && a.group_size % 4 == 0) ? norm_launch_t<float, 4>(a, p)
                                        : norm_launch_t<float, 1>(a, p);
}

int conv_launch(const ConvArgs& a) {
    // the streaming kernel (block_staged.cu) for 16-byte aligned rows of channels
    const int st = conv_staged_launch(a);
    if (st != SSD_ERR_UNSUPPORTED) return st;
    ConvParams p;
    p.L = a.seqlen; p.C = a.channels; p.x = a.x; p.w = a.weight; p.bias = a.bias;
    p.s_in = a.s_in; p.s_out = a.s_out; p.out = a.out; p.silu = a.silu;
    const bool v = vec_ok(a.x) && vec_ok(a.out) && vec_ok(a.s_in) && vec_ok(a.s_out);
    if (a.dtype == SSD_BF16)
        return (v && a.channels % 8 == 0) ? conv_launch_t<__nv_bfloat16, 8>(a, p)
                                          : conv_launch_t<__nv_bfloat16, 1>(a, p);
    return (v && a.channels % 4 == 0) ? conv_launch_t<float, 4>(a, p)
                                      : conv_launch_t<float, 1>(a, p);
}

}  // namespace ssd
