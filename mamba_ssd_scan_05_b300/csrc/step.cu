// step.cu -- ssd_step_fwd: one recurrent step of the scan per (batch row, head), for tokens
// that arrive one at a time (decoding).  It is the scan's recurrence with a single token:
//
//     h <- exp(dt A) h + dt x B^T          (h: headdim x dstate, float32, updated in HBM)
//     y  = C^T h + D x                     (y[p] = sum_n C[n] h[p][n] + D x[p])
//
// youngju.dev "Mamba / selective SSM" article, section "LTIからSelectionへの切り替え" (the
// recurrence, Abar = exp(Delta A), Bbar = Delta B); waylandz.com chapter 32, section 32.2.4 (the
// recurrent mode: constant work per generated token).
//
// The step reads and writes the whole float32 state once and touches little else, so it is
// bound by HBM bandwidth.  One CTA per (batch row, head): warp w handles state rows
// p = w, w + 8, ...; a lane holds 16-byte column vectors of a row, so a warp moves 512
// contiguous bytes per row per vector.  Each warp has kRows rows in flight before it uses any,
// and the state streams through with evict-first hints.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kWarps = 8;
constexpr int kRows = 4;     // state rows a warp loads before it uses any

struct StepParams {
    int64_t H, P, N, G;
    const void* x;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const float* s_in;
    float* s_out;
    void* y;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Four consecutive elements of T at an 8-byte (bf16) or 16-byte (float) aligned address.
template <typename T> __device__ __forceinline__ float4 load4(const T* p);
template <> __device__ __forceinline__ float4 load4<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <> __device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// The fast form: N = 128 * NV and 16-byte aligned state rows.  Lane l holds columns
// 128 v + 4 l .. 128 v + 4 l + 3 of every row (v < NV).
template <typename T, int NV>
__global__ void __launch_bounds__(kWarps * 32) step_kernel_vec(const StepParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / p.H, h = bh - b * p.H;
    const int64_t g = h / (p.H / p.G);
    const T* xr = static_cast<const T*>(p.x) + bh * p.P;
    const float dtv = to_f32(static_cast<const T*>(p.dt)[bh]);
    const float a = expf(dtv * p.A[h]);
    const float Dh = p.D ? p.D[h] : 0.f;
    const T* Bg = static_cast<const T*>(p.B) + (b * p.G + g) * p.N;
    const T* Cg = static_cast<const T*>(p.C) + (b * p.G + g) * p.N;
    float4 bv[NV], cv[NV];   // dt B and C at this lane's columns
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const float4 bb = load4<T>(Bg + v * 128 + 4 * lane);
        bv[v] = make_float4(dtv * bb.x, dtv * bb.y, dtv * bb.z, dtv * bb.w);
        cv[v] = load4<T>(Cg + v * 128 + 4 * lane);
    }
    const int64_t base = bh * p.P * p.N + 4 * lane;
    T* yr = static_cast<T*>(p.y) + bh * p.P;
    for (int p0 = warp; p0 < p.P; p0 += kWarps * kRows) {
        float4 s[kRows][NV];
        float xv[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const int r = p0 + i * kWarps;
            const bool in = r < p.P;
            xv[i] = in ? to_f32(xr[r]) : 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v)
                s[i][v] = (in && p.s_in)
                              ? __ldcs(reinterpret_cast<const float4*>(p.s_in + base + r * p.N +
                                                                       v * 128))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const int r = p0 + i * kWarps;
            float part = 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float4& q = s[i][v];
                q.x = fmaf(a, q.x, xv[i] * bv[v].x);
                q.y = fmaf(a, q.y, xv[i] * bv[v].y);
                q.z = fmaf(a, q.z, xv[i] * bv[v].z);
                q.w = fmaf(a, q.w, xv[i] * bv[v].w);
                part = fmaf(cv[v].x, q.x, part);
                part = fmaf(cv[v].y, q.y, part);
                part = fmaf(cv[v].z, q.z, part);
                part = fmaf(cv[v].w, q.w, part);
                if (r < p.P)
                    __stcs(reinterpret_cast<float4*>(p.s_out + base + r * p.N + v * 128), q);
            }
            part = warp_sum(part);
            if (lane == 0 && r < p.P) yr[r] = from_f32<T>(fmaf(Dh, xv[i], part));
        }
    }
}

// Any N and alignment: lane l handles columns l, l + 32, ... of a row.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) step_kernel_any(const StepParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / p.H, h = bh - b * p.H;
    const int64_t g = h / (p.H / p.G);
    const T* xr = static_cast<const T*>(p.x) + bh * p.P;
    const float dtv = to_f32(static_cast<const T*>(p.dt)[bh]);
    const float a = expf(dtv * p.A[h]);
    const float Dh = p.D ? p.D[h] : 0.f;
    const T* Bg = static_cast<const T*>(p.B) + (b * p.G + g) * p.N;
    const T* Cg = static_cast<const T*>(p.C) + (b * p.G + g) * p.N;
    T* yr = static_cast<T*>(p.y) + bh * p.P;
    for (int64_t r = warp; r < p.P; r += kWarps) {
        const float xd = dtv * to_f32(xr[r]);
        const int64_t row = (bh * p.P + r) * p.N;
        float part = 0.f;
        for (int64_t n = lane; n < p.N; n += 32) {
            const float s0 = p.s_in ? p.s_in[row + n] : 0.f;
            const float s1 = fmaf(a, s0, xd * to_f32(Bg[n]));
            p.s_out[row + n] = s1;
            part = fmaf(to_f32(Cg[n]), s1, part);
        }
        part = warp_sum(part);
        if (lane == 0) yr[r] = from_f32<T>(fmaf(Dh, to_f32(xr[r]), part));
    }
}

template <typename T>
int launch_t(const StepArgs& a, const StepParams& p) {
    const dim3 grid((unsigned)(a.batch * a.nheads)), block(kWarps * 32);
    const bool vec = (a.dstate == 128 || a.dstate == 256) &&
                     (reinterpret_cast<uintptr_t>(a.s_out) % 16 == 0) &&
                     (!a.s_in || reinterpret_cast<uintptr_t>(a.s_in) % 16 == 0);
    if (vec && a.dstate == 128)
        step_kernel_vec<T, 1><<<grid, block, 0, a.stream>>>(p);
    else if (vec)
        step_kernel_vec<T, 2><<<grid, block, 0, a.stream>>>(p);
    else
        step_kernel_any<T><<<grid, block, 0, a.stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

int step_launch(const StepArgs& a) {
    StepParams p;
    p.H = a.nheads; p.P = a.headdim; p.N = a.dstate; p.G = a.ngroups;
    p.x = a.x; p.dt = a.dt; p.A = a.A; p.B = a.B; p.C = a.C; p.D = a.D;
    p.s_in = a.s_in; p.s_out = a.s_out; p.y = a.y;
    return a.dtype == SSD_F32 ? launch_t<float>(a, p) : launch_t<__nv_bfloat16>(a, p);
}

}  // namespace ssd
