// common.cuh -- shared host/device definitions of libssd_scan (internal; not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ssd_scan.h"

namespace ssd {

// Workspace layout shared by all paths: the first 256 bytes hold the status word (int32 at
// offset 0) and reserved space; path-specific regions follow at 256-byte aligned offsets.
constexpr size_t kWsHeaderBytes = 256;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Arguments of one scan, after validation, as the kernels see them.
struct ScanArgs {
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups;
    int32_t dtype;
    int chunk;                 // Q
    const void* x;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;            // may be null
    const float* h0;           // may be null
    void* y;
    float* hT;                 // may be null
    uint8_t* ws;               // workspace base (256-byte aligned)
    size_t ws_bytes;
    cudaStream_t stream;
    // tensor-core path: at most this many CTAs (0: one per SM), and the status word to record
    // a device-side failure in (null: the workspace's own)
    int max_ctas = 0;
    uint8_t* status = nullptr;
    // the gated RMSNorm fused into the output (tc128_launch with gated = 1 only): y receives
    // rmsnorm(scan) * w * silu(z) over groups of `group` features
    int gated = 0;
    const void* z = nullptr;
    const float* norm_w = nullptr;
    float eps = 0.f;
    int group = 0;
};

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);   // round to nearest even
}

// Records an error code in the status word (first writer wins).
__device__ __forceinline__ void set_status(uint8_t* ws, int code) {
    atomicCAS(reinterpret_cast<int*>(ws), 0, code);
}

// Chunked path (chunked.cu).
size_t chunked_workspace_bytes(int64_t b, int64_t L, int64_t H, int64_t P, int64_t N, int Q);
bool chunked_supports(int64_t P, int64_t N, int Q);
int chunked_launch(const ScanArgs& a);

// Arguments of one recurrent step (ssd_step_fwd), after validation.
struct StepArgs {
    int64_t batch, nheads, headdim, dstate, ngroups;
    int32_t dtype;
    const void* x;             // [batch, nheads, headdim]
    const void* dt;            // [batch, nheads]
    const float* A;
    const void* B;             // [batch, ngroups, dstate]
    const void* C;
    const float* D;            // may be null
    const float* s_in;         // [batch, nheads, headdim, dstate]; null = zeros; may equal s_out
    float* s_out;
    void* y;                   // [batch, nheads, headdim]
    cudaStream_t stream;
};

// Recurrent step (step.cu).
int step_launch(const StepArgs& a);

// Causal depthwise conv1d + SiLU (block.cu), after validation.
struct ConvArgs {
    int64_t batch, seqlen, channels;
    int width;                 // 1..8
    int32_t dtype;
    const void* x;             // [batch, seqlen, channels]
    const float* weight;       // [channels, width]
    const float* bias;         // [channels] or null
    const void* s_in;          // [batch, width - 1, channels] or null (zeros)
    void* s_out;               // [batch, width - 1, channels] or null
    int silu;
    void* out;                 // [batch, seqlen, channels]
    cudaStream_t stream;
};
int conv_launch(const ConvArgs& a);
// The shared-memory streaming form (block_staged.cu); SSD_ERR_UNSUPPORTED where it does not
// apply (nothing launched).
int conv_staged_launch(const ConvArgs& a);

// Gated RMSNorm (block.cu), after validation.
struct NormArgs {
    int64_t rows, dim, group_size;
    int32_t dtype;
    const void* y;             // [rows, dim]
    const void* z;             // [rows, dim] or null
    const float* weight;       // [dim] or null
    float eps;
    void* out;                 // [rows, dim]
    cudaStream_t stream;
};
int norm_launch(const NormArgs& a);
int norm_staged_launch(const NormArgs& a);

// Tensor-core path (tc.cu; the d_state 128 kernel in tc128.cu).
// Cycles a single device-side wait of the tensor-core kernels may take (process-wide setting,
// ssd_scan_set_wait_cycles).
long long tc_wait_budget();
int tc128_launch(const ScanArgs& a);
// The d_state 128 grid on `nsm` SMs (capped at max_ctas when > 0) and its plan mode: 1 when
// ranges are no longer than a chain, so the state-only passes run first as a kernel of their own.
void tc128_grid(int64_t batch, int64_t L, int64_t H, int64_t P, int nsm, int max_ctas,
                int* n_ctas, int* pass1_mode);
// Kernels one ungated or gated d_state 128 call launches on the current device (1 or 2), or a
// negative SSD_ERR_* code.
int tc128_kernels_per_call(int64_t batch, int64_t L, int64_t H, int64_t P);
// Whether the d_state 128 kernel fuses the gated RMSNorm for this headdim and group size.
bool tc128_gated_supports(int64_t P, int group);
size_t tc_workspace_bytes(int64_t b, int64_t L, int64_t H, int64_t P, int64_t N, int Q);
// The tensor-core workspace of a launch capped at `ctas` CTAs (hand-off slots for those only).
size_t tc_workspace_bytes_ctas(int64_t N, int ctas);
bool tc_supports(int32_t dtype, int64_t P, int64_t N, int Q);
int tc_launch(const ScanArgs& a);

}  // namespace ssd
