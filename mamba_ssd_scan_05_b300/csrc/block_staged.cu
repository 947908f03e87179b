// block_staged.cu -- the causal conv1d and the gated RMSNorm (see block.cu for what they
// compute) as persistent kernels that stream through shared memory.
//
// Both steps move every byte once and do a few flops per element, so they are bound by HBM if
// each SM keeps enough bytes in flight and spends few instructions per element.  Here one
// thread per CTA keeps a ring of whole rows (norm) or tiles (conv) in flight with asynchronous
// bulk copies while the CTA works on the oldest one, and the arithmetic runs on pairs of
// values with the packed fp32x2 instructions (block_math.cuh).
//   norm: one row (y and, when gated, z) per ring stage, fetched with two contiguous
//         cp.async.bulk copies.  Thread t owns the 16-byte vectors t, t + NT, ... of every
//         row (NT threads, VPT vectors each, NT * VPT = the row), so its weights stay in
//         registers for the whole kernel; it moves its vectors from the stage to registers,
//         adds its squares to the group sums, and after the CTA's one barrier of the row (from
//         then on the stage is refilled) scales, weights, gates and stores them.
//   conv: a tile of 64 tokens x 256 bytes of channels, fetched with a 3-D TMA load whose box
//         starts width - 1 tokens early (rows before the sequence start arrive as zeros, the
//         causal padding); the outputs are staged in shared memory and written by a TMA store
//         (which clips the channel and token tails).  A CTA keeps one channel tile for all its
//         tiles, so its weights are loaded once.
// Every wait on a copy is bounded (the tensor-core kernels' wait budget); a wait that gives up
// makes the CTA stop after draining its copies and records SSD_ERR_TIMEOUT in a device word
// that ssd_block_get_status reads.  Shapes or pointers these kernels do not take go to the
// register kernels of block.cu.
#include "block_math.cuh"
#include "tc_common.cuh"

namespace ssd {

// SSD_OK, or SSD_ERR_TIMEOUT after a staged conv / norm kernel gave up a wait.
__device__ int g_block_status;

namespace {

using bm::ffma2;
using bm::fmul2;
using bm::silu1;
using bm::silu2;

constexpr int kStMaxStages = 8;

struct StCtl {                 // at the start of dynamic shared memory (128 bytes)
    uint64_t full[kStMaxStages];
    int abort;
};
constexpr uint32_t kStCtlBytes = 128;
static_assert(sizeof(StCtl) <= kStCtlBytes, "control block");

__device__ __forceinline__ void st_flag_abort(StCtl* ctl) {
    *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
    atomicExch(&g_block_status, SSD_ERR_TIMEOUT);
}

// Bounded wait of one thread for a ring stage.  False if it gave up (this thread's timeout,
// which raises the CTA's abort flag, or another thread's abort flag).  The CTA decides to stop
// with __syncthreads_or over these results, so that every thread leaves the loop together.
// A poll suspends the thread for at most hint_ns (wait_hint); budgets too short for the
// hardware's suspension granularity (spin) poll without suspending, so that no poll outlasts
// the budget.
__device__ __forceinline__ bool st_poll(uint64_t* bar, uint32_t parity, uint32_t hint_ns,
                                        bool spin) {
    return spin ? mbar_test_wait(bar, parity) : mbar_try_wait_ns(bar, parity, hint_ns);
}
__device__ __forceinline__ bool st_wait(StCtl* ctl, int s, uint32_t parity, long long budget,
                                        uint32_t hint_ns, bool spin) {
    if (__builtin_expect(st_poll(&ctl->full[s], parity, hint_ns, spin), 1)) return true;
    const long long t0 = clock64();
    while (!st_poll(&ctl->full[s], parity, hint_ns, spin)) {
        if (*reinterpret_cast<volatile int*>(&ctl->abort)) return false;
        if (clock64() - t0 > budget) {
            st_flag_abort(ctl);
            return false;
        }
    }
    return true;
}

// After an abort (one thread): wait, with the fixed drain limit, for every issued copy of ring
// items first .. issued - 1, so that none lands after the CTA has exited.
__device__ __noinline__ void st_drain(StCtl* ctl, int64_t first, int64_t issued, int stages) {
    for (int64_t k = first; k < issued; ++k) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&ctl->full[k % stages], (uint32_t)(k / stages) & 1u)) {
            if (clock64() - t0 > kDrainCycles) {
                atomicExch(&g_block_status, SSD_ERR_TIMEOUT);
                return;
            }
        }
    }
}

// 16 bytes of T as raw words, read as pairs of floats
template <typename T> struct V16;
template <> struct V16<__nv_bfloat16> {
    static constexpr int N = 8;       // elements
    static __device__ __forceinline__ float2 pair(const uint4& q, int i) {
        const uint32_t w = i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w;
        return make_float2(bf16lo_to_f32(w), bf16hi_to_f32(w));
    }
    static __device__ __forceinline__ uint4 pack(const float2 (&o)[4]) {
        return make_uint4(pack_bf16x2(o[0].x, o[0].y), pack_bf16x2(o[1].x, o[1].y),
                          pack_bf16x2(o[2].x, o[2].y), pack_bf16x2(o[3].x, o[3].y));
    }
};
template <> struct V16<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ float2 pair(const uint4& q, int i) {
        return i == 0 ? make_float2(__uint_as_float(q.x), __uint_as_float(q.y))
                      : make_float2(__uint_as_float(q.z), __uint_as_float(q.w));
    }
    static __device__ __forceinline__ uint4 pack(const float2 (&o)[2]) {
        return make_uint4(__float_as_uint(o[0].x), __float_as_uint(o[0].y),
                          __float_as_uint(o[1].x), __float_as_uint(o[1].y));
    }
};

// ---- gated RMSNorm -------------------------------------------------------------------------

struct NormStParams {
    int64_t rows, D, g;
    const void* y;
    const void* z;            // or null
    const float* w;           // or null
    float eps;
    void* out;
    uint32_t row_bytes;       // D * sizeof(T): a multiple of 16
    int stages;
    long long budget;         // wait limit, SM cycles
    uint32_t hint_ns;         // longest hardware suspension of one poll
    bool spin;                // poll without suspending (short budgets)
};

constexpr int kNormMaxThreads = 384;

// Shared memory: StCtl | stages x (y row | z row) | group sums [3][D / g] (row j accumulates
// into buffer j % 3; after row j's barrier, buffer (j + 2) % 3 -- last read by row j - 1 -- is
// cleared for row j + 2, whose additions come after the next barrier).
// CTA c takes rows c, c + grid, c + 2 grid, ...; blockDim.x = NT, a multiple of 32, with
// NT * VPT 16-byte vectors = a row.
template <typename T, bool kZ, int VPT>
__global__ void __launch_bounds__(kNormMaxThreads)
    norm_staged_kernel(const __grid_constant__ NormStParams p) {
    constexpr int VEC = V16<T>::N, NP = VEC / 2;     // elements, pairs per vector
    extern __shared__ __align__(128) uint8_t smem[];
    StCtl* ctl = reinterpret_cast<StCtl*>(smem);
    uint8_t* ring = smem + kStCtlBytes;
    const uint32_t stage_bytes = p.row_bytes * (kZ ? 2u : 1u);
    float* gsum = reinterpret_cast<float*>(ring + (size_t)p.stages * stage_bytes);
    const int NT = blockDim.x, tid = threadIdx.x, lane = tid & 31;
    const int64_t ng = p.D / p.g;
    const int64_t G = gridDim.x;
    const int64_t nmine = (p.rows - (int64_t)blockIdx.x + G - 1) / G;
    const int stages = p.stages;
    const uint32_t vg = (uint32_t)(p.g / VEC);   // vectors per group

    // this thread's vectors: group, whether the warp's 32 vectors share it, weights
    uint32_t gk[VPT];
    bool warp_one[VPT];
    float2 wv[VPT][NP];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const uint32_t i = (uint32_t)(tid + k * NT), i0 = i - lane;
        gk[k] = ng == 1 ? 0u : i / vg;
        warp_one[k] = ng == 1 || i0 / vg == (i0 + 31) / vg;
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            wv[k][q] = p.w ? __ldg(reinterpret_cast<const float2*>(p.w + (size_t)i * VEC) + q)
                           : make_float2(1.f, 1.f);
        }
    }

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&ctl->full[s], 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    for (int64_t i = tid; i < 3 * ng; i += NT) gsum[i] = 0.f;
    __syncthreads();

    // ring positions are counted incrementally (no 64-bit division in the loop)
    int64_t issued = 0;        // thread 0: ring items whose copies have been issued
    int is = 0;                // thread 0: the stage of the next issue
    auto issue = [&]() {
        const int64_t row = (int64_t)blockIdx.x + issued * G;
        uint8_t* dst = ring + (size_t)is * stage_bytes;
        mbar_arrive_expect_tx(&ctl->full[is], stage_bytes);
        bulk_load(dst, static_cast<const uint8_t*>(p.y) + row * p.row_bytes, p.row_bytes,
                  &ctl->full[is]);
        if constexpr (kZ)
            bulk_load(dst + p.row_bytes, static_cast<const uint8_t*>(p.z) + row * p.row_bytes,
                      p.row_bytes, &ctl->full[is]);
        ++issued;
        is = is + 1 == stages ? 0 : is + 1;
    };
    if (tid == 0)
        while (issued < min((int64_t)stages, nmine)) issue();

    const float inv_g = 1.f / (float)p.g;
    int s = 0, gb = 0;         // stage of row j, sums buffer j % 3
    uint32_t par = 0;          // phase parity of the stage's barrier for row j
    int64_t j = 0;
    for (; j < nmine; ++j) {
        const uint4* ys = reinterpret_cast<const uint4*>(ring + (size_t)s * stage_bytes);
        const uint4* zs = reinterpret_cast<const uint4*>(ring + (size_t)s * stage_bytes +
                                                         p.row_bytes);
        float* gs = gsum + gb * ng;
        const bool ok = st_wait(ctl, s, par, p.budget, p.hint_ns, p.spin);
        uint4 yv[VPT], zv[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            yv[k] = ys[tid + k * NT];
            if constexpr (kZ) zv[k] = zs[tid + k * NT];
        }
        // sums of squares: one warp sum and one shared atomic per group a warp's vectors share
        float ssum = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float2 v = V16<T>::pair(yv[k], q);
                acc = ffma2(v, v, acc);
            }
            float ss = acc.x + acc.y;
            if (ng == 1) {
                ssum += ss;
            } else if (warp_one[k]) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                if (lane == 0) atomicAdd(&gs[gk[k]], ss);
            } else {
                atomicAdd(&gs[gk[k]], ss);
            }
        }
        if (ng == 1) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
            if (lane == 0) atomicAdd(&gs[0], ssum);
        }
        if (__syncthreads_or(!ok)) break;   // sums complete; stop together if a wait gave up
        // the stage is in registers: refill it; clear the sums of row j + 2
        if (tid == 0 && issued < nmine) issue();
        float* gn = gsum + (gb == 0 ? 2 : gb - 1) * ng;
        for (int64_t i = tid; i < ng; i += NT) gn[i] = 0.f;
        // y * rsqrt(mean square + eps) * w * silu(z)
        const int64_t row = (int64_t)blockIdx.x + j * G;
        uint4* orow = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + row * p.row_bytes);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const float r = rsqrtf(fmaf(gs[gk[k]], inv_g, p.eps));
            float2 o[NP];
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                o[q] = fmul2(fmul2(V16<T>::pair(yv[k], q), make_float2(r, r)), wv[k][q]);
                if constexpr (kZ) o[q] = fmul2(o[q], silu2(V16<T>::pair(zv[k], q)));
            }
            orow[tid + k * NT] = V16<T>::pack(o);
        }
        if (++s == stages) {
            s = 0;
            par ^= 1u;
        }
        gb = gb == 2 ? 0 : gb + 1;
    }
    if (j < nmine && tid == 0) st_drain(ctl, j, issued, stages);
}

// ---- causal depthwise conv1d + SiLU --------------------------------------------------------

constexpr int kCvThreads = 256;
constexpr int kCvTok = 64;            // tokens per tile
constexpr int kCvRowBytes = 256;      // bytes of channels per tile row
constexpr int kCvWords = kCvRowBytes / 4;
constexpr int kCvStages = 4;
constexpr int kCvGroups = kCvThreads / kCvWords;   // token groups per tile (4)
constexpr int kCvGroupTok = kCvTok / kCvGroups;    // tokens per thread (16)
static_assert(kCvGroups * kCvWords == kCvThreads && kCvGroupTok * kCvGroups == kCvTok, "tiling");

struct ConvStParams {
    int64_t L, C;
    int64_t nct, ntt, rows;   // channel tiles; token tiles per batch row; batch * ntt
    const float* w;           // [C, K]
    const float* bias;        // [C] or null
    const void* s_in;         // [b, K-1, C] or null
    void* s_out;              // [b, K-1, C] or null
    void* out;                // [b, L, C]
    long long budget;         // wait limit, SM cycles
    uint32_t hint_ns;         // longest hardware suspension of one poll
    bool spin;                // poll without suspending (short budgets)
};

template <int K>
constexpr uint32_t conv_in_bytes() { return (uint32_t)(kCvTok + K - 1) * kCvRowBytes; }
template <int K>
constexpr uint32_t conv_smem_bytes() {
    return kStCtlBytes + kCvStages * conv_in_bytes<K>() + 2u * kCvTok * kCvRowBytes;
}

// A 4-byte word of the tile holds PER channels: a pair of bf16 (computed as a float2 with the
// packed instructions) or one fp32.
template <typename T> struct Word;
template <> struct Word<__nv_bfloat16> {
    static constexpr int PER = 2;
    using V = float2;
    static __device__ __forceinline__ V get(uint32_t u) {
        return make_float2(bf16lo_to_f32(u), bf16hi_to_f32(u));
    }
    static __device__ __forceinline__ uint32_t put(V v) { return pack_bf16x2(v.x, v.y); }
    static __device__ __forceinline__ V fma(V a, V b, V c) { return ffma2(a, b, c); }
    static __device__ __forceinline__ V silu(V v) { return silu2(v); }
    static __device__ __forceinline__ V load(const float* p, int64_t c, int stride) {
        return make_float2(__ldg(p + c * stride), __ldg(p + (c + 1) * stride));
    }
    static __device__ __forceinline__ V zero() { return make_float2(0.f, 0.f); }
};
template <> struct Word<float> {
    static constexpr int PER = 1;
    using V = float;
    static __device__ __forceinline__ V get(uint32_t u) { return __uint_as_float(u); }
    static __device__ __forceinline__ uint32_t put(V v) { return __float_as_uint(v); }
    static __device__ __forceinline__ V fma(V a, V b, V c) { return fmaf(a, b, c); }
    static __device__ __forceinline__ V silu(V v) { return silu1(v); }
    static __device__ __forceinline__ V load(const float* p, int64_t c, int stride) {
        return __ldg(p + c * stride);
    }
    static __device__ __forceinline__ V zero() { return 0.f; }
};

// grid = nct * m CTAs.  CTA c: channel tile c % nct, token-tile rows q = c / nct, q + m, ...
// of the batch * ntt (batch row, token tile) pairs.  Thread: word column tid % 64 of the tile,
// tokens 16 (tid / 64) .. + 15.  Input stage row r holds token t0 - (K-1) + r; the outputs go
// to one of two shared buffers that a TMA store writes out (clipping the tails).
template <typename T, int K, bool kSilu>
__global__ void __launch_bounds__(kCvThreads) conv_staged_kernel(
    const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmo,
    const __grid_constant__ ConvStParams p) {
    using W = Word<T>;
    using V = typename W::V;
    constexpr int PER = W::PER;
    constexpr int CPT = kCvRowBytes / (int)sizeof(T);      // channels per tile
    constexpr uint32_t kIn = conv_in_bytes<K>();
    extern __shared__ __align__(128) uint8_t smem[];
    StCtl* ctl = reinterpret_cast<StCtl*>(smem);
    uint8_t* ring = smem + kStCtlBytes;
    uint8_t* obuf = ring + kCvStages * kIn;
    const int tid = threadIdx.x, wc = tid % kCvWords, tg = tid / kCvWords;
    // tile bookkeeping in 32 bits (rows, grid and token tiles < 2^31)
    const int nct = (int)p.nct, ntt = (int)p.ntt, m = (int)gridDim.x / nct;
    const int ct = (int)blockIdx.x % nct, q = (int)blockIdx.x / nct;
    const int nmine = q < (int)p.rows ? ((int)p.rows - q + m - 1) / m : 0;
    const int64_t c = (int64_t)ct * CPT + wc * PER;        // this thread's first channel
    const bool cin = c < p.C;
    const int r0 = tg * kCvGroupTok;                       // stage row of token t0 + r0 - (K-1)

    if (tid == 0) {
        prefetch_tmap(&tmx);
        prefetch_tmap(&tmo);
        for (int s = 0; s < kCvStages; ++s) mbar_init(&ctl->full[s], 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // (batch row, token tile) of ring item j: q + j m, advanced incrementally (m < 2^31)
    struct Pos {
        int b, tt;
        __device__ __forceinline__ void next(int m_, int ntt_) {
            tt += m_;
            while (tt >= ntt_) {
                tt -= ntt_;
                ++b;
            }
        }
    };
    int issued = 0;            // thread 0: ring items whose copies have been issued
    int is = 0;                // thread 0: the stage of the next issue
    Pos ip{q / ntt, q % ntt};  // thread 0: the position of the next issue
    auto issue = [&]() {
        mbar_arrive_expect_tx(&ctl->full[is], kIn);
        tma_load_3d(ring + (size_t)is * kIn, &tmx, &ctl->full[is], ct * CPT,
                    ip.tt * kCvTok - (K - 1), ip.b);
        ++issued;
        is = is + 1 == kCvStages ? 0 : is + 1;
        ip.next(m, ntt);
    };
    if (tid == 0)
        while (issued < min(kCvStages, nmine)) issue();

    // the channel tile's weights and bias (the first channel's where past the end)
    V w[K], bias;
    {
        const int64_t ce = cin ? c : 0;
#pragma unroll
        for (int k = 0; k < K; ++k) w[k] = W::load(p.w + k, ce, K);
        bias = p.bias ? W::load(p.bias, ce, 1) : W::zero();
    }

    bool failed = false;       // this thread's wait gave up (kept until the CTA stops)
    int s = 0;                 // stage of tile j
    uint32_t par = 0;          // phase parity of its barrier
    Pos pos{q / ntt, q % ntt};
    int j = 0;
    for (; j < nmine; ++j) {
        uint32_t* ob = reinterpret_cast<uint32_t*>(obuf + (size_t)(j & 1) * kCvTok * kCvRowBytes);
        if (tid == 0 && j >= 2) bulk_wait_read<1>();   // tile j-2's store has read this buffer
        // tile j-1 is done with its stage; stop together if a wait of tile j-1 gave up
        if (__syncthreads_or(failed)) break;
        // into the stage tile j-1 freed (tiles below j + stages fit in the ring)
        if (tid == 0 && issued < nmine && issued < j + kCvStages) issue();
        const int t0 = pos.tt * kCvTok, b = pos.b;
        failed = !st_wait(ctl, s, par, p.budget, p.hint_ns, p.spin);
        const uint32_t* in = reinterpret_cast<const uint32_t*>(ring + (size_t)s * kIn);
        V win[K > 1 ? K - 1 : 1];
#pragma unroll
        for (int k = 0; k < K - 1; ++k) win[k] = W::get(in[(r0 + k) * kCvWords + wc]);
        if (K > 1 && t0 + r0 == 0 && p.s_in) {   // the window before the sequence start: state
#pragma unroll
            for (int k = 0; k < K - 1; ++k) {
                const uint32_t u = cin ? *reinterpret_cast<const uint32_t*>(
                                             static_cast<const T*>(p.s_in) +
                                             ((int64_t)b * (K - 1) + k) * p.C + c)
                                       : 0u;
                win[k] = W::get(u);
            }
        }
#pragma unroll
        for (int i = 0; i < kCvGroupTok; ++i) {
            const V cur = W::get(in[(r0 + K - 1 + i) * kCvWords + wc]);
            V a = W::fma(w[K - 1], cur, bias);
#pragma unroll
            for (int k = 0; k < K - 1; ++k) a = W::fma(w[k], win[k], a);
            if constexpr (kSilu) a = W::silu(a);
            ob[(r0 + i) * kCvWords + wc] = W::put(a);
#pragma unroll
            for (int k = 0; k + 1 < K - 1; ++k) win[k] = win[k + 1];
            if constexpr (K > 1) win[K - 2] = cur;
        }
        // the batch row's last token tile writes the new state: inputs L-(K-1) .. L-1
        if (p.s_out && tg == 0 && cin && pos.tt == ntt - 1) {
#pragma unroll
            for (int k = 0; k < K - 1; ++k) {
                const int64_t t = p.L - (K - 1) + k;
                uint32_t u;
                if (t >= 0) u = in[(t - t0 + K - 1) * kCvWords + wc];
                else if (p.s_in)
                    u = *reinterpret_cast<const uint32_t*>(
                        static_cast<const T*>(p.s_in) + ((int64_t)b * (K - 1) + t + K - 1) * p.C + c);
                else u = 0u;
                *reinterpret_cast<uint32_t*>(static_cast<T*>(p.s_out) +
                                             ((int64_t)b * (K - 1) + k) * p.C + c) = u;
            }
        }
        fence_proxy_async_smem();   // this thread's output words, before the TMA store reads them
        __syncthreads();
        if (tid == 0) {
            tma_store_3d(&tmo, ob, ct * CPT, t0, b);
            bulk_commit();
        }
        if (++s == kCvStages) {
            s = 0;
            par ^= 1u;
        }
        pos.next(m, ntt);
    }
    // a wait that gave up in the last tile ends the loop without the break
    const bool any_failed = __syncthreads_or(failed);
    if (tid == 0) {
        bulk_wait_all();
        if (any_failed) st_drain(ctl, j > 0 ? j - 1 : 0, issued, kCvStages);
    }
}

// ---- host side -----------------------------------------------------------------------------

constexpr size_t kStMaxSmem = 200u << 10;
constexpr long long kSpinBudget = 1 << 16;   // budgets up to this many cycles poll without suspending

// budget / 4 nanoseconds (at most 1 ms, at least 1): below the budget at any SM clock >= 1 GHz
uint32_t wait_hint(long long budget) {
    return (uint32_t)std::max<long long>(1, std::min<long long>(budget / 4, 1000000));
}

// CTAs of the kernel per SM with `threads` threads and `smem` bytes of dynamic shared memory
// (0: it does not fit; -1: a CUDA call failed).
template <typename K_>
int occupancy(K_ kernel, int threads, size_t smem) {
    if (smem > kStMaxSmem) return 0;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
        return -1;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem) != cudaSuccess)
        return -1;
    return occ;
}

template <typename T, bool kZ, int VPT>
int norm_staged_v(const NormArgs& a, int threads) {
    NormStParams p;
    p.rows = a.rows; p.D = a.dim; p.g = a.group_size; p.y = a.y; p.z = a.z; p.w = a.weight;
    p.eps = a.eps; p.out = a.out;
    p.row_bytes = (uint32_t)(a.dim * (int64_t)sizeof(T));
    const size_t stage = (size_t)p.row_bytes * (kZ ? 2 : 1);
    // up to 64 KB of rows in flight per CTA (two or more CTAs per SM), at least two stages
    p.stages = (int)std::min<size_t>(kStMaxStages, std::max<size_t>(2, (64u << 10) / stage));
    p.budget = tc_wait_budget();
    p.hint_ns = wait_hint(p.budget);
    p.spin = p.budget <= kSpinBudget;
    const size_t smem =
        kStCtlBytes + p.stages * stage + 3 * sizeof(float) * (size_t)(a.dim / a.group_size);
    auto kernel = norm_staged_kernel<T, kZ, VPT>;
    const int occ = occupancy(kernel, threads, smem), sms = sm_count();
    if (occ < 0 || sms < 1) return SSD_ERR_CUDA;
    if (occ == 0) return SSD_ERR_UNSUPPORTED;
    const int64_t grid = std::min<int64_t>(a.rows, (int64_t)occ * sms);
    kernel<<<(unsigned)grid, threads, smem, a.stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

template <typename T, bool kZ>
int norm_staged_t(const NormArgs& a) {
    // a row of nv 16-byte vectors over NT = nv / VPT threads: the smallest VPT in {1, 2, 4, 8}
    // that gives at most 384 threads, NT a multiple of 32
    const int64_t nv = a.dim * (int64_t)sizeof(T) / 16;
    for (int vpt : {1, 2, 4, 8}) {
        if (nv % vpt != 0) continue;
        const int64_t nt = nv / vpt;
        if (nt > kNormMaxThreads) continue;
        if (nt % 32 != 0) return SSD_ERR_UNSUPPORTED;
        switch (vpt) {
            case 1: return norm_staged_v<T, kZ, 1>(a, (int)nt);
            case 2: return norm_staged_v<T, kZ, 2>(a, (int)nt);
            case 4: return norm_staged_v<T, kZ, 4>(a, (int)nt);
            default: return norm_staged_v<T, kZ, 8>(a, (int)nt);
        }
    }
    return SSD_ERR_UNSUPPORTED;
}

// 3-D map over [b][L][C] (C innermost) of T with a (CPT, rows, 1) box, no swizzle, zero fill.
template <typename T>
bool make_conv_map(CUtensorMap* m, const void* base, int64_t C, int64_t L, int64_t B, int rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)L, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)C * sizeof(T), (cuuint64_t)(C * L) * sizeof(T)};
    const cuuint32_t box[3] = {(cuuint32_t)(kCvRowBytes / sizeof(T)), (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <typename T, int K, bool kSilu>
int conv_staged_k(const ConvArgs& a) {
    ConvStParams p;
    p.L = a.seqlen; p.C = a.channels;
    p.nct = (a.channels * (int64_t)sizeof(T) + kCvRowBytes - 1) / kCvRowBytes;
    p.ntt = (a.seqlen + kCvTok - 1) / kCvTok;
    p.rows = p.ntt * a.batch;
    p.w = a.weight; p.bias = a.bias; p.s_in = a.s_in; p.s_out = a.s_out; p.out = a.out;
    p.budget = tc_wait_budget();
    p.hint_ns = wait_hint(p.budget);
    p.spin = p.budget <= kSpinBudget;
    if (p.rows == 0) return SSD_OK;
    CUtensorMap tmx, tmo;
    if (!make_conv_map<T>(&tmx, a.x, a.channels, a.seqlen, a.batch, kCvTok + K - 1) ||
        !make_conv_map<T>(&tmo, a.out, a.channels, a.seqlen, a.batch, kCvTok))
        return SSD_ERR_UNSUPPORTED;
    constexpr size_t smem = conv_smem_bytes<K>();
    auto kernel = conv_staged_kernel<T, K, kSilu>;
    const int occ = occupancy(kernel, kCvThreads, smem), sms = sm_count();
    if (occ < 0 || sms < 1) return SSD_ERR_CUDA;
    if (occ == 0) return SSD_ERR_UNSUPPORTED;
    // m CTAs per channel tile: fill the resident slots, but no more CTAs than token tiles
    const int64_t slots = (int64_t)occ * sms;
    const int64_t m = std::max<int64_t>(1, std::min<int64_t>(slots / p.nct, p.rows));
    const int64_t grid = p.nct * m;
    if (grid > 0x7fffffffll) return SSD_ERR_UNSUPPORTED;
    kernel<<<(unsigned)grid, kCvThreads, smem, a.stream>>>(tmx, tmo, p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

template <typename T, bool kSilu>
int conv_staged_s(const ConvArgs& a) {
    switch (a.width) {
        case 1: return conv_staged_k<T, 1, kSilu>(a);
        case 2: return conv_staged_k<T, 2, kSilu>(a);
        case 3: return conv_staged_k<T, 3, kSilu>(a);
        case 4: return conv_staged_k<T, 4, kSilu>(a);
        case 5: return conv_staged_k<T, 5, kSilu>(a);
        case 6: return conv_staged_k<T, 6, kSilu>(a);
        case 7: return conv_staged_k<T, 7, kSilu>(a);
        case 8: return conv_staged_k<T, 8, kSilu>(a);
        default: return SSD_ERR_UNSUPPORTED;
    }
}

template <typename T>
int conv_staged_t(const ConvArgs& a) {
    return a.silu ? conv_staged_s<T, true>(a) : conv_staged_s<T, false>(a);
}

bool al16(const void* p) { return !p || reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace

int norm_staged_launch(const NormArgs& a) {
    const int64_t vec = a.dtype == SSD_BF16 ? 8 : 4;
    if (!al16(a.y) || !al16(a.z) || !al16(a.out) || !al16(a.weight) || a.group_size % vec != 0 ||
        a.rows > 0x7fffffffll)
        return SSD_ERR_UNSUPPORTED;
    if (a.dtype == SSD_BF16)
        return a.z ? norm_staged_t<__nv_bfloat16, true>(a) : norm_staged_t<__nv_bfloat16, false>(a);
    return a.z ? norm_staged_t<float, true>(a) : norm_staged_t<float, false>(a);
}

int conv_staged_launch(const ConvArgs& a) {
    const size_t eb = a.dtype == SSD_BF16 ? 2 : 4;
    // tensor-map rules: 16-byte aligned base, row pitch a multiple of 16 bytes, coordinates in
    // int32; the state words are 4-byte accesses
    if (!al16(a.x) || !al16(a.out) || (a.channels * (int64_t)eb) % 16 != 0 ||
        a.seqlen > 0x7fff0000ll || a.channels > 0x7fff0000ll || !al16(a.s_in) || !al16(a.s_out))
        return SSD_ERR_UNSUPPORTED;
    const int64_t rows = (a.seqlen + kCvTok - 1) / kCvTok * a.batch;
    if (rows > 0x7fffffffll) return SSD_ERR_UNSUPPORTED;
    return a.dtype == SSD_BF16 ? conv_staged_t<__nv_bfloat16>(a) : conv_staged_t<float>(a);
}

}  // namespace ssd

extern "C" int ssd_block_get_status(void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess ||
        cudaMemcpyFromSymbol(&v, ssd::g_block_status, sizeof(int)) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (v != SSD_OK) {
        const int zero = SSD_OK;
        if (cudaMemcpyToSymbol(ssd::g_block_status, &zero, sizeof(int)) != cudaSuccess)
            return SSD_ERR_CUDA;
    }
    return v;
}
