// tc.cu -- the tensor-core path: one fused, warp-specialised sm_103a kernel per scan.
//
// What it computes is the SSD chunk algorithm (Qiita "Mamba-2 / SSD" article section 4.2;
// youngju.dev Mamba article, sections "State Space Dualityの発見" and "SSDアルゴリズムとチャンク分割"),
// evaluated in 128-token tiles that walk the sequence in order with the running state on chip:
//
//   S1  cum_i = sum_{k<=i} dt_k A  (inside the tile); L_ij = exp(cum_i - cum_j) for i >= j
//   S2  G = C B^T                         tcgen05.mma  M=128 N=128 K=d_state   (TMEM)
//       P = L o G o dt_j  -> bf16 (smem)  CUDA cores (mask first, then exp)
//       Y_diag = P X                      tcgen05.mma  M=128 N=64  K=128
//       S^T = B^T (diag(exp(cum_last - cum) dt) X)   M=d_state N=64 K=128
//   S3  H = exp(cum_last) H + S^T         CUDA cores, H (= h^T, fp32) lives in TMEM
//   S4  Y_off = C h_prev^T                tcgen05.mma  M=128 N=64  K=d_state
//       y = Y_diag + exp(cum) Y_off + D x -> bf16, 16-byte stores
//
// For a chunk length Q that is a multiple of 128 the tile is a sub-block of the chunk; the
// block of L o (C B^T) below the tile's diagonal block is applied through its low-rank factor
// (the state at the tile boundary), which the semiseparable structure of M makes exact.
// The result does not depend on Q (chunk-size invariance), so every Q that is a multiple of
// 64 runs the same tiles.
//
// One CTA owns one unit = (batch row b, head h, 64-wide slice of headdim).  Warp roles
// (320 threads):
//   warp 0      TMA producer: x / B / C tiles of 128 tokens into a ring of smem stages
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer
//   warps 2-5   "A" warpgroup: cumsum of dt*A, scaled copy of x for the state GEMM, P = L o G
//   warps 6-9   "B" warpgroup: state recurrence in TMEM, bf16 h^T for the next tile, y epilogue
// Every wait is bounded (clock64 budget); a timeout sets SSD_ERR_TIMEOUT in the workspace
// status word, makes every role stop, drains in-flight copies and frees TMEM before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace ptx;

constexpr int kTile = 128;          // tokens per tile (MMA M)
constexpr int kPS = 64;             // headdim columns per unit (MMA N of Y, Y_off, S)
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTileBytes = kTile * 128;   // a 128-row x 128-byte swizzled tile (16 KB)
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpB = 6;   // warps 2-5: the A warpgroup
constexpr float kLog2e = 1.4426950408889634f;

template <int NS>
struct Cfg {
    static constexpr int kNReg = NS / 64;             // 64-column regions of a B / C tile
    static constexpr int kStages = NS == 128 ? 2 : 1;
    static constexpr int kGBuf = NS == 128 ? 2 : 1;
    static constexpr int kMB = NS / 128;               // 128-row blocks of the state
    // shared memory (byte offsets from a 1024-aligned base)
    static constexpr uint32_t kOffX = 0;
    static constexpr uint32_t kOffB = kOffX + kStages * kTileBytes;
    static constexpr uint32_t kOffC = kOffB + kStages * kNReg * kTileBytes;
    static constexpr uint32_t kOffXt = kOffC + kStages * kNReg * kTileBytes;
    static constexpr uint32_t kOffP = kOffXt + kTileBytes;
    static constexpr uint32_t kOffHt = kOffP + 2 * kTileBytes;
    static constexpr uint32_t kOffSmall = kOffHt + NS * 128;
    // TMEM columns
    static constexpr uint32_t kColG = 0;
    static constexpr uint32_t kColY = kGBuf * 128;
    static constexpr uint32_t kColYoff = kColY + kPS;
    static constexpr uint32_t kColS = kColYoff + kPS;
    static constexpr uint32_t kColH = kColS + kMB * kPS;
    static_assert(kColH + kMB * kPS <= kTmemCols, "TMEM budget");
    static constexpr uint32_t kStageTx = kTileBytes * (1 + 2 * kNReg);
};

struct Small {
    uint64_t full[2], empty[2], g_full[2], g_empty[2];
    uint64_t xt_full, xt_empty, p_full, p_empty, s_full, s_empty, h_full, h_empty;
    uint64_t y_full, y_empty, a_sync, b_sync, mma_done;
    uint32_t tmem_base;
    int abort_flag;
    float a_cum2[kTile];     // cum * log2(e), "A" warpgroup
    float a_dt[kTile];
    float a_wsum[4];
    float b_wsum[4];
    float b_clast2;          // cum * log2(e) at the tile's last row, "B" warpgroup
};

struct TcParams {
    int64_t batch, L, H, P, N, G;
    int n_ps;           // P / 64
    int n_tiles;        // ceil(L / 128)
    const __nv_bfloat16* dt;
    const float* A;
    const float* D;
    const float* h0;
    __nv_bfloat16* y;
    float* hT;
    uint8_t* ws;
    long long budget;   // clock64 cycles a single wait may take
};

__device__ __forceinline__ void flag_abort(Small& sm, uint8_t* ws) {
    *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
    set_status(ws, SSD_ERR_TIMEOUT);
}

// Bounded wait for the completion of the phase with `parity`.  False on timeout or abort.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Small& sm,
                                         const TcParams& p) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) return false;
        if (clock64() - t0 > p.budget) {
            flag_abort(sm, p.ws);
            return false;
        }
    }
}

// wait_bar for the 32 lanes of a warp, with one verdict for the whole warp, so the warp stays
// converged for the .sync.aligned TMEM instructions that follow.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, Small& sm,
                                          const TcParams& p) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, sm, p));
}

// Intra-warpgroup barrier on an mbarrier of count 128 (bounded, unlike bar.sync).
__device__ __forceinline__ bool wg_sync(uint64_t* bar, uint32_t& phase, Small& sm,
                                        const TcParams& p) {
    mbar_arrive(bar);
    const bool ok = wait_warp(bar, phase, sm, p);
    phase ^= 1u;
    return ok;
}

// Inclusive prefix sum of `v` over the warpgroup's 128 rows (row = 32 * quarter + lane).
__device__ __forceinline__ bool wg_scan(float& v, int quarter, int lane, float* wsum,
                                        uint64_t* bar, uint32_t& phase, Small& sm,
                                        const TcParams& p) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (!wg_sync(bar, phase, sm, p)) return false;        // previous readers of wsum are done
    if (lane == 31) wsum[quarter] = v;
    if (!wg_sync(bar, phase, sm, p)) return false;
    float off = 0.f;
    for (int q = 0; q < quarter; ++q) off += wsum[q];
    v += off;
    return true;
}

template <int NS>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmC, const TcParams p) {
    using K = Cfg<NS>;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms and TMA destinations need 1024-byte aligned shared addresses
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Small& sm = *reinterpret_cast<Small*>(smem + K::kOffSmall);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x;
    const int ps = unit % p.n_ps;
    const int64_t bh = unit / p.n_ps;
    const int64_t h = bh % p.H, b = bh / p.H;
    const int64_t g = h / (p.H / p.G);
    const int n_tiles = p.n_tiles;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1 + 128);
            mbar_init(&sm.g_full[i], 1);
            mbar_init(&sm.g_empty[i], 128);
        }
        mbar_init(&sm.xt_full, 128);
        mbar_init(&sm.xt_empty, 1);
        mbar_init(&sm.p_full, 128);
        mbar_init(&sm.p_empty, 1);
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_empty, 128);
        mbar_init(&sm.h_full, 128);
        mbar_init(&sm.h_empty, 1);
        mbar_init(&sm.y_full, 1);
        mbar_init(&sm.y_empty, 128);
        mbar_init(&sm.a_sync, 128);
        mbar_init(&sm.b_sync, 128);
        mbar_init(&sm.mma_done, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpTma && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == kWarpTma) {
        // ---------------------------------------------------------------- TMA producer ----
        if (lane == 0) {
            int issued = 0;
            for (int k = 0; k < n_tiles; ++k) {
                const int s = k % K::kStages;
                const uint32_t use = k / K::kStages;
                if (!wait_bar(&sm.empty[s], (use & 1u) ^ 1u, sm, p)) break;
                mbar_arrive_expect_tx(&sm.full[s], K::kStageTx);
                const int t0 = k * kTile;
                tma_load_4d(smem + K::kOffX + s * kTileBytes, &tmX, &sm.full[s], ps * kPS, (int)h,
                            t0, (int)b);
                for (int r = 0; r < K::kNReg; ++r) {
                    tma_load_4d(smem + K::kOffB + (s * K::kNReg + r) * kTileBytes, &tmB,
                                &sm.full[s], r * 64, (int)g, t0, (int)b);
                    tma_load_4d(smem + K::kOffC + (s * K::kNReg + r) * kTileBytes, &tmC,
                                &sm.full[s], r * 64, (int)g, t0, (int)b);
                }
                ++issued;
            }
            if (sm.abort_flag) {
                // drain: every issued load must land before the CTA's smem goes away
                const long long t0 = clock64();
                for (int k = issued - K::kStages; k < issued; ++k) {
                    if (k < 0) continue;
                    const int s = k % K::kStages;
                    const uint32_t use = k / K::kStages;
                    while (!mbar_try_wait(&sm.full[s], use & 1u) && clock64() - t0 < p.budget) {
                    }
                }
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------------- MMA issuer ------
        if (lane == 0) {
            constexpr uint32_t idG = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idS = idesc_bf16(128, kPS, 1, 1);
            constexpr uint32_t idYoff = idesc_bf16(128, kPS, 0, 1);
            constexpr uint32_t idYd = idesc_bf16(128, kPS, 0, 1);
            bool ok = true;
            auto issue_G = [&](int k) -> bool {
                const int s = k % K::kStages;
                const int gb = k % K::kGBuf;
                if (!wait_bar(&sm.full[s], (uint32_t)(k / K::kStages) & 1u, sm, p)) return false;
                if (!wait_bar(&sm.g_empty[gb], ((uint32_t)(k / K::kGBuf) & 1u) ^ 1u, sm, p))
                    return false;
                tc_fence_after();
                const uint32_t cbase = sbase + K::kOffC + s * K::kNReg * kTileBytes;
                const uint32_t bbase = sbase + K::kOffB + s * K::kNReg * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < NS / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
                    mma_f16(tmem + K::kColG + gb * 128, smem_desc_sw128(cbase + off, 16, 1024),
                            smem_desc_sw128(bbase + off, 16, 1024), idG, kk > 0);
                }
                mma_commit(&sm.g_full[gb]);
                return true;
            };
            if (n_tiles > 0) ok = issue_G(0);
            for (int k = 0; k < n_tiles && ok; ++k) {
                const int s = k % K::kStages;
                const uint32_t par = (uint32_t)k & 1u;
                // chunk state S^T = B^T (w o X)
                if (!wait_bar(&sm.xt_full, par, sm, p) || !wait_bar(&sm.s_empty, par ^ 1u, sm, p)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    const uint32_t bbase = sbase + K::kOffB + s * K::kNReg * kTileBytes;
                    const uint32_t xt = sbase + K::kOffXt;
#pragma unroll
                    for (int mb = 0; mb < K::kMB; ++mb)
#pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_f16(tmem + K::kColS + mb * kPS,
                                    smem_desc_sw128(bbase + 2 * mb * kTileBytes + kk * 2048,
                                                    kTileBytes, 1024),
                                    smem_desc_sw128(xt + kk * 2048, 1024, 1024), idS, kk > 0);
                }
                mma_commit(&sm.s_full);
                mma_commit(&sm.xt_empty);
                // off-diagonal Y_off = C h_prev^T
                if (!wait_bar(&sm.h_full, par, sm, p) || !wait_bar(&sm.y_empty, par ^ 1u, sm, p)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    const uint32_t cbase = sbase + K::kOffC + s * K::kNReg * kTileBytes;
                    const uint32_t ht = sbase + K::kOffHt;
#pragma unroll
                    for (int kk = 0; kk < NS / 16; ++kk)
                        mma_f16(tmem + K::kColYoff,
                                smem_desc_sw128(cbase + (kk >> 2) * kTileBytes + (kk & 3) * 32, 16,
                                                1024),
                                smem_desc_sw128(ht + kk * 2048, 1024, 1024), idYoff, kk > 0);
                }
                mma_commit(&sm.h_empty);
                // next tile's C B^T while the A warpgroup builds this tile's P (with a single
                // smem stage the next tile can only land after this tile releases it, below)
                if (K::kStages > 1 && k + 1 < n_tiles && !issue_G(k + 1)) {
                    ok = false;
                    break;
                }
                // Y_diag = P X
                if (!wait_bar(&sm.p_full, par, sm, p)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    const uint32_t pb = sbase + K::kOffP;
                    const uint32_t xb = sbase + K::kOffX + s * kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        mma_f16(tmem + K::kColY,
                                smem_desc_sw128(pb + (kk >> 2) * kTileBytes + (kk & 3) * 32, 16,
                                                1024),
                                smem_desc_sw128(xb + kk * 2048, 1024, 1024), idYd, kk > 0);
                }
                mma_commit(&sm.p_empty);
                mma_commit(&sm.y_full);
                mma_commit(&sm.empty[s]);
                if (K::kStages == 1 && k + 1 < n_tiles && !issue_G(k + 1)) {
                    ok = false;
                    break;
                }
            }
            // every MMA issued above has completed once this barrier's phase 0 completes
            mma_commit(&sm.mma_done);
            const long long t0 = clock64();
            while (!mbar_try_wait(&sm.mma_done, 0) && clock64() - t0 < p.budget) {
            }
        }
    } else if (warp < kWarpB) {
        // ---------------------------------------------------------------- "A" warpgroup ---
        const int q = warp & 3;                 // TMEM lane quarter
        const int r = q * 32 + lane;            // tile row
        const float A2 = p.A[h] * kLog2e;
        uint32_t sync_phase = 0;
        for (int k = 0; k < n_tiles; ++k) {
            const int s = k % K::kStages;
            const int gb = k % K::kGBuf;
            const uint32_t par = (uint32_t)k & 1u;
            const int64_t t = (int64_t)k * kTile + r;
            const float dtv = t < p.L ? __bfloat162float(p.dt[(b * p.L + t) * p.H + h]) : 0.f;
            float c2 = dtv * A2;                // log2-domain cumsum
            if (!wg_scan(c2, q, lane, sm.a_wsum, &sm.a_sync, sync_phase, sm, p)) break;
            sm.a_cum2[r] = c2;
            sm.a_dt[r] = dtv;
            if (!wg_sync(&sm.a_sync, sync_phase, sm, p)) break;
            const float clast2 = sm.a_cum2[kTile - 1];

            // w o X for the chunk-state GEMM: row r scaled by exp(cum_last - cum_r) dt_r
            if (!wait_warp(&sm.full[s], (uint32_t)(k / K::kStages) & 1u, sm, p)) break;
            if (!wait_warp(&sm.xt_empty, par ^ 1u, sm, p)) break;
            {
                const float wr = ex2(clast2 - c2) * dtv;
                const uint32_t xrow = sbase + K::kOffX + s * kTileBytes;
                const uint32_t xtrow = sbase + K::kOffXt;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t off = sw128_off(r, c);
                    const uint4 v = ld_shared_v4(xrow + off);
                    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[e] = pack_bf16x2(wr * bf16lo_to_f32(in[e]), wr * bf16hi_to_f32(in[e]));
                    st_shared_v4(xtrow + off, o[0], o[1], o[2], o[3]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&sm.xt_full);

            // P = L o G o dt_j (bf16, K-major swizzled), L masked before exp
            if (!wait_warp(&sm.p_empty, par ^ 1u, sm, p)) break;
            if (!wait_warp(&sm.g_full[gb], (uint32_t)(k / K::kGBuf) & 1u, sm, p)) break;
            tc_fence_after();
            {
                const uint32_t prow = sbase + K::kOffP;
#pragma unroll
                for (int jb = 0; jb < 4; ++jb) {
                    const uint32_t atom = prow + (jb >> 1) * kTileBytes;
                    if (jb > q) {   // strictly above the diagonal for the whole warp
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            st_shared_v4(atom + sw128_off(r, (jb & 1) * 4 + c), 0, 0, 0, 0);
                        continue;
                    }
                    float gv[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + K::kColG + gb * 128 + jb * 32,
                              gv);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float pv[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int jj = c * 8 + e * 2 + u;
                                const int j = jb * 32 + jj;
                                pv[u] = (j <= r) ? ex2(c2 - sm.a_cum2[j]) * sm.a_dt[j] * gv[jj]
                                                 : 0.f;
                            }
                            o[e] = pack_bf16x2(pv[0], pv[1]);
                        }
                        st_shared_v4(atom + sw128_off(r, (jb & 1) * 4 + c), o[0], o[1], o[2],
                                     o[3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.g_empty[gb]);
            fence_proxy_async_smem();
            mbar_arrive(&sm.p_full);
        }
    } else {
        // ---------------------------------------------------------------- "B" warpgroup ---
        const int q = warp & 3;
        const int r = q * 32 + lane;             // tile row, and state row inside a 128-block
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const float A2 = p.A[h] * kLog2e;
        const float Dh = p.D ? p.D[h] : 0.f;
        const int64_t hbase = (bh * p.P + (int64_t)ps * kPS) * p.N;   // [p][n] of this slice
        uint32_t sync_phase = 0;
        bool ok = true;

        // initial state: H (TMEM, fp32) and h^T (smem, bf16) for the first tile's Y_off
#pragma unroll
        for (int mb = 0; mb < K::kMB; ++mb) {
            const int n = mb * 128 + r;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = p.h0 ? p.h0[hbase + (int64_t)(half * 32 + i) * p.N + n] : 0.f;
                tmem_st32(tmem + lane_base + K::kColH + mb * kPS + half * 32, v);
                const uint32_t hrow = sbase + K::kOffHt;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st_shared_v4(hrow + sw128_off(n, half * 4 + c),
                                 pack_bf16x2(v[c * 8 + 0], v[c * 8 + 1]),
                                 pack_bf16x2(v[c * 8 + 2], v[c * 8 + 3]),
                                 pack_bf16x2(v[c * 8 + 4], v[c * 8 + 5]),
                                 pack_bf16x2(v[c * 8 + 6], v[c * 8 + 7]));
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(&sm.h_full);

        for (int k = 0; k < n_tiles && ok; ++k) {
            const int s = k % K::kStages;
            const uint32_t par = (uint32_t)k & 1u;
            const int64_t t = (int64_t)k * kTile + r;
            const float dtv = t < p.L ? __bfloat162float(p.dt[(b * p.L + t) * p.H + h]) : 0.f;
            float c2 = dtv * A2;
            if (!wg_scan(c2, q, lane, sm.b_wsum, &sm.b_sync, sync_phase, sm, p)) break;
            // cum at the tile's last row lives in the last warp quarter's last lane
            if (lane == 31 && q == 3) sm.b_clast2 = c2;
            if (!wg_sync(&sm.b_sync, sync_phase, sm, p)) break;
            const float clast2 = sm.b_clast2;
            const float e_r = ex2(c2);          // exp(cum_r)
            const float decay = ex2(clast2);    // exp(cum_last)

            // S3: H = exp(cum_last) H + S^T
            if (!wait_warp(&sm.s_full, par, sm, p)) break;
            tc_fence_after();
#pragma unroll
            for (int mb = 0; mb < K::kMB; ++mb)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float sv[32], hv[32];
                    tmem_ld32(tmem + lane_base + K::kColS + mb * kPS + half * 32, sv);
                    tmem_ld32(tmem + lane_base + K::kColH + mb * kPS + half * 32, hv);
#pragma unroll
                    for (int i = 0; i < 32; ++i) hv[i] = fmaf(decay, hv[i], sv[i]);
                    tmem_st32(tmem + lane_base + K::kColH + mb * kPS + half * 32, hv);
                }
            tc_fence_before();
            mbar_arrive(&sm.s_empty);
            // h^T (bf16) for the next tile's Y_off, once this tile's Y_off has read the old one
            if (!wait_warp(&sm.h_empty, par, sm, p)) break;
#pragma unroll
            for (int mb = 0; mb < K::kMB; ++mb) {
                const int n = mb * 128 + r;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float hv[32];
                    tmem_ld32(tmem + lane_base + K::kColH + mb * kPS + half * 32, hv);
                    const uint32_t hrow = sbase + K::kOffHt;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        st_shared_v4(hrow + sw128_off(n, half * 4 + c),
                                     pack_bf16x2(hv[c * 8 + 0], hv[c * 8 + 1]),
                                     pack_bf16x2(hv[c * 8 + 2], hv[c * 8 + 3]),
                                     pack_bf16x2(hv[c * 8 + 4], hv[c * 8 + 5]),
                                     pack_bf16x2(hv[c * 8 + 6], hv[c * 8 + 7]));
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&sm.h_full);

            // S4: y = Y_diag + exp(cum) Y_off + D x
            if (!wait_warp(&sm.y_full, par, sm, p)) break;
            if (!wait_warp(&sm.full[s], (uint32_t)(k / K::kStages) & 1u, sm, p)) break;
            tc_fence_after();
            {
                const uint32_t xrow = sbase + K::kOffX + s * kTileBytes;
                __nv_bfloat16* yrow = p.y + ((b * p.L + t) * p.H + h) * p.P + ps * kPS;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float yd[32], yo[32];
                    tmem_ld32(tmem + lane_base + K::kColY + half * 32, yd);
                    tmem_ld32(tmem + lane_base + K::kColYoff + half * 32, yo);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 xv = ld_shared_v4(xrow + sw128_off(r, half * 4 + c));
                        const uint32_t xin[4] = {xv.x, xv.y, xv.z, xv.w};
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i0 = c * 8 + e * 2;
                            const float v0 =
                                fmaf(Dh, bf16lo_to_f32(xin[e]), fmaf(e_r, yo[i0], yd[i0]));
                            const float v1 =
                                fmaf(Dh, bf16hi_to_f32(xin[e]), fmaf(e_r, yo[i0 + 1], yd[i0 + 1]));
                            o[e] = pack_bf16x2(v0, v1);
                        }
                        if (t < p.L)
                            *reinterpret_cast<uint4*>(yrow + half * 32 + c * 8) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.y_empty);
            mbar_arrive(&sm.empty[s]);
        }
        // final state h_{L-1} (fp32)
        if (p.hT && !sm.abort_flag) {
#pragma unroll
            for (int mb = 0; mb < K::kMB; ++mb) {
                const int n = mb * 128 + r;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float hv[32];
                    tmem_ld32(tmem + lane_base + K::kColH + mb * kPS + half * 32, hv);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        p.hT[hbase + (int64_t)(half * 32 + i) * p.N + n] = hv[i];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int NS>
constexpr size_t smem_bytes() {
    return Cfg<NS>::kOffSmall + sizeof(Small) + 1024;   // + alignment slack
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// 4-D bf16 tensor map over [d3][d2][d1][d0] (d0 innermost) with a (64, 1, 128, 1) box.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t d3) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {d0, d1, d2, d3};
    const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)kTile, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int NS>
int launch_ns(const ScanArgs& a) {
    CUtensorMap tmX, tmB, tmC;
    if (!make_map(&tmX, a.x, a.headdim, a.nheads, a.seqlen, a.batch) ||
        !make_map(&tmB, a.B, a.dstate, a.ngroups, a.seqlen, a.batch) ||
        !make_map(&tmC, a.C, a.dstate, a.ngroups, a.seqlen, a.batch))
        return SSD_ERR_CUDA;
    TcParams p;
    p.batch = a.batch; p.L = a.seqlen; p.H = a.nheads; p.P = a.headdim; p.N = a.dstate;
    p.G = a.ngroups;
    p.n_ps = (int)(a.headdim / kPS);
    p.n_tiles = (int)((a.seqlen + kTile - 1) / kTile);
    p.dt = static_cast<const __nv_bfloat16*>(a.dt);
    p.A = a.A; p.D = a.D; p.h0 = a.h0;
    p.y = static_cast<__nv_bfloat16*>(a.y);
    p.hT = a.hT;
    p.ws = a.ws;
    p.budget = 4ll << 30;   // ~2 s at the B300's maximum SM clock
    const size_t smem = smem_bytes<NS>();
    if (cudaFuncSetAttribute(ssd_tc_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return SSD_ERR_CUDA;
    const int64_t units = a.batch * a.nheads * p.n_ps;
    ssd_tc_kernel<NS><<<(unsigned)units, kThreads, smem, a.stream>>>(tmX, tmB, tmC, p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

bool tc_supports(int32_t dtype, int64_t P, int64_t N, int Q) {
    return dtype == SSD_BF16 && P % kPS == 0 && (N == 128 || N == 256) && Q % 64 == 0;
}

size_t tc_workspace_bytes(int64_t, int64_t, int64_t, int64_t, int64_t, int) {
    return kWsHeaderBytes;
}

int tc_launch(const ScanArgs& a) {
    if (a.batch * a.nheads * (a.headdim / kPS) > 0x7fffffffLL || a.seqlen > 0x7fffffffLL)
        return SSD_ERR_UNSUPPORTED;
    if (a.dstate == 128) return launch_ns<128>(a);
    if (a.dstate == 256) return launch_ns<256>(a);
    return SSD_ERR_UNSUPPORTED;
}

}  // namespace ssd
