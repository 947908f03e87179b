// tc.cu -- the tensor-core path for d_state 256 (the d_state 128 kernel is in tc128.cu) and the
// tensor-core entry points of the library: one fused, warp-specialised, persistent sm_103a
// kernel per scan.
//
// What it computes is the SSD chunk algorithm (Qiita "Mamba-2 / SSD" article section 4.2;
// youngju.dev Mamba article, sections "State Space Dualityの発見" and "SSDアルゴリズムとチャンク分割"),
// evaluated in 128-token tiles that walk each sequence in order with the running state on chip:
//
//   S1  cum_i = sum_{k<=i} dt_k A  (inside the tile); L_ij = exp(cum_i - cum_j) for i >= j
//   S2  G = C B^T                         tcgen05.mma  M=128 N=128 K=d_state   (TMEM)
//       P = L o G o dt_j  -> bf16 in TMEM (CUDA cores, mask first, then exp)
//       Y_diag = P X                      tcgen05.mma  A = P from TMEM, M=128 N=64 K=128
//       S^T = B^T (diag(exp(cum_last - cum) dt) X)   M=d_state N=64 K=128
//   S3  H = exp(cum_last) H + S^T         CUDA cores, H (= h^T, fp32) in registers
//   S4  Y_off = C h_prev^T                tcgen05.mma  M=128 N=64  K=d_state
//       y = Y_diag + exp(cum) Y_off + D x -> bf16, 16-byte stores
//
// For a chunk length Q that is a multiple of 128 the tile is a sub-block of the chunk; the
// block of L o (C B^T) below the tile's diagonal block is applied through its low-rank factor
// (the state at the tile boundary), which the semiseparable structure of M makes exact.
// The result does not depend on Q (chunk-size invariance), so every Q that is a multiple of
// 64 runs the same tiles.
//
// Work: a unit is (batch row b, head h, 64-wide slice of headdim); its chain is its T tiles in
// sequence order.  The chains are laid end to end and cut into one equal range of tiles per SM
// (persistent grid, one CTA per SM).  A range that starts inside a chain takes the state its
// predecessor range ends with through a decoupled look-back over per-CTA slots in the
// workspace (inclusive states, or aggregates (decay, local state) of range pieces).
//
// Warp roles (384 threads; setmaxnreg gives the producer warpgroup 88 registers per thread and
// the compute warpgroups 208):
//   warp 0      TMA producer of the B / C ring (1 stage)
//   warp 1      TMEM allocator and MMA issuer (whole warp, one elected lane issues)
//   warp 2      producer of the x / decay ring: TMA of the x tile, and from dt the tile's
//               log2-domain cumsum and every exponential factor the other roles need
//   warp 3      idle (completes the producer warpgroup)
//   warps 4-11  two identical compute warpgroups; warpgroup g (warps 4+4g .. 7+4g) owns
//               headdim columns 32g .. 32g+31 of x, the state and y, and half of P's column
//               blocks.  Per tile: scaled copy of x for the state GEMM, its P blocks, the
//               state recurrence in registers and bf16 h^T for the next off-diagonal GEMM;
//               the y epilogue of a tile runs one tile later
// The configuration below is written for both d_state values; the d_state 256 instance is the
// one launched.
// Every wait is bounded (clock64 budget); a timeout sets SSD_ERR_TIMEOUT in the workspace
// status word, makes every role stop, drains in-flight copies and MMAs (with a fixed limit of
// their own) and frees TMEM before exit.
#include <atomic>

#include "tc_common.cuh"

namespace ssd {
namespace {

using namespace ptx;
using namespace plan;

template <int NS>
struct Cfg {
    static constexpr int kNReg = NS / 64;             // 64-column regions of a B / C tile
    static constexpr int kXSt = NS == 128 ? 3 : 2;    // x / decay ring depth
    static constexpr int kBCStages = NS == 128 ? 2 : 1;
    static constexpr int kYBuf = NS == 128 ? 2 : 1;   // Y / Y_off accumulator buffers
    static constexpr int kMB = NS / 128;               // 128-row blocks of the state
    // compute warpgroups; each owns kCW of the unit's 64 headdim columns (and kPB of P's
    // 32-column blocks per lane quarter)
    static constexpr int kWG = NS == 128 ? 4 : 2;
    static constexpr int kCW = kPS / kWG;
    static constexpr int kPB = 4 / kWG;
    static constexpr int kHReg = kMB * kCW;            // state values per compute thread
    static constexpr int kComputeThreads = 128 * kWG;
    static constexpr int kThreads = 128 + kComputeThreads;
    // registers per thread: launch budget, producer warpgroup, compute warpgroups
    static constexpr int kRegsLaunch = NS == 128 ? 96 : 168;
    static constexpr int kRegsProducer = NS == 128 ? 64 : 88;
    static constexpr int kRegsCompute = NS == 128 ? 104 : 208;
    static_assert(128 * kRegsProducer + kComputeThreads * kRegsCompute <= kThreads * kRegsLaunch,
                  "registers");
    static_assert(kThreads * kRegsLaunch <= 65536, "register file");
    static constexpr uint32_t kBCBytes = 2 * kNReg * kTileBytes;
    // shared memory (byte offsets from a 1024-aligned base)
    static constexpr uint32_t kOffX = 0;
    static constexpr uint32_t kOffBC = kOffX + kXSt * kTileBytes;
    static constexpr uint32_t kOffXt = kOffBC + kBCStages * kBCBytes;
    static constexpr uint32_t kOffHt = kOffXt + kTileBytes;
    static constexpr uint32_t kOffDt = kOffHt + NS * 128;
    static constexpr uint32_t kOffSmall = kOffDt + kXSt * sizeof(DtSlot);
    static_assert(kOffDt % 16 == 0 && kOffSmall % 16 == 0, "16-byte aligned slots and barriers");
    // TMEM columns
    static constexpr uint32_t kColG = 0;                       // C B^T, fp32, 128 columns
    static constexpr uint32_t kColP = 128;                     // P, bf16 pairs, 64 columns
    static constexpr uint32_t kColY = 192;                     // Y_diag, kYBuf x 64
    static constexpr uint32_t kColYoff = kColY + kYBuf * kPS;  // Y_off, kYBuf x 64
    static constexpr uint32_t kColS = kColYoff + kYBuf * kPS;  // S^T, kMB x 64
    static_assert(kColS + kMB * kPS <= kTmemCols, "TMEM budget");
    static_assert(kXSt <= kXStagesMax, "x ring");
};

// P column block (0..3) number bi of compute warpgroup wg: with two warpgroups each takes two
// blocks, paired so that every lane quarter's lower-triangle blocks split evenly.
template <int WG>
__device__ __forceinline__ int p_col_block(int wg, int bi) {
    if constexpr (WG == 4) return wg;
    else return bi ? (wg ? 2 : 3) : (wg ? 1 : 0);
}

template <int NS>
__global__ void __launch_bounds__(Cfg<NS>::kThreads, 1)
    ssd_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmC,
                  const __grid_constant__ TcParams p) {
    using K = Cfg<NS>;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms and TMA destinations need 1024-byte aligned shared addresses
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Small& sm = *reinterpret_cast<Small*>(smem + K::kOffSmall);
    DtSlot* slots = reinterpret_cast<DtSlot*>(smem + K::kOffDt);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < K::kXSt; ++i) {
            mbar_init(&sm.x_full[i], 1 + 32);
            mbar_init(&sm.x_empty[i], 1 + K::kComputeThreads);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.bc_full[i], 1);
            mbar_init(&sm.bc_empty[i], 1);
            mbar_init(&sm.y_full[i], 1);
            mbar_init(&sm.y_empty[i], K::kComputeThreads);
        }
        mbar_init(&sm.g_full, 1);
        mbar_init(&sm.g_empty, K::kComputeThreads);
        mbar_init(&sm.p_full, K::kComputeThreads);
        mbar_init(&sm.p_empty, 1);
        mbar_init(&sm.xt_full, K::kComputeThreads);
        mbar_init(&sm.xt_empty, 1);
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_empty, K::kComputeThreads);
        mbar_init(&sm.h_full, K::kComputeThreads);
        mbar_init(&sm.h_empty, 1);
        mbar_init(&sm.mma_done, 1);
        sm.abort_flag = 0;
        sm.plan = make_plan(p, blockIdx.x);
        const int us[3] = {sm.plan.u0, sm.plan.u1, sm.plan.f_lo};
        int* dst[3] = {sm.uc_u0, sm.uc_u1, sm.uc_flo};
        for (int i = 0; i < 3; ++i) {
            const UnitCoords c = unit_coords(p, us[i]);
            dst[i][0] = c.b;
            dst[i][1] = c.h;
            dst[i][2] = c.g;
            dst[i][3] = c.bh;
            dst[i][4] = c.ps;
            dst[i][5] = c.hr;
        }
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpTma && lane == 0) {
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
    }
    if (warp == kWarpDt && lane == 0) prefetch_tmap(&tmX);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const Plan& plan = sm.plan;

    // P's blocks above the diagonal are zero in every tile: written once
    if (warp >= kWarpC) {
        const int q = warp & 3, wg = (warp - kWarpC) >> 2;
        const uint32_t tp = tmem + ((uint32_t)(q * 32) << 16) + K::kColP;
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
        for (int bi = 0; bi < K::kPB; ++bi) {
            const int jb = p_col_block<K::kWG>(wg, bi);
            if (jb > q) tmem_st16(tp + 16 * jb, z);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp < kWarpC) {
    regs_dec<K::kRegsProducer>();
    if (warp == kWarpTma) {
        // ------------------------------------------------------- B / C TMA producer ----
        if (lane == 0) {
            int nt = 0;
            for (Cursor c = first_tile(plan, sm, p); c.valid; advance_p(c, plan, sm, p), ++nt) {
                const int s = nt % K::kBCStages;
                const uint32_t use = nt / K::kBCStages;
                if (!wait_bar_p(&sm.bc_empty[s], (use & 1u) ^ 1u, sm, p)) break;
                const int t0 = c.k * kTile;
                // a state-only tile needs B; a full tile also C
                mbar_arrive_expect_tx(&sm.bc_full[s],
                                      (c.it.pass1 ? 1 : 2) * K::kNReg * kTileBytes);
                uint8_t* dst = smem + K::kOffBC + s * K::kBCBytes;
                for (int r = 0; r < K::kNReg; ++r) {
                    tma_load_4d(dst + r * kTileBytes, &tmB, &sm.bc_full[s], r * 64, c.uc.g, t0,
                                c.uc.b);
                    if (!c.it.pass1)
                        tma_load_4d(dst + (K::kNReg + r) * kTileBytes, &tmC, &sm.bc_full[s],
                                    r * 64, c.uc.g, t0, c.uc.b);
                }
            }
            if (sm.abort_flag) {
                // drain: every issued load must land before the CTA's smem goes away
                for (int j = nt - K::kBCStages; j < nt; ++j) {
                    if (j < 0) continue;
                    drain_wait(&sm.bc_full[j % K::kBCStages], (uint32_t)(j / K::kBCStages) & 1u,
                               p.ws);
                }
            }
        }
    } else if (warp == kWarpDt) {
        // ------------------------------------------ x TMA + decay-factor producer ----
        int nt = 0;
        int a_u = -1;
        float A2 = 0.f;
        // dt of tile k of the cursor's unit, 4 consecutive tokens per lane
        auto load_dt = [&](const Cursor& c, int k, float (&d)[4]) {
            const int64_t t = (int64_t)k * kTile + 4 * lane;
            const __nv_bfloat16* src = p.dt + ((int64_t)c.uc.b * p.L + t) * p.H + c.uc.h;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                d[i] = t + i < p.L ? __bfloat162float(src[(int64_t)i * p.H]) : 0.f;
        };
        // the next tile's dt is loaded one tile ahead (when it belongs to the same unit), so
        // its memory latency overlaps this tile's work
        float dn[4] = {0.f, 0.f, 0.f, 0.f};
        bool have_next = false;
        for (Cursor c = first_tile(plan, sm, p); c.valid; advance_p(c, plan, sm, p), ++nt) {
            float d0[4];
            if (have_next) {
#pragma unroll
                for (int i = 0; i < 4; ++i) d0[i] = dn[i];
            } else {
                load_dt(c, c.k, d0);
            }
            have_next = c.k + 1 < c.it.k1;
            if (have_next) load_dt(c, c.k + 1, dn);
            if (c.it.u != a_u) {
                a_u = c.it.u;
                A2 = p.A[c.uc.h] * kLog2e;
            }
            const int s = nt % K::kXSt;
            const uint32_t use = nt / K::kXSt;
            if (!wait_warp(&sm.x_empty[s], (use & 1u) ^ 1u, sm, p)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&sm.x_full[s], kTileBytes);
                tma_load_4d(smem + K::kOffX + s * kTileBytes, &tmX, &sm.x_full[s],
                            c.uc.ps * kPS, c.uc.h, c.k * kTile, c.uc.b);
            }
            fill_dt_slot<false>(slots[s], d0, A2, lane);
            mbar_arrive(&sm.x_full[s]);
        }
        if (sm.abort_flag && lane == 0) {
            // drain: the x loads of every tile this loop completed must land before exit
            for (int j = nt - K::kXSt; j < nt; ++j) {
                if (j < 0) continue;
                drain_wait(&sm.x_full[j % K::kXSt], (uint32_t)(j / K::kXSt) & 1u, p.ws);
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------------- MMA issuer ------
        // the whole warp runs this role in converged control flow; one elected lane issues
        {
            constexpr uint32_t idG = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idS = idesc_bf16(128, kPS, 1, 1);
            constexpr uint32_t idYoff = idesc_bf16(128, kPS, 0, 1);
            constexpr uint32_t idYd = idesc_bf16(128, kPS, 0, 1);
            // Each K = 128 GEMM goes out as one block of 8 back-to-back MMAs from converged
            // code (issued one by one from a loop, the tensor core takes them at about half
            // its rate).
            // G = C B^T of tile number nt (the j-th full tile), once the P builders have read
            // the previous G
            auto issue_G = [&](int nt, int j) -> bool {
                const int s = nt % K::kBCStages;
                if (!wait_warp_p(&sm.bc_full[s], (uint32_t)(nt / K::kBCStages) & 1u, sm, p))
                    return false;
                if (!wait_warp_p(&sm.g_empty, ((uint32_t)j & 1u) ^ 1u, sm, p)) return false;
                tc_fence_after();
                const uint32_t bbase = sbase + K::kOffBC + s * K::kBCBytes;
                const uint32_t cbase = bbase + K::kNReg * kTileBytes;
#pragma unroll
                for (int kb = 0; kb < NS / 128; ++kb)
                    mma8_ss_e<kStepCols, kStepCols>(
                        tmem + K::kColG, smem_desc_sw128(cbase + 2 * kb * kTileBytes, 16, 1024),
                        smem_desc_sw128(bbase + 2 * kb * kTileBytes, 16, 1024), idG, kb > 0);
                mma_commit_e(&sm.g_full);
                return true;
            };
            int nt = 0, j = 0;           // tiles issued, full (non state-only) tiles issued
            bool g_ahead = false;        // G of the current tile was issued one tile early
            Cursor c = first_tile(plan, sm, p);
            for (; c.valid; ++nt) {
                const int s = nt % K::kBCStages;
                const int xs = nt % K::kXSt;
                const uint32_t par = (uint32_t)nt & 1u;
                const bool full_tile = !c.it.pass1;
                const bool next_full =
                    (c.k + 1 < c.it.k1)
                        ? !c.it.pass1
                        : (c.item + 1 < plan.n_items &&
                           !plan_item(plan, c.item + 1, p.n_tiles).pass1);
                if (full_tile && !g_ahead && !issue_G(nt, j)) break;
                g_ahead = false;
                // chunk state S^T = B^T (w o X)
                if (!wait_warp_p(&sm.xt_full, par, sm, p) || !wait_warp_p(&sm.s_empty, par ^ 1u, sm, p))
                    break;
                if (!full_tile &&
                    !wait_warp_p(&sm.bc_full[s], (uint32_t)(nt / K::kBCStages) & 1u, sm, p))
                    break;
                tc_fence_after();
                {
                    const uint32_t bbase = sbase + K::kOffBC + s * K::kBCBytes;
                    const uint32_t xt = sbase + K::kOffXt;
#pragma unroll
                    for (int mb = 0; mb < K::kMB; ++mb)
                        mma8_ss_e<kStepRows, kStepRows>(
                            tmem + K::kColS + mb * kPS,
                            smem_desc_sw128(bbase + 2 * mb * kTileBytes, kTileBytes, 1024),
                            smem_desc_sw128(xt, 1024, 1024), idS, 0u);
                }
                mma_commit_e(&sm.s_full);
                mma_commit_e(&sm.xt_empty);
                if (!full_tile) {
                    mma_commit_e(&sm.bc_empty[s]);
                    mma_commit_e(&sm.x_empty[xs]);
                    advance_p(c, plan, sm, p);
                    continue;
                }
                const int yb = j % K::kYBuf;
                const uint32_t ypar = (uint32_t)(j / K::kYBuf) & 1u;
                // off-diagonal Y_off = C h_prev^T, into the accumulator buffer of this tile
                if (!wait_warp_p(&sm.h_full, (uint32_t)j & 1u, sm, p) ||
                    !wait_warp_p(&sm.y_empty[yb], ypar ^ 1u, sm, p))
                    break;
                tc_fence_after();
                {
                    const uint32_t cbase = sbase + K::kOffBC + s * K::kBCBytes +
                                           K::kNReg * kTileBytes;
                    const uint32_t ht = sbase + K::kOffHt;
#pragma unroll
                    for (int kb = 0; kb < NS / 128; ++kb)
                        mma8_ss_e<kStepCols, kStepRows>(
                            tmem + K::kColYoff + yb * kPS,
                            smem_desc_sw128(cbase + 2 * kb * kTileBytes, 16, 1024),
                            smem_desc_sw128(ht + kb * 8 * 2048, 1024, 1024), idYoff, kb > 0);
                }
                mma_commit_e(&sm.h_empty);
                mma_commit_e(&sm.bc_empty[s]);   // G, S^T and Y_off have read this B / C stage
                // next tile's C B^T while this tile's P is built
                if (K::kBCStages > 1 && next_full) {
                    if (!issue_G(nt + 1, j + 1)) break;
                    g_ahead = true;
                }
                // Y_diag = P X, P read from TMEM
                if (!wait_warp_p(&sm.p_full, (uint32_t)j & 1u, sm, p)) break;
                tc_fence_after();
                {
                    const uint32_t xb = sbase + K::kOffX + xs * kTileBytes;
                    mma8_ts_e<kStepRows>(tmem + K::kColY + yb * kPS, tmem + K::kColP,
                                         smem_desc_sw128(xb, 1024, 1024), idYd, 0u);
                }
                mma_commit_e(&sm.y_full[yb]);
                mma_commit_e(&sm.p_empty);
                mma_commit_e(&sm.x_empty[xs]);
                if (K::kBCStages == 1 && next_full) {
                    if (!issue_G(nt + 1, j + 1)) break;
                    g_ahead = true;
                }
                ++j;
                advance_p(c, plan, sm, p);
            }
            // every MMA issued above has completed once this barrier's phase 0 completes
            mma_commit_e(&sm.mma_done);
            if (lane == 0) drain_wait(&sm.mma_done, 0, p.ws);
            __syncwarp();
        }
    }
    } else {
        regs_inc<K::kRegsCompute>();
        // ------------------------------------------------------------- compute warps -----
        constexpr int CW = K::kCW;
        const int w = warp - kWarpC;             // 0 .. 4 kWG - 1
        const int q = warp & 3;                  // TMEM lane quarter
        const int wg = w >> 2;                   // column block
        const int r = q * 32 + lane;             // tile row, and state row inside a 128-block
        const int c0 = wg * CW;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        float h[K::kHReg];
        PendingY<CW> pend;
        bool have_pend = false;
        // the deferred y epilogue of full tile pj: y = Y_diag + exp(cum) Y_off + D x for this
        // thread's row and column block, in 16-column steps
        auto epilogue = [&](int pj) -> bool {
            const int yb = pj % K::kYBuf;
            if (!wait_warp(&sm.y_full[yb], (uint32_t)(pj / K::kYBuf) & 1u, sm, p)) return false;
            tc_fence_after();
            float yd[CW], yo[CW];
            tmem_ld_pair<CW>(tmem + lane_base + K::kColY + yb * kPS + c0, yd,
                             tmem + lane_base + K::kColYoff + yb * kPS + c0, yo);
#pragma unroll
            for (int qc = 0; qc < CW / 16; ++qc) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const uint4 xv = pend.x[qc * 2 + cc];
                    const uint32_t xin[4] = {xv.x, xv.y, xv.z, xv.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = qc * 16 + cc * 8 + e * 2;
                        const float v0 =
                            fmaf(pend.d, bf16lo_to_f32(xin[e]), fmaf(pend.e, yo[i0], yd[i0]));
                        const float v1 = fmaf(pend.d, bf16hi_to_f32(xin[e]),
                                              fmaf(pend.e, yo[i0 + 1], yd[i0 + 1]));
                        o[e] = pack_bf16x2(v0, v1);
                    }
                    if (pend.row)
                        *reinterpret_cast<uint4*>(pend.row + qc * 16 + cc * 8) =
                            make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.y_empty[yb]);
            return true;
        };
        int nt = 0, j = 0;
        int d_u = -1;
        float Dh = 0.f;
        float item_logd = 0.f;                   // sum of log2 tile decays over the item
        bool ok = true;
        for (Cursor c = first_tile(plan, sm, p); c.valid; advance(c, plan, sm, p), ++nt) {
            const UnitCoords& uc = c.uc;
            const bool full_tile = !c.it.pass1;
            const int xs = nt % K::kXSt;
            const uint32_t par = (uint32_t)nt & 1u;
            const bool last_of_item = c.k + 1 == c.it.k1;
            if (c.k == c.it.k0) {
                // ---- start of an item: the entering state (a deferred epilogue of the previous
                // item runs after this item's first P, like any other)
                item_logd = 0.f;
                if (c.it.u != d_u) {
                    d_u = c.it.u;
                    Dh = p.D ? p.D[uc.h] : 0.f;
                }
                if (c.it.init == kInitLookback) {
                    if (!look_back<NS, CW>(h, p, sm, w, lane, r, c0, c.it.u)) { ok = false; break; }
                } else {
                    const float* src = (c.it.init == kInitH0 && p.h0)
                                           ? p.h0 + ((int64_t)uc.bh * p.P + (int64_t)uc.ps * kPS) * NS
                                           : nullptr;
                    h_from<NS, CW>(h, src, r, c0, 0.f, false, false);
                }
                if (full_tile) {
                    // h^T for the item's first Y_off, once the previous full tile's Y_off is done
                    if (j > 0 && !wait_warp(&sm.h_empty, (uint32_t)(j - 1) & 1u, sm, p)) {
                        ok = false;
                        break;
                    }
                    ht_write<NS, CW>(h, smem + K::kOffHt, r, wg);
                    fence_proxy_async_smem();
                    mbar_arrive(&sm.h_full);
                }
            }
            if (!wait_warp(&sm.x_full[xs], (uint32_t)(nt / K::kXSt) & 1u, sm, p)) { ok = false; break; }
            const DtSlot& sl = slots[xs];

            // w o X for the chunk-state GEMM: row r scaled by exp(cum_last - cum_r) dt_r; the raw
            // x row stays in registers for this tile's (deferred) D x term
            if (!wait_warp(&sm.xt_empty, par ^ 1u, sm, p)) { ok = false; break; }
            uint4 xk[CW / 8];
            {
                const float wr = sl.w[r];
                const uint8_t* xrow = smem + K::kOffX + xs * kTileBytes;
                uint8_t* xtrow = smem + K::kOffXt;
#pragma unroll
                for (int cc = 0; cc < CW / 8; ++cc)
                    xk[cc] = *reinterpret_cast<const uint4*>(xrow + sw128_off(r, wg * (CW / 8) + cc));
#pragma unroll
                for (int cc = 0; cc < CW / 8; ++cc) {
                    const uint32_t in[4] = {xk[cc].x, xk[cc].y, xk[cc].z, xk[cc].w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[e] = pack_bf16x2(wr * bf16lo_to_f32(in[e]), wr * bf16hi_to_f32(in[e]));
                    *reinterpret_cast<uint4*>(xtrow + sw128_off(r, wg * (CW / 8) + cc)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&sm.xt_full);

            if (full_tile) {
                // this warp's column blocks of P (those above the diagonal stay zero)
                if (!wait_warp(&sm.g_full, (uint32_t)j & 1u, sm, p)) { ok = false; break; }
                if (!wait_warp(&sm.p_empty, ((uint32_t)j & 1u) ^ 1u, sm, p)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tg = tmem + lane_base + K::kColG;
                const uint32_t tp = tmem + lane_base + K::kColP;
#pragma unroll 1
                for (int bi = 0; bi < K::kPB; ++bi) {
                    const int jb = p_col_block<K::kWG>(wg, bi);
                    if (jb > q) continue;
                    float g[32];
                    tmem_ld32(tg + 32 * jb, g);
                    uint32_t pk[16];
                    p_block(pk, g, jb, q, lane, r, sl);
                    tmem_st16(tp + 16 * jb, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sm.g_empty);
                mbar_arrive(&sm.p_full);
                // the previous full tile's y (its Y_diag has completed: P was free)
                if (have_pend) {
                    if (!epilogue(j - 1)) { ok = false; break; }
                    have_pend = false;
                }
            }

            // S3: H = exp(cum_last) H + S^T, and (on a full tile that is not the item's last)
            // bf16 h^T for the next tile's Y_off, once this tile's Y_off has read the old one
            const float clast2 = sl.clast2;
            const float decay = ex2(clast2);    // exp(cum_last)
            item_logd += clast2;
            const bool write_ht = full_tile && !last_of_item;
            if (!wait_warp(&sm.s_full, par, sm, p)) { ok = false; break; }
            if (write_ht && !wait_warp(&sm.h_empty, (uint32_t)j & 1u, sm, p)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int mb = 0; mb < K::kMB; ++mb) {
                float sv[CW];
                tmem_ld_cols<CW>(tmem + lane_base + K::kColS + mb * kPS + c0, sv);
#pragma unroll
                for (int i = 0; i < CW; ++i) h[mb * CW + i] = fmaf(decay, h[mb * CW + i], sv[i]);
            }
            tc_fence_before();
            mbar_arrive(&sm.s_empty);
            if (write_ht) {
                ht_write<NS, CW>(h, smem + K::kOffHt, r, wg);
                fence_proxy_async_smem();
                mbar_arrive(&sm.h_full);
            }
            const float e_r = sl.e[r];
            mbar_arrive(&sm.x_empty[xs]);        // the MMA adds its own arrival after Y_diag

            // this tile's y is deferred to the next full tile
            if (full_tile) {
                const int64_t t = (int64_t)c.k * kTile + r;
                pend.row = t < p.L ? p.y + (((int64_t)uc.b * p.L + t) * p.H + uc.h) * p.P +
                                         uc.ps * kPS + c0
                                   : nullptr;
                pend.e = e_r;
                pend.d = Dh;
#pragma unroll
                for (int cc = 0; cc < CW / 8; ++cc) pend.x[cc] = xk[cc];
                have_pend = true;
                ++j;
            }

            if (last_of_item && c.it.fin != kFinNone) {
                // ---- end of an item: final state, or publish for the next range
                if (c.it.fin == kFinFinal) {
                    if (p.hT)
                        h_to<NS, CW>(h, p.hT + ((int64_t)uc.bh * p.P + (int64_t)uc.ps * kPS) * NS, r,
                                 c0);
                } else {
                    publish<NS, CW>(h, p, w, lane, r, c0, c.it.fin, item_logd);
                }
            }
        }
        if (ok && have_pend) epilogue(j - 1);
    }

    // single-lane roles (TMA, MMA issue) reconverge their warp before the CTA barrier
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

template <int NS>
constexpr size_t smem_bytes() {
    return Cfg<NS>::kOffSmall + sizeof(Small) + 1024;   // + alignment slack
}
// at most 227 KB of dynamic shared memory per CTA on sm_103a
static_assert(smem_bytes<256>() <= 232448, "shared memory");

template <int NS>
int launch_ns(const ScanArgs& a) {
    CUtensorMap tmX, tmB, tmC;
    if (!make_map(&tmX, a.x, a.headdim, a.nheads, a.seqlen, a.batch) ||
        !make_map(&tmB, a.B, a.dstate, a.ngroups, a.seqlen, a.batch) ||
        !make_map(&tmC, a.C, a.dstate, a.ngroups, a.seqlen, a.batch))
        return SSD_ERR_CUDA;
    const int nsm = sm_count();
    if (nsm <= 0) return SSD_ERR_CUDA;
    TcParams p;
    p.batch = a.batch; p.L = a.seqlen; p.H = a.nheads; p.P = a.headdim; p.N = a.dstate;
    p.G = a.ngroups;
    p.n_ps = (int)(a.headdim / kPS);
    p.n_tiles = (int)((a.seqlen + kTile - 1) / kTile);
    p.n_units = a.batch * a.nheads * p.n_ps;
    const int64_t total = p.n_units * p.n_tiles;
    p.n_ctas = (int)std::min<int64_t>(std::min(nsm, kMaxCtas), total);
    if (a.max_ctas > 0) p.n_ctas = std::min(p.n_ctas, a.max_ctas);
    // Without a state-only pass, a range's head piece is published before its successor's
    // tail piece is needed as long as every range is longer than a chain.
    p.pass1_mode = (total / p.n_ctas) > p.n_tiles ? 0 : 1;
    p.dt = static_cast<const __nv_bfloat16*>(a.dt);
    p.A = a.A; p.D = a.D; p.h0 = a.h0;
    p.y = static_cast<__nv_bfloat16*>(a.y);
    p.hT = a.hT;
    p.ws = a.status ? a.status : a.ws;
    p.flags = reinterpret_cast<int*>(a.ws + kWsHeaderBytes);
    p.slots = reinterpret_cast<float*>(a.ws + kWsHeaderBytes + flags_bytes());
    p.budget = tc_wait_budget();
    if (cudaMemsetAsync(p.flags, 0, sizeof(int) * kFlagsPerCta * (size_t)p.n_ctas, a.stream) !=
        cudaSuccess)
        return SSD_ERR_CUDA;
    const size_t smem = smem_bytes<NS>();
    if (cudaFuncSetAttribute(ssd_tc_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return SSD_ERR_CUDA;
    ssd_tc_kernel<NS><<<(unsigned)p.n_ctas, Cfg<NS>::kThreads, smem, a.stream>>>(tmX, tmB, tmC, p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

namespace {
constexpr long long kDefaultWaitCycles = 4ll << 30;   // ~2 s at the B300's maximum SM clock
std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};
}  // namespace

long long tc_wait_budget() { return g_wait_cycles.load(std::memory_order_relaxed); }

bool tc_supports(int32_t dtype, int64_t P, int64_t N, int Q) {
    return dtype == SSD_BF16 && P % kPS == 0 && (N == 128 || N == 256) && Q % 64 == 0;
}

size_t tc_workspace_bytes(int64_t b, int64_t L, int64_t H, int64_t P, int64_t N, int) {
    size_t bytes = kWsHeaderBytes + flags_bytes() + slots_bytes(N);
    if (N == 128) {
        // segment records of the separate state-only pass
        const int64_t tiles = (L + kTile - 1) / kTile;
        bytes += (size_t)seg_records(b * H * (P / kPS) * tiles, kMaxCtas) * kSegRecBytes;
    }
    return bytes;
}

size_t tc_workspace_bytes_ctas(int64_t N, int ctas) {
    size_t bytes = kWsHeaderBytes + flags_bytes() + sizeof(float) * 2 * (size_t)ctas * kPS * (size_t)N;
    if (N == 128) bytes += (size_t)5 * ctas * kSegRecBytes;
    return bytes;
}

int tc_launch(const ScanArgs& a) {
    if (a.batch * a.nheads * (a.headdim / kPS) > 0x7fffffffLL || a.seqlen > 0x7fffffffLL)
        return SSD_ERR_UNSUPPORTED;
    if (a.dstate == 128) return tc128_launch(a);
    if (a.dstate == 256) return launch_ns<256>(a);
    return SSD_ERR_UNSUPPORTED;
}

}  // namespace ssd

extern "C" int64_t ssd_scan_set_wait_cycles(int64_t cycles) {
    const long long v = cycles > 0 ? (long long)cycles : ssd::kDefaultWaitCycles;
    return (int64_t)ssd::g_wait_cycles.exchange(v, std::memory_order_relaxed);
}
