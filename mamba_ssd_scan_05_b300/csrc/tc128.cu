// tc128.cu -- the tensor-core scan for d_state 128: one fused, warp-specialised, persistent
// sm_103a kernel per scan.
//
// What it computes is the SSD chunk algorithm (Qiita "Mamba-2 / SSD" article section 4.2;
// youngju.dev Mamba article, sections "State Space Dualityの発見" and "SSDアルゴリズムとチャンク分割"),
// evaluated in 128-token tiles that walk each sequence in order with the running state on chip:
//
//   S1  cum_i = sum_{k<=i} dt_k A  (inside the tile); L_ij = exp(cum_i - cum_j) for i >= j
//   S2  G = C B^T                                       tcgen05.mma  M=128 N=128 K=128
//       Y_diag = (L o G o dt_j) X,  chunk state S^T = B^T (exp(cum_last - cum) dt o X)
//   S3  H = exp(cum_last) H + S^T                       CUDA cores, H (= h^T, fp32) in registers
//   S4  y = Y_diag + exp(cum) C h_prev^T + D x          bf16, 16-byte stores
//
// Two ways to evaluate a tile, chosen per (head, tile) by the decay producer:
//
// Factored (almost every tile: the decay over the tile stays within 2^-160 and every dt is at
// most 2^20).  With a reference m (half the tile's log2 decay, an integer), the decay mask
// factors exactly as L_ij dt_j = 2^(cum_i - m) * 2^(m - cum_j) dt_j, so
//       y_i = 2^(cum_i - m) * [ ((G o mask) Xs)_i + (C (2^m h_prev)^T)_i ] + D x_i,
//       Xs  = diag(2^(m - cum_j) dt_j) X,    S^T = 2^(cum_last - m) B^T Xs.
// The diagonal term and the off-diagonal term accumulate into ONE TMEM accumulator, the
// P operand is G with the causal mask (no exponentials per element), and the one scaled copy
// Xs of the x tile feeds both the state GEMM and Y_diag.  Every factor lies in [2^-100, 2^100].
//
// Fallback (any other tile, e.g. a step size so large that the state resets inside it): P is
// L o G o dt_j built per element (masked before the exponential; factored around a
// 32-token block's row where the block allows it), Y_diag = P X with the raw x tile, the
// off-diagonal term C h^T goes to an accumulator of its own and is scaled by exp(cum_i) in the
// epilogue, and the state GEMM uses exp(cum_last - cum_j) dt_j X.
//
// The tile and the chunk: for a chunk length Q that is a multiple of 128 the tile is a
// sub-block of the chunk; the block of L o (C B^T) below the tile's diagonal block is applied
// through its low-rank factor (the state at the tile boundary), which the semiseparable
// structure of M makes exact; the result does not depend on Q, so every Q that is a multiple of
// 64 runs the same tiles.
//
// Work: a unit is (batch row b, head h, 64-wide slice of headdim); its chain is its T tiles in
// sequence order.  The chains are laid end to end and cut into one equal range of tiles per SM
// (persistent grid, one CTA per SM); a range that starts inside a chain takes its entering
// state through a look-back over per-CTA slots in the workspace.
//
// Warp roles (640 threads; setmaxnreg gives the producer warpgroup 64 registers per thread
// and the compute warpgroups 104):
//   warp 0      TMA producer of the B / C ring (2 stages)
//   warp 1      TMEM allocator and MMA issuer (whole warp, one elected lane issues); per tile:
//               S^T, the off-diagonal GEMM, Y_diag, then C B^T of the next tile
//   warp 2      x TMA and decay producer: the tile's log2-domain cumsum of dt A and every
//               factor the other roles need, and the tile's mode
//   warp 3      idle (completes the producer warpgroup, which setmaxnreg needs whole)
//   warps 4-19  four identical compute warpgroups; warpgroup g owns headdim columns
//               16g .. 16g+15 of x, the state and y, and P's column block g.  Per tile: the
//               scaled x tile, its P block, the previous tile's y epilogue, the state
//               recurrence in registers and bf16 h^T for the next off-diagonal GEMM.
// TMEM (512 columns): C B^T 128 | P 2 x 64 (bf16, double-buffered) | Y 2 x 64 | S^T 64 |
// fallback off-diagonal accumulator 64.
// Every wait is bounded (a clock64 budget); a timeout sets SSD_ERR_TIMEOUT in the workspace
// status word, makes every role stop, drains in-flight copies and MMAs (with a fixed limit of
// their own) and frees TMEM before exit.
#include "tc_common.cuh"
#include "tc_state.cuh"

namespace ssd {
namespace {

using namespace ptx;
using namespace plan;

struct K3 {
    static constexpr int NS = 128;
    static constexpr int kNReg = NS / 64;              // 64-column regions of a B / C tile
    static constexpr int kXSt = 3;                     // x / decay ring depth
    static constexpr int kBCStages = 2;
    static constexpr int kWG = 4;                      // compute warpgroups
    static constexpr int kCW = kPS / kWG;              // headdim columns per compute warpgroup
    static constexpr int kComputeThreads = 128 * kWG;
    static constexpr int kThreads = 128 + kComputeThreads;
    // registers per thread: at launch, and the setmaxnreg split
    static constexpr int kRegsLaunch = 96, kRegsProducer = 64, kRegsCompute = 104;
    static_assert(128 * kRegsProducer + kComputeThreads * kRegsCompute <=
                      kThreads * kRegsLaunch, "registers");
    static_assert(kThreads * kRegsLaunch <= 65536, "register file");
    static constexpr uint32_t kBCBytes = 2 * kNReg * kTileBytes;
    // shared memory (byte offsets from a 1024-aligned base)
    static constexpr uint32_t kOffX = 0;
    static constexpr uint32_t kOffBC = kOffX + kXSt * kTileBytes;
    static constexpr uint32_t kOffXs = kOffBC + kBCStages * kBCBytes;   // scaled x tile
    static constexpr uint32_t kOffHt = kOffXs + kTileBytes;
    static constexpr uint32_t kOffDt = kOffHt + NS * 128;
    static constexpr uint32_t kOffSmall = kOffDt + kXSt * sizeof(DtSlot);
    static_assert(kOffDt % 16 == 0 && kOffSmall % 16 == 0, "16-byte aligned slots and barriers");
    static constexpr size_t kSmemBytes = kOffSmall + sizeof(Small) + 1024;   // + alignment slack
    // the instance with the fused gated RMSNorm adds the row-sum exchange [128 rows][4] floats
    static constexpr uint32_t kOffRed = (kOffSmall + sizeof(Small) + 15) / 16 * 16;
    static constexpr size_t kSmemBytesGated = kOffRed + 128 * 4 * sizeof(float) + 1024;
    // TMEM columns
    static constexpr uint32_t kColG = 0;        // C B^T, fp32, 128 columns
    static constexpr uint32_t kColP = 128;      // P, bf16 pairs, 2 buffers x 64
    static constexpr uint32_t kColY = 256;      // output accumulator, 2 buffers x 64
    static constexpr uint32_t kColS = 384;      // S^T, 64
    static constexpr uint32_t kColYoff = 448;   // fallback tiles' off-diagonal term, 64
    static_assert(kColYoff + kPS <= kTmemCols, "TMEM budget");
    static_assert(kXSt <= kXStagesMax, "x ring");
    // at most 227 KB of dynamic shared memory per CTA on sm_103a
    static_assert(kSmemBytes <= 232448 && kSmemBytesGated <= 232448, "shared memory");
};

// ------------------------------------------------------------------- producer roles ----------

// Warp 0, one lane: B and C tiles of every tile of the CTA's plan into the B / C ring (a
// state-only tile needs B only).
template <bool kExt>
__device__ __forceinline__ void role_bc_producer(const Plan& plan, Small& sm, const TcParams& p,
                                                 uint8_t* smem, const CUtensorMap* tmB,
                                                 const CUtensorMap* tmC) {
    using K = K3;
    int nt = 0;
    for (Cursor c = first_tile<kExt>(plan, sm, p); c.valid; advance_p<kExt>(c, plan, sm, p), ++nt) {
        const int s = nt % K::kBCStages;
        const uint32_t use = nt / K::kBCStages;
        if (!wait_bar_p(&sm.bc_empty[s], (use & 1u) ^ 1u, sm, p)) break;
        SSD_TC_TRACE_POINT(60, nt);
        const int t0 = c.k * kTile;
        mbar_arrive_expect_tx(&sm.bc_full[s], (c.it.pass1 ? 1 : 2) * K::kNReg * kTileBytes);
        uint8_t* dst = smem + K::kOffBC + s * K::kBCBytes;
        for (int r = 0; r < K::kNReg; ++r) {
            tma_load_4d(dst + r * kTileBytes, tmB, &sm.bc_full[s], r * 64, c.uc.g, t0, c.uc.b);
            if (!c.it.pass1)
                tma_load_4d(dst + (K::kNReg + r) * kTileBytes, tmC, &sm.bc_full[s], r * 64,
                            c.uc.g, t0, c.uc.b);
        }
    }
    if (sm.abort_flag) {
        // drain: every issued load must land before the CTA's shared memory goes away
        for (int j = nt - K::kBCStages; j < nt; ++j)
            if (j >= 0)
                drain_wait(&sm.bc_full[j % K::kBCStages], (uint32_t)(j / K::kBCStages) & 1u, p.ws);
    }
}

// Warp 2, all lanes: the x tile (TMA) and the tile's decay factors and mode (DtSlot).
template <bool kExt>
__device__ __forceinline__ void role_x_producer(const Plan& plan, Small& sm, const TcParams& p,
                                                uint8_t* smem, DtSlot* slots,
                                                const CUtensorMap* tmX, int lane) {
    using K = K3;
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
    // the next tile's dt is loaded one tile ahead (when it belongs to the same unit), so its
    // memory latency overlaps this tile's work
    float dn[4] = {0.f, 0.f, 0.f, 0.f};
    bool have_next = false;
    for (Cursor c = first_tile<kExt>(plan, sm, p); c.valid; advance_p<kExt>(c, plan, sm, p), ++nt) {
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
        if (!wait_warp_p(&sm.x_empty[s], (use & 1u) ^ 1u, sm, p)) break;
        SSD_TC_TRACE_POINT(50, nt);
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.x_full[s], kTileBytes);
            tma_load_4d(smem + K::kOffX + s * kTileBytes, tmX, &sm.x_full[s], c.uc.ps * kPS,
                        c.uc.h, c.k * kTile, c.uc.b);
        }
        fill_dt_slot<true>(slots[s], d0, A2, lane);
        mbar_arrive(&sm.x_full[s]);
        SSD_TC_TRACE_POINT(51, nt);
    }
    if (sm.abort_flag && lane == 0) {
        // drain: the x loads of every tile this loop completed must land before exit
        for (int j = nt - K::kXSt; j < nt; ++j)
            if (j >= 0) drain_wait(&sm.x_full[j % K::kXSt], (uint32_t)(j / K::kXSt) & 1u, p.ws);
    }
}

// Warp 1, the whole warp in converged control flow (one elected lane issues).  Per full tile
// k: S^T_k, the off-diagonal GEMM (into the output accumulator on a factored tile, into its own
// accumulator on a fallback tile), Y_diag_k (A = P from TMEM; B = the scaled x tile on a
// factored tile, the raw x tile on a fallback tile), then G_{k+1} = C B^T of the next tile once
// the compute warps have read G_k.  Per state-only tile: S^T_k alone.  Each K = 128 GEMM goes
// out as one block of 8 back-to-back MMAs.
template <bool kExt>
__device__ __forceinline__ void role_mma(const Plan& plan, Small& sm, const TcParams& p,
                                         const DtSlot* slots, uint32_t sbase, uint32_t tmem,
                                         int lane) {
    using K = K3;
    constexpr uint32_t idG = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idS = idesc_bf16(128, kPS, 1, 1);
    constexpr uint32_t idYoff = idesc_bf16(128, kPS, 0, 1);
    constexpr uint32_t idYd = idesc_bf16(128, kPS, 0, 1);
    // G = C B^T of tile number nt (the j-th full tile), once the compute warps have read G_{j-1}
    auto issue_G = [&](int nt, int j) -> bool {
        const int s = nt % K::kBCStages;
        if (!wait_warp_p(&sm.bc_full[s], (uint32_t)(nt / K::kBCStages) & 1u, sm, p)) return false;
        if (!wait_warp_p(&sm.g_empty, ((uint32_t)j & 1u) ^ 1u, sm, p)) return false;
        SSD_TC_TRACE_POINT(13, nt);
        tc_fence_after();
        const uint32_t bbase = sbase + K::kOffBC + s * K::kBCBytes;
        const uint32_t cbase = bbase + K::kNReg * kTileBytes;
        mma8_ss_e<kStepCols, kStepCols>(tmem + K::kColG, smem_desc_sw128(cbase, 16, 1024),
                                        smem_desc_sw128(bbase, 16, 1024), idG, 0u);
        mma_commit_e(&sm.g_full);
        return true;
    };
    int nt = 0, j = 0;        // tiles issued, full (non state-only) tiles issued
    int nf = 0;               // fallback full tiles issued
    bool g_ahead = false;     // G of the current tile was issued during the previous tile
    Cursor c = first_tile<kExt>(plan, sm, p);
    for (; c.valid; ++nt) {
        const int s = nt % K::kBCStages;
        const int xs = nt % K::kXSt;
        const uint32_t par = (uint32_t)nt & 1u;
        const bool full_tile = !c.it.pass1;
        const bool next_full =
            (c.k + 1 < c.it.k1)
                ? !c.it.pass1
                : (c.item + 1 < plan.n_items && !plan_item<kExt>(plan, c.item + 1, p.n_tiles).pass1);
        if (full_tile && !g_ahead && !issue_G(nt, j)) break;
        g_ahead = false;
        // chunk state S^T = B^T Xs, once the compute warps have built Xs and read S^T_{k-1}
        if (!wait_warp_p(&sm.xt_full, par, sm, p) || !wait_warp_p(&sm.s_empty, par ^ 1u, sm, p))
            break;
        if (!full_tile &&
            !wait_warp_p(&sm.bc_full[s], (uint32_t)(nt / K::kBCStages) & 1u, sm, p))
            break;
        SSD_TC_TRACE_POINT(10, nt);
        tc_fence_after();
        const uint32_t bbase = sbase + K::kOffBC + s * K::kBCBytes;
        const uint32_t xsb = sbase + K::kOffXs;
        mma8_ss_e<kStepRows, kStepRows>(tmem + K::kColS, smem_desc_sw128(bbase, kTileBytes, 1024),
                                        smem_desc_sw128(xsb, 1024, 1024), idS, 0u);
        mma_commit_e(&sm.s_full);
        if (!full_tile) {
            mma_commit_e(&sm.xt_empty);
            mma_commit_e(&sm.bc_empty[s]);
            mma_commit_e(&sm.x_empty[xs]);
            advance_p<kExt>(c, plan, sm, p);
            continue;
        }
        // the tile's mode, written by the decay producer before x_full completed
        if (!wait_warp_p(&sm.x_full[xs], (uint32_t)(nt / K::kXSt) & 1u, sm, p)) break;
        const bool fac = slots[xs].fac != 0;
        const int yb = j & 1;
        const uint32_t ypar = (uint32_t)(j >> 1) & 1u;
        // off-diagonal C (s_h h)^T, with s_h = 2^m (factored) or 1 (fallback)
        if (!wait_warp_p(&sm.h_full, (uint32_t)j & 1u, sm, p) ||
            !wait_warp_p(&sm.y_empty[yb], ypar ^ 1u, sm, p))
            break;
        if (!fac && !wait_warp_p(&sm.yoff_empty, ((uint32_t)nf & 1u) ^ 1u, sm, p)) break;
        SSD_TC_TRACE_POINT(11, nt);
        tc_fence_after();
        const uint32_t dy = tmem + K::kColY + yb * kPS;
        mma8_ss_e<kStepCols, kStepRows>(fac ? dy : tmem + K::kColYoff,
                                        smem_desc_sw128(bbase + K::kNReg * kTileBytes, 16, 1024),
                                        smem_desc_sw128(sbase + K::kOffHt, 1024, 1024), idYoff, 0u);
        mma_commit_e(&sm.h_empty);
        mma_commit_e(&sm.bc_empty[s]);   // G, S^T and the off-diagonal GEMM have read this stage
        // Y_diag = P Xs (factored, accumulated onto the off-diagonal term) or P X (fallback)
        if (!wait_warp_p(&sm.p_full, (uint32_t)j & 1u, sm, p)) break;
        SSD_TC_TRACE_POINT(12, nt);
        tc_fence_after();
        const uint32_t bx = fac ? xsb : sbase + K::kOffX + xs * kTileBytes;
        mma8_ts_e<kStepRows>(dy, tmem + K::kColP + yb * kPS, smem_desc_sw128(bx, 1024, 1024), idYd,
                             fac ? 1u : 0u);
        mma_commit_e(&sm.y_full[yb]);
        mma_commit_e(&sm.pb_empty[yb]);
        mma_commit_e(&sm.xt_empty);
        mma_commit_e(&sm.x_empty[xs]);
        if (!fac) ++nf;
        // the next tile's C B^T while this tile's epilogue and the next S^T / h^T run
        if (next_full) {
            if (!issue_G(nt + 1, j + 1)) break;
            g_ahead = true;
        }
        ++j;
        advance_p<kExt>(c, plan, sm, p);
    }
    // every MMA issued above has completed once this barrier's phase 0 completes
    mma_commit_e(&sm.mma_done);
    if (lane == 0) drain_wait(&sm.mma_done, 0, p.ws);
    __syncwarp();
}

// bf16 (s h)^T into the MN-major, 128-byte swizzled h^T tile (128 rows x 64 columns): the B
// operand of the off-diagonal GEMM; s = 2^m (a power of two, exact) or 1.
template <int CW>
__device__ __forceinline__ void ht_write_scaled(const float (&h)[CW], float s, uint8_t* ht, int r,
                                                int wg) {
#pragma unroll
    for (int cc = 0; cc < CW / 8; ++cc) {
        const float* v = &h[cc * 8];
        *reinterpret_cast<uint4*>(ht + sw128_off(r, wg * (CW / 8) + cc)) =
            make_uint4(pack_bf16x2(s * v[0], s * v[1]), pack_bf16x2(s * v[2], s * v[3]),
                       pack_bf16x2(s * v[4], s * v[5]), pack_bf16x2(s * v[6], s * v[7]));
    }
}

// A tile whose y epilogue is deferred to the next full tile.  Its x stage (the x row for the
// D x term) and decay slot (the row factor, the mode) stay held until that epilogue has run.
struct Pend {
    int64_t off;            // element offset of this thread's y (and z) row and column block,
                            // or -1 past the sequence end
    int64_t wcol;           // feature index of its first column (h * P + column)
    float d;                // D of the head
    int xs;                 // x / decay stage of the tile
};

// ---- paths taken once per item, per fallback block or per CTA ---------------------------------

// A compute thread's part of the running state, passed by value to and from the cold paths.
struct HState {
    float v[K3::kCW];
    int ok;
};

// The state an item starts from: the look-back over the preceding ranges, the initial state,
// or zeros.  ok = 0 on a timeout or abort.
__device__ __forceinline__ HState item_entry_state(const TcParams* p, Small* sm, int init, int u,
                                                int bh, int ps, int w, int lane, int r, int c0) {
    HState s;
    s.ok = 1;
    if (init == kInitLookback) {
        if (!look_back<K3::NS, K3::kCW>(s.v, *p, *sm, w, lane, r, c0, u)) s.ok = 0;
    } else {
        const float* src = (init == kInitH0 && p->h0)
                               ? p->h0 + ((int64_t)bh * p->P + (int64_t)ps * kPS) * K3::NS
                               : nullptr;
        h_from<K3::NS, K3::kCW>(s.v, src, r, c0, 0.f, false, false);
    }
    return s;
}

// The state an item ends with: the final state, or published for the next range.
__device__ __forceinline__ void item_exit_state(HState h, const TcParams* p, int fin, int bh, int ps,
                                             int w, int lane, int r, int c0, float item_logd) {
    if (fin == kFinFinal) {
        if (p->hT)
            h_to<K3::NS, K3::kCW>(h.v, p->hT + ((int64_t)bh * p->P + (int64_t)ps * kPS) * K3::NS,
                                  r, c0);
    } else {
        publish<K3::NS, K3::kCW>(h.v, *p, w, lane, r, c0, fin, item_logd);
    }
}

struct G16 {
    float v[16];
};
struct P8 {
    uint32_t v[8];
};

// Half a block of P on a fallback tile (L o G o dt_j with the decay factors of the slot).
__device__ __forceinline__ P8 p_half_fallback(G16 g, int jb, int hf, int q, int lane, int r,
                                           const DtSlot* sl) {
    P8 o;
    p_half(o.v, g.v, jb, hf, q, lane, r, *sl);
    return o;
}

// silu(v) = v / (1 + exp(-v)) with the fast exponential and division (0 for v < -88).
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.f + __expf(-v)); }

// The output of this thread's 16 columns of a token row: y = s Y + D x (s = the row factor on
// a factored tile, 1 on a fallback tile, whose Y already holds Y_diag + e Y_off).  Plain: y is
// rounded to bf16 and stored.  Gated (kGated): out = y rsqrt(mean_group(y^2) + eps) w silu(z)
// over groups of p.gsize consecutive features (Qiita "Mamba-2 / SSD" article, section 4.2,
// step 4), from the float32 y; a group wider than the thread's 16 columns is summed across the
// warps of the TMEM lane quarter through `red` (row sums) and red_bar[q] (bounded waits, two
// phases: sums written, sums read).  Returns false on a timeout or abort.
template <bool kGated>
__device__ __forceinline__ bool emit(const Pend& pend, float sc, const float (&yv)[16],
                                     const uint4 (&xv)[2], const TcParams& p, Small& sm,
                                     float* red, int r, int wg, int q) {
    float y[16];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const uint32_t xin[4] = {xv[cc].x, xv[cc].y, xv[cc].z, xv[cc].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i0 = cc * 8 + k * 2;
            y[i0] = fmaf(pend.d, bf16lo_to_f32(xin[k]), sc * yv[i0]);
            y[i0 + 1] = fmaf(pend.d, bf16hi_to_f32(xin[k]), sc * yv[i0 + 1]);
        }
    }
    if constexpr (kGated) {
        uint4 zv[2] = {};
        if (pend.off >= 0) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
                zv[cc] = *reinterpret_cast<const uint4*>(p.z + pend.off + cc * 8);
        }
        float s0 = 0.f, s1 = 0.f;     // sums of squares of columns 0-7 and 8-15
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            s0 = fmaf(y[i], y[i], s0);
            s1 = fmaf(y[8 + i], y[8 + i], s1);
        }
        float ss0 = s0, ss1 = s1;     // the sums over each column's group
        if (p.gsize >= 16) ss0 = ss1 = s0 + s1;
        if (p.gsize > 16) {
            red[r * 4 + wg] = ss0;
            mbar_arrive(&sm.red_bar[q]);
            if (!wait_warp(&sm.red_bar[q], 0u, sm, p)) return false;
            const float* rr = red + r * 4;
            ss0 = ss1 = p.gsize == 32 ? rr[wg & 2] + rr[(wg & 2) + 1] : (rr[0] + rr[1]) + (rr[2] + rr[3]);
            mbar_arrive(&sm.red_bar[q]);
            if (!wait_warp(&sm.red_bar[q], 1u, sm, p)) return false;
        }
        const float inv = 1.f / (float)p.gsize;
        const float rs0 = rsqrtf(fmaf(ss0, inv, p.eps)), rs1 = rsqrtf(fmaf(ss1, inv, p.eps));
        float wv[16];
        if (p.nw) {
            const float4* wp = reinterpret_cast<const float4*>(p.nw + pend.wcol);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 f = wp[i];
                wv[4 * i] = f.x; wv[4 * i + 1] = f.y; wv[4 * i + 2] = f.z; wv[4 * i + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) wv[i] = 1.f;
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const uint32_t zin[4] = {zv[cc].x, zv[cc].y, zv[cc].z, zv[cc].w};
            const float rsc = cc ? rs1 : rs0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i0 = cc * 8 + k * 2;
                y[i0] *= rsc * wv[i0] * silu_fast(bf16lo_to_f32(zin[k]));
                y[i0 + 1] *= rsc * wv[i0 + 1] * silu_fast(bf16hi_to_f32(zin[k]));
            }
        }
    }
    if (pend.off >= 0) {
        __nv_bfloat16* row = p.y + pend.off;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
            *reinterpret_cast<uint4*>(row + cc * 8) =
                make_uint4(pack_bf16x2(y[cc * 8 + 0], y[cc * 8 + 1]),
                           pack_bf16x2(y[cc * 8 + 2], y[cc * 8 + 3]),
                           pack_bf16x2(y[cc * 8 + 4], y[cc * 8 + 5]),
                           pack_bf16x2(y[cc * 8 + 6], y[cc * 8 + 7]));
    }
    return true;
}

// The last pending epilogue of the CTA (after its loop).
template <bool kGated>
__device__ __forceinline__ bool last_epilogue(Pend pend, int pj, Small* sm, const TcParams* p,
                                              const DtSlot* slots, const uint8_t* smem,
                                              float* red, uint32_t tmem, uint32_t lane_base,
                                              int r, int wg, int q) {
    const int yb = pj & 1;
    const DtSlot& ps = slots[pend.xs];
    const float e = ps.e[r];
    const bool fac = ps.fac != 0;
    uint4 xv[2];
    const uint8_t* xrow = smem + K3::kOffX + pend.xs * kTileBytes;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc)
        xv[cc] = *reinterpret_cast<const uint4*>(xrow + sw128_off(r, wg * 2 + cc));
    if (!wait_warp(&sm->y_full[yb], (uint32_t)(pj >> 1) & 1u, *sm, *p)) return false;
    tc_fence_after();
    float yv[16], yo[16];
    tmem_ld16x2(tmem + lane_base + K3::kColY + yb * kPS + wg * 16, yv,
                tmem + lane_base + K3::kColYoff + wg * 16, yo);
    if (!fac) {
#pragma unroll
        for (int i = 0; i < 16; ++i) yv[i] = fmaf(e, yo[i], yv[i]);
    }
    tc_fence_before();
    mbar_arrive(&sm->y_empty[yb]);
    if (!fac) mbar_arrive(&sm->yoff_empty);
    mbar_arrive(&sm->x_empty[pend.xs]);
    return emit<kGated>(pend, fac ? e : 1.f, yv, xv, *p, *sm, red, r, wg, q);
}

// bf16 (s h)^T into the MN-major, 128-byte swizzled h^T tile (128 rows x 64 columns): the B
// operand of the off-diagonal GEMM; s = 2^m (a power of two, exact) or 1.
__device__ __forceinline__ void ht_write_scaled(const float (&h)[16], float s, uint8_t* ht, int r,
                                                int wg) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const float* v = &h[cc * 8];
        *reinterpret_cast<uint4*>(ht + sw128_off(r, wg * 2 + cc)) =
            make_uint4(pack_bf16x2(s * v[0], s * v[1]), pack_bf16x2(s * v[2], s * v[3]),
                       pack_bf16x2(s * v[4], s * v[5]), pack_bf16x2(s * v[6], s * v[7]));
    }
}

// Warps 4-19: compute warpgroup wg (headdim columns c0 = 16 wg ..), lane quarter q (TMEM lanes,
// tile rows and state rows 32q .. 32q+31).  Per tile: the scaled x tile, this tile's P block,
// the previous tile's y, the state.  Returns false on a timeout or abort.
template <bool kGated, bool kExt>
__device__ __forceinline__ bool role_compute(const Plan& plan, Small& sm, const TcParams& p,
                                             uint8_t* smem, const DtSlot* slots, uint32_t tmem,
                                             int w, int lane) {
    using K = K3;
    constexpr int CW = K::kCW;
    static_assert(CW == 16, "one 16-column block per compute warpgroup");
    const int q = w & 3;                     // TMEM lane quarter (= warp index mod 4)
    const int wg = w >> 2;                   // column block, and P's column block
    const int r = q * 32 + lane;             // tile row, and state row
    const int c0 = wg * CW;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + K::kOffRed);   // gated instance only
    float h[CW];
    Pend pend{};
    bool have_pend = false;
    int nt = 0, j = 0;
    int d_u = -1;
    float Dh = 0.f;
    float item_logd = 0.f;                   // sum of log2 tile decays over the item
    for (Cursor c = first_tile<kExt>(plan, sm, p); c.valid; advance<kExt>(c, plan, sm, p), ++nt) {
        const UnitCoords& uc = c.uc;
        const bool full_tile = !c.it.pass1;
        const int xs = nt % K::kXSt;
        const uint32_t par = (uint32_t)nt & 1u;
        const bool last_of_item = c.k + 1 == c.it.k1;
        if (c.k == c.it.k0) {
            // ---- start of an item: the entering state
            item_logd = 0.f;
            if (c.it.u != d_u) {
                d_u = c.it.u;
                Dh = p.D ? p.D[uc.h] : 0.f;
            }
            const HState hs = item_entry_state(&p, &sm, c.it.init, c.it.u, uc.bh, uc.ps, w, lane,
                                               r, c0);
            if (!hs.ok) return false;
#pragma unroll
            for (int i = 0; i < CW; ++i) h[i] = hs.v[i];
        }
        if (!wait_warp(&sm.x_full[xs], (uint32_t)(nt / K::kXSt) & 1u, sm, p)) return false;
        const DtSlot& sl = slots[xs];
        if (c.k == c.it.k0 && full_tile) {
            // h^T for the item's first off-diagonal GEMM, once the previous one is done
            if (j > 0 && !wait_warp(&sm.h_empty, (uint32_t)(j - 1) & 1u, sm, p)) return false;
            ht_write_scaled(h, sl.hsc, smem + K::kOffHt, r, wg);
            fence_proxy_async_smem();
            mbar_arrive(&sm.h_full);
        }

        // ---- the scaled x tile for the state GEMM (and Y_diag on a factored tile)
        if (!wait_warp(&sm.xt_empty, par ^ 1u, sm, p)) return false;
        SSD_TC_TRACE_POINT(30, nt);
        {
            const float wr = sl.w[r];
            const uint8_t* xrow = smem + K::kOffX + xs * kTileBytes;
            uint8_t* xsrow = smem + K::kOffXs;
            uint4 xk[2];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
                xk[cc] = *reinterpret_cast<const uint4*>(xrow + sw128_off(r, wg * 2 + cc));
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const uint32_t in[4] = {xk[cc].x, xk[cc].y, xk[cc].z, xk[cc].w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = pack_bf16x2(wr * bf16lo_to_f32(in[e]), wr * bf16hi_to_f32(in[e]));
                *reinterpret_cast<uint4*>(xsrow + sw128_off(r, wg * 2 + cc)) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(&sm.xt_full);
        SSD_TC_TRACE_POINT(31, nt);

        if (full_tile) {
            // ---- this tile's P block: G with the causal mask (factored) or L o G o dt_j
            // (fallback), into this tile's P buffer; blocks above the diagonal stay zero
            const int pb = j & 1;
            if (!wait_warp(&sm.g_full, (uint32_t)j & 1u, sm, p)) return false;
            if (!wait_warp(&sm.pb_empty[pb], ((uint32_t)(j >> 1) & 1u) ^ 1u, sm, p)) return false;
            SSD_TC_TRACE_POINT(20, nt);
            tc_fence_after();
            if (wg <= q) {
                float g0[16], g1[16];
                const uint32_t tg = tmem + lane_base + K::kColG + 32 * wg;
                tmem_ld16x2(tg, g0, tg + 16, g1);
                SSD_TC_TRACE_POINT(22, nt);
                const uint32_t tp = tmem + lane_base + K::kColP + pb * kPS + 16 * wg;
                uint32_t pk[8];
                if (sl.fac) {
                    if (wg == q) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) g0[k] = k <= lane ? g0[k] : 0.f;
#pragma unroll
                        for (int k = 0; k < 16; ++k) g1[k] = 16 + k <= lane ? g1[k] : 0.f;
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(g0[2 * i], g0[2 * i + 1]);
                    tmem_st8(tp, pk);
#pragma unroll
                    for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(g1[2 * i], g1[2 * i + 1]);
                    tmem_st8(tp + 8, pk);
                } else {
                    G16 ga, gb;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        ga.v[i] = g0[i];
                        gb.v[i] = g1[i];
                    }
                    const P8 pa = p_half_fallback(ga, wg, 0, q, lane, r, &sl);
                    const P8 pc = p_half_fallback(gb, wg, 1, q, lane, r, &sl);
#pragma unroll
                    for (int i = 0; i < 8; ++i) pk[i] = pa.v[i];
                    tmem_st8(tp, pk);
#pragma unroll
                    for (int i = 0; i < 8; ++i) pk[i] = pc.v[i];
                    tmem_st8(tp + 8, pk);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&sm.g_empty);
            mbar_arrive(&sm.p_full);
            SSD_TC_TRACE_POINT(21, nt);
            // ---- the previous full tile's y (its x stage is released here)
            if (have_pend) {
                const int pyb = (j - 1) & 1;
                const DtSlot& ps = slots[pend.xs];
                const float pe = ps.e[r];
                const bool pfac = ps.fac != 0;
                uint4 xv[2];
                const uint8_t* xrow = smem + K::kOffX + pend.xs * kTileBytes;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
                    xv[cc] = *reinterpret_cast<const uint4*>(xrow + sw128_off(r, wg * 2 + cc));
                if (!wait_warp(&sm.y_full[pyb], (uint32_t)((j - 1) >> 1) & 1u, sm, p)) return false;
                SSD_TC_TRACE_POINT(40, nt);
                tc_fence_after();
                float yv[16];
                if (pfac) {
                    tmem_ld16(tmem + lane_base + K::kColY + pyb * kPS + c0, yv);
                } else {
                    float yo[16];
                    tmem_ld16x2(tmem + lane_base + K::kColY + pyb * kPS + c0, yv,
                                tmem + lane_base + K::kColYoff + c0, yo);
#pragma unroll
                    for (int i = 0; i < 16; ++i) yv[i] = fmaf(pe, yo[i], yv[i]);
                }
                SSD_TC_TRACE_POINT(42, nt);
                tc_fence_before();
                mbar_arrive(&sm.y_empty[pyb]);
                if (!pfac) mbar_arrive(&sm.yoff_empty);
                mbar_arrive(&sm.x_empty[pend.xs]);
                if (!emit<kGated>(pend, pfac ? pe : 1.f, yv, xv, p, sm, red, r, wg, q))
                    return false;
                have_pend = false;
            }
            SSD_TC_TRACE_POINT(41, nt);
        }

        // ---- S3: H = exp(cum_last) H + sigma S^T, and (on a full tile that is not the item's
        // last) bf16 (s h)^T for the next tile's off-diagonal GEMM
        const float clast2 = sl.clast2;
        const float decay = ex2(clast2);    // exp(cum_last)
        const float sigma = sl.sigma;
        item_logd += clast2;
        const bool write_ht = full_tile && !last_of_item;
        if (!wait_warp(&sm.s_full, par, sm, p)) return false;
        SSD_TC_TRACE_POINT(32, nt);
        tc_fence_after();
        {
            float sv[CW];
            tmem_ld16(tmem + lane_base + K::kColS + c0, sv);
            SSD_TC_TRACE_POINT(34, nt);
#pragma unroll
            for (int i = 0; i < CW; ++i) h[i] = fmaf(decay, h[i], sigma * sv[i]);
        }
        tc_fence_before();
        mbar_arrive(&sm.s_empty);
        if (write_ht) {
            // the next tile (same item) decides the scale of h^T: wait for its decay slot
            const int xs1 = (nt + 1) % K::kXSt;
            if (!wait_warp(&sm.x_full[xs1], (uint32_t)((nt + 1) / K::kXSt) & 1u, sm, p))
                return false;
            if (!wait_warp(&sm.h_empty, (uint32_t)j & 1u, sm, p)) return false;
            ht_write_scaled(h, slots[xs1].hsc, smem + K::kOffHt, r, wg);
            fence_proxy_async_smem();
            mbar_arrive(&sm.h_full);
        }
        SSD_TC_TRACE_POINT(33, nt);

        // this tile's y is deferred to the next full tile (which then releases the x stage);
        // a state-only tile releases its stage now
        if (full_tile) {
            const int64_t t = (int64_t)c.k * kTile + r;
            pend.wcol = (int64_t)uc.h * p.P + uc.ps * kPS + c0;
            pend.off = t < p.L ? ((int64_t)uc.b * p.L + t) * p.H * p.P + pend.wcol : -1;
            pend.d = Dh;
            pend.xs = xs;
            have_pend = true;
            ++j;
        } else {
            mbar_arrive(&sm.x_empty[xs]);
        }

        if (last_of_item && c.it.fin != kFinNone) {
            // ---- end of an item: final state, or publish for the next range
            HState hs;
#pragma unroll
            for (int i = 0; i < CW; ++i) hs.v[i] = h[i];
            hs.ok = 1;
            item_exit_state(hs, &p, c.it.fin, uc.bh, uc.ps, w, lane, r, c0, item_logd);
        }
    }
    if (have_pend &&
        !last_epilogue<kGated>(pend, j - 1, &sm, &p, slots, smem, red, tmem, lane_base, r, wg, q))
        return false;
    return true;
}

// ------------------------------------------------------------------- the kernel --------------

template <bool kGated, bool kExt>
__global__ void __launch_bounds__(K3::kThreads, 1)
    ssd_tc128_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ TcParams p) {
    using K = K3;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms and TMA destinations need 1024-byte aligned shared addresses
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Small& sm = *reinterpret_cast<Small*>(smem + K::kOffSmall);
    DtSlot* slots = reinterpret_cast<DtSlot*>(smem + K::kOffDt);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr uint32_t kC = K::kComputeThreads;

    if (threadIdx.x == 0) {
        for (int i = 0; i < K::kXSt; ++i) {
            mbar_init(&sm.x_full[i], 1 + 32);
            mbar_init(&sm.x_empty[i], 1 + kC);   // the MMA's commit and every compute thread
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.bc_full[i], 1);
            mbar_init(&sm.bc_empty[i], 1);
            mbar_init(&sm.y_full[i], 1);
            mbar_init(&sm.y_empty[i], kC);
            mbar_init(&sm.pb_empty[i], 1);
        }
        mbar_init(&sm.g_full, 1);
        mbar_init(&sm.g_empty, kC);
        mbar_init(&sm.p_full, kC);
        mbar_init(&sm.xt_full, kC);
        mbar_init(&sm.xt_empty, 1);
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_empty, kC);
        mbar_init(&sm.h_full, kC);
        mbar_init(&sm.h_empty, 1);
        mbar_init(&sm.yoff_empty, kC);
        for (int i = 0; i < 4; ++i) mbar_init(&sm.red_bar[i], 128);
        mbar_init(&sm.mma_done, 1);
        sm.abort_flag = 0;
        sm.plan = plan::make_plan<kExt>(p.n_units, p.n_tiles, p.n_ctas, p.pass1_mode, blockIdx.x);
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

    // the blocks of P above the diagonal are zero in every tile: written once, in both buffers
    if (warp >= kWarpC) {
        const int q = warp & 3, jb = (warp - kWarpC) >> 2;
        if (jb > q) {
            uint32_t z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = 0u;
            const uint32_t tp = tmem + ((uint32_t)(q * 32) << 16) + K::kColP + 16 * jb;
            tmem_st16(tp, z);
            tmem_st16(tp + kPS, z);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp < kWarpC) {
        regs_dec<K::kRegsProducer>();
        if (warp == kWarpTma) {
            if (lane == 0) role_bc_producer<kExt>(plan, sm, p, smem, &tmB, &tmC);
        } else if (warp == kWarpDt) {
            role_x_producer<kExt>(plan, sm, p, smem, slots, &tmX, lane);
        } else if (warp == kWarpMma) {
            role_mma<kExt>(plan, sm, p, slots, sbase, tmem, lane);
        }
    } else {
        regs_inc<K::kRegsCompute>();
        role_compute<kGated, kExt>(plan, sm, p, smem, slots, tmem, warp - kWarpC, lane);
    }

    // single-lane roles (B / C TMA) reconverge their warp before the CTA barrier
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

namespace {

template <bool kGated>
int launch128(const ScanArgs& a, const TcParams& p) {
    using K = K3;
    constexpr size_t smem = kGated ? K::kSmemBytesGated : K::kSmemBytes;
    // Ranges shorter than chains: the state-only passes run as a kernel of their own
    // (tc_state.cuh), then the scan instance whose plan leaves them out (kExt), which finds
    // every state it looks back for already published.
    const bool ext = p.pass1_mode == 1;
    auto kernel = ext ? ssd_tc128_kernel<kGated, true> : ssd_tc128_kernel<kGated, false>;
    // the setmaxnreg split must fit in the registers the kernel is launched with: check what
    // the compiler gave each instance before its first launch (a split that does not fit would
    // never complete)
    static int regs_ok[2] = {-1, -1};
    if (regs_ok[ext] < 0) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return SSD_ERR_CUDA;
        regs_ok[ext] =
            (fa.numRegs == K::kRegsLaunch && fa.maxThreadsPerBlock >= K::kThreads) ? 1 : 0;
    }
    if (!regs_ok[ext]) return SSD_ERR_UNSUPPORTED;
    CUtensorMap tmX, tmB, tmC;
    if (!make_map(&tmX, a.x, a.headdim, a.nheads, a.seqlen, a.batch) ||
        !make_map(&tmB, a.B, a.dstate, a.ngroups, a.seqlen, a.batch) ||
        !make_map(&tmC, a.C, a.dstate, a.ngroups, a.seqlen, a.batch))
        return SSD_ERR_CUDA;
    if (cudaMemsetAsync(p.flags, 0, sizeof(int) * kFlagsPerCta * (size_t)p.n_ctas, a.stream) !=
        cudaSuccess)
        return SSD_ERR_CUDA;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return SSD_ERR_CUDA;
    if (ext) {
        // segment records after the hand-off slots, as many as the workspace holds
        const size_t off = seg_offset(a.max_ctas > 0 ? a.max_ctas : kMaxCtas);
        const int64_t recs = a.ws_bytes > off ? (int64_t)((a.ws_bytes - off) / kSegRecBytes) : 0;
        StTable tab;
        int n_segs = 0;
        int rc = st_table(p, reinterpret_cast<float*>(a.ws + off), recs, &tab, &n_segs);
        if (rc == SSD_OK && n_segs > 0) rc = tc128_state_launch(tmX, tmB, p, tab, n_segs, a.stream);
        if (rc != SSD_OK) return rc;
    }
    kernel<<<(unsigned)p.n_ctas, K::kThreads, smem, a.stream>>>(tmX, tmB, tmC, p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

void tc128_grid(int64_t batch, int64_t L, int64_t H, int64_t P, int nsm, int max_ctas,
                int* n_ctas, int* pass1_mode) {
    const int64_t n_tiles = (L + kTile - 1) / kTile;
    const int64_t total = batch * H * (P / kPS) * n_tiles;
    int ctas = (int)std::min<int64_t>(std::min(nsm, kMaxCtas), total);
    if (max_ctas > 0) ctas = std::min(ctas, max_ctas);
    *n_ctas = ctas;
    // Without a state-only pass, a range's head piece is published before its successor's
    // tail piece is needed as long as every range is longer than a chain.
    *pass1_mode = (total / ctas) > n_tiles ? 0 : 1;
}

int tc128_kernels_per_call(int64_t batch, int64_t L, int64_t H, int64_t P) {
    const int nsm = sm_count();
    if (nsm <= 0) return -SSD_ERR_CUDA;
    int ctas = 0, mode = 0;
    tc128_grid(batch, L, H, P, nsm, 0, &ctas, &mode);
    if (mode != 1) return 1;
    // the state-only pass kernel runs when some range ends inside a chain
    static thread_local plan::StPiece pieces[kMaxCtas];
    int np = 0;
    const int64_t n_tiles = (L + kTile - 1) / kTile;
    if (plan::state_segments(batch * H * (P / kPS), (int)n_tiles, ctas, 0, pieces, kMaxCtas, &np) < 0)
        return -SSD_ERR_UNSUPPORTED;
    return np > 0 ? 2 : 1;
}

bool tc128_gated_supports(int64_t P, int group) {
    return P % kPS == 0 && (group == 8 || group == 16 || group == 32 || group == 64);
}

int tc128_launch(const ScanArgs& a) {
    if (a.gated && !tc128_gated_supports(a.headdim, a.group)) return SSD_ERR_UNSUPPORTED;
    const int nsm = sm_count();
    if (nsm <= 0) return SSD_ERR_CUDA;
    TcParams p;
    p.batch = a.batch; p.L = a.seqlen; p.H = a.nheads; p.P = a.headdim; p.N = a.dstate;
    p.G = a.ngroups;
    p.n_ps = (int)(a.headdim / kPS);
    p.n_tiles = (int)((a.seqlen + kTile - 1) / kTile);
    p.n_units = a.batch * a.nheads * p.n_ps;
    tc128_grid(a.batch, a.seqlen, a.nheads, a.headdim, nsm, a.max_ctas, &p.n_ctas, &p.pass1_mode);
    p.dt = static_cast<const __nv_bfloat16*>(a.dt);
    p.A = a.A; p.D = a.D; p.h0 = a.h0;
    p.y = static_cast<__nv_bfloat16*>(a.y);
    p.hT = a.hT;
    p.ws = a.status ? a.status : a.ws;
    p.flags = reinterpret_cast<int*>(a.ws + kWsHeaderBytes);
    p.slots = reinterpret_cast<float*>(a.ws + kWsHeaderBytes + flags_bytes());
    p.budget = tc_wait_budget();
    p.z = static_cast<const __nv_bfloat16*>(a.z);
    p.nw = a.norm_w;
    p.eps = a.eps;
    p.gsize = a.group;
    return a.gated ? launch128<true>(a, p) : launch128<false>(a, p);
}

}  // namespace ssd
