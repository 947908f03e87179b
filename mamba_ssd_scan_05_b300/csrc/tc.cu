// tc.cu -- the tensor-core path: one fused, warp-specialised, persistent sm_103a kernel per scan.
//
// What it computes is the SSD chunk algorithm (Qiita "Mamba-2 / SSD" article section 4.2;
// youngju.dev Mamba article, sections "State Space Dualityの発見" and "SSDアルゴリズムとチャンク分割"),
// evaluated in 128-token tiles that walk each sequence in order with the running state on chip:
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
// Work: a unit is (batch row b, head h, 64-wide slice of headdim); its chain is its T tiles in
// sequence order.  The chains are laid end to end and cut into one equal range of tiles per SM
// (persistent grid, one CTA per SM).  A range that starts inside a chain takes the state its
// predecessor range ends with through a decoupled look-back over per-CTA slots in the
// workspace (inclusive states, or aggregates (decay, local state) of range pieces).
//
// Warp roles (320 threads):
//   warp 0      TMA producer: x / B / C tiles of 128 tokens into a ring of smem stages
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer
//   warps 2-5   "A" warpgroup: cumsum of dt*A, scaled copy of x for the state GEMM, P = L o G
//   warps 6-9   "B" warpgroup: state recurrence in TMEM, bf16 h^T for the next tile, y epilogue,
//               state hand-off between CTAs
// Every wait is bounded (clock64 budget); a timeout sets SSD_ERR_TIMEOUT in the workspace
// status word, makes every role stop, drains in-flight copies and frees TMEM before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

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
constexpr int kMaxCtas = 256;       // grid cap (and number of hand-off slots in the workspace)

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
    float a_cp[kTile];       // cum * log2(e) - log2(dt) per row ("A" warpgroup; +inf if dt = 0)
    float a_wsum[2][4];      // per-warp scan totals, double-buffered by tile parity
    float b_wsum[2][4];
    int lb_kind;             // look-back step decided by one "B" thread: 1 inclusive, 2 aggregate
    float lb_logd;           // that step's aggregate log2 decay
};

struct TcParams {
    int64_t batch, L, H, P, N, G;
    int n_ps;           // P / 64
    int n_tiles;        // T = ceil(L / 128): tiles per unit chain
    int64_t n_units;    // U = batch * H * n_ps
    int n_ctas;         // grid size (persistent: at most one CTA per SM)
    int pass1_mode;     // 1: range pieces with a successor run a state-only pass first
    const __nv_bfloat16* dt;
    const float* A;
    const float* D;
    const float* h0;
    __nv_bfloat16* y;
    float* hT;
    uint8_t* ws;
    int* flags;         // per CTA: [0] inclusive-state flag, [1] aggregate flag, [2] log2 decay
    float* slots;       // per CTA: inclusive state [64 x N], then aggregate state [64 x N]
    long long budget;   // clock64 cycles a single wait may take
};

// ---- the work of one CTA --------------------------------------------------------------------
//
// A range holds at most a tail piece of one chain (it needs the state the previous range
// ends with), whole chains, and a head piece of another chain (its end state is needed by the
// next range); or a middle piece of one chain.  Items run in this order: [state-only pass over
// the piece with a successor, in pass1 mode], [head piece], [whole chains], [tail piece], so
// the state a successor needs is published as early as possible and the state a range needs
// is consumed as late as possible.

enum : int { kInitH0 = 0, kInitZero = 1, kInitLookback = 2 };
enum : int { kFinNone = 0, kFinFinal = 1, kFinIncl = 2, kFinAgg = 3 };

struct Item {
    int64_t u;        // unit
    int k0, k1;       // tile range of the unit's chain
    int pass1;        // 1: state-only pass (no y)
    int init;         // how the state starts: kInit*
    int fin;          // what happens to the state at the end: kFin*
};

struct Plan {
    int n_pre;
    Item pre[2];
    int64_t f_lo, n_full;   // whole chains f_lo .. f_lo + n_full - 1
    int has_post;
    Item post;
    int64_t n_items;
};

__device__ __forceinline__ Plan make_plan(const TcParams& p, int cta) {
    Plan pl;
    pl.n_pre = 0;
    pl.n_full = 0;
    pl.f_lo = 0;
    pl.has_post = 0;
    const int64_t T = p.n_tiles, total = p.n_units * T;
    const int64_t start = (int64_t)cta * total / p.n_ctas;
    const int64_t end = (int64_t)(cta + 1) * total / p.n_ctas;
    if (start >= end) {
        pl.n_items = 0;
        return pl;
    }
    const int64_t u0 = start / T, u1 = (end - 1) / T;
    const int k0 = (int)(start % T), k1 = (int)((end - 1) % T + 1);
    const bool p1 = p.pass1_mode != 0;
    if (u0 == u1 && k0 > 0 && k1 < T) {              // middle piece of one chain
        if (p1) pl.pre[pl.n_pre++] = Item{u0, k0, k1, 1, kInitZero, kFinAgg};
        pl.post = Item{u0, k0, k1, 0, kInitLookback, kFinIncl};
        pl.has_post = 1;
    } else {
        // head piece of chain u1 (starts at tile 0, ends before T)
        const bool head = (u0 == u1) ? (k0 == 0 && k1 < T) : (k1 < T);
        // tail piece of chain u0 (starts after tile 0, runs to T)
        const bool tail = k0 > 0;
        if (head) {
            if (p1) pl.pre[pl.n_pre++] = Item{u1, 0, k1, 1, kInitH0, kFinIncl};
            pl.pre[pl.n_pre++] = Item{u1, 0, k1, 0, kInitH0, p1 ? kFinNone : kFinIncl};
        }
        const int64_t f_first = tail ? u0 + 1 : u0;
        const int64_t f_last = head ? u1 - 1 : u1;
        if (f_last >= f_first) {
            pl.f_lo = f_first;
            pl.n_full = f_last - f_first + 1;
        }
        if (tail) {
            pl.post = Item{u0, k0, (u0 == u1) ? k1 : (int)T, 0, kInitLookback, kFinFinal};
            pl.has_post = 1;
        }
    }
    pl.n_items = pl.n_pre + pl.n_full + pl.has_post;
    return pl;
}

__device__ __forceinline__ Item plan_item(const Plan& pl, int64_t i, int T) {
    if (i < pl.n_pre) return pl.pre[i];
    i -= pl.n_pre;
    if (i < pl.n_full) return Item{pl.f_lo + i, 0, T, 0, kInitH0, kFinFinal};
    return pl.post;
}

// Position in a CTA's sequence of tiles.
struct Cursor {
    int64_t item;
    int k;
    Item it;
    bool valid;
};

__device__ __forceinline__ Cursor first_tile(const Plan& pl, int T) {
    Cursor c;
    c.item = 0;
    c.k = 0;
    c.valid = pl.n_items > 0;
    if (c.valid) {
        c.it = plan_item(pl, 0, T);
        c.k = c.it.k0;
    }
    return c;
}

__device__ __forceinline__ Cursor next_tile(const Plan& pl, Cursor c, int T) {
    if (c.k + 1 < c.it.k1) {
        ++c.k;
        return c;
    }
    ++c.item;
    c.valid = c.item < pl.n_items;
    if (c.valid) {
        c.it = plan_item(pl, c.item, T);
        c.k = c.it.k0;
    }
    return c;
}

struct UnitCoords {
    int64_t b, h, g, bh;
    int ps;
};

__device__ __forceinline__ UnitCoords unit_coords(const TcParams& p, int64_t u) {
    UnitCoords c;
    c.ps = (int)(u % p.n_ps);
    c.bh = u / p.n_ps;
    c.h = c.bh % p.H;
    c.b = c.bh / p.H;
    c.g = c.h / (p.H / p.G);
    return c;
}

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
// `wsum` must alternate between two buffers on consecutive calls (one barrier per scan).
// Also returns the sum over all earlier warps (`pre`, the prefix at row 32 * quarter - 1)
// and over the whole tile (`total`).
__device__ __forceinline__ bool wg_scan(float& v, int quarter, int lane, float* wsum,
                                        uint64_t* bar, uint32_t& phase, Small& sm,
                                        const TcParams& p, float& pre, float& total) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) wsum[quarter] = v;
    if (!wg_sync(bar, phase, sm, p)) return false;
    pre = 0.f;
    total = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float w = wsum[q];
        if (q < quarter) pre += w;
        total += w;
    }
    v += pre;
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
    const int T = p.n_tiles;
    const Plan plan = make_plan(p, blockIdx.x);

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
            int nt = 0;
            for (Cursor c = first_tile(plan, T); c.valid; c = next_tile(plan, c, T), ++nt) {
                const int s = nt % K::kStages;
                const uint32_t use = nt / K::kStages;
                if (!wait_bar(&sm.empty[s], (use & 1u) ^ 1u, sm, p)) break;
                const UnitCoords uc = unit_coords(p, c.it.u);
                const int t0 = c.k * kTile;
                // a state-only tile needs x and B; a full tile also C
                mbar_arrive_expect_tx(&sm.full[s],
                                      c.it.pass1 ? kTileBytes * (1 + K::kNReg) : K::kStageTx);
                tma_load_4d(smem + K::kOffX + s * kTileBytes, &tmX, &sm.full[s], uc.ps * kPS,
                            (int)uc.h, t0, (int)uc.b);
                for (int r = 0; r < K::kNReg; ++r) {
                    tma_load_4d(smem + K::kOffB + (s * K::kNReg + r) * kTileBytes, &tmB,
                                &sm.full[s], r * 64, (int)uc.g, t0, (int)uc.b);
                    if (!c.it.pass1)
                        tma_load_4d(smem + K::kOffC + (s * K::kNReg + r) * kTileBytes, &tmC,
                                    &sm.full[s], r * 64, (int)uc.g, t0, (int)uc.b);
                }
            }
            if (sm.abort_flag) {
                // drain: every issued load must land before the CTA's smem goes away
                const long long t0 = clock64();
                for (int j = nt - K::kStages; j < nt; ++j) {
                    if (j < 0) continue;
                    const int s = j % K::kStages;
                    const uint32_t use = j / K::kStages;
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
            // G = C B^T of tile number nt (the j-th full tile) into G buffer j % kGBuf
            auto issue_G = [&](int nt, int j) -> bool {
                const int s = nt % K::kStages;
                const int gb = j % K::kGBuf;
                if (!wait_bar(&sm.full[s], (uint32_t)(nt / K::kStages) & 1u, sm, p)) return false;
                if (!wait_bar(&sm.g_empty[gb], ((uint32_t)(j / K::kGBuf) & 1u) ^ 1u, sm, p))
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
            int nt = 0, j = 0;           // tiles issued, full (non state-only) tiles issued
            bool g_ahead = false;        // G of the current tile was issued one tile early
            for (Cursor c = first_tile(plan, T); c.valid; c = next_tile(plan, c, T), ++nt) {
                const int s = nt % K::kStages;
                const uint32_t par = (uint32_t)nt & 1u;
                const bool full_tile = !c.it.pass1;
                const Cursor nx = next_tile(plan, c, T);
                const bool next_full = nx.valid && !nx.it.pass1;
                if (full_tile && !g_ahead && !issue_G(nt, j)) break;
                g_ahead = false;
                // chunk state S^T = B^T (w o X)
                if (!wait_bar(&sm.xt_full, par, sm, p) || !wait_bar(&sm.s_empty, par ^ 1u, sm, p))
                    break;
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
                if (!full_tile) {
                    mma_commit(&sm.empty[s]);
                    continue;
                }
                const uint32_t jpar = (uint32_t)j & 1u;
                // off-diagonal Y_off = C h_prev^T
                if (!wait_bar(&sm.h_full, jpar, sm, p) || !wait_bar(&sm.y_empty, jpar ^ 1u, sm, p))
                    break;
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
                if (K::kStages > 1 && next_full) {
                    if (!issue_G(nt + 1, j + 1)) break;
                    g_ahead = true;
                }
                // Y_diag = P X
                if (!wait_bar(&sm.p_full, jpar, sm, p)) break;
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
                if (K::kStages == 1 && next_full) {
                    if (!issue_G(nt + 1, j + 1)) break;
                    g_ahead = true;
                }
                ++j;
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
        uint32_t sync_phase = 0;
        auto load_dt = [&](const Cursor& c) -> float {
            if (!c.valid) return 0.f;
            const UnitCoords uc = unit_coords(p, c.it.u);
            const int64_t t = (int64_t)c.k * kTile + r;
            return t < p.L ? __bfloat162float(p.dt[(uc.b * p.L + t) * p.H + uc.h]) : 0.f;
        };
        Cursor c = first_tile(plan, T);
        float dt_next = load_dt(c);
        int nt = 0, j = 0;
        for (; c.valid; ++nt) {
            const Cursor nx = next_tile(plan, c, T);
            const int s = nt % K::kStages;
            const uint32_t par = (uint32_t)nt & 1u;
            const bool full_tile = !c.it.pass1;
            const float dtv = dt_next;           // loaded one tile ahead
            dt_next = load_dt(nx);
            const float A2 = p.A[unit_coords(p, c.it.u).h] * kLog2e;
            float c2 = dtv * A2;                // log2-domain cumsum
            float pre, clast2;
            if (!wg_scan(c2, q, lane, sm.a_wsum[par], &sm.a_sync, sync_phase, sm, p, pre, clast2))
                break;
            if (full_tile) {
                sm.a_cp[r] = c2 - lg2(dtv);     // folds dt_j into the column term (+inf if 0)
                if (!wg_sync(&sm.a_sync, sync_phase, sm, p)) break;
            }

            // w o X for the chunk-state GEMM: row r scaled by exp(cum_last - cum_r) dt_r
            if (!wait_warp(&sm.full[s], (uint32_t)(nt / K::kStages) & 1u, sm, p)) break;
            if (!wait_warp(&sm.xt_empty, par ^ 1u, sm, p)) break;
            {
                const float wr = ex2(clast2 - c2) * dtv;
                const uint32_t xrow = sbase + K::kOffX + s * kTileBytes;
                const uint32_t xtrow = sbase + K::kOffXt;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint32_t off = sw128_off(r, cc);
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

            if (full_tile) {
                // P = L o G o dt_j (bf16, K-major swizzled), L masked before exp.
                // Below the warp's diagonal 32x32 block every L_ij factors exactly as
                // exp(cum_i - m) * exp(m - cum_j), m = cum at row 32q - 1, which lies between
                // cum_i and cum_j, so those blocks need one exponential per row and one per
                // column instead of one per element.
                const int gb = j % K::kGBuf;
                const uint32_t jpar = (uint32_t)j & 1u;
                if (!wait_warp(&sm.p_empty, jpar ^ 1u, sm, p)) break;
                if (!wait_warp(&sm.g_full[gb], (uint32_t)(j / K::kGBuf) & 1u, sm, p)) break;
                tc_fence_after();
                const uint32_t prow = sbase + K::kOffP;
                const float u_r = ex2(c2 - pre);    // exp(cum_r - m)
#pragma unroll
                for (int jb = 0; jb < 4; ++jb) {
                    const uint32_t atom = prow + (jb >> 1) * kTileBytes;
                    if (jb > q) {   // strictly above the diagonal for the whole warp
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc)
                            st_shared_v4(atom + sw128_off(r, (jb & 1) * 4 + cc), 0, 0, 0, 0);
                        continue;
                    }
                    float gv[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + K::kColG + gb * 128 + jb * 32,
                              gv);
                    if (jb < q) {
                        // column factor exp(m - cum_j) dt_j, one per lane, shared by shuffles
                        const float wl = ex2(pre - sm.a_cp[jb * 32 + lane]);
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            gv[jj] *= __shfl_sync(0xffffffffu, wl, jj) * u_r;
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            gv[jj] = (jj <= lane) ? ex2(c2 - sm.a_cp[jb * 32 + jj]) * gv[jj] : 0.f;
                    }
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        st_shared_v4(atom + sw128_off(r, (jb & 1) * 4 + cc),
                                     pack_bf16x2(gv[cc * 8 + 0], gv[cc * 8 + 1]),
                                     pack_bf16x2(gv[cc * 8 + 2], gv[cc * 8 + 3]),
                                     pack_bf16x2(gv[cc * 8 + 4], gv[cc * 8 + 5]),
                                     pack_bf16x2(gv[cc * 8 + 6], gv[cc * 8 + 7]));
                }
                tc_fence_before();
                mbar_arrive(&sm.g_empty[gb]);
                fence_proxy_async_smem();
                mbar_arrive(&sm.p_full);
                ++j;
            }
            c = nx;
        }
    } else {
        // ---------------------------------------------------------------- "B" warpgroup ---
        const int q = warp & 3;
        const int r = q * 32 + lane;             // tile row, and state row inside a 128-block
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int64_t slot_elems = (int64_t)kPS * NS;
        uint32_t sync_phase = 0;
        bool ok = true;
        auto load_dt = [&](const Cursor& c) -> float {
            if (!c.valid) return 0.f;
            const UnitCoords uc = unit_coords(p, c.it.u);
            const int64_t t = (int64_t)c.k * kTile + r;
            return t < p.L ? __bfloat162float(p.dt[(uc.b * p.L + t) * p.H + uc.h]) : 0.f;
        };
        // H (TMEM) <- scale * src + H when `accumulate`, else H <- src.  src is a [64 x N] fp32
        // block (element (p, n) at p * ld + n); nullptr means zeros.  `l2only` reads bypass L1
        // (for states another SM published).
        auto h_from = [&](const float* src, int64_t ld, float scale, bool accumulate,
                          bool l2only) {
#pragma unroll
            for (int mb = 0; mb < K::kMB; ++mb) {
                const int n = mb * 128 + r;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float v[32];
                    if (accumulate)
                        tmem_ld32(tmem + lane_base + K::kColH + mb * kPS + half * 32, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float x = 0.f;
                        if (src) {
                            const float* a = src + (int64_t)(half * 32 + i) * ld + n;
                            x = l2only ? __ldcg(a) : *a;
                        }
                        v[i] = accumulate ? fmaf(scale, x, v[i]) : x;
                    }
                    tmem_st32(tmem + lane_base + K::kColH + mb * kPS + half * 32, v);
                }
            }
        };
        // dst[p][n] <- H (fp32)
        auto h_to = [&](float* dst, int64_t ld) {
#pragma unroll
            for (int mb = 0; mb < K::kMB; ++mb) {
                const int n = mb * 128 + r;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float hv[32];
                    tmem_ld32(tmem + lane_base + K::kColH + mb * kPS + half * 32, hv);
#pragma unroll
                    for (int i = 0; i < 32; ++i) dst[(int64_t)(half * 32 + i) * ld + n] = hv[i];
                }
            }
        };
        // h^T (bf16, MN-major swizzled) <- H, for the next Y_off GEMM
        auto ht_from_h = [&]() {
#pragma unroll
            for (int mb = 0; mb < K::kMB; ++mb) {
                const int n = mb * 128 + r;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float hv[32];
                    tmem_ld32(tmem + lane_base + K::kColH + mb * kPS + half * 32, hv);
                    const uint32_t hrow = sbase + K::kOffHt;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        st_shared_v4(hrow + sw128_off(n, half * 4 + cc),
                                     pack_bf16x2(hv[cc * 8 + 0], hv[cc * 8 + 1]),
                                     pack_bf16x2(hv[cc * 8 + 2], hv[cc * 8 + 3]),
                                     pack_bf16x2(hv[cc * 8 + 4], hv[cc * 8 + 5]),
                                     pack_bf16x2(hv[cc * 8 + 6], hv[cc * 8 + 7]));
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&sm.h_full);
        };
        Cursor c = first_tile(plan, T);
        float dt_next = load_dt(c);
        int nt = 0, j = 0;
        int64_t cur_item = -1;
        float item_logd = 0.f;                   // sum of log2 tile decays over the item
        for (; c.valid && ok; ++nt) {
            const Cursor nx = next_tile(plan, c, T);
            const UnitCoords uc = unit_coords(p, c.it.u);
            const bool full_tile = !c.it.pass1;
            const int s = nt % K::kStages;
            const uint32_t par = (uint32_t)nt & 1u;
            if (c.item != cur_item) {
                // ---- start of an item: the state entering its first tile
                cur_item = c.item;
                item_logd = 0.f;
                const int64_t hbase = (uc.bh * p.P + (int64_t)uc.ps * kPS) * p.N;
                if (c.it.init == kInitZero) {
                    h_from(nullptr, p.N, 0.f, false, false);
                } else if (c.it.init == kInitH0) {
                    h_from(p.h0 ? p.h0 + hbase : nullptr, p.N, 0.f, false, false);
                } else {
                    // decoupled look-back over the preceding ranges' published states:
                    // h_in = D_1 (D_2 (... h_incl ...) + H_2) + H_1
                    h_from(nullptr, p.N, 0.f, false, false);
                    float acc_logd = 0.f;
                    int jp = (int)blockIdx.x - 1;
                    while (true) {
                        if (r == 0) {
                            int kind = 0;
                            const long long t0 = clock64();
                            while (jp >= 0 && kind == 0) {
                                if (ld_acquire_gpu(p.flags + 4 * jp + 0)) kind = 1;
                                else if (ld_acquire_gpu(p.flags + 4 * jp + 1)) kind = 2;
                                else if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) break;
                                else if (clock64() - t0 > p.budget) {
                                    flag_abort(sm, p.ws);
                                    break;
                                }
                            }
                            sm.lb_kind = kind;
                            sm.lb_logd = kind == 2 ? __int_as_float(__ldcg(p.flags + 4 * jp + 2))
                                                   : 0.f;
                        }
                        if (!wg_sync(&sm.b_sync, sync_phase, sm, p)) {
                            ok = false;
                            break;
                        }
                        const int kind = sm.lb_kind;
                        const float lb_logd = sm.lb_logd;
                        if (!wg_sync(&sm.b_sync, sync_phase, sm, p)) {   // lb_* consumed
                            ok = false;
                            break;
                        }
                        if (kind == 0) {
                            ok = false;
                            break;
                        }
                        const float* slot = p.slots + (int64_t)jp * 2 * slot_elems;
                        h_from(kind == 1 ? slot : slot + slot_elems, NS, ex2(acc_logd), true,
                               true);
                        if (kind == 1) break;
                        acc_logd += lb_logd;
                        --jp;
                    }
                    if (!ok) break;
                }
                if (full_tile) {
                    // h^T for the item's first Y_off, once the previous full tile's Y_off is done
                    if (j > 0 && !wait_warp(&sm.h_empty, (uint32_t)(j - 1) & 1u, sm, p)) break;
                    ht_from_h();
                }
            }
            const float dtv = dt_next;           // loaded one tile ahead
            dt_next = load_dt(nx);
            const float A2 = p.A[uc.h] * kLog2e;
            const float Dh = p.D ? p.D[uc.h] : 0.f;
            float c2 = dtv * A2;
            float pre, clast2;
            if (!wg_scan(c2, q, lane, sm.b_wsum[par], &sm.b_sync, sync_phase, sm, p, pre, clast2))
                break;
            const float e_r = ex2(c2);          // exp(cum_r)
            const float decay = ex2(clast2);    // exp(cum_last)
            item_logd += clast2;

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
            const bool last_of_item = !nx.valid || nx.item != c.item;

            if (full_tile) {
                const uint32_t jpar = (uint32_t)j & 1u;
                // h^T for the next tile's Y_off, once this tile's Y_off has read the old one
                if (!last_of_item) {
                    if (!wait_warp(&sm.h_empty, jpar, sm, p)) break;
                    ht_from_h();
                }
                // S4: y = Y_diag + exp(cum) Y_off + D x
                if (!wait_warp(&sm.y_full, jpar, sm, p)) break;
                if (!wait_warp(&sm.full[s], (uint32_t)(nt / K::kStages) & 1u, sm, p)) break;
                tc_fence_after();
                const int64_t t = (int64_t)c.k * kTile + r;
                const uint32_t xrow = sbase + K::kOffX + s * kTileBytes;
                __nv_bfloat16* yrow = p.y + ((uc.b * p.L + t) * p.H + uc.h) * p.P + uc.ps * kPS;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float yd[32], yo[32];
                    tmem_ld32(tmem + lane_base + K::kColY + half * 32, yd);
                    tmem_ld32(tmem + lane_base + K::kColYoff + half * 32, yo);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint4 xv = ld_shared_v4(xrow + sw128_off(r, half * 4 + cc));
                        const uint32_t xin[4] = {xv.x, xv.y, xv.z, xv.w};
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i0 = cc * 8 + e * 2;
                            const float v0 =
                                fmaf(Dh, bf16lo_to_f32(xin[e]), fmaf(e_r, yo[i0], yd[i0]));
                            const float v1 =
                                fmaf(Dh, bf16hi_to_f32(xin[e]), fmaf(e_r, yo[i0 + 1], yd[i0 + 1]));
                            o[e] = pack_bf16x2(v0, v1);
                        }
                        if (t < p.L)
                            *reinterpret_cast<uint4*>(yrow + half * 32 + cc * 8) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                tc_fence_before();
                mbar_arrive(&sm.y_empty);
                ++j;
            }
            mbar_arrive(&sm.empty[s]);

            if (last_of_item) {
                // ---- end of an item: final state, or publish for the next range
                const int fin = c.it.fin;
                if (fin == kFinFinal) {
                    if (p.hT) h_to(p.hT + (uc.bh * p.P + (int64_t)uc.ps * kPS) * p.N, p.N);
                } else if (fin == kFinIncl || fin == kFinAgg) {
                    float* slot = p.slots + (int64_t)blockIdx.x * 2 * slot_elems +
                                  (fin == kFinAgg ? slot_elems : 0);
                    h_to(slot, NS);
                    __threadfence();
                    if (!wg_sync(&sm.b_sync, sync_phase, sm, p)) break;
                    if (r == 0) {
                        if (fin == kFinAgg)
                            st_relaxed_gpu(p.flags + 4 * blockIdx.x + 2, __float_as_int(item_logd));
                        st_release_gpu(p.flags + 4 * blockIdx.x + (fin == kFinAgg ? 1 : 0), 1);
                    }
                }
            }
            c = nx;
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

size_t flags_bytes() { return align_up(sizeof(int) * 4 * kMaxCtas, 256); }
size_t slots_bytes(int64_t N) { return sizeof(float) * 2 * (size_t)kMaxCtas * kPS * (size_t)N; }

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return -1;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

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
    // Without a state-only pass, a range's head piece is published before its successor's
    // tail piece is needed as long as every range is longer than a chain.
    p.pass1_mode = (total / p.n_ctas) > p.n_tiles ? 0 : 1;
    p.dt = static_cast<const __nv_bfloat16*>(a.dt);
    p.A = a.A; p.D = a.D; p.h0 = a.h0;
    p.y = static_cast<__nv_bfloat16*>(a.y);
    p.hT = a.hT;
    p.ws = a.ws;
    p.flags = reinterpret_cast<int*>(a.ws + kWsHeaderBytes);
    p.slots = reinterpret_cast<float*>(a.ws + kWsHeaderBytes + flags_bytes());
    p.budget = 4ll << 30;   // ~2 s at the B300's maximum SM clock
    if (cudaMemsetAsync(p.flags, 0, sizeof(int) * 4 * (size_t)p.n_ctas, a.stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    const size_t smem = smem_bytes<NS>();
    if (cudaFuncSetAttribute(ssd_tc_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return SSD_ERR_CUDA;
    ssd_tc_kernel<NS><<<(unsigned)p.n_ctas, kThreads, smem, a.stream>>>(tmX, tmB, tmC, p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

bool tc_supports(int32_t dtype, int64_t P, int64_t N, int Q) {
    return dtype == SSD_BF16 && P % kPS == 0 && (N == 128 || N == 256) && Q % 64 == 0;
}

size_t tc_workspace_bytes(int64_t, int64_t, int64_t, int64_t, int64_t N, int) {
    return kWsHeaderBytes + flags_bytes() + slots_bytes(N);
}

int tc_launch(const ScanArgs& a) {
    if (a.batch * a.nheads * (a.headdim / kPS) > 0x7fffffffLL || a.seqlen > 0x7fffffffLL)
        return SSD_ERR_UNSUPPORTED;
    if (a.dstate == 128) return launch_ns<128>(a);
    if (a.dstate == 256) return launch_ns<256>(a);
    return SSD_ERR_UNSUPPORTED;
}

}  // namespace ssd
