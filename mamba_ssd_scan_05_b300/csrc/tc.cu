// tc.cu -- the tensor-core path: one fused, warp-specialised, persistent sm_103a kernel per scan.
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
// Warp roles (384 threads; the producer warpgroup runs with 72 registers per thread so that
// the compute warpgroups get 216):
//   warp 0      TMA producer of the B / C ring (2 stages for d_state 128)
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer
//   warp 2      producer of the x / decay ring: TMA of the x tile, and from dt the tile's
//               log2-domain cumsum and every exponential factor the other roles need
//   warp 3      idle (completes the producer warpgroup)
//   warps 4-11  two identical compute warpgroups; warpgroup g (warps 4+4g .. 7+4g) owns
//               headdim columns 32g .. 32g+31 of x, the state and y, and half of P's column
//               blocks.  Per tile: scaled copy of x for the state GEMM, its P blocks, the
//               state recurrence in registers and bf16 h^T for the next off-diagonal GEMM;
//               the y epilogue of a tile runs one tile later, so the tensor core never
//               waits for it (Y and Y_off are double-buffered in TMEM)
// Every wait is bounded (clock64 budget); a timeout sets SSD_ERR_TIMEOUT in the workspace
// status word, makes every role stop, drains in-flight copies and frees TMEM before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "tc_plan.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace ptx;
using namespace plan;

constexpr int kTile = 128;          // tokens per tile (MMA M)
constexpr int kPS = 64;             // headdim columns per unit (MMA N of Y, Y_off, S)
// warps 0-3: producers (warp 3 idle); warps 4 ...: compute warpgroups
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpDt = 2, kWarpC = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTileBytes = kTile * 128;   // a 128-row x 128-byte swizzled tile (16 KB)
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxCtas = 256;       // grid cap (and number of hand-off slots in the workspace)
constexpr int kXStagesMax = 3;      // x / decay ring depth (at most)

// Per-tile decay factors (log2 domain: cum2 = cum * log2(e)), written by the decay producer.
struct DtSlot {
    float cum2[kTile];      // inclusive cumsum of dt * A * log2(e) inside the tile
    float pcol[kTile];      // cum2 - log2(dt) (+inf where dt = 0): column term of L o dt
    float w[kTile];         // exp2(cum2_last - cum2) * dt: decay to the tile end, times dt
    float e[kTile];         // exp2(cum2): decay from the tile start (off-diagonal rows)
    float urow[kTile];      // exp2(cum2 - m_q), m_q = cum2[32 q - 1], q = row / 32 >= 1
    float colf[3][kTile];   // exp2(m_q - pcol), q = 1..3 (used for columns j < 32 q)
    float rd[kTile];        // exp2(cum2 - d_q), d_q = cum2[32 q + 15]: diagonal-block row factor
    float cd[kTile];        // exp2(d_q - pcol): diagonal-block column factor
    float clast2;           // cum2[kTile - 1]
    int dfac[3];            // bit q: the diagonal block of quarter q uses rd / cd (its decay
                            // range is small enough for both factors to stay in fp32 range)
};

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
    // TMEM columns
    static constexpr uint32_t kColG = 0;                       // C B^T, fp32, 128 columns
    static constexpr uint32_t kColP = 128;                     // P, bf16 pairs, 64 columns
    static constexpr uint32_t kColY = 192;                     // Y_diag, kYBuf x 64
    static constexpr uint32_t kColYoff = kColY + kYBuf * kPS;  // Y_off, kYBuf x 64
    static constexpr uint32_t kColS = kColYoff + kYBuf * kPS;  // S^T, kMB x 64
    static_assert(kColS + kMB * kPS <= kTmemCols, "TMEM budget");
    static_assert(kXSt <= kXStagesMax, "x ring");
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
    int* flags;         // per CTA and compute warp: inclusive flag, aggregate flag, log2 decay
    float* slots;       // per CTA: inclusive state [64 x N], then aggregate state [64 x N]
    long long budget;   // clock64 cycles a single wait may take
};

struct Small {
    uint64_t x_full[kXStagesMax], x_empty[kXStagesMax];   // x tile + decay slot
    uint64_t bc_full[2], bc_empty[2];                      // B / C tiles
    uint64_t g_full, g_empty;       // C B^T written / read by the P builders
    uint64_t p_full, p_empty;       // P written / read by Y_diag
    uint64_t xt_full, xt_empty, s_full, s_empty, h_full, h_empty;
    uint64_t y_full[2], y_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    Plan plan;
    int uc_u0[6], uc_u1[6], uc_flo[6];   // coordinates of the plan's anchor units
};

__device__ __forceinline__ Plan make_plan(const TcParams& p, int cta) {
    return plan::make_plan(p.n_units, p.n_tiles, p.n_ctas, p.pass1_mode, cta);
}

struct UnitCoords {
    int b, h, g, bh, ps;
    int hr;             // h % (H / G): position of h inside its group
};

// Coordinates of unit u (divisions: computed once per CTA, for the plan's anchor units).
__device__ __forceinline__ UnitCoords unit_coords(const TcParams& p, int u) {
    const int H = (int)p.H, R = (int)(p.H / p.G);
    UnitCoords c;
    c.ps = u % p.n_ps;
    c.bh = u / p.n_ps;
    c.h = c.bh % H;
    c.b = c.bh / H;
    c.g = c.h / R;
    c.hr = c.h % R;
    return c;
}

// Coordinates of unit u + 1 from those of u (no divisions).
__device__ __forceinline__ void next_unit(UnitCoords& c, const TcParams& p) {
    if (++c.ps < p.n_ps) return;
    c.ps = 0;
    ++c.bh;
    ++c.h;
    if (++c.hr == (int)(p.H / p.G)) {
        c.hr = 0;
        ++c.g;
    }
    if (c.h == (int)p.H) {
        c.h = 0;
        c.g = 0;
        c.hr = 0;
        ++c.b;
    }
}

// Position in a CTA's sequence of tiles; the unit's coordinates are refreshed only when the
// item changes.
struct Cursor {
    int item;
    int k;
    bool valid;
    Item it;
    UnitCoords uc;
};

// Coordinates of an item's unit: one of the plan's anchors (u0, u1, f_lo), else the unit after
// the previous item's (whole chains run in unit order).
__device__ __forceinline__ void item_coords(Cursor& c, const Plan& pl, const Small& sm,
                                            int prev_u, const TcParams& p) {
    const int* a = c.it.u == pl.u0
                       ? sm.uc_u0
                       : (c.it.u == pl.u1 ? sm.uc_u1 : (c.it.u == pl.f_lo ? sm.uc_flo : nullptr));
    if (a) {
        c.uc = UnitCoords{a[0], a[1], a[2], a[3], a[4], a[5]};
    } else if (c.it.u != prev_u) {
        next_unit(c.uc, p);
    }
}

__device__ __forceinline__ Cursor first_tile(const Plan& pl, const Small& sm, const TcParams& p) {
    Cursor c;
    c.item = 0;
    c.valid = pl.n_items > 0;
    c.it = plan_item(pl, 0, p.n_tiles);
    c.k = c.it.k0;
    c.uc = UnitCoords{0, 0, 0, 0, 0, 0};
    item_coords(c, pl, sm, -1, p);
    return c;
}

__device__ __forceinline__ void advance(Cursor& c, const Plan& pl, const Small& sm,
                                        const TcParams& p) {
    if (!c.valid) return;
    if (c.k + 1 < c.it.k1) {
        ++c.k;
        return;
    }
    ++c.item;
    c.valid = c.item < pl.n_items;
    if (c.valid) {
        const int prev_u = c.it.u;
        c.it = plan_item(pl, c.item, p.n_tiles);
        c.k = c.it.k0;
        item_coords(c, pl, sm, prev_u, p);
    }
}

// advance for the producer roles: the item change is one out-of-line copy.
__device__ __noinline__ Cursor next_item(Cursor c, const Plan* pl, const Small* sm,
                                         const TcParams* p) {
    advance(c, *pl, *sm, *p);
    return c;
}
__device__ __forceinline__ void advance_p(Cursor& c, const Plan& pl, const Small& sm,
                                          const TcParams& p) {
    if (__builtin_expect(c.valid && c.k + 1 < c.it.k1, 1)) {
        ++c.k;
        return;
    }
    c = next_item(c, &pl, &sm, &p);
}

__device__ __forceinline__ void flag_abort(Small& sm, uint8_t* ws) {
    *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
    set_status(ws, SSD_ERR_TIMEOUT);
}

// Bounded wait for the completion of the phase with `parity`.  False on timeout or abort.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Small& sm,
                                         const TcParams& p) {
    if (__builtin_expect(mbar_try_wait(bar, parity), 1)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (__builtin_expect(*reinterpret_cast<volatile int*>(&sm.abort_flag), 0)) return false;
        if (__builtin_expect(clock64() - t0 > p.budget, 0)) {
            flag_abort(sm, p.ws);
            return false;
        }
    }
    return true;
}

// wait_bar for the single-lane producer roles: the slow path is one out-of-line copy (a call
// is cheap there, with few live registers), which keeps their hot code small.
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, Small* sm,
                                           const TcParams* p) {
    return wait_bar(bar, parity, *sm, *p);
}
__device__ __forceinline__ bool wait_bar_p(uint64_t* bar, uint32_t parity, Small& sm,
                                           const TcParams& p) {
    if (__builtin_expect(mbar_try_wait(bar, parity), 1)) return true;
    return wait_bar_slow(bar, parity, &sm, &p);
}

// wait_bar for the 32 lanes of a warp, with one verdict for the whole warp, so the warp stays
// converged for the .sync.aligned TMEM instructions that follow.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, Small& sm,
                                          const TcParams& p) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, sm, p));
}

// wait_warp for a producer role run by a whole warp, with the slow path out of line.
__device__ __forceinline__ bool wait_warp_p(uint64_t* bar, uint32_t parity, Small& sm,
                                            const TcParams& p) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__builtin_expect(__all_sync(0xffffffffu, ok), 1)) return true;
    return __all_sync(0xffffffffu, ok || wait_bar_slow(bar, parity, &sm, &p));
}

// One 32 x 32 block (rows 32q .. 32q+31, columns 32jb .. 32jb+31) of P = L o G o dt_j for this
// lane's row: g holds G's block (read from TMEM by the caller); the bf16 pairs go to pk.  Strictly
// below the diagonal block every L_ij factors exactly as exp(cum_i - m) exp(m - cum_j) with
// m = cum at row 32q - 1 (between cum_i and cum_j), so the block needs no exponential; the
// diagonal block is masked before the exponential.  (Blocks above the diagonal are zero and
// are written once, at kernel start.)
__device__ __forceinline__ void p_block(uint32_t (&pk)[16], float (&g)[32], int jb, int q, int lane,
                                        int r, const DtSlot& sl) {
    if (jb < q) {
        const float ur = sl.urow[r];
        const float4* cf = reinterpret_cast<const float4*>(&sl.colf[q - 1][jb * 32]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 c = cf[i];
            g[4 * i + 0] *= c.x * ur;
            g[4 * i + 1] *= c.y * ur;
            g[4 * i + 2] *= c.z * ur;
            g[4 * i + 3] *= c.w * ur;
        }
    } else if (__builtin_expect((sl.dfac[0] >> q) & 1, 1)) {
        // diagonal block with factors around its middle row: L_ij dt_j = rd_i cd_j (j <= i)
        const float rr = sl.rd[r];
        const float4* cf = reinterpret_cast<const float4*>(&sl.cd[jb * 32]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 c = cf[i];
            const float cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int jj = 4 * i + e;
                g[jj] = (jj <= lane) ? g[jj] * cv[e] * rr : 0.f;
            }
        }
    } else {
        const float c2 = sl.cum2[r];
        const float4* pc = reinterpret_cast<const float4*>(&sl.pcol[jb * 32]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 c = pc[i];
            const float cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int jj = 4 * i + e;
                g[jj] = (jj <= lane) ? ex2(c2 - cv[e]) * g[jj] : 0.f;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(g[2 * i], g[2 * i + 1]);
}

// ---- the state in registers of the compute threads -------------------------------------------
// Compute thread (row r, column block c0) holds h^T rows n = 128 mb + r, columns
// p = c0 .. c0 + CW - 1 (CW headdim columns per compute warpgroup).

// h <- scale * src + h when `accumulate`, else h <- src.  src is a [64 x NS] fp32 block
// (element (p, n) at p * NS + n: the state layout, whose row length is d_state); nullptr means
// zeros.  `l2only` reads bypass L1 (for states another SM published).  The element offsets
// are compile-time constants from one base address.
template <int NS, int CW>
__device__ __forceinline__ void h_from(float (&h)[NS / 128 * CW], const float* src, int r, int c0,
                                       float scale, bool accumulate, bool l2only) {
    if (!src) {
#pragma unroll
        for (int i = 0; i < NS / 128 * CW; ++i) h[i] = accumulate ? h[i] : 0.f;
        return;
    }
    const float* base = src + (int64_t)c0 * NS + r;
#pragma unroll
    for (int mb = 0; mb < NS / 128; ++mb)
#pragma unroll
        for (int i = 0; i < CW; ++i) {
            const float* a = base + i * NS + mb * 128;
            const float x = l2only ? __ldcg(a) : *a;
            h[mb * CW + i] = accumulate ? fmaf(scale, x, h[mb * CW + i]) : x;
        }
}

// dst[p][n] <- h (fp32), dst a [64 x NS] block with rows of d_state elements
template <int NS, int CW>
__device__ __forceinline__ void h_to(const float (&h)[NS / 128 * CW], float* dst, int r, int c0) {
    float* base = dst + (int64_t)c0 * NS + r;
#pragma unroll
    for (int mb = 0; mb < NS / 128; ++mb)
#pragma unroll
        for (int i = 0; i < CW; ++i) base[i * NS + mb * 128] = h[mb * CW + i];
}

// bf16 h^T into the MN-major, 128-byte swizzled tile (N rows x 64 columns) at ht: the B operand
// of the next off-diagonal GEMM.
// wg is the thread's column block (its 16-byte chunks are wg * CW / 8 ...).
template <int NS, int CW>
__device__ __forceinline__ void ht_write(const float (&h)[NS / 128 * CW], uint8_t* ht, int r,
                                         int wg) {
#pragma unroll
    for (int mb = 0; mb < NS / 128; ++mb)
#pragma unroll
        for (int cc = 0; cc < CW / 8; ++cc) {
            const float* v = &h[mb * CW + cc * 8];
            *reinterpret_cast<uint4*>(ht + sw128_off(mb * 128 + r, wg * (CW / 8) + cc)) =
                make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                           pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
        }
}

// Flags of the state hand-off between CTAs, per CTA and per compute warp w (the warp that owns
// state rows 32q .. 32q+31 of every 128-row block and one column block): [0] inclusive state
// published, [1] aggregate published, [2] the aggregate's log2 decay.  A warp only needs the
// same part of its predecessor's state, so publishing and looking back are per warp.
constexpr int kFlagsPerCta = 64;   // 4 words for each of up to 16 compute warps

// Decoupled look-back over the preceding ranges' published states (per compute warp):
//     h_in = D_1 (D_2 (... h_incl ...) + H_2) + H_1.
// False on timeout or abort.
template <int NS, int CW>
__device__ __forceinline__ bool look_back(float (&h)[NS / 128 * CW], const TcParams& p, Small& sm,
                                          int w, int lane, int r, int c0) {
    const int64_t slot_elems = (int64_t)kPS * NS;
    h_from<NS, CW>(h, nullptr, r, c0, 0.f, false, false);
    float acc_logd = 0.f;
#pragma unroll 1
    for (int jp = (int)blockIdx.x - 1; jp >= 0; --jp) {
        const int* f = p.flags + jp * kFlagsPerCta + w * 4;
        int kind = 0;
        if (lane == 0) {
            const long long t0 = clock64();
            while (kind == 0) {
                if (ld_acquire_gpu(f + 0)) kind = 1;
                else if (ld_acquire_gpu(f + 1)) kind = 2;
                else if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) break;
                else if (clock64() - t0 > p.budget) {
                    flag_abort(sm, p.ws);
                    break;
                }
            }
        }
        kind = __shfl_sync(0xffffffffu, kind, 0);
        if (kind == 0) return false;
        // every lane acquires the flag itself before it reads the published state
        (void)ld_acquire_gpu(f + kind - 1);
        const float* slot = p.slots + (int64_t)jp * 2 * slot_elems + (kind == 2 ? slot_elems : 0);
        h_from<NS, CW>(h, slot, r, c0, ex2(acc_logd), true, true);
        if (kind == 1) return true;
        acc_logd += __int_as_float(__ldcg(f + 2));
    }
    return false;   // no inclusive state before this range: cannot happen for a valid plan
}

// This warp's part of the CTA's inclusive state (kFinIncl) or aggregate (kFinAgg), published
// for the next range.
template <int NS, int CW>
__device__ __forceinline__ void publish(const float (&h)[NS / 128 * CW], const TcParams& p, int w,
                                        int lane, int r, int c0, int fin, float item_logd) {
    const int64_t slot_elems = (int64_t)kPS * NS;
    float* slot = p.slots + (int64_t)blockIdx.x * 2 * slot_elems + (fin == kFinAgg ? slot_elems : 0);
    h_to<NS, CW>(h, slot, r, c0);
    __threadfence();
    __syncwarp();
    if (lane == 0) {
        int* f = p.flags + (int)blockIdx.x * kFlagsPerCta + w * 4;
        if (fin == kFinAgg) st_relaxed_gpu(f + 2, __float_as_int(item_logd));
        st_release_gpu(f + (fin == kFinAgg ? 1 : 0), 1);
    }
    __syncwarp();
}

// A tile whose y epilogue is deferred by one tile (always the previous full tile).
template <int CW>
struct PendingY {
    __nv_bfloat16* row;     // y row at this thread's column block, or null past the sequence end
    float e;                // exp(cum) of the row
    float d;                // D of the head
    uint4 x[CW / 8];        // x row, this thread's column block (bf16 pairs)
};

// CW consecutive fp32 TMEM columns at ta and at tb, one wait for both
template <int CW>
__device__ __forceinline__ void tmem_ld_pair(uint32_t ta, float (&va)[CW], uint32_t tb,
                                             float (&vb)[CW]) {
    if constexpr (CW == 32) tmem_ld32x2(ta, va, tb, vb);
    else tmem_ld16x2(ta, va, tb, vb);
}
template <int CW>
__device__ __forceinline__ void tmem_ld_cols(uint32_t ta, float (&v)[CW]) {
    if constexpr (CW == 32) tmem_ld32(ta, v);
    else tmem_ld16(ta, v);
}

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
                const long long t0 = clock64();
                for (int j = nt - K::kBCStages; j < nt; ++j) {
                    if (j < 0) continue;
                    const int s = j % K::kBCStages;
                    const uint32_t use = j / K::kBCStages;
                    while (!mbar_try_wait(&sm.bc_full[s], use & 1u) &&
                           clock64() - t0 < p.budget) {
                    }
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
            // log2-domain cumsum: 4 consecutive tokens per lane, then a warp scan
            float cs[4];
            cs[0] = d0[0] * A2;
#pragma unroll
            for (int i = 1; i < 4; ++i) cs[i] = fmaf(d0[i], A2, cs[i - 1]);
            float incl = cs[3];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            float excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0) excl = 0.f;
            const float clast2 = __shfl_sync(0xffffffffu, incl, 31);
            const float m1 = __shfl_sync(0xffffffffu, incl, 7);    // cum2 at token 31
            const float m2 = __shfl_sync(0xffffffffu, incl, 15);   // token 63
            const float m3 = __shfl_sync(0xffffffffu, incl, 23);   // token 95
            const int q = lane >> 3;
            const float mq = q == 1 ? m1 : (q == 2 ? m2 : m3);
            // middle of this lane's 32-token block (token 32 q + 15 = lane 8 q + 3, entry 3)
            const float dq = __shfl_sync(0xffffffffu, incl, 8 * q + 3);
            // decay range of each 32-token block, in log2 units (cum2 is non-increasing)
            const float blk_first = __shfl_sync(0xffffffffu, excl + cs[0], 8 * q);
            const float blk_last = __shfl_sync(0xffffffffu, incl, 8 * q + 7);
            DtSlot& sl = slots[s];
            const int o = 4 * lane;
            float c2[4], pc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                c2[i] = excl + cs[i];
                pc[i] = d0[i] > 0.f ? c2[i] - lg2(d0[i]) : __int_as_float(0x7f800000);
            }
            // each factor is stored as soon as its four values exist (few live registers)
            auto put = [&](float* dst, auto f) {
                *reinterpret_cast<float4*>(dst + o) = make_float4(f(0), f(1), f(2), f(3));
            };
            put(sl.cum2, [&](int i) { return c2[i]; });
            put(sl.pcol, [&](int i) { return pc[i]; });
            put(sl.w, [&](int i) { return ex2(clast2 - c2[i]) * d0[i]; });
            put(sl.e, [&](int i) { return ex2(c2[i]); });
            put(sl.urow, [&](int i) { return q > 0 ? ex2(c2[i] - mq) : 1.f; });
            put(sl.colf[0], [&](int i) { return ex2(m1 - pc[i]); });
            put(sl.colf[1], [&](int i) { return ex2(m2 - pc[i]); });
            put(sl.colf[2], [&](int i) { return ex2(m3 - pc[i]); });
            put(sl.rd, [&](int i) { return ex2(c2[i] - dq); });
            put(sl.cd, [&](int i) { return ex2(dq - pc[i]); });
            // |cum2_i - d_q| and |d_q - cum2_j| stay below 100 when the block's range does;
            // dt <= 2^20 keeps cd below 2^120
            const unsigned small = __ballot_sync(0xffffffffu, (lane & 7) == 0 &&
                                                                  blk_first - blk_last < 100.f &&
                                                                  blk_first - blk_last >= 0.f);
            if (lane == 0) {
                sl.clast2 = clast2;
                sl.dfac[0] = (int)((small & 1u) | ((small >> 8) & 1u) << 1 |
                                   ((small >> 16) & 1u) << 2 | ((small >> 24) & 1u) << 3);
            }
            mbar_arrive(&sm.x_full[s]);
        }
        if (sm.abort_flag && lane == 0) {
            // drain: the x loads of every tile this loop completed must land before exit
            const long long t0 = clock64();
            for (int j = nt - K::kXSt; j < nt; ++j) {
                if (j < 0) continue;
                const int s = j % K::kXSt;
                const uint32_t use = j / K::kXSt;
                while (!mbar_try_wait(&sm.x_full[s], use & 1u) && clock64() - t0 < p.budget) {
                }
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
            const long long t0 = clock64();
            while (!mbar_try_wait(&sm.mma_done, 0) && clock64() - t0 < p.budget) {
            }
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
                    if (!look_back<NS, CW>(h, p, sm, w, lane, r, c0)) { ok = false; break; }
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
static_assert(smem_bytes<128>() <= 232448 && smem_bytes<256>() <= 232448, "shared memory");

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

size_t flags_bytes() { return align_up(sizeof(int) * kFlagsPerCta * kMaxCtas, 256); }
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
