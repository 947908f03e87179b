// tc_common.cuh -- pieces shared by the tensor-core scan kernels (tc.cu: d_state 256,
// tc128.cu: d_state 128): tile constants, the per-tile decay factors, kernel parameters and
// barriers, the work-plan cursor, bounded waits, the P-block builder, the register-held state
// and its cross-CTA hand-off, and the host-side tensor-map / grid helpers.  Internal to
// libssd_scan.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "tc_plan.cuh"
#include "tc_ptx.cuh"
// Timing hook for profiling builds: a no-op unless the build defines
// SSD_TC_TRACE_POINT(event, tile) (then it records a per-role clock64 timeline).
#ifndef SSD_TC_TRACE_POINT
#define SSD_TC_TRACE_POINT(event, tile) ((void)0)
#endif

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
// The slots sit back to back in shared memory and their arrays are read and written as float4,
// so the struct is padded to a multiple of 16 bytes.
struct alignas(16) DtSlot {
    float cum2[kTile];      // inclusive cumsum of dt * A * log2(e) inside the tile
    float lgdt[kTile];      // log2(dt) (-inf where dt = 0): column term of L o dt
    float w[kTile];         // exp2(cum2_last - cum2) * dt: decay to the tile end, times dt
                            // (factored mode: 2^(m - cum2) dt)
    float e[kTile];         // exp2(cum2): decay from the tile start (off-diagonal rows)
                            // (factored mode: 2^(cum2 - m))
    float urow[kTile];      // exp2(cum2 - m_q), m_q = cum2[32 q - 1], q = row / 32 >= 1
    float colf[3][kTile];   // exp2((m_q - cum2) + lgdt), q = 1..3 (for columns j < 32 q)
    float rd[kTile];        // exp2(cum2 - d_q), d_q = cum2[32 q + 15]: diagonal-block row factor
    float cd[kTile];        // exp2((d_q - cum2) + lgdt): diagonal-block column factor
    float clast2;           // cum2[kTile - 1]
    int dfac[3];            // bit q: the diagonal block of quarter q uses rd / cd (its decay
                            // range is small enough for both factors to stay in fp32 range)
    // Factored mode (filled when fill_dt_slot is asked for it; else fac = 0): the whole tile's
    // decay from its start stays within 2^-160 and every dt <= 2^20, so with the reference
    // m = round(cum2_last / 2) every factor below lies in [2^-100, 2^100] and
    //   L_ij dt_j = 2^(cum2_i - m) * 2^(m - cum2_j) dt_j:
    // w holds 2^(m - cum2_j) dt_j (the column factor of x), e holds 2^(cum2_i - m) (the row
    // factor of the output), sigma = 2^(cum2_last - m) turns the state GEMM of the scaled x
    // into the chunk state, and hsc = 2^m scales h^T for the off-diagonal GEMM, so that the
    // diagonal and off-diagonal terms share one accumulator.
    int fac;
    float sigma;
    float hsc;
};
static_assert(sizeof(DtSlot) % 16 == 0 && alignof(DtSlot) == 16, "DtSlot arrays need 16-byte alignment");

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
    // the gated RMSNorm applied in the epilogue (the kernel instance that fuses it): z as y,
    // the norm weight [H * P] (or null), eps, and the group size (8, 16, 32 or 64 features)
    const __nv_bfloat16* z;
    const float* nw;
    float eps;
    int gsize;
};

struct Small {
    uint64_t x_full[kXStagesMax], x_empty[kXStagesMax];   // x tile + decay slot
    uint64_t bc_full[2], bc_empty[2];                      // B / C tiles
    uint64_t g_full, g_empty;       // C B^T written / read by the P builders
    uint64_t p_full, p_empty;       // P written / read by Y_diag
    uint64_t xt_full, xt_empty, s_full, s_empty, h_full, h_empty;
    uint64_t y_full[2], y_empty[2];
    uint64_t pb_empty[2];           // P buffer free (double-buffered P)
    uint64_t yoff_empty;            // separate off-diagonal accumulator free (fallback tiles)
    uint64_t red_bar[4];            // per TMEM lane quarter: the fused norm's row sums exchanged
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

template <bool kExt = false>
__device__ __forceinline__ Cursor first_tile(const Plan& pl, const Small& sm, const TcParams& p) {
    Cursor c;
    c.item = 0;
    c.valid = pl.n_items > 0;
    c.it = plan_item<kExt>(pl, 0, p.n_tiles);
    c.k = c.it.k0;
    c.uc = UnitCoords{0, 0, 0, 0, 0, 0};
    item_coords(c, pl, sm, -1, p);
    return c;
}

template <bool kExt = false>
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
        c.it = plan_item<kExt>(pl, c.item, p.n_tiles);
        c.k = c.it.k0;
        item_coords(c, pl, sm, prev_u, p);
    }
}

// advance for the producer roles: the item change is one out-of-line copy.
template <bool kExt = false>
__device__ __noinline__ Cursor next_item(Cursor c, const Plan* pl, const Small* sm,
                                         const TcParams* p) {
    advance<kExt>(c, *pl, *sm, *p);
    return c;
}
template <bool kExt = false>
__device__ __forceinline__ void advance_p(Cursor& c, const Plan& pl, const Small& sm,
                                          const TcParams& p) {
    if (__builtin_expect(c.valid && c.k + 1 < c.it.k1, 1)) {
        ++c.k;
        return;
    }
    c = next_item<kExt>(c, &pl, &sm, &p);
}

// Limit of the waits that run after an abort (issued TMA loads landing, issued MMAs
// completing): fixed and generous, independent of the wait budget that may have triggered the
// abort, so that an aborting CTA does not release shared memory or TMEM that is still being
// written.  A drain that gives up anyway records SSD_ERR_TIMEOUT.
constexpr long long kDrainCycles = 4ll << 30;   // ~2 s at the B300's maximum SM clock

// Drain wait (single thread): true once the phase with `parity` has completed.
__device__ __noinline__ bool drain_wait(uint64_t* bar, uint32_t parity, uint8_t* ws) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kDrainCycles) {
            set_status(ws, SSD_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
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

// The decay producer's per-tile work (one warp, lane l holds tokens 4l .. 4l + 3 of the tile,
// d0 their dt): the log2-domain inclusive cumsum of dt * A * log2(e) and every factor of the
// decay mask and of the state / off-diagonal terms, stored into the tile's DtSlot.  With
// kFactored, tiles that allow it get the factored-mode w, e, sigma and hsc (see DtSlot).
template <bool kFactored>
__device__ __forceinline__ void fill_dt_slot(DtSlot& sl, const float (&d0)[4], float A2,
                                             int lane) {
    // log2-domain cumsum: 4 consecutive tokens per lane, then a warp scan, in 64-bit fixed
    // point (units of 2^-32).  Integer addition is associative, so every scan order gives the
    // same prefix sums: a run of dt = 0 tokens keeps an identical cumsum on both sides of a
    // lane boundary, which a float32 tree scan does not guarantee.  Each token's term is
    // clamped to [-2^23, 2^23] (a decay beyond 2^-(2^23) per token is 0 either way) so that
    // a tile's sum stays inside the 64-bit range.  Every exponent below is a difference of two
    // of the per-token values (plus log2(dt), added last); the reference points (tile end,
    // block starts and middles) are taken from the very same values, so a difference of equal
    // tokens, or of tokens separated only by dt = 0, is exactly 0.
    long long cs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = fminf(fmaxf(d0[i] * A2, -8388608.f), 8388608.f);
        const long long qa = __float2ll_rn(a * 4294967296.f);
        cs[i] = i == 0 ? qa : cs[i - 1] + qa;
    }
    long long incl = cs[3];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    long long excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0;
    float c2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c2[i] = __ll2float_rn(excl + cs[i]) * 2.3283064365386963e-10f;
    const float clast2 = __shfl_sync(0xffffffffu, c2[3], 31);
    const int o = 4 * lane;
    // each factor is stored as soon as its four values exist (few live registers)
    auto put = [&](float* dst, auto f) {
        *reinterpret_cast<float4*>(dst + o) = make_float4(f(0), f(1), f(2), f(3));
    };
    if constexpr (kFactored) {
        float tmax = fmaxf(fmaxf(d0[0], d0[1]), fmaxf(d0[2], d0[3]));
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, m));
        // (false for NaN); warp-uniform
        if (clast2 >= -160.f && clast2 <= 0.f && tmax <= 1048576.f) {
            // factored tile: only w, e, sigma and hsc are read
            const int mi = __float2int_rn(0.5f * clast2);            // -80 .. 0
            const float mf = (float)mi;
            put(sl.w, [&](int i) { return ex2(mf - c2[i]) * d0[i]; });
            put(sl.e, [&](int i) { return ex2(c2[i] - mf); });
            if (lane == 0) {
                sl.fac = 1;
                sl.sigma = ex2(clast2 - mf);
                sl.hsc = __int_as_float((mi + 127) << 23);           // 2^m, exact
                sl.clast2 = clast2;
            }
            return;
        }
    }
    float lg[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) lg[i] = d0[i] > 0.f ? lg2(d0[i]) : -__int_as_float(0x7f800000);
    const float m1 = __shfl_sync(0xffffffffu, c2[3], 7);    // cum2 at token 31
    const float m2 = __shfl_sync(0xffffffffu, c2[3], 15);   // token 63
    const float m3 = __shfl_sync(0xffffffffu, c2[3], 23);   // token 95
    const int q = lane >> 3;
    const float mq = q == 1 ? m1 : (q == 2 ? m2 : m3);
    // middle of this lane's 32-token block (token 32 q + 15 = lane 8 q + 3, entry 3)
    const float dq = __shfl_sync(0xffffffffu, c2[3], 8 * q + 3);
    // decay range of each 32-token block, in log2 units (cum2 is non-increasing)
    const float blk_first = __shfl_sync(0xffffffffu, c2[0], 8 * q);
    const float blk_last = __shfl_sync(0xffffffffu, c2[3], 8 * q + 7);
    put(sl.cum2, [&](int i) { return c2[i]; });
    put(sl.lgdt, [&](int i) { return lg[i]; });
    put(sl.w, [&](int i) { return ex2(clast2 - c2[i]) * d0[i]; });
    put(sl.e, [&](int i) { return ex2(c2[i]); });
    if (lane == 0) {
        sl.fac = 0;
        sl.sigma = 1.f;
        sl.hsc = 1.f;
    }
    put(sl.urow, [&](int i) { return q > 0 ? ex2(c2[i] - mq) : 1.f; });
    put(sl.colf[0], [&](int i) { return ex2((m1 - c2[i]) + lg[i]); });
    put(sl.colf[1], [&](int i) { return ex2((m2 - c2[i]) + lg[i]); });
    put(sl.colf[2], [&](int i) { return ex2((m3 - c2[i]) + lg[i]); });
    put(sl.rd, [&](int i) { return ex2(c2[i] - dq); });
    put(sl.cd, [&](int i) { return ex2((dq - c2[i]) + lg[i]); });
    // |cum2_i - d_q| and |d_q - cum2_j| stay below 100 when the block's range does, and
    // dt <= 2^20 keeps cd below 2^120: blocks that meet both use the factored form
    float dmax = fmaxf(fmaxf(d0[0], d0[1]), fmaxf(d0[2], d0[3]));
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, m));
    const unsigned small = __ballot_sync(0xffffffffu, (lane & 7) == 0 &&
                                                          blk_first - blk_last < 100.f &&
                                                          blk_first - blk_last >= 0.f &&
                                                          dmax <= 1048576.f);
    if (lane == 0) {
        sl.clast2 = clast2;
        sl.dfac[0] = (int)((small & 1u) | ((small >> 8) & 1u) << 1 |
                           ((small >> 16) & 1u) << 2 | ((small >> 24) & 1u) << 3);
    }
}

// Grouping of state-only tiles (tc_state.cuh): a tile joins a group while the group's decay from
// its start stays within 2^-64 and dt <= 2^20, so that its weights 2^-C_t dt_t (C_t the log2
// cumsum from the group's start) lie in [dt_t, 2^84] and a group's accumulated state stays far
// inside the fp32 range.
constexpr float kGroupRange2 = 64.f;
constexpr float kGroupDtMax = 1048576.f;

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
        // per element: exp2((cum2_i - cum2_j) + log2 dt_j), the cumsum difference formed first
        const float c2 = sl.cum2[r];
        const float4* cc = reinterpret_cast<const float4*>(&sl.cum2[jb * 32]);
        const float4* lc = reinterpret_cast<const float4*>(&sl.lgdt[jb * 32]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 c = cc[i], l = lc[i];
            const float cv[4] = {c.x, c.y, c.z, c.w};
            const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int jj = 4 * i + e;
                g[jj] = (jj <= lane) ? ex2((c2 - cv[e]) + lv[e]) * g[jj] : 0.f;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(g[2 * i], g[2 * i + 1]);
}

// Half (16 columns: hf = 0 or 1) of the 32 x 32 block of p_block, for a caller that loads and
// stores G and P in 16-column pieces (fewer live registers): the same arithmetic per element.
__device__ __forceinline__ void p_half(uint32_t (&pk)[8], float (&g)[16], int jb, int hf, int q,
                                       int lane, int r, const DtSlot& sl) {
    const int j0 = jb * 32 + hf * 16;
    if (jb < q) {
        const float ur = sl.urow[r];
        const float4* cf = reinterpret_cast<const float4*>(&sl.colf[q - 1][j0]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 c = cf[i];
            g[4 * i + 0] *= c.x * ur;
            g[4 * i + 1] *= c.y * ur;
            g[4 * i + 2] *= c.z * ur;
            g[4 * i + 3] *= c.w * ur;
        }
    } else if (__builtin_expect((sl.dfac[0] >> q) & 1, 1)) {
        const float rr = sl.rd[r];
        const float4* cf = reinterpret_cast<const float4*>(&sl.cd[j0]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 c = cf[i];
            const float cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int jj = hf * 16 + 4 * i + e;
                g[4 * i + e] = (jj <= lane) ? g[4 * i + e] * cv[e] * rr : 0.f;
            }
        }
    } else {
        const float c2 = sl.cum2[r];
        const float4* cc = reinterpret_cast<const float4*>(&sl.cum2[j0]);
        const float4* lc = reinterpret_cast<const float4*>(&sl.lgdt[j0]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 c = cc[i], l = lc[i];
            const float cv[4] = {c.x, c.y, c.z, c.w};
            const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int jj = hf * 16 + 4 * i + e;
                g[4 * i + e] = (jj <= lane) ? ex2((c2 - cv[e]) + lv[e]) * g[4 * i + e] : 0.f;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(g[2 * i], g[2 * i + 1]);
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

// Look-back over the preceding ranges' published states (per compute warp), for a range whose
// first item continues chain u:
//     h_in = D_1 (D_2 (... h_incl ...) + H_2) + H_1.
// Which part each predecessor contributes is fixed by the plan (lookback_uses_aggregate), not
// by timing, so the result is the same on every run: aggregates (log2 decay D, local state H)
// of the predecessors holding middle pieces of chain u, then the inclusive state of the one
// holding its head piece.  False on timeout or abort.
template <int NS, int CW>
__device__ __forceinline__ bool look_back(float (&h)[NS / 128 * CW], const TcParams& p, Small& sm,
                                          int w, int lane, int r, int c0, int u) {
    const int64_t slot_elems = (int64_t)kPS * NS;
    h_from<NS, CW>(h, nullptr, r, c0, 0.f, false, false);
    float acc_logd = 0.f;
#pragma unroll 1
    for (int jp = (int)blockIdx.x - 1; jp >= 0; --jp) {
        const int* f = p.flags + jp * kFlagsPerCta + w * 4;
        const bool middle = lookback_uses_aggregate(p.n_units, p.n_tiles, p.n_ctas, p.pass1_mode, jp, u);
        const int* flag = f + (middle ? 1 : 0);
        bool ok = true;
        if (lane == 0) {
            const long long t0 = clock64();
            while (!ld_acquire_gpu(flag)) {
                if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) {
                    ok = false;
                    break;
                }
                if (clock64() - t0 > p.budget) {
                    flag_abort(sm, p.ws);
                    ok = false;
                    break;
                }
            }
        }
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) return false;
        // every lane acquires the flag itself before it reads the published state
        (void)ld_acquire_gpu(flag);
        const float* slot = p.slots + (int64_t)jp * 2 * slot_elems + (middle ? slot_elems : 0);
        h_from<NS, CW>(h, slot, r, c0, ex2(acc_logd), true, true);
        if (!middle) return true;
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

// Segment records of the d_state-128 state-only pass (plan::seg_records of them), after the
// hand-off slots of a grid capped at `cap` CTAs: each a local state [64 x 128] (slot layout)
// and its log2 decay, padded to 16 bytes.
constexpr size_t kSegRecBytes = sizeof(float) * kPS * 128 + 16;
size_t seg_offset(int cap) {
    return kWsHeaderBytes + flags_bytes() + sizeof(float) * 2 * (size_t)cap * kPS * 128;
}

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

}  // namespace
}  // namespace ssd
