// tc_state.cuh -- the state-only pass of the d_state-128 scan as a kernel of its own
// (included by tc128.cu, which launches it; internal to libssd_scan).
//
// When the tile ranges of the CTAs are shorter than the units' chains (the 128K-token
// workload), a range that ends inside a chain must publish the state its successor starts
// from: the head piece of a chain its inclusive state (from the initial state), a middle piece
// its aggregate (log2 decay, local state from zero); see tc_plan.cuh.  This kernel computes
// exactly those publications, for every CTA of the scan's plan, before the scan kernel runs
// (which then runs in plan mode 2 and finds every state it looks back for already published).
//
// Only the state is needed, so a piece reduces to the chunk-state GEMMs of its tiles,
//     h_end = exp(cum_end) h_0 + sum_t exp(cum_end - cum_t) dt_t x_t B_t^T,
// and consecutive tiles are grouped: inside a group the state GEMMs S^T = B^T Xs accumulate in
// TMEM with the weights 2^-C_t dt_t of the group (C_t the log2 cumsum from the group's start,
// the group kept within 2^-64 of decay so that every weight lies in [dt_t, 2^84]), and the
// register-held state is updated once per group, h = 2^C_end (h + S).  A tile whose own decay
// exceeds the group range is a group of one with the per-tile weights 2^(clast - c_t) dt_t and
// h = 2^clast h + S.
//
// Roles (384 threads): warp 0 loads x and B by TMA (lane 0); warp 1 issues the MMAs; warp 2
// computes each tile's weights and grouping from dt; warps 4-11 (two warpgroups of 32 headdim
// columns) scale x into Xs and keep the state, row n = 32 (warp % 4) + lane of S^T.
// Every wait is bounded; on a timeout the CTA records SSD_ERR_TIMEOUT, drains its copies and
// MMAs and publishes nothing (the scan kernel's look-back then times out too).
#pragma once

#include "tc_common.cuh"
// Timing hook for profiling builds: a no-op unless the build defines
// SSD_ST_TRACE_POINT(event, tile) (then it records a per-role clock64 timeline).
#ifndef SSD_ST_TRACE_POINT
#define SSD_ST_TRACE_POINT(event, tile) ((void)0)
#endif

namespace ssd {
namespace {

struct alignas(16) StSlot {
    float w[kTile];           // weight of each token's x row in the state GEMM
    float udec2;              // at a group's last tile: H = 2^udec2 H + sigma S
    float sigma;
    float clast2;             // the tile's own log2 decay
    int sflags;               // bit 0 first tile of its group, bit 1 last
};
static_assert(sizeof(StSlot) % 16 == 0, "slot alignment");

struct SK {
    static constexpr int kStages = 3;
    static constexpr int kNReg = 2;                             // 64-column regions of a B tile
    static constexpr uint32_t kXBytes = kTileBytes;             // x [128 tokens x 64]
    static constexpr uint32_t kBBytes = kNReg * kTileBytes;     // B [128 tokens x 128]
    static constexpr uint32_t kStageBytes = kXBytes + kBBytes;
    static constexpr int kThreads = 384;
    static constexpr int kWarpC = 4, kCompute = 256;
    static constexpr uint32_t kOffStage = 0;
    static constexpr uint32_t kOffXs = kStages * kStageBytes;           // 2 buffers
    static constexpr uint32_t kOffSlot = kOffXs + 2 * kTileBytes;
    static constexpr uint32_t kOffDt = kOffSlot + kStages * sizeof(StSlot);   // dt ring
    static constexpr int kDtRing = 8, kDtAhead = 4;     // ring tiles; tiles loaded ahead
    static constexpr uint32_t kOffBar = kOffDt + kDtRing * kTile * 4;
    static constexpr size_t kSmem = kOffBar + 256 + 1024;             // + alignment slack
    static constexpr uint32_t kTmemCols = 64;                          // S^T [128 x 64]
};

struct StBars {
    uint64_t full[SK::kStages], empty[SK::kStages];
    uint64_t xs_full[2], xs_empty[2];
    uint64_t s_full, s_empty, done;
    uint32_t tmem;
    int abort;
    int tma_n, dt_n;          // tiles loaded / tiles whose weights arrived
};
static_assert(sizeof(StBars) <= 256, "barrier block");

__device__ __forceinline__ bool st_abort_set(StBars& b) {
    return *reinterpret_cast<volatile int*>(&b.abort) != 0;
}

// Bounded wait of the whole warp (one verdict).  On timeout: abort flag and status word.  A
// budget of at most 2^16 cycles (a test of the failure path) is polled without suspending, since
// the hardware may park a try_wait for longer than that.
__device__ __forceinline__ bool sp_wait(uint64_t* bar, uint32_t parity, StBars& b,
                                        const TcParams& p) {
    const bool spin = p.budget <= (1ll << 16);
    auto poll = [&]() { return spin ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity); };
    bool ok = poll();
    if (!__all_sync(0xffffffffu, ok)) {
        const long long t0 = clock64();
        while (!ok) {
            if (st_abort_set(b)) break;
            if (clock64() - t0 > p.budget) {
                *reinterpret_cast<volatile int*>(&b.abort) = 1;
                set_status(p.ws, SSD_ERR_TIMEOUT);
                break;
            }
            ok = poll();
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// A tile's log2 cumsum (4 tokens per lane) as a float32 warp scan, and (returned) its last
// value.  The state pass needs weights and group decays that agree with each other, not the
// scan kernel's bit-exact 64-bit form; the float scan's rounding (about 1e-5 in log2 over a
// tile) is far below bf16's.
__device__ __forceinline__ float tile_scan2f(const float (&d0)[4], float A2, int lane,
                                             float (&c2)[4]) {
    float cs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) cs[i] = (i == 0 ? 0.f : cs[i - 1]) + d0[i] * A2;
    float incl = cs[3];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    const float excl = incl - cs[3];
#pragma unroll
    for (int i = 0; i < 4; ++i) c2[i] = excl + cs[i];
    return __shfl_sync(0xffffffffu, incl, 31);
}

// A tile's largest dt (warp-uniform) by one integer reduction: floats mapped to signed integers
// in the same order (negative values with their magnitude bits flipped).
__device__ __forceinline__ float tile_dtmax_r(const float (&d0)[4]) {
    const float m = fmaxf(fmaxf(d0[0], d0[1]), fmaxf(d0[2], d0[3]));
    int key = __float_as_int(m);
    key = key >= 0 ? key : key ^ 0x7fffffff;
    key = __reduce_max_sync(0xffffffffu, key);
    return __int_as_float(key >= 0 ? key : key ^ 0x7fffffff);
}

// The pieces of plan mode 1 whose end state the state-only pass publishes, each cut into
// segments of about equal length (one CTA each, so that the hardware's block scheduler
// balances the work over SMs of unequal speed and pieces of unequal length).  A segment
// computes its local state from zero into a record; the piece's last segment to finish (a
// counter in the piece's flag words) combines the records in order, h = 2^C_s h + S_s from the
// initial state (head piece) or zero (middle piece), and publishes.  A piece of one segment
// starts from its own initial state and publishes directly.
struct StTable {
    int n_pieces;
    float* seg;         // segment records (kSegRecBytes each) in the workspace
    StPiece piece[kMaxCtas];
};

// ---- warp 0: x and B tiles by TMA ------------------------------------------------------------

__device__ __forceinline__ void sp_load(const Item& it, const UnitCoords& uc, StBars& b,
                                        const TcParams& p, uint8_t* smem,
                                        const CUtensorMap* tmX, const CUtensorMap* tmB, int lane) {
    const int n = it.k1 - it.k0;
    for (int j = 0; j < n; ++j) {
        const int k = it.k0 + j, s = j % SK::kStages;
        if (!sp_wait(&b.empty[s], ((uint32_t)(j / SK::kStages) & 1u) ^ 1u, b, p)) break;
        if (lane == 0) {
            uint8_t* st = smem + SK::kOffStage + s * SK::kStageBytes;
            mbar_arrive_expect_tx(&b.full[s], SK::kStageBytes);
            tma_load_4d(st, tmX, &b.full[s], uc.ps * kPS, uc.h, k * kTile, uc.b);
            for (int r = 0; r < SK::kNReg; ++r)
                tma_load_4d(st + SK::kXBytes + r * kTileBytes, tmB, &b.full[s], r * 64, uc.g,
                            k * kTile, uc.b);
            b.tma_n = j + 1;   // tiles issued (read after the CTA's last barrier)
        }
    }
}

// A tile's weights (4 tokens per lane) and its slot's scalars, computed ahead of the slot wait:
// per-tile mode 2^(clast - c_t) dt_t, then H = 2^clast H + S; grouped 2^-(goff + c_t) dt_t, and at
// the group's last tile H = 2^u (H + S) with u = goff + clast (the group's log2 decay).
struct StW {
    float w[4];
    float udec2, sigma, clast2;
    int sflags;
};
__device__ __forceinline__ StW st_weights(const float (&d0)[4], const float (&c2)[4], float clast2,
                                          bool grouped, float goff, int sflags) {
    StW r;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        r.w[i] = (grouped ? ex2(-(goff + c2[i])) : ex2(clast2 - c2[i])) * d0[i];
    r.clast2 = clast2;
    r.sflags = sflags;
    r.udec2 = grouped ? goff + clast2 : clast2;
    r.sigma = grouped ? ex2(r.udec2) : 1.f;
    return r;
}
__device__ __forceinline__ void st_store(StSlot& sl, const StW& r, int lane) {
    *reinterpret_cast<float4*>(sl.w + 4 * lane) = make_float4(r.w[0], r.w[1], r.w[2], r.w[3]);
    if (lane == 0) {
        sl.udec2 = r.udec2;
        sl.sigma = r.sigma;
        sl.clast2 = r.clast2;
        sl.sflags = r.sflags;
    }
}

// ---- warp 2: each tile's weights and grouping, from dt ---------------------------------------

__device__ __forceinline__ void sp_weights(const Item& it, const UnitCoords& uc, StBars& b,
                                           const TcParams& p, uint8_t* smem, StSlot* slots,
                                           int lane) {
    const float A2 = p.A[uc.h] * kLog2e;
    // dt of tile k, 4 consecutive tokens per lane, copied asynchronously (cp.async) into a ring
    // in shared memory kDtAhead tiles ahead: the aligned 4-byte word holding each token's bf16
    // value (it lies inside the tensor's allocation, whose bounds are 4-byte aligned).  Loads into
    // registers would stall the warp wherever the value is first moved or used.
    uint32_t* ring = reinterpret_cast<uint32_t*>(smem + SK::kOffDt);
    // token t's dt at byte a0 + t * stride; which half of its word does not depend on the tile
    // (a tile advances the address by 256 H bytes)
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p.dt) +
                         2 * (uintptr_t)((int64_t)uc.b * p.L * p.H + uc.h);
    const uintptr_t stride = 2 * (uintptr_t)p.H;
    int hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        hi |= (int)(((a0 + (uintptr_t)(4 * lane + i) * stride) >> 1) & 1u) << i;
    auto issue_dt = [&](int k) {
        if (k < it.k1) {
            const int64_t t = (int64_t)k * kTile + 4 * lane;
            uint32_t* dst = ring + (k % SK::kDtRing) * kTile + 4 * lane;
            uintptr_t a = a0 + (uintptr_t)t * stride;
#pragma unroll
            for (int i = 0; i < 4; ++i, a += stride) {
                if (t + i < p.L) cp_async4(dst + i, reinterpret_cast<const void*>(a & ~(uintptr_t)3));
                else dst[i] = 0u;
            }
        }
        cp_async_commit();   // one group per tile, empty past the piece's end
    };
    auto read_dt = [&](int k, float (&d)[4]) {
        const uint32_t* src = ring + (k % SK::kDtRing) * kTile + 4 * lane;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t v = src[i];
            d[i] = __uint_as_float((((hi >> i) & 1) ? (v >> 16) : (v & 0xffffu)) << 16);
        }
    };
    const int n = it.k1 - it.k0;
#pragma unroll 1
    for (int q = 0; q < SK::kDtAhead; ++q) issue_dt(it.k0 + q);
    auto groupable = [](float cl, float dmx) { return cl >= -kGroupRange2 && dmx <= kGroupDtMax; };
    // Tiles go in pairs (j, j + 1): both the pair's next tiles are scanned together (independent
    // shuffle chains), and both weights are computed before the slot waits; only the flag that
    // ends a group needs the tile after.  Tile j's cumsum was scanned by the previous pair.
    float dA[4], cA[4], clA, dmA;
    cp_async_wait<SK::kDtAhead - 1>();   // tile k0 has landed
    read_dt(it.k0, dA);
    clA = tile_scan2f(dA, A2, lane, cA);
    dmA = tile_dtmax_r(dA);
    int mode = groupable(clA, dmA) ? 1 : 0;   // tile j: 0 per-tile update, 1 new group, 2 joins
    float goff = 0.f;                         // the group's log2 decay before the current tile
    for (int j = 0; j < n; j += 2) {
        const int k = it.k0 + j;
        const bool has1 = j + 1 < n, has2 = j + 2 < n;
        issue_dt(k + SK::kDtAhead);
        issue_dt(k + 1 + SK::kDtAhead);
        cp_async_wait<SK::kDtAhead - 1>();   // tiles k + 1 and k + 2 have landed
        float dB[4], cB[4], dC[4], cC[4];
        read_dt(k + 1, dB);
        read_dt(k + 2, dC);
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // past the piece's end the ring holds stale words
            dB[i] = has1 ? dB[i] : 0.f;
            dC[i] = has2 ? dC[i] : 0.f;
        }
        const float clB = tile_scan2f(dB, A2, lane, cB);
        const float clC = tile_scan2f(dC, A2, lane, cC);
        const float dmB = tile_dtmax_r(dB), dmC = tile_dtmax_r(dC);
        // tile j
        const bool gA = mode != 0, fA = mode != 2;
        if (fA) goff = 0.f;
        const int modeB = !(has1 && groupable(clB, dmB))                  ? 0
                          : (gA && goff + clA + clB >= -kGroupRange2)     ? 2
                                                                          : 1;
        const bool lA = !has1 || modeB != 2;
        const StW wA = st_weights(dA, cA, clA, gA, goff, (fA ? 1 : 0) | (lA ? 2 : 0));
        if (gA) goff += clA;
        // tile j + 1
        const bool gB = modeB != 0, fB = modeB != 2;
        if (fB) goff = 0.f;
        const int modeC = !(has2 && groupable(clC, dmC))                  ? 0
                          : (gB && goff + clB + clC >= -kGroupRange2)     ? 2
                                                                          : 1;
        const bool lB = !has2 || modeC != 2;
        const StW wB = st_weights(dB, cB, clB, gB, goff, (fB ? 1 : 0) | (lB ? 2 : 0));
        if (gB) goff += clB;
        mode = modeC;
        const int sA = j % SK::kStages;
        SSD_ST_TRACE_POINT(0, j);
        if (!sp_wait(&b.empty[sA], ((uint32_t)(j / SK::kStages) & 1u) ^ 1u, b, p)) break;
        SSD_ST_TRACE_POINT(1, j);
        st_store(slots[sA], wA, lane);
        mbar_arrive(&b.full[sA]);
        if (lane == 0) b.dt_n = j + 1;   // tiles whose weights arrived
        SSD_ST_TRACE_POINT(2, j);
        if (has1) {
            const int sB = (j + 1) % SK::kStages;
            if (!sp_wait(&b.empty[sB], ((uint32_t)((j + 1) / SK::kStages) & 1u) ^ 1u, b, p)) break;
            st_store(slots[sB], wB, lane);
            mbar_arrive(&b.full[sB]);
            if (lane == 0) b.dt_n = j + 2;
            SSD_ST_TRACE_POINT(2, j + 1);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            dA[i] = dC[i];
            cA[i] = cC[i];
        }
        clA = clC;
        dmA = dmC;
    }
    cp_async_wait<0>();
    __syncwarp();
}

// ---- warp 1: the state GEMMs, accumulated over each group ------------------------------------

__device__ __forceinline__ void sp_mma(const Item& it, StBars& b, const TcParams& p,
                                       const StSlot* slots, uint32_t sbase, uint32_t tmem,
                                       int lane) {
    constexpr uint32_t idS = idesc_bf16(128, kPS, 1, 1);   // S^T [N x P] = B^T Xs
    const int n = it.k1 - it.k0;
    int g = -1;               // group of the current tile
    for (int j = 0; j < n; ++j) {
        const int s = j % SK::kStages, xb = j & 1;
        SSD_ST_TRACE_POINT(3, j);
        if (!sp_wait(&b.xs_full[xb], (uint32_t)(j >> 1) & 1u, b, p)) break;
        SSD_ST_TRACE_POINT(4, j);
        if (!sp_wait(&b.full[s], (uint32_t)(j / SK::kStages) & 1u, b, p)) break;
        const int fl = slots[s].sflags;
        if (fl & 1) {
            ++g;
            if (!sp_wait(&b.s_empty, ((uint32_t)g & 1u) ^ 1u, b, p)) break;
        }
        tc_fence_after();
        const uint32_t bb = sbase + SK::kOffStage + s * SK::kStageBytes + SK::kXBytes;
        const uint32_t xsb = sbase + SK::kOffXs + xb * kTileBytes;
        mma8_ss_e<kStepRows, kStepRows>(tmem, smem_desc_sw128(bb, kTileBytes, 1024),
                                        smem_desc_sw128(xsb, 1024, 1024), idS,
                                        (fl & 1) ? 0u : 1u);
        mma_commit_e(&b.xs_empty[xb]);
        mma_commit_e(&b.empty[s]);
        if (fl & 2) mma_commit_e(&b.s_full);
        SSD_ST_TRACE_POINT(5, j);
    }
    // every MMA issued above has completed once this barrier's phase 0 completes
    mma_commit_e(&b.done);
    if (lane == 0) drain_wait(&b.done, 0, p.ws);
    __syncwarp();
}

// ---- warps 4-11: Xs and the state ------------------------------------------------------------

// Thread: token row (and state row) r = 32 (warp % 4) + lane; headdim columns c0 .. c0 + 31 of
// its warpgroup.  Returns false on a timeout or abort; else leaves its part of the published
// state in the CTA's slot and the piece's log2 decay in *logd_out.
__device__ __forceinline__ bool sp_compute(const Item& it, StBars& b, const TcParams& p,
                                           uint8_t* smem, const StSlot* slots, uint32_t tmem,
                                           int cw, int lane, const float* h0, float* out,
                                           float* logd_out) {
    const int q = cw & 3, wg = cw >> 2;
    const int r = 32 * q + lane, c0 = 32 * wg;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    // entering state: h0 (the initial state of the unit's 64 headdim rows, element (p, n) at
    // p * d_state + n), or zero
    float h[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) h[i] = h0 ? h0[(c0 + i) * 128 + r] : 0.f;
    float logd = 0.f;
    int g = -1;
    const int n = it.k1 - it.k0;
    for (int j = 0; j < n; ++j) {
        const int s = j % SK::kStages, xb = j & 1;
        SSD_ST_TRACE_POINT(6, j);
        if (!sp_wait(&b.full[s], (uint32_t)(j / SK::kStages) & 1u, b, p)) return false;
        SSD_ST_TRACE_POINT(7, j);
        if (!sp_wait(&b.xs_empty[xb], ((uint32_t)(j >> 1) & 1u) ^ 1u, b, p)) return false;
        SSD_ST_TRACE_POINT(8, j);
        // every field of the slot is read before xs_full: after it the MMA may complete and
        // the producer refill the stage
        const StSlot& sl = slots[s];
        const float wr = sl.w[r], clast2 = sl.clast2, udec2 = sl.udec2, sigma = sl.sigma;
        const int fl = sl.sflags;
        const uint8_t* xrow = smem + SK::kOffStage + s * SK::kStageBytes;
        uint8_t* xsrow = smem + SK::kOffXs + xb * kTileBytes;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const uint4 v = *reinterpret_cast<const uint4*>(xrow + sw128_off(r, wg * 4 + cc));
            const uint32_t in[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[e] = pack_bf16x2(wr * bf16lo_to_f32(in[e]), wr * bf16hi_to_f32(in[e]));
            *reinterpret_cast<uint4*>(xsrow + sw128_off(r, wg * 4 + cc)) =
                make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&b.xs_full[xb]);
        SSD_ST_TRACE_POINT(9, j);
        logd += clast2;
        if (fl & 2) {
            ++g;
            const float decay = ex2(udec2);
            if (!sp_wait(&b.s_full, (uint32_t)g & 1u, b, p)) return false;
            tc_fence_after();
            float sv[32];
            tmem_ld32(tmem + lane_base + c0, sv);
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = fmaf(decay, h[i], sigma * sv[i]);
            tc_fence_before();
            mbar_arrive(&b.s_empty);
        }
    }
    // this thread's part of the state, in the scan kernel's slot layout (element (p, n) at
    // p * d_state + n)
#pragma unroll
    for (int i = 0; i < 32; ++i) out[(c0 + i) * 128 + r] = h[i];
    __threadfence();
    *logd_out = logd;
    return true;
}

// The last segment of a multi-segment piece: combines the records of the piece's segments in
// order into the scan's slot and returns the piece's log2 decay.  All threads; each owns
// float4 columns tid, tid + kThreads, ... of the [64 x 128] state.
__device__ __forceinline__ float st_combine(const StPiece& pc, const StTable& tab,
                                            const float* h0, float* slot) {
    constexpr int kE = kPS * 128, kE4 = kE / 4;
    constexpr int kPer = (kE4 + SK::kThreads - 1) / SK::kThreads;
    constexpr int kRec = (int)(kSegRecBytes / sizeof(float));
    float4 h[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int e = 4 * ((int)threadIdx.x + k * SK::kThreads);
        h[k] = (h0 && e < kE) ? make_float4(h0[e], h0[e + 1], h0[e + 2], h0[e + 3])
                              : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float logd = 0.f;
#pragma unroll 1
    for (int q = 0; q < pc.nseg; ++q) {
        const float* rec = tab.seg + (int64_t)(pc.rec0 + q) * kRec;
        const float ls = __ldcg(rec + kE);
        const float d = ex2(ls);
        logd += ls;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int e4 = (int)threadIdx.x + k * SK::kThreads;
            if (e4 < kE4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(rec) + e4);
                h[k] = make_float4(fmaf(d, h[k].x, v.x), fmaf(d, h[k].y, v.y),
                                   fmaf(d, h[k].z, v.z), fmaf(d, h[k].w, v.w));
            }
        }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int e4 = (int)threadIdx.x + k * SK::kThreads;
        if (e4 < kE4) reinterpret_cast<float4*>(slot)[e4] = h[k];
    }
    __threadfence();
    return logd;
}

__global__ void __launch_bounds__(SK::kThreads, 1)
    ssd_state_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ TcParams p, const __grid_constant__ StTable tab) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    StBars& b = *reinterpret_cast<StBars*>(smem + SK::kOffBar);
    StSlot* slots = reinterpret_cast<StSlot*>(smem + SK::kOffSlot);
    __shared__ float logd_sh;
    __shared__ int last_sh;
    // this CTA's segment, of the last piece whose first segment is at most blockIdx.x
    int c = 0;
    for (int hi = tab.n_pieces - 1; c < hi;) {
        const int mid = (c + hi + 1) >> 1;
        if (tab.piece[mid].seg0 <= (int)blockIdx.x) c = mid;
        else hi = mid - 1;
    }
    const StPiece& pc = tab.piece[c];
    const int si = (int)blockIdx.x - pc.seg0, len = pc.k1 - pc.k0;
    Item it;
    it.u = pc.u;
    it.k0 = pc.k0 + (int)((int64_t)si * len / pc.nseg);
    it.k1 = pc.k0 + (int)((int64_t)(si + 1) * len / pc.nseg);
    it.pass1 = 1;
    it.init = kInitZero;
    it.fin = kFinAgg;
    const UnitCoords uc = unit_coords(p, it.u);
    const bool direct = pc.nseg == 1;
    constexpr int64_t kE = (int64_t)kPS * 128;
    float* slot = p.slots + (int64_t)pc.cta * 2 * kE + (pc.agg ? kE : 0);
    float* rec = tab.seg + (int64_t)(pc.rec0 + si) * (int64_t)(kSegRecBytes / sizeof(float));
    // the unit's initial state, where the piece (a head piece) starts from it
    const float* h0 = (!pc.agg && p.h0) ? p.h0 + ((int64_t)uc.bh * p.P + (int64_t)uc.ps * kPS) * 128
                                        : nullptr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < SK::kStages; ++i) {
            mbar_init(&b.full[i], 1 + 32);
            mbar_init(&b.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&b.xs_full[i], SK::kCompute);
            mbar_init(&b.xs_empty[i], 1);
        }
        mbar_init(&b.s_full, 1);
        mbar_init(&b.s_empty, SK::kCompute);
        mbar_init(&b.done, 1);
        b.abort = 0;
        b.tma_n = 0;
        b.dt_n = 0;
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&b.tmem, SK::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b.tmem;
    bool ok = true;
    if (warp == 0) {
        sp_load(it, uc, b, p, smem, &tmX, &tmB, lane);
    } else if (warp == 1) {
        sp_mma(it, b, p, slots, smem_u32(smem), tmem, lane);
    } else if (warp == 2) {
        sp_weights(it, uc, b, p, smem, slots, lane);
    } else if (warp >= SK::kWarpC) {
        float logd = 0.f;
        ok = sp_compute(it, b, p, smem, slots, tmem, warp - SK::kWarpC, lane,
                        direct ? h0 : nullptr, direct ? slot : rec, &logd);
        if (warp == SK::kWarpC && lane == 0) logd_sh = logd;
    }
    ok = __syncthreads_and(ok) && !st_abort_set(b);
    if (!ok && threadIdx.x == 0) {
        // after an abort the loads of the last tiles issued must land before the CTA exits.  A
        // stage whose weights never arrived gets stand-in arrivals so that its phase can
        // complete; the loads run at most kStages tiles ahead of the weights (a stage is
        // refilled only after the MMA of its previous tile, which waited for that tile's weights).
        const int nt = b.tma_n;
        for (int q = b.dt_n; q < nt; ++q) mbar_arrive_cnt(&b.full[q % SK::kStages], 32);
        for (int q = nt - SK::kStages; q < nt; ++q)
            if (q >= 0) drain_wait(&b.full[q % SK::kStages], (uint32_t)(q / SK::kStages) & 1u, p.ws);
    }
    if (threadIdx.x == 0) {
        // a multi-segment piece: the record's log2 decay, then the count of finished segments
        // (release); the last one to finish (acquire) combines
        int last = ok ? 1 : 0;
        if (ok && !direct) {
            rec[kE] = logd_sh;
            __threadfence();
            last = atomicAdd(p.flags + pc.cta * kFlagsPerCta + 3, 1) == pc.nseg - 1;
            if (last) __threadfence();
        }
        last_sh = last;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, SK::kTmemCols);
    if (!last_sh) return;
    const float logd = direct ? logd_sh : st_combine(pc, tab, h0, slot);
    __syncthreads();
    if (threadIdx.x == 0) {
        // every thread's part of the state is written: publish it for all 16 warps of the scan
        // kernel (the aggregate's log2 decay first)
        __threadfence();
        for (int w = 0; w < 16; ++w) {
            int* f = p.flags + pc.cta * kFlagsPerCta + w * 4;
            if (pc.agg) st_relaxed_gpu(f + 2, __float_as_int(logd));
            st_release_gpu(f + (pc.agg ? 1 : 0), 1);
        }
    }
}

// Host: the table of the state-only pass, its segments within the `recs` records of `seg`.
inline int st_table(const TcParams& p, float* seg, int64_t recs, StTable* tab, int* n_segs) {
    const int s = state_segments(p.n_units, p.n_tiles, p.n_ctas, recs, tab->piece, kMaxCtas,
                                 &tab->n_pieces);
    if (s < 0) return SSD_ERR_UNSUPPORTED;
    tab->seg = seg;
    *n_segs = s;
    return SSD_OK;
}

// The state-only pass of the d_state-128 scan for plan `p` (launched before the scan kernel,
// whose plan then leaves these items out): one CTA per segment of `tab`.  tmX / tmB are the
// scan's tensor maps.
int tc128_state_launch(const CUtensorMap& tmX, const CUtensorMap& tmB, const TcParams& p,
                       const StTable& tab, int n_segs, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(ssd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SK::kSmem) != cudaSuccess)
            return SSD_ERR_CUDA;
        attr = true;
    }
    ssd_state_kernel<<<(unsigned)n_segs, SK::kThreads, SK::kSmem, st>>>(tmX, tmB, p, tab);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace
}  // namespace ssd
