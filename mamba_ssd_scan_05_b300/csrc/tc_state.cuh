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
// Roles (384 threads): warp 0 loads x and B by TMA (lane 0) and computes the tile's weights and
// grouping (all lanes); warp 1 issues the MMAs; warps 4-11 (two warpgroups of 32 headdim
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
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) c2[i] = excl + cs[i];
    return __shfl_sync(0xffffffffu, incl, 31);
}

// The CTA's state-only item under plan mode 1 (the piece whose state it must publish), if any.
__device__ __forceinline__ bool pass1_item(const TcParams& p, Item& out) {
    const Plan pl = plan::make_plan(p.n_units, p.n_tiles, p.n_ctas, 1, (int)blockIdx.x);
    for (int i = 0; i < pl.n_items; ++i) {
        const Item it = plan_item(pl, i, p.n_tiles);
        if (it.pass1) {
            out = it;
            return true;
        }
    }
    return false;
}

// ---- warp 0: x and B tiles, weights and grouping --------------------------------------------

__device__ __forceinline__ void sp_producer(const Item& it, const UnitCoords& uc, StBars& b,
                                            const TcParams& p, uint8_t* smem, StSlot* slots,
                                            const CUtensorMap* tmX, const CUtensorMap* tmB,
                                            int lane) {
    const float A2 = p.A[uc.h] * kLog2e;
    // dt of tile k, 4 consecutive tokens per lane, copied asynchronously (cp.async) into a ring
    // in shared memory kDtAhead tiles ahead: the aligned 4-byte word holding each token's bf16
    // value (it lies inside the tensor's allocation, whose bounds are 4-byte aligned).  Loads into
    // registers would stall the warp wherever the value is first moved or used.
    uint32_t* ring = reinterpret_cast<uint32_t*>(smem + SK::kOffDt);
    const uintptr_t dt_base = reinterpret_cast<uintptr_t>(p.dt);
    auto dt_addr = [&](int64_t t) {       // byte address of token t's dt
        return dt_base + 2 * (uintptr_t)(((int64_t)uc.b * p.L + t) * p.H + uc.h);
    };
    auto issue_dt = [&](int k) {
        if (k < it.k1) {
            const int64_t t = (int64_t)k * kTile + 4 * lane;
            uint32_t* dst = ring + (k % SK::kDtRing) * kTile + 4 * lane;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (t + i < p.L) cp_async4(dst + i, reinterpret_cast<const void*>(dt_addr(t + i) & ~(uintptr_t)3));
                else dst[i] = 0u;
            }
        }
        cp_async_commit();   // one group per tile, empty past the piece's end
    };
    auto read_dt = [&](int k, float (&d)[4]) {
        const int64_t t = (int64_t)k * kTile + 4 * lane;
        const uint32_t* src = ring + (k % SK::kDtRing) * kTile + 4 * lane;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t v = src[i];
            const bool hi = (dt_addr(t + i) & 2) != 0;
            d[i] = __uint_as_float((hi ? (v >> 16) : (v & 0xffffu)) << 16);
        }
    };
    const int n = it.k1 - it.k0;
#pragma unroll 1
    for (int q = 0; q < SK::kDtAhead; ++q) issue_dt(it.k0 + q);
    int nmode = 0;            // the next tile: 0 per-tile update, 1 new group, 2 joins
    float goff = 0.f;         // the group's log2 decay before the current tile
    // each tile's cumsum is scanned once, as the previous iteration's look at the next tile
    float dcur[4], c2cur[4], clcur, dmxcur;
    cp_async_wait<SK::kDtAhead - 1>();
    read_dt(it.k0, dcur);
    clcur = tile_scan2f(dcur, A2, lane, c2cur);
    dmxcur = tile_dtmax(dcur);
    int j = 0;
    for (; j < n; ++j) {
        const int k = it.k0 + j, s = j % SK::kStages;
        const bool has1 = j + 1 < n;
        issue_dt(k + SK::kDtAhead);   // the ring slot of tile k - (ring - ahead) is free
        SSD_ST_TRACE_POINT(0, j);
        if (!sp_wait(&b.empty[s], ((uint32_t)(j / SK::kStages) & 1u) ^ 1u, b, p)) break;
        SSD_ST_TRACE_POINT(1, j);
        uint8_t* st = smem + SK::kOffStage + s * SK::kStageBytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(&b.full[s], SK::kStageBytes);
            tma_load_4d(st, tmX, &b.full[s], uc.ps * kPS, uc.h, k * kTile, uc.b);
            for (int r = 0; r < SK::kNReg; ++r)
                tma_load_4d(st + SK::kXBytes + r * kTileBytes, tmB, &b.full[s], r * 64, uc.g,
                            k * kTile, uc.b);
        }
        // grouping: this tile joins the current group unless it starts one (or is on its own)
        int mode = nmode;
        if (j == 0) mode = (clcur >= -kGroupRange2 && dmxcur <= kGroupDtMax) ? 1 : 0;
        const bool grouped = mode != 0, first = mode != 2;
        if (first) goff = 0.f;
        bool last = true;
        float dn[4], c2n[4], cln = 0.f, dmxn = 0.f;
        if (has1) {
            cp_async_wait<SK::kDtAhead - 1>();   // tile k + 1 has landed
            read_dt(k + 1, dn);
            cln = tile_scan2f(dn, A2, lane, c2n);
            dmxn = tile_dtmax(dn);
            nmode = !(cln >= -kGroupRange2 && dmxn <= kGroupDtMax)      ? 0
                    : (grouped && goff + clcur + cln >= -kGroupRange2)  ? 2
                                                                        : 1;
            last = nmode != 2;
        }
        state_weights(slots[s].w, slots[s].udec2, slots[s].sigma, slots[s].clast2,
                      slots[s].sflags, dcur, c2cur, clcur, lane, grouped, goff,
                      (first ? 1 : 0) | (last ? 2 : 0));
        if (grouped) goff += clcur;
        mbar_arrive(&b.full[s]);
        SSD_ST_TRACE_POINT(2, j);
        if (has1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dcur[i] = dn[i];
                c2cur[i] = c2n[i];
            }
            clcur = cln;
            dmxcur = dmxn;
        }
    }
    cp_async_wait<0>();
    if (st_abort_set(b) && lane == 0) {
        // the loads of every tile this loop issued must land before the CTA exits
        for (int q = j - SK::kStages; q < j; ++q)
            if (q >= 0) drain_wait(&b.full[q % SK::kStages], (uint32_t)(q / SK::kStages) & 1u, p.ws);
    }
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
__device__ __forceinline__ bool sp_compute(const Item& it, const UnitCoords& uc, StBars& b,
                                           const TcParams& p, uint8_t* smem,
                                           const StSlot* slots, uint32_t tmem, int cw, int lane,
                                           float* logd_out) {
    const int q = cw & 3, wg = cw >> 2;
    const int r = 32 * q + lane, c0 = 32 * wg;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    // entering state: the chain's initial state (head piece) or zero (middle piece); element
    // (p, n) of a head's state at p * d_state + n
    float h[32];
    const float* h0 = (it.init == kInitH0 && p.h0)
                          ? p.h0 + ((int64_t)uc.bh * p.P + (int64_t)uc.ps * kPS) * 128
                          : nullptr;
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
    // this thread's part of the publication, in the scan kernel's slot layout (element (p, n) at
    // p * d_state + n of the CTA's inclusive or aggregate slot)
    const int64_t slot_elems = (int64_t)kPS * 128;
    float* slot = p.slots + (int64_t)blockIdx.x * 2 * slot_elems +
                  (it.fin == kFinAgg ? slot_elems : 0);
#pragma unroll
    for (int i = 0; i < 32; ++i) slot[(c0 + i) * 128 + r] = h[i];
    __threadfence();
    *logd_out = logd;
    return true;
}

__global__ void __launch_bounds__(SK::kThreads, 1)
    ssd_state_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    StBars& b = *reinterpret_cast<StBars*>(smem + SK::kOffBar);
    StSlot* slots = reinterpret_cast<StSlot*>(smem + SK::kOffSlot);
    __shared__ float logd_sh;
    Item it;
    if (!pass1_item(p, it)) return;          // this CTA's range publishes nothing
    const UnitCoords uc = unit_coords(p, it.u);
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
        sp_producer(it, uc, b, p, smem, slots, &tmX, &tmB, lane);
    } else if (warp == 1) {
        sp_mma(it, b, p, slots, smem_u32(smem), tmem, lane);
    } else if (warp >= SK::kWarpC) {
        float logd = 0.f;
        ok = sp_compute(it, uc, b, p, smem, slots, tmem, warp - SK::kWarpC, lane, &logd);
        if (warp == SK::kWarpC && lane == 0) logd_sh = logd;
    }
    ok = __syncthreads_and(ok) && !st_abort_set(b);
    if (ok && threadIdx.x == 0) {
        // every compute warp's part of the state is written: publish it for all 16 warps of
        // the scan kernel (the aggregate's log2 decay first)
        __threadfence();
        for (int w = 0; w < 16; ++w) {
            int* f = p.flags + (int)blockIdx.x * kFlagsPerCta + w * 4;
            if (it.fin == kFinAgg) st_relaxed_gpu(f + 2, __float_as_int(logd_sh));
            st_release_gpu(f + (it.fin == kFinAgg ? 1 : 0), 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, SK::kTmemCols);
}

// The state-only pass of the d_state-128 scan for the CTAs of plan `p` (launched before the
// scan kernel, which then runs in plan mode 2).  tmX / tmB are the scan's tensor maps.
int tc128_state_launch(const CUtensorMap& tmX, const CUtensorMap& tmB, const TcParams& p,
                       cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(ssd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SK::kSmem) != cudaSuccess)
            return SSD_ERR_CUDA;
        attr = true;
    }
    ssd_state_kernel<<<(unsigned)p.n_ctas, SK::kThreads, SK::kSmem, st>>>(tmX, tmB, p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace
}  // namespace ssd
