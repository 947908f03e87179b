// tc_plan.cuh -- the work plan of the tensor-core scan kernel: how the tile chains of all
// units are cut into one contiguous range per CTA, and the items (chain pieces) each CTA runs.
// Plain integer arithmetic, compiled for the device (the kernel) and for the host (the plan
// checks in the tests).  Internal to libssd_scan.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define SSD_HD __host__ __device__ __forceinline__
#else
#define SSD_HD inline
#endif

namespace ssd {
namespace plan {

enum : int { kInitH0 = 0, kInitZero = 1, kInitLookback = 2 };
enum : int { kFinNone = 0, kFinFinal = 1, kFinIncl = 2, kFinAgg = 3 };

// Unit indices and coordinates fit in 32 bits (the launcher checks batch * H * P/64).
struct Item {
    int u;            // unit
    int k0, k1;       // tile range of the unit's chain
    int pass1;        // 1: state-only pass (no y)
    int init;         // how the state starts: kInit*
    int fin;          // what happens to the state at the end: kFin*
};

// A CTA's range, as scalars (no arrays, so nothing of it lives in local memory).
//
// A range holds at most a tail piece of one chain (it needs the state the previous range
// ends with), whole chains, and a head piece of another chain (its end state is needed by the
// next range); or a middle piece of one chain.  Items run in this order: [state-only pass over
// the piece with a successor, in pass1 mode], [head piece], [whole chains], [tail piece], so
// the state a successor needs is published as early as possible and the state a range needs
// is consumed as late as possible.
//
// kExt (the plan of a kernel launched after the separate state-only pass, tc_state.cuh): the
// same plan as pass1_mode 1 without the state-only items, which that pass has run already,
// publishing what they publish.
struct Plan {
    int u0, u1, f_lo, n_full, n_items;
    int k0, k1, n_pre, middle, p1;
};

template <bool kExt = false>
SSD_HD Plan make_plan(int64_t n_units, int n_tiles, int n_ctas, int pass1_mode, int cta) {
    Plan pl;
    pl.u0 = pl.u1 = pl.f_lo = pl.n_full = pl.n_items = 0;
    pl.k0 = pl.k1 = pl.n_pre = pl.middle = 0;
    pl.p1 = pass1_mode != 0;
    const int64_t T = n_tiles, total = n_units * T;
    const int64_t start = (int64_t)cta * total / n_ctas;
    const int64_t end = (int64_t)(cta + 1) * total / n_ctas;
    if (start >= end) return pl;
    pl.u0 = (int)(start / T);
    pl.u1 = (int)((end - 1) / T);
    pl.k0 = (int)(start % T);
    pl.k1 = (int)((end - 1) % T + 1);
    if (pl.u0 == pl.u1 && pl.k0 > 0 && pl.k1 < T) {     // middle piece of one chain
        pl.middle = 1;
        pl.n_pre = kExt ? 0 : pl.p1;
        pl.n_items = pl.n_pre + 1;
        return pl;
    }
    // head piece of chain u1 (starts at tile 0, ends before T); tail piece of chain u0
    const bool head = (pl.u0 == pl.u1) ? (pl.k0 == 0 && pl.k1 < T) : (pl.k1 < T);
    const bool tail = pl.k0 > 0;
    pl.n_pre = head ? 1 + (kExt ? 0 : pl.p1) : 0;
    const int f_first = tail ? pl.u0 + 1 : pl.u0;
    const int f_last = head ? pl.u1 - 1 : pl.u1;
    if (f_last >= f_first) {
        pl.f_lo = f_first;
        pl.n_full = f_last - f_first + 1;
    }
    pl.n_items = pl.n_pre + pl.n_full + (tail ? 1 : 0);
    return pl;
}

template <bool kExt = false>
SSD_HD Item plan_item(const Plan& pl, int i, int T) {
    if (pl.middle) {
        if (pl.n_pre > 0 && i == 0) return Item{pl.u0, pl.k0, pl.k1, 1, kInitZero, kFinAgg};
        return Item{pl.u0, pl.k0, pl.k1, 0, kInitLookback, kFinIncl};
    }
    if (i < pl.n_pre) {
        if (!kExt && pl.p1 && i == 0) return Item{pl.u1, 0, pl.k1, 1, kInitH0, kFinIncl};
        return Item{pl.u1, 0, pl.k1, 0, kInitH0, pl.p1 ? kFinNone : kFinIncl};
    }
    i -= pl.n_pre;
    if (i < pl.n_full) return Item{pl.f_lo + i, 0, T, 0, kInitH0, kFinFinal};
    return Item{pl.u0, pl.k0, (pl.u0 == pl.u1) ? pl.k1 : T, 0, kInitLookback, kFinFinal};
}

// The look-back's choice for predecessor CTA jp of a range that continues chain u: true takes
// jp's aggregate and goes on to jp - 1, false takes jp's inclusive state and stops.  With the
// state-only pass, a CTA whose range starts inside chain u holds a middle piece of it, whose
// aggregate that pass publishes early; the CTA whose range starts at or before the chain's
// first tile holds the head piece.  Without it, every piece publishes its inclusive state.
// Fixed by the plan, so every run combines the same states in the same order.
SSD_HD bool lookback_uses_aggregate(int64_t n_units, int n_tiles, int n_ctas, int pass1_mode,
                                    int jp, int u) {
    const int64_t total = n_units * n_tiles;
    return pass1_mode != 0 && (int64_t)jp * total / n_ctas > (int64_t)u * n_tiles;
}

// The work of the separate state-only pass (d_state 128): the pieces of the plan in mode 1
// whose end state it publishes, each cut into nseg segments of about equal length; segment s
// of a piece covers tiles k0 + s len / nseg .. k0 + (s + 1) len / nseg (len = k1 - k0).  The
// segments of a piece cut into several keep their local states in records rec0 .. rec0 +
// nseg - 1 of the workspace.
struct StPiece {
    int u, k0, k1;      // unit and tile range
    int cta;            // the scan CTA whose slot and flags receive the state
    int agg;            // 1: aggregate (middle piece), 0: inclusive state (head piece)
    int seg0, nseg;     // segments seg0 .. seg0 + nseg - 1 (grid indices)
    int rec0;           // first record (pieces with nseg > 1)
};
constexpr int kSegMinTiles = 32;

// Records a problem of `total_tiles` tiles may use on a grid of at most `cap` CTAs: with the
// segment length z chosen below, the cut pieces (longer than z) hold at most 2 t / z records,
// t the state-only tiles (at most total_tiles), and at most 5 per CTA (4 from the length, one
// more per piece).  Monotone in the problem size, so a part of a problem never needs more.
SSD_HD int64_t seg_records(int64_t total_tiles, int cap) {
    const int64_t a = 5 * (int64_t)cap, b = total_tiles / (kSegMinTiles / 2);
    return a < b ? a : b;
}

// Fills pieces[0 .. *n_pieces) for a grid of n_ctas CTAs and returns the number of segments
// (-1 if more than max_pieces pieces).  Segments are at least kSegMinTiles long, about 4 per CTA
// in all, and long enough that the cut pieces use at most `recs` records (none: every piece
// stays whole).
inline int state_segments(int64_t n_units, int n_tiles, int n_ctas, int64_t recs,
                          StPiece* pieces, int max_pieces, int* n_pieces) {
    int np = 0;
    int64_t t1 = 0;
    for (int c = 0; c < n_ctas; ++c) {
        const Plan pl = make_plan(n_units, n_tiles, n_ctas, 1, c);
        for (int i = 0; i < pl.n_items; ++i) {
            const Item it = plan_item(pl, i, n_tiles);
            if (!it.pass1) continue;
            if (np >= max_pieces) return -1;
            pieces[np++] = StPiece{it.u, it.k0, it.k1, c, it.fin == kFinAgg ? 1 : 0, 0, 1, 0};
            t1 += it.k1 - it.k0;
        }
    }
    const int64_t per = 4 * (int64_t)n_ctas;
    int64_t z = t1 / per + (t1 % per != 0);
    if (z < kSegMinTiles) z = kSegMinTiles;
    if (recs > 0) {
        // a cut piece (len > z) has ceil(len / z) < 2 len / z segments
        const int64_t zr = (2 * t1) / recs + ((2 * t1) % recs != 0);
        if (zr > z) z = zr;
    } else {
        z = (int64_t)1 << 40;   // no records: every piece stays whole
    }
    int s = 0, r = 0;
    for (int q = 0; q < np; ++q) {
        const int64_t len = pieces[q].k1 - pieces[q].k0;
        const int64_t n = (len + z - 1) / z;
        pieces[q].nseg = n < 1 ? 1 : (int)n;
        pieces[q].seg0 = s;
        pieces[q].rec0 = r;
        s += pieces[q].nseg;
        if (pieces[q].nseg > 1) r += pieces[q].nseg;
    }
    *n_pieces = np;
    return s;
}

}  // namespace plan
}  // namespace ssd
