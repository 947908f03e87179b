// Host checks of the tensor-core kernel's work plan (mamba_ssd_scan_05_b300/csrc/tc_plan.cuh):
// for many (units, tiles per chain, CTAs, state-only-pass mode) it runs make_plan / plan_item
// for every CTA, exactly as the kernel does, and checks that
//   1. each CTA's items stay inside its contiguous tile range;
//   2. every tile of every chain is produced (non state-only) exactly once;
//   3. a piece that starts at tile 0 starts from the initial state, any other piece looks
//      back, and the look-back walk over the preceding CTAs' publications, taking from each
//      the publication lookback_uses_aggregate names, reaches an inclusive state through
//      pieces that end exactly where the next begins;
//   4. a CTA publishes for one chain only (its flags are per CTA), at most one inclusive state
//      and one aggregate;
//   5. every chain ends in exactly one final-state item, at its last tile;
//   6. a state-only pass covers the same tiles as the piece it precedes;
//   7. the separate state-only pass's segments (state_segments): its pieces are exactly the
//      state-only items of mode 1, each cut into non-empty segments that tile it in order,
//      with contiguous grid indices; the segments of cut pieces take consecutive records and
//      fit the records the workspace holds (the count it reserves, or fewer), segments of a
//      cut piece are at least half the minimum length, and there are at most 5 per CTA.
// Prints the first violations and exits non-zero if there are any.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "../mamba_ssd_scan_05_b300/csrc/tc_plan.cuh"

using namespace ssd::plan;

namespace {

int g_fail = 0;

void fail(const char* what, long U, int T, int C, int p1, int cta, long detail) {
    if (g_fail < 20)
        std::printf("FAIL %s: U=%ld T=%d C=%d p1=%d cta=%d (%ld)\n", what, U, T, C, p1, cta,
                    detail);
    ++g_fail;
}

struct Pub {
    int u = -1, k0 = 0, k1 = 0;
    bool set = false;
};

void check(long U, int T, int C, int p1) {
    const long total = U * T;
    std::vector<int> cover((size_t)total, 0);
    std::vector<int> finals((size_t)U, 0);
    std::vector<Pub> incl((size_t)C), agg((size_t)C);
    struct Look {
        int cta, u, k0;
    };
    std::vector<Look> looks;
    for (int c = 0; c < C; ++c) {
        const long start = (long)c * total / C, end = (long)(c + 1) * total / C;
        // mode 2: the plan of the kernel launched after the separate state-only pass
        const Plan pl = p1 == 2 ? make_plan<true>(U, T, C, 1, c) : make_plan(U, T, C, p1, c);
        int pub_unit = -1;
        if (p1 == 2) {
            // the separate state-only kernel runs mode 1's state-only items of this range and
            // publishes what they publish; the plan itself must hold none of them
            const Plan ext = make_plan(U, T, C, 1, c);
            for (int i = 0; i < ext.n_items; ++i) {
                const Item it = plan_item(ext, i, T);
                if (!it.pass1) continue;
                Pub& pb = (it.fin == kFinIncl) ? incl[c] : agg[c];
                if (pb.set) fail("two publications of one kind", U, T, C, p1, c, i);
                pb.set = true;
                pb.u = it.u;
                pb.k0 = it.k0;
                pb.k1 = it.k1;
                pub_unit = it.u;
            }
            for (int i = 0; i < pl.n_items; ++i)
                if (plan_item<true>(pl, i, T).pass1)
                    fail("state-only item in mode 2", U, T, C, p1, c, i);
        }
        for (int i = 0; i < pl.n_items; ++i) {
            const Item it = p1 == 2 ? plan_item<true>(pl, i, T) : plan_item(pl, i, T);
            if (it.u < 0 || it.u >= U || it.k0 < 0 || it.k1 > T || it.k0 >= it.k1) {
                fail("item range", U, T, C, p1, c, i);
                continue;
            }
            if ((long)it.u * T + it.k0 < start || (long)it.u * T + it.k1 > end)
                fail("item outside the CTA range", U, T, C, p1, c, i);
            if (it.pass1) {
                // 6: the next item is the full pass over the same tiles
                if (i + 1 >= pl.n_items) {
                    fail("state-only pass without its piece", U, T, C, p1, c, i);
                } else {
                    const Item nx = plan_item(pl, i + 1, T);
                    if (nx.u != it.u || nx.k0 != it.k0 || nx.k1 != it.k1 || nx.pass1)
                        fail("state-only pass and its piece differ", U, T, C, p1, c, i);
                }
            } else {
                for (int k = it.k0; k < it.k1; ++k) ++cover[(size_t)it.u * T + k];
            }
            // 3: initial state versus look-back
            if (it.init == kInitH0 && it.k0 != 0) fail("initial state mid-chain", U, T, C, p1, c, i);
            if (it.init == kInitLookback) {
                if (it.k0 == 0) fail("look-back at a chain start", U, T, C, p1, c, i);
                looks.push_back({c, it.u, it.k0});
            }
            if (it.init == kInitZero && !it.pass1)
                fail("zero start on a full pass", U, T, C, p1, c, i);
            // 4, 5: publications and final states
            if (it.fin == kFinIncl || it.fin == kFinAgg) {
                if (pub_unit >= 0 && pub_unit != it.u)
                    fail("publishes for two chains", U, T, C, p1, c, i);
                pub_unit = it.u;
                Pub& pb = (it.fin == kFinIncl) ? incl[c] : agg[c];
                if (pb.set) fail("two publications of one kind", U, T, C, p1, c, i);
                pb.set = true;
                pb.u = it.u;
                pb.k0 = it.k0;
                pb.k1 = it.k1;
                if (it.k1 == T) fail("publishes at a chain end", U, T, C, p1, c, i);
            }
            if (it.fin == kFinFinal) {
                if (it.pass1 || it.k1 != T) fail("final state not at the chain end", U, T, C, p1, c, i);
                ++finals[(size_t)it.u];
            }
        }
    }
    for (long t = 0; t < total; ++t)
        if (cover[(size_t)t] != 1) {
            fail("tile not produced exactly once", U, T, C, p1, -1, t);
            break;
        }
    for (long u = 0; u < U; ++u)
        if (finals[(size_t)u] != 1) {
            fail("chain without exactly one final state", U, T, C, p1, -1, u);
            break;
        }
    // 3: the look-back walk, with the kernel's rule for which publication each predecessor
    // contributes (aggregate: compose and go on; inclusive state: stop)
    for (const Look& lk : looks) {
        int pos = lk.k0;
        bool done = false;
        for (int jp = lk.cta - 1; jp >= 0 && !done; --jp) {
            const Pub& in = incl[jp];
            const Pub& ag = agg[jp];
            if (!lookback_uses_aggregate(U, T, C, p1 == 2 ? 1 : p1, jp, lk.u)) {
                if (!(in.set && in.u == lk.u && in.k1 == pos)) {
                    fail("look-back wants an inclusive state that is not there", U, T, C, p1,
                         lk.cta, jp);
                    break;
                }
                done = true;
            } else {
                if (!(ag.set && ag.u == lk.u && ag.k1 == pos)) {
                    fail("look-back wants an aggregate that is not there", U, T, C, p1, lk.cta,
                         jp);
                    break;
                }
                pos = ag.k0;
            }
            // a CTA that has both publishes them over the same tiles
            if (in.set && ag.set && (in.k0 != ag.k0 || in.k1 != ag.k1))
                fail("aggregate and inclusive state differ", U, T, C, p1, jp, 0);
        }
        if (!done && pos > 0) fail("look-back runs out of CTAs", U, T, C, p1, lk.cta, pos);
    }
}

// 7: segments for a grid of C CTAs with `recs` records in the workspace
void check_segments(long U, int T, int C, long recs) {
    std::vector<StPiece> pieces(256);
    int np = 0;
    const int s = state_segments(U, T, C, recs, pieces.data(), 256, &np);
    if (s < 0) {
        fail("segments: too many pieces", U, T, C, 2, -1, recs);
        return;
    }
    // the pieces are the state-only items of mode 1, in CTA order
    int q = 0;
    for (int c = 0; c < C; ++c) {
        const Plan pl = make_plan(U, T, C, 1, c);
        for (int i = 0; i < pl.n_items; ++i) {
            const Item it = plan_item(pl, i, T);
            if (!it.pass1) continue;
            if (q >= np) {
                fail("segments: a state-only item without a piece", U, T, C, 2, c, i);
                return;
            }
            const StPiece& pc = pieces[(size_t)q++];
            if (pc.u != it.u || pc.k0 != it.k0 || pc.k1 != it.k1 || pc.cta != c ||
                pc.agg != (it.fin == kFinAgg ? 1 : 0))
                fail("segments: piece differs from its state-only item", U, T, C, 2, c, i);
        }
    }
    if (q != np) fail("segments: extra pieces", U, T, C, 2, -1, np - q);
    int next = 0, rec = 0;
    long cut = 0;
    for (int i = 0; i < np; ++i) {
        const StPiece& pc = pieces[(size_t)i];
        const int len = pc.k1 - pc.k0;
        if (pc.seg0 != next || pc.nseg < 1 || pc.nseg > len)
            fail("segments: indices or count", U, T, C, 2, pc.cta, pc.nseg);
        int pos = pc.k0;
        for (int g = 0; g < pc.nseg; ++g) {
            const int a = pc.k0 + (int)((long)g * len / pc.nseg);
            const int b = pc.k0 + (int)((long)(g + 1) * len / pc.nseg);
            if (a != pos || b <= a) fail("segments: do not tile the piece", U, T, C, 2, pc.cta, g);
            if (pc.nseg > 1 && b - a < kSegMinTiles / 2)
                fail("segments: too short", U, T, C, 2, pc.cta, b - a);
            pos = b;
        }
        if (pos != pc.k1) fail("segments: piece not covered", U, T, C, 2, pc.cta, pos);
        if (pc.nseg > 1) {
            if (pc.rec0 != rec) fail("segments: record indices", U, T, C, 2, pc.cta, pc.rec0);
            rec += pc.nseg;
            cut += pc.nseg;
        }
        next += pc.nseg;
    }
    if (next != s) fail("segments: count returned", U, T, C, 2, -1, s);
    if (cut > recs) fail("segments: records overflow", U, T, C, 2, -1, cut);
    if (s > 5L * C) fail("segments: more than 5 per CTA", U, T, C, 2, -1, s);
}

}  // namespace

int main() {
    const long units[] = {1, 2, 3, 5, 8, 24, 80, 192, 320, 1000, 10240};
    const int tiles[] = {1, 2, 3, 7, 16, 32, 129, 1024};
    const int ctas[] = {1, 2, 3, 7, 148, 256};
    long cases = 0;
    for (long U : units)
        for (int T : tiles)
            for (int C0 : ctas) {
                const long total = U * T;
                const int C = (int)(C0 < total ? C0 : total);   // the launcher's clamp
                for (int p1 = 0; p1 < 3; ++p1) {
                    check(U, T, C, p1);
                    ++cases;
                }
                // the records a workspace reserves for C CTAs (5 per CTA, fewer for short
                // problems), none, as many as pieces, and one more
                for (long recs : {(long)seg_records(total, C), 0L, 1L, 7L, (long)C, 100000L})
                    check_segments(U, T, C, recs);
            }
    std::printf("%ld plans checked, %d violations\n", cases, g_fail);
    return g_fail ? 1 : 0;
}
