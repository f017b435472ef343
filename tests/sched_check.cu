// Host-side check of the GEMM's persistent / stream-K schedule (Sched,
// SegIter from gemm.cuh), compiled by tests/test_sched_cpu.py and run on the
// CPU.  For each (tiles, K blocks, CTAs) case it walks every CTA's segments
// and checks what the kernels rely on:
//   * every (tile, K block) is done exactly once;
//   * a tile done whole by one CTA is a single segment (rel = -1);
//   * the pieces of a cut tile belong to CTAs cta_of(first block) ..
//     cta_of(last block), in K order with the CTA index, each piece's slot is
//     the one slot_in_tile() names, and no two pieces share a slot;
//   * slots stay below 2 * CTAs and cut tiles number at most 2 * CTAs (the
//     workspace holds that many partial tiles and counter rows).
// Prints "ok <cases>" and exits 0, or prints the first violation and exits 1.
#include <cstdio>
#include <map>
#include <set>
#include <vector>

#include "gemm.cuh"

using namespace fp8q;

static int fail(const char* what, int tiles, int kb, int g) {
    std::printf("FAIL %s (tiles %d, K blocks %d, CTAs %d)\n", what, tiles, kb, g);
    return 1;
}

static int check(int tiles, int Kb, int G, bool allow_sk) {
    Sched sc{};
    sc.plan(tiles, Kb, G, allow_sk);
    if (sc.dp_tiles % G != 0 && sc.dp_tiles != tiles) return fail("whole-tile count", tiles, Kb, G);
    if (tiles - sc.dp_tiles > 2 * G) return fail("cut-tile capacity", tiles, Kb, G);
    std::vector<std::vector<int>> done(tiles, std::vector<int>(Kb, 0));
    struct Piece { int cta, kb0, kb1, slot; };
    std::map<int, std::vector<Piece>> pieces;          // by stream-K tile rel
    std::set<int> slots;
    for (int c = 0; c < G; ++c) {
        SegIter si;
        si.start(&sc, c);
        Seg sg;
        int guard = 0;
        while (si.next(sg)) {
            if (++guard > tiles + 4) return fail("runaway segment walk", tiles, Kb, G);
            if (sg.t < 0 || sg.t >= tiles || sg.kb0 < 0 || sg.kb1 > Kb || sg.kb0 >= sg.kb1)
                return fail("segment out of range", tiles, Kb, G);
            for (int k = sg.kb0; k < sg.kb1; ++k) done[sg.t][k]++;
            if (sg.rel < 0) {
                if (sg.kb0 != 0 || sg.kb1 != Kb) return fail("partial segment marked whole", tiles, Kb, G);
            } else {
                if (sg.t != sc.dp_tiles + sg.rel) return fail("rel / tile mismatch", tiles, Kb, G);
                if (sg.slot < 0 || sg.slot >= 2 * G) return fail("slot out of range", tiles, Kb, G);
                if (!slots.insert(sg.slot).second) return fail("slot used twice", tiles, Kb, G);
                pieces[sg.rel].push_back({c, sg.kb0, sg.kb1, sg.slot});
            }
        }
    }
    for (int t = 0; t < tiles; ++t)
        for (int k = 0; k < Kb; ++k)
            if (done[t][k] != 1) return fail("block not done exactly once", tiles, Kb, G);
    for (auto& kv : pieces) {
        const int rel = kv.first;
        auto& ps = kv.second;
        const long long ts = static_cast<long long>(rel) * Kb;
        const int c_lo = sc.cta_of(ts), c_hi = sc.cta_of(ts + Kb - 1);
        const bool before = sc.lo(c_lo) < ts;
        if (static_cast<int>(ps.size()) != c_hi - c_lo + 1) return fail("piece count", tiles, Kb, G);
        for (size_t j = 0; j < ps.size(); ++j) {
            if (ps[j].cta != c_lo + static_cast<int>(j)) return fail("pieces not in CTA order", tiles, Kb, G);
            if (j > 0 && ps[j].kb0 != ps[j - 1].kb1) return fail("pieces not in K order", tiles, Kb, G);
            if (ps[j].slot != sc.slot_in_tile(ps[j].cta, c_lo, before)) return fail("slot_in_tile", tiles, Kb, G);
        }
        if (ps.front().kb0 != 0 || ps.back().kb1 != Kb) return fail("pieces do not span the tile", tiles, Kb, G);
    }
    return 0;
}

int main() {
    const int kbs[] = {1, 2, 3, 7, 8, 9, 16, 40, 56, 64, 128};
    const int gs[] = {1, 2, 16, 132, 148, 160};
    int cases = 0;
    for (int g : gs)
        for (int kb : kbs)
            for (int tiles = 1; tiles <= 700; tiles += (tiles < 64 ? 1 : 13))
                for (int allow = 0; allow < 2; ++allow) {
                    if (check(tiles, kb, g, allow != 0)) return 1;
                    ++cases;
                }
    // the bench's shapes: forward, grouped, wgrad, accumulation, Dgrad
    const int shapes[][3] = {{256, 56, 148}, {1144, 56, 148}, {448, 64, 148}, {32, 128, 148}, {896, 16, 148}};
    for (auto& s : shapes) {
        if (check(s[0], s[1], s[2], true)) return 1;
        ++cases;
    }
    std::printf("ok %d\n", cases);
    return 0;
}
