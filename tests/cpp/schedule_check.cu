// Host-only check of the tile schedule (no CUDA call is made at run time).
// Invariants, for several problem sets, tile widths and grid caps:
//  * every tile's K-stages 0..nk-1 are covered exactly once, by segments in K order;
//  * a split tile has nseg > 1 segments with seg = 0..nseg-1 and consecutive workspace
//    slots; a whole tile has split = -1;
//  * with split_tail on and uniform K, the CTAs' stage counts differ by at most one
//    plus one tile's worth less than the whole-tile share, i.e. max - min <= nk;
//  * the small-grid fill keeps the whole grid when there are fewer tiles than CTAs and
//    leaves every CTA within one stage of the even share;
//  * the list offsets are monotone and end at the item count;
//  * M-fusion runs form where A rows follow one another, and only there.
#include "nvfp4_gemm.cu"
#include "prepack.cu"

#include <cstdio>
#include <map>
#include <tuple>

static int fails = 0;
#define CHECK(cond, ...)                         \
    do {                                         \
        if (!(cond)) {                           \
            ++fails;                             \
            std::printf("FAIL %s: ", #cond);     \
            std::printf(__VA_ARGS__);            \
            std::printf("\n");                   \
        }                                        \
    } while (0)

static void check(const std::vector<ActiveGroup> &gs, int bm, int bn, int cap, int split)
{
    Schedule sc = build_schedule(gs, bm, bn, cap, split);
    const int lists = sc.grid * kPipes;
    CHECK((int)sc.list_begin.size() == lists + 1, "lists");
    CHECK(sc.list_begin[lists] == sc.items.size(), "end");
    std::map<std::tuple<int, int, int>, std::vector<WorkItem>> by_tile;
    std::vector<int64_t> load(lists, 0);
    bool any_split = false;
    for (int l = 0; l < lists; ++l) {
        CHECK(sc.list_begin[l] <= sc.list_begin[l + 1], "monotone");
        bool seen_whole = false;
        for (uint32_t i = sc.list_begin[l]; i < sc.list_begin[l + 1]; ++i) {
            const WorkItem &w = sc.items[i];
            any_split = any_split || w.split >= 0;
            CHECK(!(seen_whole && w.split >= 0), "split segment after a whole tile in list %d", l);
            seen_whole = seen_whole || w.split < 0;
            by_tile[{w.group, w.tile_m, w.tile_n}].push_back(w);
            load[l] += w.kb_end - w.kb_begin;
            CHECK(w.kb_end > w.kb_begin, "empty segment");
        }
    }
    size_t tiles = 0;
    bool uniform = true;
    int nk0 = -1;
    for (size_t g = 0; g < gs.size(); ++g) {
        const int tm = (gs[g].M + bm - 1) / bm, tn = (gs[g].N + bn - 1) / bn, nk = (gs[g].K / 64 + 3) / 4;
        uniform = uniform && (nk0 < 0 || nk == nk0);
        nk0 = nk;
        tiles += (size_t)tm * tn;
        for (int n = 0; n < tn; ++n)
            for (int m = 0; m < tm; ++m) {
                auto it = by_tile.find({(int)g, m, n});
                CHECK(it != by_tile.end(), "tile missing g=%zu m=%d n=%d", g, m, n);
                if (it == by_tile.end())
                    continue;
                auto segs = it->second;
                std::sort(segs.begin(), segs.end(), [](const WorkItem &a, const WorkItem &b) { return a.seg < b.seg; });
                int k = 0;
                for (size_t j = 0; j < segs.size(); ++j) {
                    CHECK(segs[j].seg == (int)j && segs[j].nseg == (int)segs.size(), "seg numbering");
                    CHECK(segs[j].kb_begin == k, "gap or overlap at k=%d", k);
                    k = segs[j].kb_end;
                    if (segs.size() > 1)
                        CHECK(segs[j].split >= 0 && segs[j].ws_slot == segs[0].ws_slot + (int)j &&
                                  segs[j].split == segs[0].split, "split bookkeeping");
                    else
                        CHECK(segs[j].split == -1, "whole tile marked split");
                }
                CHECK(k == nk, "K not covered: %d of %d", k, nk);
            }
    }
    CHECK(by_tile.size() == tiles, "extra tiles");
    CHECK(split || !any_split, "split with split_tail off");
    const int64_t mx = *std::max_element(load.begin(), load.end()), mn = *std::min_element(load.begin(), load.end());
    if (any_split) {
        CHECK(mx - mn <= 1, "imbalance %lld..%lld (bn %d cap %d)", (long long)mn, (long long)mx, bn, cap);
    } else if (uniform) {
        // whole tiles dealt round-robin: tile counts differ by at most one
        CHECK(mx - mn <= nk0, "whole-tile imbalance %lld..%lld", (long long)mn, (long long)mx);
        // and where splitting was on, it was skipped only when it would save little
        const int64_t G = sc.grid, unb = (int64_t)((tiles + G - 1) / G) * nk0, bal = ((int64_t)tiles * nk0 + G - 1) / G;
        if (split && (int64_t)tiles > G && tiles % G != 0)
            CHECK(unb - bal < 2 || (unb - bal) * 8 < unb, "split skipped though it saves %lld of %lld", (long long)(unb - bal),
                  (long long)unb);
    }
}

static ActiveGroup G(int M, int N, int K) { return ActiveGroup{M, N, K, 0, nullptr, nullptr, nullptr, nullptr, nullptr}; }

// The swapped-operand kernel's schedule: items of one 128-row B tile against one or two
// 128-row A tiles, whole or cut along K (stream-K).
//  * every (group, B tile, A tile pair) is covered over K exactly once, by segments in K
//    order, each at least kSwapMinSeg K-stages long when the tile is cut;
//  * split bookkeeping: one split id per tile with ntok counters, consecutive slots per
//    segment (ntok each);
//  * the item's MMA widths and A box follow from M;
//  * each list walks its items in tile order;
//  * with stream-K the lists' stage counts differ by at most one tile's worth.
// Returns the busiest list's shared-memory stages.
static int64_t check_swap(const std::vector<ActiveGroup> &gs, int cap, bool stream_k)
{
    Schedule sc = build_swap_schedule(gs, cap, stream_k);
    const int G = sc.grid;
    CHECK(G >= 1 && G <= cap, "grid %d of %d", G, cap);
    CHECK((int)sc.list_begin.size() == G + 1 && sc.list_begin[G] == sc.items.size(), "lists");
    std::map<std::tuple<int, int, int>, std::vector<WorkItem>> by_tile;
    std::vector<int64_t> load(G, 0);
    int64_t max_tile = 0;
    int splits = 0, slots = 0;
    bool any_split = false;
    for (int l = 0; l < G; ++l) {
        CHECK(sc.list_begin[l] <= sc.list_begin[l + 1], "monotone");
        std::tuple<int, int, int> prev{-1, -1, -1};
        for (uint32_t i = sc.list_begin[l]; i < sc.list_begin[l + 1]; ++i) {
            const WorkItem &w = sc.items[i];
            const std::tuple<int, int, int> key{w.group, w.tile_n, w.tile_m};
            CHECK(prev < key, "list %d not in tile order", l);
            prev = key;
            by_tile[{w.group, w.tile_n, w.tile_m}].push_back(w);
            const int ntok = swap_ntok(w.flags);
            load[l] += (int64_t)(w.kb_end - w.kb_begin) * ntok;
            CHECK(w.kb_end > w.kb_begin, "empty segment");
            any_split = any_split || w.split >= 0;
        }
    }
    size_t tiles = 0;
    for (size_t g = 0; g < gs.size(); ++g) {
        const int M = gs[g].M, ntt = (M + 127) / 128, tw = (gs[g].N + 127) / 128, nk = (gs[g].K / 64 + 3) / 4;
        for (int wt = 0; wt < tw; ++wt)
            for (int t0 = 0; t0 < ntt; t0 += 2) {
                ++tiles;
                auto it = by_tile.find({(int)g, wt, t0});
                CHECK(it != by_tile.end(), "tile missing g=%zu w=%d t0=%d", g, wt, t0);
                if (it == by_tile.end())
                    continue;
                auto segs = it->second;
                std::sort(segs.begin(), segs.end(), [](const WorkItem &a, const WorkItem &b) { return a.seg < b.seg; });
                const int ntok = std::min(2, ntt - t0);
                max_tile = std::max<int64_t>(max_tile, (int64_t)nk * ntok);
                int k = 0;
                for (size_t j = 0; j < segs.size(); ++j) {
                    const WorkItem &w = segs[j];
                    CHECK(swap_ntok(w.flags) == ntok, "ntok");
                    CHECK(swap_nt(w.flags, 0) == round16(std::min(128, M - 128 * t0)), "nt0");
                    CHECK(ntok == 1 || swap_nt(w.flags, 1) == round16(std::min(128, M - 128 * (t0 + 1))), "nt1");
                    CHECK(swap_box_rows(w.flags) == (M <= 128 ? round16(M) : 128), "box");
                    CHECK(w.a_row == 128 * t0 && w.tile_m == t0, "a rows");
                    CHECK(w.seg == (int)j && w.nseg == (int)segs.size(), "seg numbering");
                    CHECK(w.kb_begin == k, "gap or overlap at k=%d", k);
                    k = w.kb_end;
                    if (segs.size() > 1) {
                        CHECK(w.kb_end - w.kb_begin >= kSwapMinSeg, "segment of %d stages", w.kb_end - w.kb_begin);
                        CHECK(w.split == segs[0].split && w.ws_slot == segs[0].ws_slot + (int)j * ntok, "split bookkeeping");
                    } else {
                        CHECK(w.split == -1, "whole tile marked split");
                    }
                }
                CHECK(k == nk, "K not covered: %d of %d", k, nk);
                if (segs.size() > 1) {
                    splits += ntok;
                    slots += (int)segs.size() * ntok;
                }
            }
    }
    CHECK(by_tile.size() == tiles, "extra tiles");
    CHECK(sc.splits == splits && sc.ws_slots == slots, "split counts %d/%d slots %d/%d", sc.splits, splits, sc.ws_slots,
          slots);
    CHECK(stream_k || !any_split, "split with stream-K off");
    const int64_t mx = *std::max_element(load.begin(), load.end()), mn = *std::min_element(load.begin(), load.end());
    if (any_split)
        CHECK(mx - mn <= max_tile, "stream-K imbalance %lld..%lld", (long long)mn, (long long)mx);
    return mx;
}

int main()
{
    std::vector<std::vector<ActiveGroup>> sets = {
        {G(80, 4096, 7168), G(176, 4096, 7168), G(128, 4096, 7168), G(72, 4096, 7168), G(64, 4096, 7168),
         G(248, 4096, 7168), G(96, 4096, 7168), G(160, 4096, 7168)},
        {G(40, 7168, 2048), G(76, 7168, 2048), G(168, 7168, 2048), G(72, 7168, 2048), G(164, 7168, 2048),
         G(148, 7168, 2048), G(196, 7168, 2048), G(160, 7168, 2048)},
        {G(192, 3072, 4096), G(320, 3072, 4096)},
        {G(128, 4096, 1536), G(384, 4096, 1536)},
        {G(130, 2048, 1024), G(60, 1024, 1024), G(200, 1536, 1024), G(129, 520, 1024)},
        {G(200, 384, 1536), G(64, 256, 512), G(129, 136, 768)},
        {G(1, 8, 64)},
        {G(300, 72, 2304), G(5, 8, 64)},
    };
    // single-CTA tiles 128 x 128 and 128 x 256; CTA-pair tiles 256 x 256 (grid = pairs)
    const int shapes[3][2] = {{128, 128}, {128, 256}, {256, 256}};
    for (auto &gs : sets)
        for (auto &sh : shapes)
            for (int cap : {152, 148, 76, 40, 7, 1})
                for (bool split : {true, false})
                    check(gs, sh[0], sh[1], cap, split);
    for (auto &gs : sets)
        for (int cap : {152, 148, 76, 40, 7, 1})
            for (bool sk : {true, false})
                check_swap(gs, cap, sk);
    // the CTA-pair swapped kernel's schedule: tiles of 256 rows of B x up to 256 rows of A,
    // covered over K exactly once, split bookkeeping consistent, lists in tile order
    for (auto &gs : sets)
        for (int cap : {76, 40, 7, 1})
            for (bool sk : {true, false}) {
                const Schedule sc = build_swap_pair_schedule(gs, cap, sk);
                CHECK(sc.grid >= 1 && sc.grid <= cap && sc.list_begin[sc.grid] == sc.items.size(), "pair lists");
                std::map<std::tuple<int, int, int>, std::vector<WorkItem>> by_tile;
                int splits = 0, slots = 0;
                for (int l = 0; l < sc.grid; ++l) {
                    std::tuple<int, int, int> prev{-1, -1, -1};
                    for (uint32_t i = sc.list_begin[l]; i < sc.list_begin[l + 1]; ++i) {
                        const WorkItem &w = sc.items[i];
                        const std::tuple<int, int, int> key{w.group, w.tile_n, w.tile_m};
                        CHECK(prev < key, "pair list %d order", l);
                        prev = key;
                        by_tile[key].push_back(w);
                        CHECK(swap_pair_nt(w.flags) == round16(std::min(gs[w.group].M, 256)), "pair nt");
                    }
                }
                size_t tiles = 0;
                for (size_t g = 0; g < gs.size(); ++g) {
                    const int nk = (gs[g].K / 64 + 3) / 4;
                    for (int wt = 0; wt < (gs[g].N + 255) / 256; ++wt)
                        for (int t = 0; t < (gs[g].M + 255) / 256; ++t) {
                            ++tiles;
                            auto segs = by_tile[{(int)g, wt, t}];
                            std::sort(segs.begin(), segs.end(),
                                      [](const WorkItem &a, const WorkItem &b) { return a.seg < b.seg; });
                            int k = 0;
                            for (size_t j = 0; j < segs.size(); ++j) {
                                CHECK(segs[j].kb_begin == k && segs[j].seg == (int)j, "pair coverage");
                                k = segs[j].kb_end;
                                if (segs.size() > 1)
                                    CHECK(segs[j].ws_slot == segs[0].ws_slot + (int)j && segs[j].split == segs[0].split,
                                          "pair split bookkeeping");
                            }
                            CHECK(k == nk, "pair K coverage");
                            if (segs.size() > 1) {
                                splits += 1;
                                slots += (int)segs.size();
                            }
                        }
                }
                CHECK(by_tile.size() == tiles && sc.splits == splits && sc.ws_slots == slots, "pair counts");
            }
    // the K = 7168 MoE set goes stream-K on 152 SMs (whole items would leave a short last
    // wave); the K = 2048 set's whole items already balance within a stage or two. Both
    // stay within a few stages of the even share.
    CHECK(build_swap_schedule(sets[0], 152, true).splits > 0, "moe K=7168: stream-K");
    for (int i = 0; i < 2; ++i) {
        const Schedule sc = build_swap_schedule(sets[i], 152, true);
        CHECK(sc.grid == 152, "moe set %d: grid %d", i, sc.grid);
        const int64_t mx = check_swap(sets[i], 152, true);
        int64_t total = 0;
        for (const WorkItem &w : sc.items)
            total += (int64_t)(w.kb_end - w.kb_begin) * swap_ntok(w.flags);
        CHECK(mx <= (total + 151) / 152 + 2 * kSwapMinSeg, "moe set %d: busiest list %lld of %lld", i, (long long)mx,
              (long long)total);
        std::printf("swap-AB moe set %d: %lld stages over 152 CTAs, busiest %lld, %d split tiles\n", i, (long long)total,
                    (long long)mx, sc.splits);
    }
    // the two MoE sets split at both tile widths, and the K=2048 set at width 128 does not
    auto splits = [](const std::vector<ActiveGroup> &gs, int bn) {
        Schedule sc = build_schedule(gs, 128, bn, 152, true);
        return sc.splits;
    };
    CHECK(splits(sets[0], 128) > 0 && splits(sets[0], 256) > 0, "moe K=7168 should split");
    CHECK(splits(sets[1], 128) == 0 && splits(sets[1], 256) > 0, "moe K=2048 split choice");
    // the problem set of the GPU split test: splits at grids 70, 72 (width 128) and 36, 37
    // (width 256), not at 152 or 7
    const std::vector<ActiveGroup> t4 = {G(130, 2048, 2048), G(60, 1024, 2048), G(200, 1536, 2048), G(129, 520, 2048)};
    CHECK(build_schedule(t4, 128, 128, 70, true).splits > 0 && build_schedule(t4, 128, 128, 72, true).splits > 0, "t4 128");
    CHECK(build_schedule(t4, 128, 256, 36, true).splits > 0 && build_schedule(t4, 128, 256, 37, true).splits > 0, "t4 256");
    CHECK(build_schedule(t4, 128, 128, 152, true).splits == 0 && build_schedule(t4, 128, 256, 7, true).splits == 0, "t4 none");
    {
        const Schedule sc = build_schedule(t4, 128, 128, 72, true);
        int mx = 0;
        for (const WorkItem &w : sc.items)
            mx = std::max(mx, w.nseg);
        CHECK(mx == 8, "t4 at 72 CTAs: one-stage segments, %d per tile", mx);
    }
    for (auto cap : {70, 72, 36, 37, 7, 152})
        for (auto &sh : shapes)
            check(t4, sh[0], sh[1], cap, true);
    // the small-grid fill (split mode 3 on single CTAs): the two-group K = 4096 set's 120
    // tiles of 128 x 128 spread over all 152 CTAs, every CTA within one stage of the even
    // share; with the tail mode alone the grid stays at 120 CTAs of whole tiles
    {
        const std::vector<ActiveGroup> g2 = {G(192, 3072, 4096), G(320, 3072, 4096)};
        const Schedule f = build_schedule(g2, 128, 128, 152, kSplitFill);
        CHECK(f.grid == 152 && f.splits > 0, "fill: grid %d, %d split tiles", f.grid, f.splits);
        const Schedule t = build_schedule(g2, 128, 128, 152, kSplitTail);
        CHECK(t.grid == 120 && t.splits == 0, "tail: grid %d, %d split tiles", t.grid, t.splits);
        check(g2, 128, 128, 152, kSplitFill);
        // one tile: spread where it pays (16 stages over 152 CTAs saves 15), at least the tile itself
        const std::vector<ActiveGroup> one = {G(100, 128, 4096)};
        CHECK(build_schedule(one, 128, 128, 152, kSplitFill).grid > 1, "fill of a single tile");
        for (auto cap : {152, 100, 37, 1})
            for (auto &sh : shapes)
                check(t4, sh[0], sh[1], cap, kSplitFill);
        CHECK(split_for(0, 3) == kSplitFill && split_for(kVariantPair, 3) == kSplitNone && split_for(0, 1) == kSplitTail &&
                  split_for(kVariantPair, 2) == kSplitTail && split_for(0, 0) == kSplitNone,
              "split_for");
    }
    // the pair kernel's split test set (256 x 256 tiles): 8 + 4 + 6 + 3 = 21 tiles at K = 2048,
    // so 19 and 20 pairs split the short last wave, 21 and more do not
    CHECK(build_schedule(t4, 256, 256, 19, true).splits > 0 && build_schedule(t4, 256, 256, 20, true).splits > 0, "pair split");
    CHECK(build_schedule(t4, 256, 256, 76, true).splits == 0, "pair no split");
    // the MoE sets on 76 pairs: K=7168 splits (128 tiles), K=2048 splits (224 tiles)
    CHECK(build_schedule(sets[0], 256, 256, 76, true).splits > 0, "pair moe K=7168");
    // the automatic choice on a 152-SM device that fits 76 CTA pairs: pairs for the two
    // MoE-shaped sets, single CTAs for the two-group sets and the tiny one
    {
        DeviceState ds;
        ds.sm_count = 152;
        ds.pair_clusters = 76;
        const std::vector<ActiveGroup> g2a = {G(128, 4096, 1536), G(384, 4096, 1536)};
        const std::vector<ActiveGroup> g2b = {G(192, 3072, 4096), G(320, 3072, 4096)};
        const std::vector<ActiveGroup> tiny = {G(64, 512, 512), G(128, 512, 512)};
        CHECK(choose_variant(sets[0], ds, 0, 1) == kVariantPair, "moe K=7168 -> pairs");
        CHECK(choose_variant(sets[1], ds, 0, 1) == kVariantPair, "moe K=2048 -> pairs");
        CHECK(choose_variant(g2a, ds, 0, 1) == 0, "g2 K=1536 -> single");
        CHECK(choose_variant(g2b, ds, 0, 1) == 0, "g2 K=4096 -> single");
        CHECK(choose_variant(tiny, ds, 0, 1) == 0, "tiny -> single");
        // decode-sized sets (every group at most 32 rows of A): the swapped-operand kernel
        const std::vector<ActiveGroup> dec = {G(8, 4096, 7168), G(32, 4096, 7168), G(1, 4096, 7168)};
        CHECK(choose_variant(dec, ds, 0, 1) == kVariantSwap, "decode -> swap-AB");
        const std::vector<ActiveGroup> mid = {G(33, 4096, 7168), G(8, 4096, 7168)};
        CHECK(choose_variant(mid, ds, 0, 1) != kVariantSwap, "33 rows -> not swap-AB");
    }
    // M-fusion runs (a_runs): A rows that follow one another with the same K join the
    // previous group's run; a gap, a change of K or of the scale layout, row-major SFA rows
    // that do not follow, or a run longer than 32-bit row coordinates starts a new one.
    {
        auto P = [](uintptr_t x) { return reinterpret_cast<const void *>(x); };
        auto AG = [&](int M, int K, uintptr_t a, int rm = 0, uintptr_t sfa = 0x100000) {
            return ActiveGroup{M, 256, K, rm, P(a), P(0x1000), P(sfa), P(0x2000), nullptr};
        };
        const uintptr_t base = 0x10000000;
        // 3 contiguous groups (K = 1024: 512 bytes per row), then a gap, then 2 contiguous
        std::vector<ActiveGroup> gs = {AG(100, 1024, base), AG(37, 1024, base + 100 * 512),
                                       AG(5, 1024, base + 137 * 512), AG(64, 1024, base + 142 * 512 + 4096),
                                       AG(1, 1024, base + 206 * 512 + 4096)};
        ARuns r = a_runs(gs, true);
        CHECK(r.maps == 2, "runs: %d maps", r.maps);
        CHECK(r.head[0] == 0 && r.head[1] == 0 && r.head[2] == 0 && r.head[3] == 3 && r.head[4] == 3, "run heads");
        CHECK(r.row0[1] == 100 && r.row0[2] == 137 && r.row0[4] == 64, "run rows");
        CHECK(r.rows[0] == 142 && r.rows[3] == 65, "run lengths");
        r = a_runs(gs, false);
        CHECK(r.maps == 5 && r.head[2] == 2 && r.row0[2] == 0 && r.rows[2] == 5, "fusion off");
        // a change of K breaks a run even where the bytes follow
        gs = {AG(100, 1024, base), AG(50, 512, base + 100 * 512)};
        CHECK(a_runs(gs, true).maps == 2, "K change");
        // row-major scales: SFA rows (K/16 bytes each) must follow too; a layout change breaks
        gs = {AG(100, 1024, base, 1, 0x200000), AG(50, 1024, base + 100 * 512, 1, 0x200000 + 100 * 64)};
        CHECK(a_runs(gs, true).maps == 1, "row-major SFA follows");
        gs[1].SFA = P(0x200000 + 100 * 64 + 16);
        CHECK(a_runs(gs, true).maps == 2, "row-major SFA gap");
        gs = {AG(100, 1024, base, 0), AG(50, 1024, base + 100 * 512, 1)};
        CHECK(a_runs(gs, true).maps == 2, "layout change");
        // 32-bit row coordinates: a run stops before passing INT32_MAX rows
        gs.clear();
        uintptr_t a = base;
        for (int i = 0; i < 200; ++i) {
            gs.push_back(AG(1 << 24, 64, a));
            a += (size_t)(1 << 24) * 32;
        }
        r = a_runs(gs, true);
        CHECK(r.maps == 2 && r.rows[0] == 127LL * (1 << 24) && r.head[127] == 127, "row limit: %d maps", r.maps);
    }
    std::printf(fails ? "FAILED %d\n" : "ok\n", fails);
    return fails ? 1 : 0;
}
