// fanout_plan.cu -- host-side planning of a fan-out launch: how many chunks the
// shared prefix is split into and where their boundaries lie.
//
// The units of a fan-out launch are (prefix chunk, KV head, row pair), launched
// chunk-major with the row pair fastest; each writes one partial per row, and
// the merge joins them ("AHBM Agentic Runtime Architecture", sections 3.3-3.4:
// every sequence shard produces a partial state, merged by row).  A unit costs
// its prefix tiles, the suffix tiles folded into its chunk (branch b's suffix
// goes to chunk b % n_chunks) and a fixed cost of about 4.3 tiles (set-up,
// first loads from HBM, epilogue: per-CTA clock stamps on GB300); every chunk
// adds a partial per row to the join, about one tile more.
//
// The plan is chosen by simulating the block scheduler: units in launch order,
// each started on the SM that frees first, the makespan minimised.  The
// simulation reproduced a measured launch's timeline to within 3% (SMs running
// dry at 163 / 227 / 241 us simulated against 172 / 215 / 247 us measured).
// Besides equal chunks it tries shaped splits (one longer chunk, one shorter)
// and longest-first plans: when per-chunk units fit the SMs k times with SMs
// left over, k long chunks keep k x units SMs busy for the whole launch and
// the remaining tiles go to a few shorter chunks, longest first, for the other
// SMs (R = 147 stacked rows, 40 units per chunk, 152 SMs: chunks of 140, 140,
// 140, 66 and 26 tiles, 250 -> 236 us against the previous best of 7 chunks;
// the 8 x 20 prefill 248 -> 234 us).  A short local search moving tiles between
// chunks refines the best plan.  The first call of a shape spends up to a few
// milliseconds of host time planning; plans are cached per shape.
//
// Units that hold a single row tile (all stacked rows of a KV head in one
// 128-row tile: few rows, a decode) are bound by HBM bandwidth, not by their
// SM: the prefix bytes leave HBM at the same rate whether 112 or 152 CTAs
// read them, while every extra chunk adds a partial to write and merge and a
// unit's fixed cost.  Their chunk count is capped so that the units take at
// most 4/5 of the SMs (measured on GB300, 65536-token prefix, 8 KV heads,
// 16 rows: 14-15 chunks 59.9 us, 16 chunks 61.9 us, 19 chunks 64.0 us, the
// launch and its merge).  Not over a paged KV cache: small pages arrive in
// small TMA boxes, which bound each SM's read rate, so a paged launch wants
// every SM (16-token pages: 74 us with 19 chunks, 88 us with 15).
#include <algorithm>
#include <cmath>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include "ra_internal.h"

namespace ra {

namespace {

constexpr int kTileRows = 128;  // query rows of an M tile / keys of a KV tile
constexpr int kMaxPlanChunks = 64;
constexpr double kUnitFixedTiles = 4.3;     // a unit's set-up, first loads and epilogue, in tiles
constexpr double kMergeTilesPerChunk = 1.0;  // the join's extra cost per partial, in tiles

struct Shape {
    int n_tiles;       // prefix KV tiles
    double s_tiles;    // suffix tiles of one branch
    int n_branches, n_mpairs, Hkv, n_sm;
    bool one_tile;     // the stacked rows fit one row tile (bandwidth-bound units)
};

// Largest chunk count the plan may use.
int max_chunks(const Shape& sh) {
    int c = std::min(sh.n_tiles, kMaxPlanChunks);
    if (sh.one_tile) c = std::min(c, std::max(1, 4 * sh.n_sm / (5 * sh.Hkv * sh.n_mpairs)));
    return c;
}

// Folded suffix tiles an average unit of chunk c carries.
double folded(const Shape& sh, int n_chunks, int c) {
    if (sh.s_tiles == 0) return 0;
    const int nbr = sh.n_branches / n_chunks + (c < sh.n_branches % n_chunks ? 1 : 0);
    return sh.s_tiles * nbr / sh.n_mpairs;
}

// Makespan (in tile units) of the greedy schedule of a plan.
double simulate(const Shape& sh, const std::vector<int>& prefix_tiles) {
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < sh.n_sm; ++i) free_at.push(0.0);
    double makespan = 0;
    const int n = static_cast<int>(prefix_tiles.size());
    for (int c = 0; c < n; ++c) {
        const double cost = prefix_tiles[c] + folded(sh, n, c) + kUnitFixedTiles;
        for (long long u = 0; u < static_cast<long long>(sh.Hkv) * sh.n_mpairs; ++u) {
            const double t = free_at.top() + cost;
            free_at.pop();
            free_at.push(t);
            makespan = std::max(makespan, t);
        }
    }
    return makespan;
}

// Prefix tiles per chunk for target work weights (prefix + folded suffix), at
// least one tile each, summing to n_tiles (cumulative rounding).
std::vector<int> split(const Shape& sh, const std::vector<double>& weight) {
    const int n = static_cast<int>(weight.size());
    double wsum = 0;
    for (double w : weight) wsum += w;
    double total = sh.n_tiles;
    for (int c = 0; c < n; ++c) total += folded(sh, n, c);
    std::vector<double> want(n);
    double sum = 0;
    for (int c = 0; c < n; ++c) {
        want[c] = std::max(1.0, total * weight[c] / wsum - folded(sh, n, c));
        sum += want[c];
    }
    std::vector<int> tiles(n);
    double acc = 0;
    int prev = 0;
    for (int c = 0; c < n; ++c) {
        acc += want[c] * sh.n_tiles / sum;
        int e = static_cast<int>(acc + 0.5);
        e = std::max(e, prev + 1);
        e = std::min(e, sh.n_tiles - (n - 1 - c));
        if (c == n - 1) e = sh.n_tiles;
        tiles[c] = e - prev;
        prev = e;
    }
    return tiles;
}

struct Plan {
    double cost = -1;
    std::vector<int> tiles;
};

Plan search(const Shape& sh) {
    Plan best;
    const int max_c = max_chunks(sh);
    const long long per_chunk = static_cast<long long>(sh.Hkv) * sh.n_mpairs;
    auto consider = [&](const std::vector<int>& tiles, double penalty) {
        const double cost = simulate(sh, tiles) + penalty + kMergeTilesPerChunk * tiles.size();
        if (best.cost < 0 || cost < best.cost) {
            best.cost = cost;
            best.tiles = tiles;
        }
    };
    // equal chunks: with equal units the greedy schedule is whole waves, so the
    // scan uses that closed form, then simulates the best three counts
    const double work = sh.n_tiles + sh.s_tiles * sh.n_branches / sh.n_mpairs;  // tiles per (KV head, row pair)
    int c0 = 1;
    double c0_cost = -1;
    for (int c = 1; c <= max_c; ++c) {
        const long long waves = (per_chunk * c + sh.n_sm - 1) / sh.n_sm;
        const double cost = waves * (work / c + kUnitFixedTiles) + kMergeTilesPerChunk * c;
        if (c0_cost < 0 || cost < c0_cost) {
            c0_cost = cost;
            c0 = c;
        }
    }
    const int c_lo = std::max(1, c0 - 1), c_hi = std::min(max_c, c0 + 1);
    for (int c = c_lo; c <= c_hi; ++c) consider(split(sh, std::vector<double>(c, 1.0)), 0);
    // shaped splits (chunk 0 or 1 longer, the last shorter) where the last wave is
    // partial and the waves are few enough for it to matter
    for (int c = std::max(2, c_lo); c <= c_hi; ++c) {
        const long long units = per_chunk * c;
        if (units % sh.n_sm == 0 || units > 4LL * sh.n_sm) continue;
        for (int big_at = 0; big_at <= 1; ++big_at)
            for (int ib = 0; ib <= 10; ++ib)
                for (int is = 0; is <= 4; ++is) {
                    std::vector<double> w(c, 1.0);
                    w[big_at] = 1.0 + 0.2 * ib;
                    w[c - 1] = std::min(w[c - 1], 0.2 + 0.2 * is);
                    // a shaped plan must beat the equal one clearly: the model is approximate
                    consider(split(sh, w), 1.0);
                }
    }
    // Longest-first plans for a chunk count that leaves SMs over: k long chunks
    // whose k * per_chunk units keep that many SMs busy for the whole launch,
    // their size the balanced makespan less a unit's fixed and folded cost, and
    // the remaining tiles in m shorter chunks of decreasing size for the other
    // SMs, each tried at a few sizes of the long chunks and decay ratios.
    const int q = static_cast<int>(sh.n_sm / per_chunk);
    for (int k = std::max(1, q - 1); k <= q; ++k)
        for (int m = 1; m <= 4; ++m) {
            const int n = k + m;
            if (n > max_c) continue;
            double fold_sum = 0;
            for (int c = 0; c < n; ++c) fold_sum += folded(sh, n, c);
            const double work_all = per_chunk * (sh.n_tiles + fold_sum + n * kUnitFixedTiles);
            const double long_tiles = work_all / sh.n_sm - fold_sum / n - kUnitFixedTiles;
            for (int ia = -2; ia <= 1; ++ia) {
                const int L = static_cast<int>(long_tiles * (1.0 + 0.02 * ia) + 0.5);
                const int rest = sh.n_tiles - k * L;
                if (L < 1 || rest < m) continue;
                for (int ir = 0; ir < 6; ++ir) {
                    const double rho = 0.25 + 0.15 * ir;
                    std::vector<double> w(m);
                    double wsum = 0;
                    for (int i = 0; i < m; ++i) wsum += (w[i] = std::pow(rho, i));
                    std::vector<int> tiles(k, L);
                    int left = rest;
                    for (int i = 0; i < m; ++i) {
                        int t = (i == m - 1) ? left : std::max(1, static_cast<int>(rest * w[i] / wsum + 0.5));
                        t = std::min(t, left - (m - 1 - i));
                        tiles.push_back(t);
                        left -= t;
                    }
                    if (left != 0 || tiles.back() < 1) continue;
                    consider(tiles, 1.0);
                }
            }
        }
    // Refinement: move tiles between two chunks while that shortens the
    // simulated makespan (longest chunks first), a bounded number of trials.
    if (best.tiles.size() > 1) {
        int trials = 0;
        for (int d = 8; d >= 1 && trials < 200; d /= 2) {
            bool moved = true;
            while (moved && trials < 200) {
                moved = false;
                const int n = static_cast<int>(best.tiles.size());
                for (int i = 0; i < n && !moved; ++i)
                    for (int j = 0; j < n && !moved; ++j) {
                        if (i == j || best.tiles[i] - d < 1) continue;
                        std::vector<int> t = best.tiles;
                        t[i] -= d;
                        t[j] += d;
                        std::sort(t.begin(), t.end(), std::greater<int>());
                        const double before = best.cost;
                        consider(t, 1.0);
                        ++trials;
                        moved = best.cost < before;
                    }
            }
        }
    }
    return best;
}

std::mutex g_plan_mu;
std::map<std::tuple<int, int, int, int, int, int>, std::vector<int>> g_plans;

}  // namespace

int fanout_slots(int R, int Hq, int Hkv, int n_chunks, int S_prefix, int S_suffix, int* split_prefix,
                 int* suffix_slot0) {
    const int rows_per_tile = kTileRows / (Hq / Hkv);
    if (split_prefix) *split_prefix = (R <= rows_per_tile) ? 1 : 0;
    if (suffix_slot0) *suffix_slot0 = 0;
    // with a prefix the suffixes are folded into prefix units; without one,
    // suffix units write slot 0
    return S_prefix > 0 ? n_chunks : (S_suffix > 0 ? 1 : 0);
}

void fanout_plan(int R, int S_prefix, int S_suffix, int n_branches, int Hq, int Hkv, int n_sm, int* n_chunks,
                 int* chunk_start, bool paged) {
    const int rows_per_tile = kTileRows / (Hq / Hkv);
    Shape sh;
    sh.n_mpairs = (R + 2 * rows_per_tile - 1) / (2 * rows_per_tile);
    sh.n_tiles = (S_prefix + kTileRows - 1) / kTileRows;
    sh.s_tiles = (S_suffix > 0 && S_prefix > 0) ? (S_suffix + kTileRows - 1) / kTileRows : 0;
    sh.n_branches = n_branches;
    sh.Hkv = Hkv;
    sh.n_sm = n_sm > 0 ? n_sm : 1;
    sh.one_tile = R <= rows_per_tile && !paged;
    if (sh.n_tiles == 0 || sh.n_mpairs == 0) {
        *n_chunks = 0;
        if (chunk_start) chunk_start[0] = 0;
        return;
    }
    const auto key = std::make_tuple(sh.n_mpairs, sh.n_tiles, static_cast<int>(sh.s_tiles), n_branches, Hkv,
                                     sh.n_sm * 2 + (sh.one_tile ? 1 : 0));
    std::vector<int> tiles;
    {
        std::lock_guard<std::mutex> lock(g_plan_mu);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) tiles = it->second;
    }
    if (tiles.empty()) {
        tiles = search(sh).tiles;
        std::lock_guard<std::mutex> lock(g_plan_mu);
        if (g_plans.size() > 4096) g_plans.clear();
        g_plans[key] = tiles;
    }
    *n_chunks = static_cast<int>(tiles.size());
    if (chunk_start) {
        chunk_start[0] = 0;
        for (size_t c = 0; c < tiles.size(); ++c) chunk_start[c + 1] = chunk_start[c] + tiles[c];
    }
}

void fanout_split_equal(int n_chunks, int R, int S_prefix, int S_suffix, int n_branches, int Hq, int Hkv,
                        int* chunk_start) {
    const int rows_per_tile = kTileRows / (Hq / Hkv);
    Shape sh;
    sh.n_mpairs = std::max(1, (R + 2 * rows_per_tile - 1) / (2 * rows_per_tile));
    sh.n_tiles = (S_prefix + kTileRows - 1) / kTileRows;
    sh.s_tiles = (S_suffix > 0 && S_prefix > 0) ? (S_suffix + kTileRows - 1) / kTileRows : 0;
    sh.n_branches = n_branches;
    sh.Hkv = Hkv;
    sh.n_sm = 1;
    sh.one_tile = R <= rows_per_tile;
    const std::vector<int> tiles = split(sh, std::vector<double>(n_chunks, 1.0));
    chunk_start[0] = 0;
    for (int c = 0; c < n_chunks; ++c) chunk_start[c + 1] = chunk_start[c] + tiles[c];
}

}  // namespace ra
