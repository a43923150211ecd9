// ra_walk.h -- the ring-order KV walk, shared by the host (inspection API,
// launch sizing) and every kernel role (producer, MMA issuer, softmax).
//
// "RingAttention and Context Parallelism: Mathematical Foundations", section 3:
// the sequence is cut into N shards of L = S/N tokens and the query block of
// shard k holds, at ring step t, the KV shard (k - t) mod N.  Section 5: with a
// causal mask the keys a query cannot see are skipped.  On one GPU the ring
// becomes the order in which a query tile streams KV tiles from HBM: shard k
// first, then k-1, ..., 0, N-1, ..., k+1.
//
// Shard layouts (same page, section 5).  Storage row p of the q/k/v tensors
// sits in shard s = p / L at offset o = p % L; its position in the sequence
// (the one the causal mask compares) is
//   contiguous : p                          (shard k holds tokens [kL, (k+1)L))
//   zigzag     : o <  L/2 -> s*L/2 + o       (the sequence cut into 2N chunks of
//                o >= L/2 -> (2N-1-s)*L/2 + o - L/2   L/2; shard k holds chunks k
//                                                      and 2N-1-k, in that order)
//   striped    : o*N + s                    (shard k holds the tokens i with
//                                            i mod N = k, in increasing order)
// In all three, positions increase along the rows of a shard, so the keys of a
// shard that a query can see under the causal mask are a prefix of the shard's
// rows, and a query tile walks one contiguous range of tiles per shard.
#pragma once

#ifdef __CUDACC__
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

namespace ra {

enum : int { kLayoutContiguous = 0, kLayoutZigzag = 1, kLayoutStriped = 2 };

RA_HD int clampi(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

// Sequence position of storage row p.
RA_HD int layout_pos(int layout, int L, int n_shards, int p) {
    const int s = p / L, o = p - s * L;
    if (layout == kLayoutZigzag) {
        const int H = L / 2;
        return o < H ? s * H + o : (2 * n_shards - 1 - s) * H + (o - H);
    }
    if (layout == kLayoutStriped) return o * n_shards + s;
    return p;
}

// Keys of shard j whose sequence position is <= pos (a prefix of its rows).
RA_HD int shard_visible(int layout, int L, int n_shards, int j, int pos) {
    if (layout == kLayoutZigzag) {
        const int H = L / 2;
        return clampi(pos + 1 - j * H, 0, H) + clampi(pos + 1 - (2 * n_shards - 1 - j) * H, 0, H);
    }
    if (layout == kLayoutStriped) {
        if (pos < j) return 0;
        const int n = (pos - j) / n_shards + 1;  // rows o with o*N + j <= pos
        return n < L ? n : L;
    }
    return clampi(pos + 1 - j * L, 0, L);
}

// Storage row of sequence position pos in a zigzag-stored sequence of n_shards
// shards, cut into 2 n_shards chunks of `half` tokens: chunk c is the first half
// of shard c (c < n_shards) or the second half of shard 2 n_shards - 1 - c.  The
// inverse of layout_pos for the zigzag layout; half = 0 means rows are positions.
RA_HD int zigzag_row(int n_shards, int half, int pos) {
    if (half == 0) return pos;
    const int c = pos / half, o = pos - c * half;
    return (c < n_shards ? 2 * c * half : (4 * n_shards - 1 - 2 * c) * half) + o;
}

struct RingWalk {
    int n_shards;     // N
    int shard_len;    // L = S / N
    int tile;         // keys per KV tile
    int k;            // shard of the query tile
    int first_tiles;  // tiles taken from shard k
    int tiles_per_shard;
    int n_visited;    // shards visited: the first n_visited of the ring order; the rest see nothing
    int total;        // total KV tiles walked
    int causal, layout;
    int maxpos;       // sequence position of the query tile's last row (causal)
};

RA_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Tiles of shard j the walk takes (all of them unless causal).
RA_HD int shard_tiles(const RingWalk& w, int j) {
    if (!w.causal) return w.tiles_per_shard;
    return ceil_div(shard_visible(w.layout, w.shard_len, w.n_shards, j, w.maxpos), w.tile);
}

// q_row0: first storage row of the query tile; q_rows: rows in it.  The tile
// must lie inside one shard (zigzag: inside one half of it), so its rows'
// positions increase and its last row sees the most keys.  Requires
// shard_len % tile == 0 (zigzag: (shard_len / 2) % tile == 0) and
// q_row0 + q_rows <= S.
RA_HD RingWalk make_ring_walk(int S, int n_shards, int tile, int causal, int q_row0, int q_rows,
                              int layout = kLayoutContiguous) {
    RingWalk w;
    w.n_shards = n_shards;
    w.shard_len = S / n_shards;
    w.tile = tile;
    w.k = q_row0 / w.shard_len;
    w.tiles_per_shard = w.shard_len / tile;
    w.causal = causal;
    w.layout = layout;
    w.maxpos = layout_pos(layout, w.shard_len, n_shards, q_row0 + q_rows - 1);
    if (!causal) {
        w.first_tiles = w.tiles_per_shard;
        w.n_visited = n_shards;
        w.total = n_shards * w.tiles_per_shard;
        return w;
    }
    w.first_tiles = shard_tiles(w, w.k);
    const int L = w.shard_len, N = n_shards, P = w.maxpos;
    if (layout == kLayoutZigzag) {
        // chunk c = P / H holds the last row; r of its keys are visible
        const int H = L / 2, c = P / H, r = P - c * H + 1, th = H / tile;
        if (c < N) {  // first half of shard k = c: shards 0..c-1 give their first chunk
            w.n_visited = c + 1;
            w.total = c * th + ceil_div(r, tile);
        } else {      // second half of shard k = 2N-1-c: every first chunk, the second chunks of k+1..N-1
            w.n_visited = N;
            w.total = N * th + ceil_div(r, tile) + (N - 1 - w.k) * th;
        }
    } else if (layout == kLayoutStriped) {
        // last row: local index u in shard a = k; shards j <= a see u+1 keys, j > a see u
        const int u = P / N, a = P - u * N;
        w.n_visited = u == 0 ? a + 1 : N;
        w.total = (a + 1) * ceil_div(u + 1, tile) + (N - 1 - a) * ceil_div(u, tile);
    } else {
        w.n_visited = w.k + 1;
        w.total = w.first_tiles + w.k * w.tiles_per_shard;
    }
    return w;
}

// Shard visited at ring step t (t < n_visited).
RA_HD int ring_shard_at(const RingWalk& w, int t) { return (w.k - t + w.n_shards) % w.n_shards; }

// Incremental form of the same walk, for kernel loops: advancing within a
// shard costs adds and compares only.  LAYOUTS = false walks contiguous shards
// (every shard after the first is walked whole); LAYOUTS = true also handles
// causal zigzag and striped walks, where a shard switch recomputes that shard's
// visible prefix.
template <bool LAYOUTS>
struct RingIterT {
    int n_shards, L, tile, tiles_per_shard;
    int lay;    // LAYOUTS: layout when causal (contiguous otherwise)
    int maxpos; // LAYOUTS: position of the query tile's last row
    int t;      // ring step of the current shard
    int j;      // current shard
    int in;     // tile index within the current shard's visited tiles
    int count;  // visited tiles of the current shard
    int kb;     // first key (storage row) of the current tile

    RA_HD void start(const RingWalk& w) {
        n_shards = w.n_shards;
        L = w.shard_len;
        tile = w.tile;
        tiles_per_shard = w.tiles_per_shard;
        if (LAYOUTS) {
            lay = w.causal ? w.layout : kLayoutContiguous;
            maxpos = w.maxpos;
        }
        t = 0;
        j = w.k;
        in = 0;
        count = w.first_tiles;
        kb = j * L;
    }
    // A single linear range of `n_tiles` tiles starting at key kv_lo.
    RA_HD void start_linear(int kv_lo, int n_tiles, int tile_keys) {
        n_shards = 1;
        L = 0;
        tile = tile_keys;
        tiles_per_shard = n_tiles;
        if (LAYOUTS) {
            lay = kLayoutContiguous;
            maxpos = 0;
        }
        t = 0;
        j = 0;
        in = 0;
        count = n_tiles;
        kb = kv_lo;
    }
    RA_HD bool first() const { return in == 0; }
    RA_HD bool last() const { return in == count - 1; }
    // Past the walk's last tile the iterator moves on through the remaining
    // shards; callers stop after RingWalk::total tiles.
    RA_HD void next() {
        ++in;
        kb += tile;
        if (in == count && n_shards > 1) {
            ++t;
            j = (j == 0) ? n_shards - 1 : j - 1;
            in = 0;
            count = (!LAYOUTS || lay == kLayoutContiguous)
                        ? tiles_per_shard
                        : ceil_div(shard_visible(lay, L, n_shards, j, maxpos), tile);
            kb = j * L;
        }
    }
};
using RingIter = RingIterT<true>;

// Query tiles of a launch in heaviest-first order under the causal mask: the
// r-th tile launched holds the r-th largest last-row position.  n_qtiles tiles
// of `rows` rows; returns the first storage row of that tile.
RA_HD int heavy_tile_row0(int layout, int S, int n_shards, int rows, int r) {
    const int L = S / n_shards, n_qtiles = S / rows, tps = L / rows;
    if (layout == kLayoutZigzag) {
        const int g = n_qtiles - 1 - r;  // tile index in sequence order
        const int tph = tps / 2, c = g / tph, x = g - c * tph;
        const int s = c < n_shards ? c : 2 * n_shards - 1 - c;
        return s * L + (c < n_shards ? 0 : L / 2) + x * rows;
    }
    if (layout == kLayoutStriped) {
        const int x = tps - 1 - r / n_shards, a = n_shards - 1 - r % n_shards;
        return a * L + x * rows;
    }
    return (n_qtiles - 1 - r) * rows;
}

}  // namespace ra
