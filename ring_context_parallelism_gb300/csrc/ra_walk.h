// ra_walk.h -- the ring-order KV walk, shared by the host (inspection API,
// launch sizing) and every kernel role (producer, MMA issuer, softmax).
//
// "RingAttention and Context Parallelism: Mathematical Foundations", section 3:
// the sequence is cut into N contiguous shards of L = S/N tokens and the query
// block of shard k holds, at ring step t, the KV shard (k - t) mod N.  Section 5:
// with a causal mask the KV shards after k are empty and are skipped.  On one
// GPU the ring becomes the order in which a query tile streams KV tiles from
// HBM: shard k first (ascending tiles, stopping at the query tile's diagonal
// when causal), then k-1, ..., 0, N-1, ..., k+1.
#pragma once

#ifdef __CUDACC__
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

namespace ra {

struct RingWalk {
    int n_shards;     // N
    int shard_len;    // L = S / N
    int tile;         // keys per KV tile
    int k;            // shard of the query tile
    int first_tiles;  // tiles taken from shard k
    int tiles_per_shard;
    int n_visited;    // shards visited (N, or k+1 when causal)
    int total;        // total KV tiles walked
};

// q_row0: first row of the query tile; q_rows: rows in it (must not cross a
// shard boundary).  Requires shard_len % tile == 0 and q_row0 + q_rows <= S.
RA_HD RingWalk make_ring_walk(int S, int n_shards, int tile, int causal, int q_row0, int q_rows) {
    RingWalk w;
    w.n_shards = n_shards;
    w.shard_len = S / n_shards;
    w.tile = tile;
    w.k = q_row0 / w.shard_len;
    w.tiles_per_shard = w.shard_len / tile;
    if (causal) {
        const int diag_end = q_row0 + q_rows;  // keys [k*L, diag_end) of the own shard are visible
        w.first_tiles = (diag_end - w.k * w.shard_len + tile - 1) / tile;
        w.n_visited = w.k + 1;
    } else {
        w.first_tiles = w.tiles_per_shard;
        w.n_visited = n_shards;
    }
    w.total = w.first_tiles + (w.n_visited - 1) * w.tiles_per_shard;
    return w;
}

// Shard visited at ring step t (t < n_visited).
RA_HD int ring_shard_at(const RingWalk& w, int t) { return (w.k - t + w.n_shards) % w.n_shards; }

// i-th KV tile of the walk: returns its first key; *shard_pos = ring step of
// its shard; *first / *last = whether it opens / closes that shard's tiles.
RA_HD int ring_tile(const RingWalk& w, int i, int* shard_pos, bool* first, bool* last) {
    if (i < w.first_tiles) {
        *shard_pos = 0;
        *first = (i == 0);
        *last = (i == w.first_tiles - 1);
        return w.k * w.shard_len + i * w.tile;
    }
    const int r = i - w.first_tiles;
    const int t = 1 + r / w.tiles_per_shard;
    const int in = r % w.tiles_per_shard;
    *shard_pos = t;
    *first = (in == 0);
    *last = (in == w.tiles_per_shard - 1);
    return ring_shard_at(w, t) * w.shard_len + in * w.tile;
}

// Incremental form of the same walk, for kernel loops: advancing costs adds
// and compares only (no division per tile).
struct RingIter {
    int n_shards, L, tile, tiles_per_shard;
    int t;      // ring step of the current shard
    int j;      // current shard
    int in;     // tile index within the current shard's visited tiles
    int count;  // visited tiles of the current shard
    int kb;     // first key of the current tile

    RA_HD void start(const RingWalk& w) {
        n_shards = w.n_shards;
        L = w.shard_len;
        tile = w.tile;
        tiles_per_shard = w.tiles_per_shard;
        t = 0;
        j = w.k;
        in = 0;
        count = w.first_tiles;
        kb = j * L;
    }
    // A single linear range of `count` tiles starting at key kv_lo.
    RA_HD void start_linear(int kv_lo, int n_tiles, int tile_keys) {
        n_shards = 1;
        L = 0;
        tile = tile_keys;
        tiles_per_shard = n_tiles;
        t = 0;
        j = 0;
        in = 0;
        count = n_tiles;
        kb = kv_lo;
    }
    RA_HD bool first() const { return in == 0; }
    RA_HD bool last() const { return in == count - 1; }
    RA_HD void next() {
        ++in;
        kb += tile;
        if (in == count && n_shards > 1) {
            ++t;
            j = (j == 0) ? n_shards - 1 : j - 1;
            in = 0;
            count = tiles_per_shard;
            kb = j * L;
        }
    }
};

}  // namespace ra
