// attn_tc.cu -- blockwise exact attention on the sm_103a tensor cores.
//
// One CTA owns up to two 128-row query tiles that read the same K/V tiles (two
// query heads of one GQA group in the ring prefill; two row tiles of the
// stacked branch rows in the fan-out), and walks the KV tiles in ring order.
// Per KV tile, the online-softmax state transition of "RingAttention and
// Context Parallelism: Mathematical Foundations", section 2 figure, is run as:
//
//   S   = Q K^T                  tcgen05.mma (smem x smem -> TMEM, fp32)
//   m'  = max(m, rowmax(S))      softmax warps, one thread per row (TMEM lane)
//   P~  = exp(S - m')            ex2 with log2(e)/sqrt(d) folded in; bf16 into TMEM
//   l   = e^{m-m'} l + rowsum(P~)
//   O   = e^{m-m'} O + P~ V      tcgen05.mma (P~ from TMEM, V from smem)
//   A   = O / l,  lse = m + ln l epilogue
//
// The running max is only moved when a tile's max exceeds it by more than
// 2^8 (in log2 units); otherwise the stale max is kept, which changes no
// result (O and l share it) and skips the O rescale.
//
// Roles (384 threads):  warp 0 lane 0  TMA producer of Q (once) and the K ring;
// warp 2 lane 0  TMA producer of the V ring (up to three stages each for
// D = 128, four for D = 64; Cfg below);  warp 1 lane 0  MMA issuer (also
// allocates TMEM);  warps 4-7  softmax + epilogue of tile 0;  warps 8-11  same
// for tile 1.  TMEM: tile t uses columns [256t, 256t+128) for S (P~ overwrites
// its first half as packed bf16) and [256t+128, 256t+128+D) for O.
//
// Kernel modes: the ring prefill over contiguous shards (which also runs causal
// zigzag shards, through their chunk map, and causal striped shards over
// positions), the layouts' own rings (ra_walk.h) for striped shard counts that do
// not divide 128 and for per-shard partials, and the fan-out (stacked branch
// rows against a prefix chunk plus folded private suffixes; decode, prefill with
// a causal suffix, or a paged KV pool), whose units split their KV tiles over
// the two softmax slots (one row tile) or pair two row tiles.
//
// Every wait is bounded (ra::mbar_wait); a wait that runs out records
// RA_ERR_DEVICE_TIMEOUT in the status word and the CTA unwinds and returns.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "ra_device.cuh"
#include "ra_internal.h"
#include "ra_walk.h"

namespace ra {

static __device__ unsigned g_tc_status[2];

namespace {

constexpr int kTileM = 128;
constexpr int kTileN = 128;
constexpr int kThreads = 384;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kTmemCols = 512;
constexpr int kMaxChunks = 64;
constexpr int kLaunchRegs = 168;  // registers per thread at launch: 65536 / 384, rounded down to a multiple of 8

struct TcParams {
    int fanout;     // 0 ring prefill, 1 fan-out
    int causal;
    int layout;     // ring: shard layout (ra_walk.h), used when causal
    int T2;         // ring: two heads per CTA (GQA group size even)
    // ring
    int B, S, Hq, Hkv, n_shards, n_qtiles, n_head_groups;
    // fan-out
    int R, G, rows_per_tile, n_mpairs, S_prefix, n_chunks, S_suffix, n_branches,
        suffix_mpairs, n_prefix_units;
    int split_prefix;   // prefix units hold one row tile: split their KV tiles over both tile slots
    int suffix_slot0;   // partial slot of the suffix (suffix units; only without a prefix)
    int fold;           // suffixes folded into prefix units: branch b into chunk b % n_chunks
    int suffix_causal;  // fan-out prefill: a branch's rows are the last tokens of its suffix, causal inside it
    // ring over a zigzag-stored sequence walked in sequence-position order (0: rows are positions):
    // position chunk c of zz_half tokens is the first half of shard c (c < zz_n) or the
    // second half of shard 2 zz_n - 1 - c
    int zz_n, zz_half;
    // paged KV: the K/V maps address a page pool [n_pages * page_size, Hkv, D];
    // key k of the prefix lives in page prefix_pages[k >> page_shift], key k of
    // branch b's suffix in page suffix_pages[b * n_suffix_pages + (k >> page_shift)]
    int paged, page_shift, n_pages, n_prefix_pages, n_suffix_pages;
    const int* prefix_pages;
    const int* suffix_pages;
    int chunk_start[kMaxChunks + 1];  // prefix tile where chunk c starts
    const int* offsets;
    float scale_log2;
    OutDesc out;
};

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;                   // 128-byte column groups per row
    static constexpr int kTileBytes = kTileM * D * 2;        // one Q/K/V tile
    // Q tiles and K / V stages share kDataTiles tile slots: two Q tiles leave
    // room for 3 K + 2 V stages (D = 128), a split unit's single Q tile for 3 + 3.
    static constexpr int kDataTiles = D == 128 ? 7 : 10;
    static constexpr int kMaxKV = D == 128 ? 3 : 4;          // per ring
    static constexpr int kQOff = 0;
    static constexpr int kBarOff = kDataTiles * kTileBytes;
    // Iteration-done barriers (stage release in paired mode): a producer waits
    // for iteration j while the MMA issuer is at most max(stages) iterations
    // past it, so that many slots keep the parity of slot j unambiguous.
    static constexpr int kNVPair = kDataTiles - 2 - kMaxKV;  // V stages with two Q tiles
    static constexpr int kIterRing = kMaxKV > kNVPair ? kMaxKV : kNVPair;
    // Issue loop unrolled over a whole cycle of the rings (and of the two
    // tile-slot parities): every stage and iteration-done slot used equally
    // often per block.  A ring whose stages are used an odd number of times
    // per block sees its barrier parities flip from one block to the next.
    static constexpr int kGcd(int a, int b) { return b == 0 ? a : kGcd(b, a % b); }
    static constexpr int kLcm(int a, int b) { return a / kGcd(a, b) * b; }
    static constexpr int kBlk = kLcm(kLcm(kLcm(kMaxKV, kNVPair), kIterRing), 2);
    static constexpr bool kKFlip = (kBlk / kMaxKV) % 2 == 1;
    static constexpr bool kVFlip = (kBlk / kNVPair) % 2 == 1;
    static constexpr int kNumBars = 1 + 4 * kMaxKV + 7 + kIterRing;
    static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;  // + alignment slack
    static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory a CTA may use");
};

// Unit of work of one CTA, identical in every thread.
struct Unit {
    int valid;
    int T;                 // tiles (1 or 2)
    int qc1[2], qc2[2], qc3[2];  // Q tensor-map coordinates (dims 1..3) per tile
    int kv_head, kv_z;     // K/V map coordinates (dims 1 and 3)
    int suffix;            // fan-out: K/V from the suffix maps
    // ring
    int b, head[2], q_row0;
    int q_srow0;           // storage row of the query tile (q_row0 unless zigzag in position order)
    // fan-out
    int row0[2], row_hi, kv_lo, kv_hi;
    int split;             // both tiles share Q tile 0 and take alternate KV tiles
    int n_q;               // Q tiles to load
    int slot[2];           // output partial slot per tile
    int total;             // fan-out: KV tiles of the walk (prefix range + folded suffixes)
    int fold_b0;           // fan-out prefix unit: first branch whose suffix is folded in (-1: none)
    int unit_row_lo, unit_row_hi;  // stacked rows the unit's tiles cover
};

// Storage row of sequence position pos (tile-aligned runs stay inside one chunk).
__device__ __forceinline__ int zz_row(const TcParams& p, int pos) { return zigzag_row(p.zz_n, p.zz_half, pos); }

template <bool FAN, bool LAY = false, bool STR = false>
__device__ __forceinline__ Unit decode_unit(const TcParams& p) {
    Unit u;
    u.valid = 1;
    u.suffix = 0;
    u.split = 0;
    const int idx = blockIdx.x;
    if (!FAN) {
        // (batch, KV head) outermost: the CTAs resident at one time share one or
        // two KV heads, whose K and V stay in L2 while every query tile of the
        // group walks them.  Within a group the heaviest query tiles launch first.
        const int hg_per_kv = p.n_head_groups / p.Hkv;
        const int per_kv = p.n_qtiles * hg_per_kv;
        const int g = idx / per_kv;
        const int rem = idx - g * per_kv;
        const int qt_rev = rem / hg_per_kv;
        u.b = g / p.Hkv;
        const int hg = (g - u.b * p.Hkv) * hg_per_kv + (rem - qt_rev * hg_per_kv);
        u.q_row0 = !p.causal             ? qt_rev * kTileM
                   : LAY                   ? heavy_tile_row0(p.layout, p.S, p.n_shards, kTileM, qt_rev)
                   : STR                   ? heavy_tile_row0(kLayoutStriped, p.S, p.n_shards, kTileM, qt_rev)
                                           : (p.n_qtiles - 1 - qt_rev) * kTileM;
        u.q_srow0 = LAY ? u.q_row0 : zz_row(p, u.q_row0);
        u.T = p.T2 ? 2 : 1;
        for (int t = 0; t < 2; ++t) {
            u.head[t] = hg * u.T + (t < u.T ? t : 0);
            u.qc1[t] = u.head[t];
            u.qc2[t] = u.q_srow0;
            u.qc3[t] = u.b;
        }
        u.kv_head = u.head[0] / (p.Hq / p.Hkv);
        u.kv_z = u.b;
        u.n_q = u.T;
        u.slot[0] = u.slot[1] = 0;
        return u;
    }
    u.b = 0;
    int mp;
    if (idx < p.n_prefix_units) {
        // KV head varies fastest after the row pair: the CTAs of one chunk's
        // heads run together and stream the same token rows, which share DRAM
        // pages ([S, Hkv, D] layout).
        mp = idx % p.n_mpairs;
        const int rest = idx / p.n_mpairs;
        u.kv_head = rest % p.Hkv;
        const int chunk = rest / p.Hkv;
        u.kv_z = 0;
        u.kv_lo = p.chunk_start[chunk] * kTileN;
        u.kv_hi = min(p.S_prefix, p.chunk_start[chunk + 1] * kTileN);
        u.row0[0] = 2 * mp * p.rows_per_tile;
        u.row_hi = p.R;
        u.split = p.split_prefix;
        u.slot[0] = u.slot[1] = chunk;
        u.total = (u.kv_hi - u.kv_lo + kTileN - 1) / kTileN;
        u.unit_row_lo = u.row0[0];
        u.unit_row_hi = min(p.R, u.row0[0] + (u.split ? 1 : 2) * p.rows_per_tile);
        // First branch whose suffix may fold into this chunk; which ones do
        // (their rows meet the unit's) needs branch_offsets from memory, read
        // by fold_tiles() after the launch's first loads are in flight.
        u.fold_b0 = (p.fold && chunk < p.n_branches) ? chunk : -1;
    } else {
        const int j = idx - p.n_prefix_units;
        mp = j % p.suffix_mpairs;
        const int rest = j / p.suffix_mpairs;
        u.kv_head = rest % p.Hkv;
        const int br = rest / p.Hkv;
        const int lo = p.offsets[br];
        const int hi = p.offsets[br + 1];
        if (lo < 0 || hi < lo || hi > p.R || (br == 0 && lo != 0) || (br == p.n_branches - 1 && hi != p.R)) {
            if (threadIdx.x == 0) {
                atomicCAS(&g_tc_status[0], 0u, kDevInvalidArg);
                atomicCAS(&g_tc_status[1], 0u, 0x0F000000u | static_cast<unsigned>(br));
            }
            u.valid = 0;
            return u;
        }
        u.suffix = 1;
        u.kv_z = br;
        u.kv_lo = 0;
        u.kv_hi = p.S_suffix;
        u.row0[0] = lo + 2 * mp * p.rows_per_tile;
        u.row_hi = hi;
        u.split = (hi - lo <= p.rows_per_tile) ? 1 : 0;
        u.slot[0] = u.slot[1] = p.suffix_slot0;
        u.total = (p.S_suffix + kTileN - 1) / kTileN;
        u.fold_b0 = -1;
        u.unit_row_lo = lo;
        u.unit_row_hi = hi;
    }
    u.row0[1] = u.split ? u.row0[0] : u.row0[0] + p.rows_per_tile;
    if (u.row0[0] >= u.row_hi) u.valid = 0;
    u.T = (u.split || u.row0[1] < u.row_hi) ? 2 : 1;
    u.n_q = u.split ? 1 : u.T;
    for (int t = 0; t < 2; ++t) {
        u.qc1[t] = 0;
        u.qc2[t] = u.kv_head;
        u.qc3[t] = u.row0[t];
    }
    return u;
}

// KV tiles of the suffixes folded into a fan-out prefix unit: branches
// fold_b0, fold_b0 + n_chunks, ... whose rows meet the unit's rows.  A branch
// with invalid offsets is skipped and recorded in the status word.
__device__ int fold_tiles(const TcParams& p, const Unit& u, bool report) {
    if (u.fold_b0 < 0) return 0;
    const int s_tiles = (p.S_suffix + kTileN - 1) / kTileN;
    int n = 0;
    for (int b = u.fold_b0; b < p.n_branches; b += p.n_chunks) {
        const int lo = p.offsets[b], hi = p.offsets[b + 1];
        if (lo < 0 || hi < lo || hi > p.R) {
            if (report) {
                atomicCAS(&g_tc_status[0], 0u, kDevInvalidArg);
                atomicCAS(&g_tc_status[1], 0u, 0x0F000000u | static_cast<unsigned>(b));
            }
            continue;
        }
        if (hi > lo && lo < u.unit_row_hi && hi > u.unit_row_lo) n += s_tiles;
    }
    return n;
}

// Position in a unit's walk of KV tiles.  Ring prefill: the ring order of
// ra_walk.h.  Fan-out: the unit's prefix range, then the suffix of every
// branch folded into it (only that branch's rows see those keys); a suffix
// unit walks one branch's suffix.
template <bool FAN, bool LAY = false>
struct TileWalk {
    static constexpr bool fan = FAN;
    RingIterT<LAY> ring;
    int seg;              // fan-out: 0 prefix, 1 suffix
    int b;                // fan-out suffix segment: branch
    int kb, key_end;      // first key of the tile, end of the segment's keys
    int tin, tcount;      // tile within the segment, tiles in it
    int row_lo, row_hi;   // stacked rows that see the segment
    int stride;           // next folded branch: b + stride (0: none)
    bool more;            // fan-out: the walk has a current tile

    __device__ __forceinline__ bool seek_branch(const TcParams& p, const Unit& u, int from) {
        for (int bb = from; stride > 0 && bb < p.n_branches; bb += stride) {
            const int lo = p.offsets[bb], hi = p.offsets[bb + 1];
            if (lo < 0 || hi < lo || hi > p.R) continue;
            if (hi > lo && lo < u.unit_row_hi && hi > u.unit_row_lo) {
                seg = 1;
                b = bb;
                kb = 0;
                key_end = p.S_suffix;
                tin = 0;
                tcount = (p.S_suffix + kTileN - 1) / kTileN;
                row_lo = lo;
                row_hi = hi;
                return true;
            }
        }
        return false;
    }
    __device__ __forceinline__ void start(const TcParams& p, const Unit& u, const RingWalk& w) {
        if (!fan) {
            ring.start(w);
            return;
        }
        more = true;
        if (u.suffix) {  // a suffix unit: one branch's suffix, rows = the unit's branch
            seg = 1;
            b = u.kv_z;
            kb = 0;
            key_end = p.S_suffix;
            tin = 0;
            tcount = (p.S_suffix + kTileN - 1) / kTileN;
            row_lo = u.unit_row_lo;
            row_hi = u.unit_row_hi;
            stride = 0;
            return;
        }
        seg = 0;
        b = 0;
        kb = u.kv_lo;
        key_end = u.kv_hi;
        tin = 0;
        tcount = (u.kv_hi - u.kv_lo + kTileN - 1) / kTileN;
        row_lo = 0;
        row_hi = p.R;
        stride = p.fold ? p.n_chunks : 0;
        if (tcount == 0) more = u.fold_b0 >= 0 && seek_branch(p, u, u.fold_b0);
    }
    __device__ __forceinline__ void next(const TcParams& p, const Unit& u) {
        if (!fan) {
            ring.next();
            return;
        }
        ++tin;
        kb += kTileN;
        if (tin == tcount) {
            if (seg == 0)
                more = u.fold_b0 >= 0 && seek_branch(p, u, u.fold_b0);
            else
                more = seek_branch(p, u, b + stride);
        }
    }
    __device__ __forceinline__ int key() const { return fan ? kb : ring.kb; }
};

// S = Q K^T for one 128x128 tile: D/16 MMAs, both operands K-major in smem.
// q_lo / k_lo: low descriptor words of the tiles (LBO field 16 B).
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tS, uint32_t q_lo, uint32_t k_lo) {
    constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kTileN, false, false);
    asm volatile("" : "+r"(q_lo), "+r"(k_lo));  // descriptor words formed here, next to their MMAs
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * (16384 >> 4) + (kk & 3) * (32 >> 4);
        mma_ss(tS, sw128_desc(q_lo + off), sw128_desc(k_lo + off), idesc, kk > 0 ? 1u : 0u);
    }
}

// O (+)= P~ V: 8 MMAs of 16 keys, P~ from TMEM (packed bf16 over S), V MN-major
// in smem (v_lo: low descriptor word with LBO = 16 KB between 64-column groups).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint32_t v_lo, bool accumulate_first) {
    constexpr uint32_t idesc = idesc_bf16_f32(kTileM, D, false, true);
    asm volatile("" : "+r"(tP), "+r"(v_lo));
#pragma unroll
    for (int kk = 0; kk < kTileN / 16; ++kk)
        mma_ts(tO, tP + kk * 8, sw128_desc(v_lo + kk * (2048 >> 4)), idesc, (kk > 0 || accumulate_first) ? 1u : 0u);
}

template <int D>
__device__ __forceinline__ void store_row(const OutDesc& out, long long o_base, int chunk, const float* vals,
                                          float inv_l) {
    if (out.o_f32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out.o) + o_base + chunk * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(vals[4 * j] * inv_l, vals[4 * j + 1] * inv_l, vals[4 * j + 2] * inv_l,
                                 vals[4 * j + 3] * inv_l);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out.o) + o_base + chunk * 32);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(pack_bf16x2(vals[8 * j] * inv_l, vals[8 * j + 1] * inv_l),
                                pack_bf16x2(vals[8 * j + 2] * inv_l, vals[8 * j + 3] * inv_l),
                                pack_bf16x2(vals[8 * j + 4] * inv_l, vals[8 * j + 5] * inv_l),
                                pack_bf16x2(vals[8 * j + 6] * inv_l, vals[8 * j + 7] * inv_l));
    }
}

// The same values written to a row of shared memory (the final flush stages
// each row there and hands it to one bulk copy: a thread per row writing its
// row straight to global memory touches 32 lines per warp instruction).
template <int D>
__device__ __forceinline__ void stage_row(const OutDesc& out, uint8_t* srow, int chunk, const float* vals,
                                          float inv_l) {
    if (out.o_f32) {
        float4* dst = reinterpret_cast<float4*>(srow) + chunk * 8;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(vals[4 * j] * inv_l, vals[4 * j + 1] * inv_l, vals[4 * j + 2] * inv_l,
                                 vals[4 * j + 3] * inv_l);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(srow) + chunk * 4;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(pack_bf16x2(vals[8 * j] * inv_l, vals[8 * j + 1] * inv_l),
                                pack_bf16x2(vals[8 * j + 2] * inv_l, vals[8 * j + 3] * inv_l),
                                pack_bf16x2(vals[8 * j + 4] * inv_l, vals[8 * j + 5] * inv_l),
                                pack_bf16x2(vals[8 * j + 6] * inv_l, vals[8 * j + 7] * inv_l));
    }
}

// Stage and phase of a ring of n slots, advanced without division.
struct StageCtr {
    int s = 0, ph = 0;
    __device__ __forceinline__ void next(int n) {
        if (++s == n) {
            s = 0;
            ph ^= 1;
        }
    }
};

// Kernel variants: ring prefill, and fan-out launches whose units all split
// their KV tiles over the two tile slots (one row tile), all pair two row
// tiles, or mix both (suffix units without a prefix).  The uniform fan-out
// variants compile only their own issue and softmax paths.
// A causal ring over zigzag shards runs the contiguous variant (its tiles
// addressed through the layout's chunk map), one over striped shards the
// contiguous walk over positions with tiles gathered by 5-D boxes
// (kModeRingStripedPos; N dividing 128) or else the layout's ring
// (kModeRingStriped); the per-shard partials over either layout walk the
// layout's ring in kModeRingLayoutPartials.  The
// fan-out modes over a paged KV pool (kModeFan*Paged) are the same three
// fan-out variants with the producers' page-table path compiled in.  The ring
// walks that write one partial per KV shard (kModeRing*Partials) are compiled
// apart from the single-output ones: the flush inside the tile loop made the
// contiguous prefill 7% slower (5.30 against 4.95 ms) where it is never taken.
enum KernelMode : int {
    kModeRing = 0,
    kModeFanMixed = 1,
    kModeFanSplit = 2,
    kModeFanPaired = 3,
    kModeFanMixedPaged = 5,
    kModeFanSplitPaged = 6,
    kModeFanPairedPaged = 7,
    kModeRingPartials = 8,
    kModeRingLayoutPartials = 9,
    kModeRingStriped = 10,
    kModeRingStripedPos = 11
};

// Register split per warpgroup: the producer / MMA warpgroup's registers per
// thread (dec) and the two softmax warpgroups' (inc), at most the launch's
// 384 x 168 = 64512 in all.  ptxas's spill report moves erratically with the
// split, so each kernel variant takes the split that measured fastest among
// those with the fewest spilled bytes: the contiguous and striped rings 64 / 216
// (the unrolled MMA loop spilled at 48), the fan-out split and paired
// variants 40 / 232 and 80 / 208 (3% faster than 56 / 224 on the R = 147
// decode and the 8 x 20 prefill); the rest by the spill report alone.
template <int MODE>
struct RegSplit {
    static constexpr int dec = MODE == kModeRing                ? 64
                               : MODE == kModeRingStriped        ? 64
                               : MODE == kModeRingStripedPos     ? 64
                               : MODE == kModeFanMixed           ? 80
                               : MODE == kModeFanSplit           ? 40
                               : MODE == kModeFanPaired          ? 80
                               : MODE == kModeFanMixedPaged      ? 72
                               : MODE == kModeRingPartials       ? 64
                               : MODE == kModeRingLayoutPartials ? 48
                                                                 : 56;
    static constexpr int inc = MODE == kModeRing                ? 216
                               : MODE == kModeRingStriped        ? 216
                               : MODE == kModeRingStripedPos     ? 216
                               : MODE == kModeFanMixed           ? 208
                               : MODE == kModeFanSplit           ? 232
                               : MODE == kModeFanPaired          ? 208
                               : MODE == kModeFanMixedPaged      ? 216
                               : MODE == kModeRingPartials       ? 216
                                                                 : 224;
    static_assert(128 * dec + 256 * inc <= kThreads * kLaunchRegs, "register split exceeds the launch's registers");
};
template <int MODE>
__device__ __forceinline__ void reg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RegSplit<MODE>::dec) : "memory");
}
template <int MODE>
__device__ __forceinline__ void reg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(RegSplit<MODE>::inc) : "memory");
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_k2,
                   const __grid_constant__ CUtensorMap tm_v2, const TcParams p) {
    using C = Cfg<D>;
    constexpr bool PART = MODE == kModeRingPartials || MODE == kModeRingLayoutPartials;  // one partial per KV shard
    // causal striped shards with one output: the contiguous variant's code with the
    // striped walk's per-shard tile counts and diagonal masks
    constexpr bool STR = MODE == kModeRingStriped;
    // causal striped shards with one output, N dividing 128: the contiguous causal walk over
    // sequence positions, every 128-position tile gathered by one 5-D TMA box per 64
    // columns (shard index the faster box dimension, so rows land in position order)
    constexpr bool SPOS = MODE == kModeRingStripedPos;
    constexpr bool RING = MODE == kModeRing || PART || STR || SPOS;
    constexpr bool FAN = !RING;
    constexpr bool LAY = MODE == kModeRingLayoutPartials;
    // single-output ring variants: the Unit's per-slot arrays indexed with constants
    // only (a runtime index keeps the Unit in local memory; the ring prefill measured
    // 0.6-1.3% faster without, the fan-out variants 2-7% slower, so they keep it)
    constexpr bool CSEL = MODE == kModeRing || STR || SPOS;
    constexpr bool PG = MODE >= kModeFanMixedPaged && MODE <= kModeFanPairedPaged;  // paged KV pool
    constexpr int FMODE = PG ? MODE - kModeFanMixedPaged + kModeFanMixed : MODE;  // its unpaged fan-out mode
    const Unit u = decode_unit<FAN, LAY, STR>(p);
    if (!u.valid) return;
    const bool split = FMODE == kModeFanSplit ? true : (RING || FMODE == kModeFanPaired) ? false : u.split != 0;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* q_smem = smem + C::kQOff;
    // K and V rings after the Q tiles the unit loads
    const int nK = C::kMaxKV;
    const int nV = (u.n_q == 1) ? C::kMaxKV : C::kDataTiles - 2 - C::kMaxKV;
    uint8_t* kv_smem = smem + C::kQOff + u.n_q * C::kTileBytes;
    uint8_t* k_smem = kv_smem;
    uint8_t* v_smem = kv_smem + nK * C::kTileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + C::kMaxKV;
    uint64_t* v_full = k_empty + C::kMaxKV;
    uint64_t* v_empty = v_full + C::kMaxKV;
    uint64_t* s_full = v_empty + C::kMaxKV;    // [2]
    uint64_t* p_full = s_full + 2;             // [2]
    uint64_t* o_done = p_full + 2;             // [2]
    uint64_t* drain = o_done + 2;
    uint64_t* iter_done = drain + 1;           // [kIterRing]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    RingWalk w{};
    int total;
    if (!FAN) {
        w = make_ring_walk(p.S, p.n_shards, kTileN, p.causal, u.q_row0, kTileM, LAY ? p.layout : kLayoutContiguous);
        if (STR) {
            // the same walk as the striped layout's: each of the N shards, in ring
            // order, up to the tile at the query tile's own in-shard index
            const int n = (u.q_row0 - w.k * w.shard_len) / kTileN + 1;
            w.first_tiles = w.tiles_per_shard = n;
            w.n_visited = p.n_shards;
            w.total = p.n_shards * n;
        }
        total = w.total;
    } else {
        total = u.total;
    }

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < C::kMaxKV; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 128);
            mbar_init(&o_done[t], 1);
        }
        mbar_init(drain, 1);
        for (int r = 0; r < C::kIterRing; ++r) mbar_init(&iter_done[r], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int T = u.T;
    unsigned* status = g_tc_status;
    // Folded suffix tiles extend the walk.  The producers find them as they
    // walk (their first loads are issued before branch_offsets is read); the
    // other roles count them here, while those loads are in flight.
    if (FAN && u.fold_b0 >= 0 && warp != 0 && warp != 2) total += fold_tiles(p, u, threadIdx.x == 32);

    // Register split, set inside each role (reg_dec / reg_inc).

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers
        // Lane 0 of warp 0 loads Q and streams the K ring, lane 0 of warp 2 the
        // V ring: one issuing thread alone cannot keep both rings filled at the
        // rate the MMAs (or HBM, for the fan-out) consume them.  A paged fan-out
        // tile arrives in one small box per page and column chunk (16 for
        // 16-token pages), and the TMA unit takes small boxes slowly from a
        // single issuing thread: there every lane of the warp walks the tiles,
        // lane 0 sets the stage's expected bytes and each lane issues one box.
        reg_dec<MODE>();
        constexpr bool warp_issue = PG;
        if (lane == 0 || warp_issue) {
            const bool lead = lane == 0;
            const bool is_k = (warp == 0);
            uint64_t* full = is_k ? k_full : v_full;
            uint64_t* empty = is_k ? k_empty : v_empty;
            uint8_t* ring = is_k ? k_smem : v_smem;
            const int n_stages = is_k ? nK : nV;
            const CUtensorMap* map1 = is_k ? &tm_k : &tm_v;
            const CUtensorMap* map2 = is_k ? &tm_k2 : &tm_v2;
            if (lead) {
                tma_prefetch_desc(map1);
                if (FAN) tma_prefetch_desc(map2);
            }
            if (is_k && lead) {
                tma_prefetch_desc(&tm_q);
                mbar_arrive_expect_tx(q_full, u.n_q * C::kTileBytes);
                if (SPOS) {
#pragma unroll
                    for (int t = 0; t < 2; ++t)
                        if (t < u.n_q)
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_5d(&tm_q, q_full, q_smem + t * C::kTileBytes + c * 16384, c * 64,
                                            u.qc1[t], 0, u.q_row0 / p.n_shards, u.qc3[t]);
                } else if (CSEL) {
#pragma unroll
                    for (int t = 0; t < 2; ++t)
                        if (t < u.n_q)
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_4d(&tm_q, q_full, q_smem + t * C::kTileBytes + c * 16384, c * 64,
                                            u.qc1[t], u.qc2[t], u.qc3[t]);
                } else {
                    for (int t = 0; t < u.n_q; ++t)
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_4d(&tm_q, q_full, q_smem + t * C::kTileBytes + c * 16384, c * 64, u.qc1[t],
                                        u.qc2[t], u.qc3[t]);
                }
            }
            int issued = 0;
            StageCtr cs;
            TileWalk<FAN, LAY> wi;
            wi.start(p, u, w);
            bool ok = true;
            for (int i = 0; ok && (FAN ? wi.more : i < total); ++i, wi.next(p, u)) {
                const bool from_suffix = FAN && wi.seg == 1;
                const CUtensorMap* map = from_suffix ? map2 : map1;
                const int z = FAN ? (from_suffix ? wi.b : 0) : u.kv_z;
                // Stage free: split units release K and V stages one by one; paired
                // units once per MMA iteration (K tile j is done with after
                // iteration j, V tile j after iteration j + 1).
                const unsigned where = 0x01000000u | (2 * i + (is_k ? 0 : 1));
                if (split) {
                    ok = mbar_wait(&empty[cs.s], cs.ph ^ 1, abort_flag, status, where);
                } else if (i >= n_stages) {
                    const int j = is_k ? i - n_stages : i - n_stages + 1;
                    ok = mbar_wait(&iter_done[j % C::kIterRing], (j / C::kIterRing) & 1, abort_flag, status, where);
                }
                if (warp_issue) ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (lead) mbar_arrive_expect_tx(&full[cs.s], C::kTileBytes);
                if (PG) {
                    __syncwarp();  // the expected bytes are set before any box of the stage can land
                    // one box per page (or per 128 rows of a larger page); a 128B-swizzled
                    // tile is the same bytes whether it lands in one box or several
                    // (every sub-box starts on a 1024-byte swizzle atom).  Pages past
                    // the listed ones, and invalid page indices, load zeros from past
                    // the pool (those keys are masked, or reported).
                    const int* table = from_suffix ? p.suffix_pages + static_cast<long long>(wi.b) * p.n_suffix_pages
                                                   : p.prefix_pages;
                    const int n_listed = from_suffix ? p.n_suffix_pages : p.n_prefix_pages;
                    const int page_size = 1 << p.page_shift;
                    const int sub_rows = page_size < kTileN ? page_size : kTileN;
                    const int n_boxes = (kTileN / sub_rows) * C::kChunks;  // at most 16 x 2 (8-token pages)
                    for (int b = lane; b < n_boxes; b += 32) {
                        const int r0 = (b / C::kChunks) * sub_rows;
                        const int c = b % C::kChunks;
                        const int lk = wi.key() + r0;
                        const int lp = lk >> p.page_shift;
                        int row = p.n_pages << p.page_shift;
                        if (lp < n_listed) {
                            const int pg = table[lp];
                            if (pg >= 0 && pg < p.n_pages) {
                                row = (pg << p.page_shift) + (lk - (lp << p.page_shift));
                            } else {
                                atomicCAS(&g_tc_status[0], 0u, kDevInvalidArg);
                                atomicCAS(&g_tc_status[1], 0u, 0x0E000000u | static_cast<unsigned>(lp & 0xFFFFFF));
                            }
                        }
                        tma_load_4d(map, &full[cs.s], ring + cs.s * C::kTileBytes + c * 16384 + r0 * 128, c * 64,
                                    u.kv_head, row, 0);
                    }
                } else if (SPOS) {
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_5d(map, &full[cs.s], ring + cs.s * C::kTileBytes + c * 16384, c * 64, u.kv_head, 0,
                                    wi.key() / p.n_shards, z);
                } else {
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_4d(map, &full[cs.s], ring + cs.s * C::kTileBytes + c * 16384, c * 64, u.kv_head,
                                    (RING && !LAY) ? zz_row(p, wi.key()) : wi.key(), z);
                }
                cs.next(n_stages);
                ++issued;
            }
            if (lead && *abort_flag) {
                // let copies already in flight land before the CTA exits: the
                // last n_stages loads of this ring (and Q)
                StageCtr ls;
                for (int n = 0; n < issued; ++n) {
                    if (n >= issued - n_stages) mbar_wait_landing(&full[ls.s], ls.ph);
                    ls.next(n_stages);
                }
                if (is_k) mbar_wait_landing(q_full, 0);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        reg_dec<MODE>();
        if (lane == 0) {
            const uint32_t q_addr = smem_u32(q_smem);
            // low descriptor words: Q tiles, K stages (LBO 16 B), V stages (LBO 16 KB)
            const uint32_t q_lo0 = sw128_desc_lo(q_addr, 16);
            const uint32_t k_lo0 = sw128_desc_lo(smem_u32(k_smem), 16);
            const uint32_t v_lo0 = sw128_desc_lo(smem_u32(v_smem), 16384);
            constexpr uint32_t kStageLo = C::kTileBytes >> 4;
            StageCtr ck, cv;  // K tile i, V tile i - 1
            bool ok = mbar_wait(q_full, 0, abort_flag, status, 0x02000000u);
            tc_fence_after();
            if (split) {
                // Both tile slots use Q tile 0; KV tile i goes to slot i % 2.
                // Issue order QK(i), PV(i-1) keeps one slot's softmax running
                // while the other slot's MMAs execute.
                for (int i = 0; ok && i <= total; ++i) {
                    if (i < total) {
                        const int t = i & 1;
                        ok = mbar_wait(&k_full[ck.s], ck.ph, abort_flag, status, 0x05000000u | i);
                        if (!ok) break;
                        tc_fence_after();
                        issue_qk<D>(tmem_base + t * 256, q_lo0, k_lo0 + ck.s * kStageLo);
                        mma_commit(&s_full[t]);
                        mma_commit(&k_empty[ck.s]);
                        ck.next(nK);
                    }
                    if (i > 0) {
                        const int i2 = i - 1;
                        const int t2 = i2 & 1;
                        const int j2 = i2 >> 1;
                        const uint32_t tS2 = tmem_base + t2 * 256;
                        ok = mbar_wait(&v_full[cv.s], cv.ph, abort_flag, status, 0x03000000u | i2);
                        if (!ok) break;
                        ok = mbar_wait(&p_full[t2], j2 & 1, abort_flag, status, 0x04000000u | i2);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv<D>(tS2 + 128, tS2, v_lo0 + cv.s * kStageLo, j2 > 0);
                        mma_commit(&o_done[t2]);
                        mma_commit(&v_empty[cv.s]);
                        cv.next(nV);
                    }
                }
            }
            // Paired tiles: iteration i issues PV_t(i-1) and QK_t(i) for t = 0, 1.
            // Two tiles (the common case): straight-line issue, stage descriptor
            // words advanced in place, ring position tracked only for partials.
            if (!split && T == 2) {
                const uint32_t tS0 = tmem_base, tS1 = tmem_base + 256;
                const uint32_t q0 = q_lo0, q1 = q_lo0 + kStageLo;
                const uint32_t k_end = k_lo0 + nK * kStageLo, v_end = v_lo0 + nV * kStageLo;
                uint32_t k_lo = k_lo0, v_lo = v_lo0;
                const bool track = PART && !FAN;
                RingIterT<LAY> wp;  // tile i - 1 (shard openings restart O in partials mode)
                if (track) wp.start(w);
                // One iteration with runtime stage indices.
                auto step = [&](int i) -> bool {
                    const uint32_t par = (i - 1) & 1;
                    const bool acc_prev = track ? !wp.first() : (i != 1);
                    if (i > 0) {
                        if (!mbar_wait(&v_full[cv.s], cv.ph, abort_flag, status, 0x03000000u | (i - 1))) return false;
                        if (!mbar_wait(&p_full[0], par, abort_flag, status, 0x04000000u | (i - 1))) return false;
                        tc_fence_after();
                        issue_pv<D>(tS0 + 128, tS0, v_lo, acc_prev);
                    }
                    if (i < total) {
                        if (!mbar_wait(&k_full[ck.s], ck.ph, abort_flag, status, 0x05000000u | i)) return false;
                        tc_fence_after();
                        issue_qk<D>(tS0, q0, k_lo);
                        mma_commit(&s_full[0]);
                    }
                    if (i > 0) {
                        if (!mbar_wait(&p_full[1], par, abort_flag, status, 0x04000000u | (i - 1))) return false;
                        tc_fence_after();
                        issue_pv<D>(tS1 + 128, tS1, v_lo, acc_prev);
                    }
                    if (i < total) issue_qk<D>(tS1, q1, k_lo);
                    // One commit frees K tile i and V tile i - 1 and hands S of tile
                    // 1 to its softmax; s_full / iter_done of the next tile tell the
                    // softmax that this iteration's PV is done.
                    mma_commit(&iter_done[i % C::kIterRing]);
                    if (i > 0) {
                        cv.next(nV);
                        v_lo = (v_lo + kStageLo == v_end) ? v_lo0 : v_lo + kStageLo;
                        if (track) wp.next();
                    }
                    if (i < total) {
                        ck.next(nK);
                        k_lo = (k_lo + kStageLo == k_end) ? k_lo0 : k_lo + kStageLo;
                    }
                    return true;
                };
                int i = 0;
                ok = total < 0 || step(0);
                i = 1;
                // Steady state in blocks of kBlk iterations from i = 1: kBlk is a
                // multiple of each ring size, of the iteration-barrier ring and of
                // 2, so every stage, barrier and slot parity below is a constant;
                // a ring's phase parity is a constant up to a per-block flip.
                constexpr int kBlk = C::kBlk;
                constexpr int nKc = C::kMaxKV, nVc = C::kNVPair;
                uint32_t kflip = 0, vflip = 0;
                // (ring prefill variants only: the fan-out variants and the former
                // layout-walk variant measured slower with it -- their larger code
                // missed the instruction cache: 3x the no-instruction stalls of the
                // contiguous mode under ncu)
                for (; (MODE == kModeRing || MODE == kModeRingPartials || STR || SPOS) && ok && i + kBlk <= total;
                     i += kBlk) {
                    const uint32_t kb = k_lo0, vb = v_lo0, qa = q0, qb = q1;
#pragma unroll
                    for (int pos = 0; pos < kBlk; ++pos) {
                        const int ks = (1 + pos) % nKc;
                        const uint32_t kph = (((1 + pos) / nKc) & 1) ^ kflip;
                        const int vs = pos % nVc;
                        const uint32_t vph = ((pos / nVc) & 1) ^ vflip;
                        const uint32_t par = pos & 1;
                        const bool acc_prev = track ? !wp.first() : (i + pos != 1);
                        if (!(ok = mbar_wait(&v_full[vs], vph, abort_flag, status, 0x03000000u))) break;
                        if (!(ok = mbar_wait(&p_full[0], par, abort_flag, status, 0x04000000u))) break;
                        tc_fence_after();
                        issue_pv<D>(tS0 + 128, tS0, vb + vs * kStageLo, acc_prev);
                        if (!(ok = mbar_wait(&k_full[ks], kph, abort_flag, status, 0x05000000u))) break;
                        tc_fence_after();
                        issue_qk<D>(tS0, qa, kb + ks * kStageLo);
                        mma_commit(&s_full[0]);
                        if (!(ok = mbar_wait(&p_full[1], par, abort_flag, status, 0x04000000u))) break;
                        tc_fence_after();
                        issue_pv<D>(tS1 + 128, tS1, vb + vs * kStageLo, acc_prev);
                        issue_qk<D>(tS1, qb, kb + ks * kStageLo);
                        mma_commit(&iter_done[(1 + pos) % C::kIterRing]);
                        if (track) wp.next();
                    }
                    if (C::kKFlip) kflip ^= 1;
                    if (C::kVFlip) vflip ^= 1;
                }
                // the runtime rings resume where the blocks left them
                ck.ph ^= kflip;
                cv.ph ^= vflip;
                for (; ok && i <= total; ++i) ok = step(i);
            }
            RingIterT<LAY> wp;  // at iteration i >= 1: tile i-1 (shard openings restart O in partials mode)
            if (!FAN) wp.start(w);
            for (int i = 0; ok && !split && T == 1 && i <= total; ++i) {
                const bool fresh_prev = (PART && !FAN) ? wp.first() : (i == 1);
                for (int t = 0; t < T && ok; ++t) {
                    const uint32_t tS = tmem_base + t * 256;
                    if (i > 0) {
                        if (t == 0) {
                            ok = mbar_wait(&v_full[cv.s], cv.ph, abort_flag, status, 0x03000000u | (i - 1));
                            if (!ok) break;
                        }
                        ok = mbar_wait(&p_full[t], (i - 1) & 1, abort_flag, status, 0x04000000u | (i - 1));
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv<D>(tS + 128, tS, v_lo0 + cv.s * kStageLo, !fresh_prev);
                    }
                    if (i < total) {
                        if (t == 0) {
                            ok = mbar_wait(&k_full[ck.s], ck.ph, abort_flag, status, 0x05000000u | i);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        issue_qk<D>(tS, q_lo0 + t * kStageLo, k_lo0 + ck.s * kStageLo);
                        mma_commit(&s_full[t]);
                    }
                }
                if (!ok) break;
                // one commit frees K tile i and V tile i - 1; s_full of the next
                // tile tells the softmax that this iteration's PV is done
                mma_commit(&iter_done[i % C::kIterRing]);
                if (i > 0) cv.next(nV);
                if (i < total) ck.next(nK);
                if (i > 0 && !FAN) wp.next();
            }
            // all issued MMAs complete before TMEM is released
            mma_commit(drain);
            mbar_wait(drain, 0, abort_flag, status, 0);
        }
    } else if (warp == 3) {
        reg_dec<MODE>();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        reg_inc<MODE>();
        const int t = (warp - 4) >> 2;
        if (t < T) {
        const int quad = warp & 3;
        const int lane_row = quad * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem_base + lane_off + t * 256;
        const uint32_t tO = tS + 128;

        // this thread's output row
        int row, head;
        bool row_ok;
        if (!FAN) {
            row = u.q_row0 + lane_row;
            head = CSEL ? (t ? u.head[1] : u.head[0]) : u.head[t];
            row_ok = true;
        } else {
            row = u.row0[t] + lane_row / p.G;
            head = u.kv_head * p.G + lane_row % p.G;
            row_ok = row < u.row_hi;
        }
        const OutDesc& out = p.out;
        // storage row of the output (striped over positions: position i sits in shard i mod N
        // at row i / N)
        const int out_row = FAN    ? row
                            : SPOS ? (row % p.n_shards) * (p.S / p.n_shards) + row / p.n_shards
                                   : u.q_srow0 + lane_row;
        const long long o_row_base = static_cast<long long>(u.b) * out.o_b + static_cast<long long>(out_row) * out.o_row +
                                     static_cast<long long>(head) * out.o_h;
        const long long lse_base = static_cast<long long>(u.b) * out.lse_b + static_cast<long long>(head) * out.lse_h + out_row;

        float m_use = -INFINITY, l_sum = 0.f;
        bool ok = true;
        // zigzag / striped causal walks: this row's sequence position
        const int shard_len = LAY ? p.S / p.n_shards : 0;
        const int row_pos = LAY ? layout_pos(p.layout, shard_len, p.n_shards, row) : row;
        // the query tile's first row has its smallest position: the keys of a shard it
        // sees are seen by every row, so whole tiles of them need no mask
        const int tile_minpos = LAY ? layout_pos(p.layout, shard_len, p.n_shards, FAN ? 0 : u.q_row0) : 0;
        int lay_full = 0;  // leading tiles of the current shard every row sees whole
        const int shard_len_c = STR ? p.S / p.n_shards : 0;
        const int q_shard = STR ? u.q_row0 / shard_len_c : 0;

        // Normalise the O accumulator and write it as part `part`, once `done`
        // (if given) shows its last PV complete.
        // Rows staged in shared memory for the final flush: the K/V stages are
        // idle once every MMA has completed.  Rows are padded by 16 bytes so
        // that a warp's 16-byte writes of 32 rows spread over all banks.
        const int row_bytes = D * (out.o_f32 ? 4 : 2);
        const int stage_stride = row_bytes + 16;
        constexpr int kSplitXBytes = (D * 128 + 4 * 128) * 4;  // split combine exchange ahead of the stage
        uint8_t* srow = kv_smem + (split ? kSplitXBytes : 0) + (t * 128 + lane_row) * stage_stride;
        bool staged = false;  // a bulk store of this thread is in flight
        auto flush = [&](uint64_t* done, uint32_t phase, int part) -> bool {
            if (done) {
                if (!mbar_wait(done, phase, abort_flag, status, 0x06000000u)) return false;
                tc_fence_after();
            }
            const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
            const long long ob = o_row_base + static_cast<long long>(part) * out.o_part;
            // the final flush (after `drain`) stages the row; mid-walk flushes
            // (per-shard partials, K/V stages busy) write it directly
            const bool stage = (done == drain);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tO + c * 32, r);
                tmem_wait_ld();
                if (stage)
                    stage_row<D>(out, srow, c, reinterpret_cast<const float*>(r), inv_l);
                else if (row_ok)
                    store_row<D>(out, ob, c, reinterpret_cast<const float*>(r), inv_l);
            }
            if (stage && row_ok) {
                bulk_store(static_cast<char*>(out.o) + ob * (out.o_f32 ? 4 : 2), srow, row_bytes);
                staged = true;
            }
            if (row_ok && out.lse) {
                const float L = l_sum > 0.f ? (m_use + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
                out.lse[lse_base + static_cast<long long>(part) * out.lse_part] = L;
            }
            return true;
        };

        // Walk tiles of this slot: all of them, or every other one in split mode.
        const int i_step = split ? 2 : 1;
        int jj = 0;  // this slot's tile count so far (barrier phase index)
        TileWalk<FAN, LAY> wi;
        wi.start(p, u, w);
        if (split && t == 1) wi.next(p, u);
        int last_shard = FAN ? 0 : wi.ring.j;
        for (int i = split ? t : 0; i < total; i += i_step, ++jj) {
            if (jj > 0) {
                wi.next(p, u);
                if (split) wi.next(p, u);
            }
            const bool tile_first = !FAN && wi.ring.first();
            const int tile_kb = wi.key();
            // S of tile 1 of a two-tile unit is signalled by the iteration-done
            // commit that follows its QK (no separate commit)
            uint64_t* s_bar = &s_full[t];
            uint32_t s_par = jj & 1;
            if (t == 1 && !split && T == 2) {
                s_bar = &iter_done[jj % C::kIterRing];
                s_par = (jj / C::kIterRing) & 1;
            }
            if (!(ok = mbar_wait(s_bar, s_par, abort_flag, status, 0x07000000u | i))) break;
            tc_fence_after();
            if (PART && tile_first && jj > 0) {
                // The previous KV shard of the ring is complete (this tile's S was
                // committed after its last PV): flush it.
                flush(nullptr, 0, last_shard);
                m_use = -INFINITY;
                l_sum = 0.f;
            }
            if (!FAN) last_shard = wi.ring.j;
            // visible columns of this tile: c <= lim (only diagonal and tail tiles mask)
            int lim = kTileN - 1;
            if (!FAN) {
                // keys of this tile the row sees: a prefix of the tile (positions
                // increase along a shard), ending where the shard's visible keys end
                if (LAY) {
                    if (wi.ring.in == 0)
                        lay_full = shard_visible(p.layout, shard_len, p.n_shards, wi.ring.j, tile_minpos) / kTileN;
                    if (wi.ring.in >= lay_full)
                        lim = min(lim, shard_visible(p.layout, shard_len, p.n_shards, wi.ring.j, row_pos) -
                                           (tile_kb - wi.ring.j * shard_len) - 1);
                } else if (p.causal) {
                    // striped: key offset <= row offset in the query's shard and the
                    // shards before it in the sequence, < in the shards after it
                    lim = min(lim, STR ? row - tile_kb + (wi.ring.j - q_shard) * shard_len_c - (wi.ring.j > q_shard)
                                       : row - tile_kb);
                }
            } else {
                lim = min(lim, wi.key_end - 1 - tile_kb);
                // rows of another branch (a folded suffix) or past the stacked rows
                if (row < wi.row_lo || row >= wi.row_hi) lim = -1;
                // prefill: row t of a branch of n rows sits at suffix position S_suffix - n + t
                if (p.suffix_causal && wi.seg == 1)
                    lim = min(lim, wi.key_end - (wi.row_hi - wi.row_lo) + (row - wi.row_lo) - tile_kb);
            }
            if (FAN && __all_sync(0xffffffffu, lim < 0)) {
                // No row of this warp sees a key of this tile: P = 0 (written over
                // S, after the QK above has landed) and the running state stays.
                const uint32_t z = 0;
#pragma unroll
                for (int c0 = 0; c0 < kTileN; c0 += 32)
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                        "{%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};" ::"r"(tS + c0 / 2),
                        "r"(z)
                        : "memory");
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&p_full[t]);
                continue;
            }
            uint32_t sr[kTileN];
#pragma unroll
            for (int c = 0; c < kTileN / 32; ++c) tmem_ld32(tS + c * 32, sr + c * 32);
            tmem_wait_ld();
            // A row that sees no key of this tile keeps its state and gets P = 0
            // through the exponent (scale 0, offset -inf) rather than a masking
            // pass; only partially visible rows (diagonal, segment tails) mask.
            const bool dead_row = lim < 0;
            if (lim < kTileN - 1 && !dead_row) {
#pragma unroll
                for (int c = 0; c < kTileN; ++c)
                    if (c > lim) sr[c] = 0xff800000u;  // -inf
            }
            // row max as four independent chains (a quarter of the dependent latency)
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < kTileN; c += 8) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    m4[q] = fmax3(m4[q], __uint_as_float(sr[c + 2 * q]), __uint_as_float(sr[c + 2 * q + 1]));
            }
            const float mraw = dead_row ? -INFINITY : fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
            const float mx = mraw * p.scale_log2;  // scores in log2 units
            const bool fresh = (jj == 0) || (PART && tile_first);
            float alpha = 1.f;
            bool resc = false;
            if (fresh) {
                m_use = mx;
                l_sum = 0.f;
            } else if (mx > m_use + kRescaleLog2) {
                alpha = (m_use == -INFINITY) ? 0.f : ex2_approx(m_use - mx);
                m_use = mx;
                resc = true;
            }
            const float neg_ms = dead_row ? -INFINITY : ((m_use == -INFINITY) ? 0.f : -m_use);
            const float sc = dead_row ? 0.f : p.scale_log2;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < kTileN; c0 += 32) {
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float y0, y1;
                    ffma2(y0, y1, __uint_as_float(sr[c0 + 2 * j]), __uint_as_float(sr[c0 + 2 * j + 1]), sc, sc,
                          neg_ms, neg_ms);
                    const float p0 = ex2_approx(y0);
                    const float p1 = ex2_approx(y1);
                    if (j & 1)
                        fadd2(a2, a3, p0, p1);
                    else
                        fadd2(a0, a1, p0, p1);
                    pk[j] = pack_bf16x2(p0, p1);
                }
                asm volatile(
                    "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                    "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(tS + c0 / 2),
                    "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7]),
                    "r"(pk[8]), "r"(pk[9]), "r"(pk[10]), "r"(pk[11]), "r"(pk[12]), "r"(pk[13]), "r"(pk[14]),
                    "r"(pk[15])
                    : "memory");
            }
            const float rs = (a0 + a1) + (a2 + a3);
            l_sum = l_sum * alpha + rs;
            if (__any_sync(0xffffffffu, resc)) {
                // O of the previous tiles is complete: this tile's S was committed
                // after their PV.
                const float a = resc ? alpha : 1.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tO + c * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * a);
                    tmem_st32(tO + c * 32, r);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[t]);
        }
        if (split) {
            // The two slots hold online-softmax states of disjoint KV tiles of the
            // same rows.  Each slot combines half of the head dims: it hands the
            // other half of its O (with m and l) to the other slot through shared
            // memory (the KV stages are idle once every MMA has completed), then
            // writes the log-sum-exp combination of its half; slot 0 writes lse.
            // Both slots always meet at the named barrier (an empty or failed
            // slot offers m = -inf, which the other ignores).
            constexpr int kHalf = D / 2;
            float* xo = reinterpret_cast<float*>(kv_smem);  // [2 slots][kHalf][128], column-major: conflict-free
            float* xm = xo + 2 * kHalf * 128;               // [2][128]
            float* xl = xm + 2 * 128;                       // [2][128]
            const int give = t == 0 ? kHalf : 0;            // columns this slot hands over
            const int keep = t == 0 ? 0 : kHalf;            // columns this slot combines
            bool have = ok && jj > 0 &&
                        (t == 0 ? mbar_wait(&o_done[0], (jj - 1) & 1, abort_flag, status, 0x0A000000u | jj)
                                : mbar_wait(drain, 0, abort_flag, status, 0x09000000u));
            have = __all_sync(0xffffffffu, have);
            if (have) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kHalf / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tO + give + c * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) xo[(t * kHalf + c * 32 + j) * 128 + lane_row] = __uint_as_float(r[j]);
                }
            }
            xm[t * 128 + lane_row] = have ? m_use : -INFINITY;
            xl[t * 128 + lane_row] = have ? l_sum : 0.f;
            asm volatile("bar.sync 1, 256;" ::: "memory");
            const float m1 = xm[(t ^ 1) * 128 + lane_row], l1 = xl[(t ^ 1) * 128 + lane_row];
            const float m0 = have ? m_use : -INFINITY, l0 = have ? l_sum : 0.f;
            const float m = fmaxf(m0, m1);
            const float a0 = (m0 == -INFINITY) ? 0.f : ex2_approx(m0 - m);
            const float a1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - m);
            const float L = a0 * l0 + a1 * l1;
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const long long ob = o_row_base + static_cast<long long>(u.slot[0]) * out.o_part + keep;
            const int half_bytes = kHalf * (out.o_f32 ? 4 : 2);
            uint8_t* hrow = kv_smem + kSplitXBytes + (t * 128 + lane_row) * (half_bytes + 16);
#pragma unroll
            for (int c = 0; c < kHalf / 32; ++c) {
                uint32_t r[32];
                if (have) {
                    tmem_ld32(tO + keep + c * 32, r);
                    tmem_wait_ld();
                }
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float o0 = have ? __uint_as_float(r[j]) : 0.f;
                    const float o1 = (a1 != 0.f) ? xo[((t ^ 1) * kHalf + c * 32 + j) * 128 + lane_row] : 0.f;
                    v[j] = a0 * o0 + a1 * o1;
                }
                stage_row<D>(out, hrow, c, v, inv);
            }
            if (row_ok) {
                bulk_store(static_cast<char*>(out.o) + ob * (out.o_f32 ? 4 : 2), hrow, half_bytes);
                staged = true;
            }
            if (t == 0 && row_ok && out.lse)
                out.lse[lse_base + static_cast<long long>(u.slot[0]) * out.lse_part] =
                    L > 0.f ? (m + log2f(L)) * 0.69314718055994531f : -INFINITY;
        } else if (ok) {
            // the last PV: every MMA of the CTA is complete once `drain` is
            if (!FAN && PART) {
                ok = flush(drain, 0, last_shard);
            } else if (jj > 0) {
                ok = flush(drain, 0, FAN ? u.slot[t] : 0);
            } else if (row_ok && out.lse) {
                // a unit with no KV tile: an empty partial (its O is never read)
                out.lse[lse_base + static_cast<long long>(CSEL ? (t ? u.slot[1] : u.slot[0]) : u.slot[t]) *
                                       out.lse_part] = -INFINITY;
            }
        }
        if (ok && !FAN && PART) {
            // KV shards the causal mask empties for this tile: O = 0, lse = -inf
            for (int t2 = w.n_visited; t2 < p.n_shards; ++t2) {
                const int j = ring_shard_at(w, t2);
                const long long ob = o_row_base + static_cast<long long>(j) * out.o_part;
                float zeros[32];
#pragma unroll
                for (int z = 0; z < 32; ++z) zeros[z] = 0.f;
                for (int c = 0; c < D / 32; ++c) store_row<D>(out, ob, c, zeros, 0.f);
                if (out.lse) out.lse[lse_base + static_cast<long long>(j) * out.lse_part] = -INFINITY;
            }
        }
        if (staged) bulk_store_wait();  // the staged rows have left shared memory
        }
        tc_fence_before();
    }

    __syncthreads();
    if (threadIdx.x == 0) grid_launch_dependents();  // outputs written: the merge may start
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int D, int MODE>
cudaError_t launch(const TcParams& p, int grid, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                   const CUtensorMap& k2, const CUtensorMap& v2, cudaStream_t stream) {
    const int smem = Cfg<D>::kSmemBytes;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(attn_tc_kernel<D, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        // the softmax warpgroups' register increase draws on the launch's registers:
        // a build that launched with fewer would wait for them forever
        cudaFuncAttributes fa;
        if (attr_err == cudaSuccess) attr_err = cudaFuncGetAttributes(&fa, attn_tc_kernel<D, MODE>);
        if (attr_err == cudaSuccess && fa.numRegs < kLaunchRegs) attr_err = cudaErrorLaunchOutOfResources;
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (grid <= 0) return cudaSuccess;
    attn_tc_kernel<D, MODE><<<grid, kThreads, smem, stream>>>(q, k, v, k2, v2, p);
    return cudaGetLastError();
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// bf16 tensor map of `rank` (4 or 5) dims, innermost first, strides in bytes for
// dims 1.., box (64, b1, ...), 128-byte swizzle.
static bool make_map_nd(CUtensorMap* m, const void* base, int rank, const unsigned long long* dims,
                        const unsigned long long* strides, const unsigned* box) {
    auto fn = encode_fn();
    if (!fn || rank < 1 || rank > 5) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i > 0) gs[i - 1] = strides[i - 1];
    }
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gd, gs, bx, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D bf16 tensor map, dims innermost first, strides in bytes for dims 1..3,
// box (64, b1, b2, b3), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, const unsigned long long dims[4], const unsigned long long strides[3],
              const unsigned box[4]) {
    return make_map_nd(m, base, 4, dims, strides, box);
}

bool make_map_5d(CUtensorMap* m, const void* base, const unsigned long long dims[5],
                 const unsigned long long strides[4], const unsigned box[5]) {
    return make_map_nd(m, base, 5, dims, strides, box);
}

cudaError_t launch_ring_tc(const RingTcArgs& a, cudaStream_t stream) {
    TcParams p{};
    p.fanout = 0;
    p.causal = a.causal;
    p.layout = a.layout;
    p.B = a.B;
    p.S = a.S;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.n_shards = a.n_shards;
    p.n_qtiles = a.S / kTileM;
    p.T2 = ((a.Hq / a.Hkv) % 2 == 0) ? 1 : 0;
    p.n_head_groups = a.Hq / (p.T2 ? 2 : 1);
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.D)));
    p.out = a.out;
    const unsigned long long D = a.D, esz = 2;
    CUtensorMap tq, tk, tv;
    const unsigned long long qd[4] = {D, (unsigned long long)a.Hq, (unsigned long long)a.S, (unsigned long long)a.B};
    const unsigned long long qs[3] = {D * esz, D * esz * a.Hq, D * esz * a.Hq * a.S};
    const unsigned long long kd[4] = {D, (unsigned long long)a.Hkv, (unsigned long long)a.S, (unsigned long long)a.B};
    const unsigned long long ks[3] = {D * esz, D * esz * a.Hkv, D * esz * a.Hkv * a.S};
    const unsigned box[4] = {64, 1, 128, 1};
    if (!make_map(&tq, a.q, qd, qs, box) || !make_map(&tk, a.k, kd, ks, box) || !make_map(&tv, a.v, kd, ks, box))
        return cudaErrorInvalidValue;
    const int grid = p.n_qtiles * a.B * p.n_head_groups;
    // A causal zigzag sequence with one output is the contiguous causal problem on
    // its 2N chunks of L/2 tokens, each 128-row tile addressed through the chunk map:
    // the contiguous ring over the 2N chunks visits the same tiles and masks only
    // the diagonal one, in the contiguous variant's code (order changes rounding only).
    if (a.causal && a.layout == kLayoutZigzag && !a.partials) {
        p.layout = kLayoutContiguous;
        p.n_shards = 2 * a.n_shards;
        p.zz_n = a.n_shards;
        p.zz_half = a.S / (2 * a.n_shards);
        return a.D == 128 ? launch<128, kModeRing>(p, grid, tq, tk, tv, tk, tv, stream)
                          : launch<64, kModeRing>(p, grid, tq, tk, tv, tk, tv, stream);
    }
    // A causal striped sequence with one output: over positions (below) when N divides
    // 128, otherwise the layout's own ring walk, in a variant compiled from the contiguous
    // one with its per-shard tile counts and diagonal masks.
    if (a.causal && a.layout == kLayoutStriped && !a.partials) {
        p.layout = kLayoutContiguous;
        if (128 % a.n_shards == 0) {
            // N dividing 128: a tile of 128 consecutive positions holds 128/N rows of every
            // shard, one 5-D box [64 cols, 1 head, N shards, 128/N rows, 1 batch] per 64
            // columns (the shard the faster box dimension: rows land in position order), and
            // the contiguous causal walk runs over positions (N position-order shards of L
            // tokens; the same visible keys, one diagonal tile per query tile)
            const unsigned long long L = a.S / a.n_shards, N = a.n_shards, S = a.S, B = a.B;
            const unsigned long long qd5[5] = {D, (unsigned long long)a.Hq, N, L, B};
            const unsigned long long qs5[4] = {D * esz, L * a.Hq * D * esz, a.Hq * D * esz, S * a.Hq * D * esz};
            const unsigned long long kd5[5] = {D, (unsigned long long)a.Hkv, N, L, B};
            const unsigned long long ks5[4] = {D * esz, L * a.Hkv * D * esz, a.Hkv * D * esz, S * a.Hkv * D * esz};
            const unsigned box5[5] = {64, 1, (unsigned)N, (unsigned)(128 / N), 1};
            CUtensorMap tq5, tk5, tv5;
            if (!make_map_nd(&tq5, a.q, 5, qd5, qs5, box5) || !make_map_nd(&tk5, a.k, 5, kd5, ks5, box5) ||
                !make_map_nd(&tv5, a.v, 5, kd5, ks5, box5))
                return cudaErrorInvalidValue;
            return a.D == 128 ? launch<128, kModeRingStripedPos>(p, grid, tq5, tk5, tv5, tk5, tv5, stream)
                              : launch<64, kModeRingStripedPos>(p, grid, tq5, tk5, tv5, tk5, tv5, stream);
        }
        return a.D == 128 ? launch<128, kModeRingStriped>(p, grid, tq, tk, tv, tk, tv, stream)
                          : launch<64, kModeRingStriped>(p, grid, tq, tk, tv, tk, tv, stream);
    }
    // without a causal mask every layout is the same walk
    if (a.causal && a.layout != kLayoutContiguous)
        return a.D == 128 ? launch<128, kModeRingLayoutPartials>(p, grid, tq, tk, tv, tk, tv, stream)
                          : launch<64, kModeRingLayoutPartials>(p, grid, tq, tk, tv, tk, tv, stream);
    p.layout = kLayoutContiguous;
    if (a.partials)
        return a.D == 128 ? launch<128, kModeRingPartials>(p, grid, tq, tk, tv, tk, tv, stream)
                          : launch<64, kModeRingPartials>(p, grid, tq, tk, tv, tk, tv, stream);
    return a.D == 128 ? launch<128, kModeRing>(p, grid, tq, tk, tv, tk, tv, stream)
                      : launch<64, kModeRing>(p, grid, tq, tk, tv, tk, tv, stream);
}

cudaError_t launch_fanout_tc(const FanoutTcArgs& a, cudaStream_t stream) {
    TcParams p{};
    p.fanout = 1;
    p.causal = 0;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.R = a.R;
    p.G = a.Hq / a.Hkv;
    p.rows_per_tile = kTileM / p.G;
    p.n_mpairs = (a.R + 2 * p.rows_per_tile - 1) / (2 * p.rows_per_tile);
    p.S_prefix = a.S_prefix;
    p.n_chunks = a.n_chunks;
    for (int c = 0; c <= a.n_chunks && c <= kMaxChunks; ++c) p.chunk_start[c] = a.chunk_start[c];
    p.S_suffix = a.S_suffix;
    p.n_branches = a.n_branches;
    p.suffix_mpairs = p.n_mpairs;  // upper bound: a branch holds at most R rows
    p.offsets = a.offsets;
    p.n_prefix_units = (a.S_prefix > 0) ? a.Hkv * p.n_mpairs * a.n_chunks : 0;
    fanout_slots(a.R, a.Hq, a.Hkv, a.S_prefix > 0 ? a.n_chunks : 0, a.S_prefix, a.S_suffix, &p.split_prefix,
                 &p.suffix_slot0);
    p.fold = (a.S_prefix > 0 && a.S_suffix > 0) ? 1 : 0;
    p.suffix_causal = a.suffix_causal;
    p.paged = a.paged;
    p.page_shift = a.page_shift;
    p.n_pages = a.n_pages;
    p.n_prefix_pages = a.n_prefix_pages;
    p.n_suffix_pages = a.n_suffix_pages;
    p.prefix_pages = a.prefix_pages;
    p.suffix_pages = a.suffix_pages;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.D)));
    p.out = a.part;
    const unsigned long long D = a.D, esz = 2;
    CUtensorMap tq, tk, tv, tk2, tv2;
    const unsigned long long qd[4] = {D, (unsigned long long)p.G, (unsigned long long)a.Hkv, (unsigned long long)a.R};
    const unsigned long long qs[3] = {D * esz, D * esz * p.G, D * esz * a.Hq};
    const unsigned qbox[4] = {64, (unsigned)p.G, 1, (unsigned)p.rows_per_tile};
    const unsigned box[4] = {64, 1, 128, 1};
    if (!make_map(&tq, a.q_rows, qd, qs, qbox)) return cudaErrorInvalidValue;
    const unsigned long long kd[4] = {D, (unsigned long long)a.Hkv,
                                      (unsigned long long)(a.S_prefix > 0 ? a.S_prefix : 1), 1};
    const unsigned long long ks[3] = {D * esz, D * esz * a.Hkv, D * esz * a.Hkv * (a.S_prefix > 0 ? a.S_prefix : 1)};
    const unsigned long long sd[4] = {D, (unsigned long long)a.Hkv, (unsigned long long)(a.S_suffix > 0 ? a.S_suffix : 1),
                                      (unsigned long long)a.n_branches};
    const unsigned long long ss[3] = {D * esz, D * esz * a.Hkv, D * esz * a.Hkv * (a.S_suffix > 0 ? a.S_suffix : 1)};
    const void* kp = a.S_prefix > 0 ? a.k_prefix : a.k_suffix;
    const void* vp = a.S_prefix > 0 ? a.v_prefix : a.v_suffix;
    const void* ksf = a.S_suffix > 0 ? a.k_suffix : a.k_prefix;
    const void* vsf = a.S_suffix > 0 ? a.v_suffix : a.v_prefix;
    if (a.paged) {
        // both segments read the page pool, in boxes of one page (at most 128 rows)
        const unsigned long long rows = static_cast<unsigned long long>(a.n_pages) << a.page_shift;
        const unsigned long long pd[4] = {D, (unsigned long long)a.Hkv, rows, 1};
        const unsigned long long ps[3] = {D * esz, D * esz * a.Hkv, D * esz * a.Hkv * rows};
        const unsigned pbox[4] = {64, 1, (unsigned)((1 << a.page_shift) < 128 ? (1 << a.page_shift) : 128), 1};
        if (!make_map(&tk, a.k_prefix, pd, ps, pbox) || !make_map(&tv, a.v_prefix, pd, ps, pbox))
            return cudaErrorInvalidValue;
        tk2 = tk;
        tv2 = tv;
    } else if (a.S_prefix > 0) {
        if (!make_map(&tk, kp, kd, ks, box) || !make_map(&tv, vp, kd, ks, box)) return cudaErrorInvalidValue;
    }
    if (!a.paged && a.S_suffix > 0) {
        if (!make_map(&tk2, ksf, sd, ss, box) || !make_map(&tv2, vsf, sd, ss, box)) return cudaErrorInvalidValue;
    }
    if (!a.paged && a.S_prefix == 0) {
        tk = tk2;
        tv = tv2;
    }
    if (!a.paged && a.S_suffix == 0) {
        tk2 = tk;
        tv2 = tv;
    }
    const int n_suffix_units = (a.S_suffix > 0 && !p.fold) ? a.n_branches * a.Hkv * p.suffix_mpairs : 0;
    const int grid = p.n_prefix_units + n_suffix_units;
    // uniform launches (prefix units only) get the variant compiled for their mode
    if (a.paged) {
        if (n_suffix_units == 0 && p.split_prefix)
            return a.D == 128 ? launch<128, kModeFanSplitPaged>(p, grid, tq, tk, tv, tk2, tv2, stream)
                              : launch<64, kModeFanSplitPaged>(p, grid, tq, tk, tv, tk2, tv2, stream);
        if (n_suffix_units == 0)
            return a.D == 128 ? launch<128, kModeFanPairedPaged>(p, grid, tq, tk, tv, tk2, tv2, stream)
                              : launch<64, kModeFanPairedPaged>(p, grid, tq, tk, tv, tk2, tv2, stream);
        return a.D == 128 ? launch<128, kModeFanMixedPaged>(p, grid, tq, tk, tv, tk2, tv2, stream)
                          : launch<64, kModeFanMixedPaged>(p, grid, tq, tk, tv, tk2, tv2, stream);
    }
    if (n_suffix_units == 0 && p.split_prefix)
        return a.D == 128 ? launch<128, kModeFanSplit>(p, grid, tq, tk, tv, tk2, tv2, stream)
                          : launch<64, kModeFanSplit>(p, grid, tq, tk, tv, tk2, tv2, stream);
    if (n_suffix_units == 0)
        return a.D == 128 ? launch<128, kModeFanPaired>(p, grid, tq, tk, tv, tk2, tv2, stream)
                          : launch<64, kModeFanPaired>(p, grid, tq, tk, tv, tk2, tv2, stream);
    return a.D == 128 ? launch<128, kModeFanMixed>(p, grid, tq, tk, tv, tk2, tv2, stream)
                      : launch<64, kModeFanMixed>(p, grid, tq, tk, tv, tk2, tv2, stream);
}

unsigned read_clear_status_tc(unsigned* where) {
    unsigned h[2] = {0, 0};
    cudaMemcpyFromSymbol(h, g_tc_status, sizeof h);
    if (h[0]) {
        const unsigned z[2] = {0, 0};
        cudaMemcpyToSymbol(g_tc_status, z, sizeof z);
    }
    if (where) *where = h[1];
    return h[0];
}

}  // namespace ra
