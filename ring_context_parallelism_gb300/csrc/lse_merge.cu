// lse_merge.cu -- row-indexed log-sum-exp merge of partial attention states.
//
// "AHBM Agentic Runtime Architecture", sections 3.4-3.5: partial states of the
// same query row computed over different sequence shards are merged row by
// row (never across rows), by the same primitive at every level of the
// reduction.  With normalised partials (O_p, lse_p) the merge is
//   M = max_p lse_p,  w_p = exp(lse_p - M),
//   O = sum_p w_p O_p / sum_p w_p,  lse = M + ln(sum_p w_p),
// which is the exactness identity of "RingAttention and Context Parallelism",
// section 2, applied to whole shards.  An empty partial (lse = -inf) gets
// weight 0 and its O does not enter the result, whatever it holds.
//
// Lane l owns D/32 consecutive head dims, so a warp reads each partial row as
// one contiguous 128- to 512-byte segment.  fp32 arithmetic.  Bandwidth-bound:
// each partial row is read once.  Four kernels, chosen by shape: a tiled one
// for many rows and up to 256 partials (coalesced lse reads, weights in shared
// memory); for fewer rows, bulk copies of up to 32 partials' rows into shared
// memory (every byte a CTA needs in flight at once), a block per row for more
// partials than that, and a looping warp per row otherwise.  With heads in
// multiples of 8 and up to 32 partials, the many-row merge takes blocks of 8
// heads x 32 positions, whose per-position segments are contiguous.
#include <cmath>

#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {

static __device__ unsigned g_merge_status[2];

namespace {

constexpr int kWarps = 8;

template <int E, bool F32>
struct Vec;  // E consecutive elements of one lane
template <>
struct Vec<4, true> {
    static __device__ __forceinline__ void load(const void* p, float* x) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    static __device__ __forceinline__ void store(void* p, const float* x) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};
template <>
struct Vec<2, true> {
    static __device__ __forceinline__ void load(const void* p, float* x) {
        const float2 v = *reinterpret_cast<const float2*>(p);
        x[0] = v.x; x[1] = v.y;
    }
    static __device__ __forceinline__ void store(void* p, const float* x) {
        *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    }
};
template <>
struct Vec<4, false> {
    static __device__ __forceinline__ void load(const void* p, float* x) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
        x[0] = __low2float(a); x[1] = __high2float(a); x[2] = __low2float(b); x[3] = __high2float(b);
    }
    static __device__ __forceinline__ void store(void* p, const float* x) {
        *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    }
};
template <>
struct Vec<2, false> {
    static __device__ __forceinline__ void load(const void* p, float* x) {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(p);
        x[0] = __low2float(a); x[1] = __high2float(a);
    }
    static __device__ __forceinline__ void store(void* p, const float* x) {
        *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(x[0], x[1]);
    }
};

// N consecutive elements (N = 4 or 8) as 16-byte vector accesses.
template <int N, bool F32>
__device__ __forceinline__ void load_elems(const void* p, float* x) {
    if (F32) {
#pragma unroll
        for (int k = 0; k < N / 4; ++k) {
            const float4 v = reinterpret_cast<const float4*>(p)[k];
            x[4 * k] = v.x; x[4 * k + 1] = v.y; x[4 * k + 2] = v.z; x[4 * k + 3] = v.w;
        }
    } else if (N == 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    } else {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xFFFF0000u);
        x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xFFFF0000u);
    }
}

template <int N, bool F32>
__device__ __forceinline__ void store_elems(void* p, const float* x) {
    if (F32) {
#pragma unroll
        for (int k = 0; k < N / 4; ++k)
            reinterpret_cast<float4*>(p)[k] = make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
    } else if (N == 8) {
        *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                                  pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
    } else {
        *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    }
}

template <int D, bool PART_F32, bool OUT_F32>
__global__ void __launch_bounds__(kWarps * 32) lse_merge_kernel(const void* __restrict__ part_O,
                                                                const float* __restrict__ part_lse,
                                                                void* __restrict__ out, float* __restrict__ out_lse,
                                                                int P, int S, int H, long long rows) {
    constexpr int E = D / 32;
    grid_dependency_wait();
    const long long rid = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (rid >= rows) return;
    const int lane = threadIdx.x & 31;
    // rid = (b*S + s)*H + h
    const int h = static_cast<int>(rid % H);
    const long long bs = rid / H;
    const int s = static_cast<int>(bs % S);
    const long long b = bs / S;
    const long long lse_idx = (b * H + h) * S + s;
    const long long o_stride = rows * D;  // elements between partials
    const long long l_stride = rows;

    // Lane j holds lse of partial g*32 + j; the weights are broadcast with
    // shuffles and the partials' rows are loaded 8 at a time so that several
    // loads are in flight per lane.
    float M = -INFINITY;
    for (int g = 0; g < P; g += 32) {
        const int pp = g + lane;
        const float L = pp < P ? part_lse[pp * l_stride + lse_idx] : -INFINITY;
        M = fmaxf(M, L);
    }
#pragma unroll
    for (int x = 16; x; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (M != -INFINITY) {
        const size_t esz = PART_F32 ? 4 : 2;
        const char* base = static_cast<const char*>(part_O) + (rid * D + lane * E) * esz;
        for (int g = 0; g < P; g += 32) {
            const int pp = g + lane;
            const float L = pp < P ? part_lse[pp * l_stride + lse_idx] : -INFINITY;
            const float myw = (L == -INFINITY) ? 0.f : expf(L - M);   // empty partial: weight 0
            float ws = myw;
#pragma unroll
            for (int x = 16; x; x >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, x);
            wsum += ws;
            const int n = min(32, P - g);
            for (int j0 = 0; j0 < n; j0 += 8) {
                float w[8];
                float x[8][E];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    w[j] = __shfl_sync(0xffffffffu, myw, (j0 + j) & 31);
                    if (j0 + j >= n) w[j] = 0.f;
                    if (w[j] != 0.f) {
                        Vec<E, PART_F32>::load(base + static_cast<long long>(g + j0 + j) * o_stride * esz, x[j]);
                    } else {
#pragma unroll
                        for (int e = 0; e < E; ++e) x[j][e] = 0.f;   // O of an empty partial is not read
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[e] = fmaf(w[j], x[j][e], acc[e]);
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= inv;
    char* dst = static_cast<char*>(out) + (rid * D + lane * E) * (OUT_F32 ? 4 : 2);
    Vec<E, OUT_F32>::store(dst, acc);
    if (out_lse && lane == 0) out_lse[lse_idx] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

// Tiled variant (P <= kMaxTiledP): a block owns 32 consecutive positions s of
// one (b, h).  Phase 1: lane l of every warp reads lse of position s0 + l for
// a subset of the partials -- consecutive lanes, consecutive addresses -- and
// the block forms the max, the weights and their sum in shared memory.
// Phase 2: each warp merges four of the 32 rows, streaming each non-empty
// partial row (D contiguous elements) with eight loads in flight.
constexpr int kMaxTiledP = 256;

// Few rows, up to 32 partials: a CTA takes rb <= 8 consecutive rows.  The
// rows of one partial are contiguous, so thread 0 fetches each partial's rb
// rows with one bulk copy into shared memory (all P copies in flight at once,
// no register or L1 miss slots held), while warp w reads lse of its row, one
// partial per lane.  Warp w then combines row w from shared memory.  Rows of
// empty partials are copied (they lie inside the caller's buffer) but dropped
// by a select, never multiplied in, so whatever they hold (NaN included)
// cannot reach the result.
constexpr int kBulkMaxP = 32;
template <int D, bool PART_F32, bool OUT_F32>
__global__ void __launch_bounds__(kWarps * 32) lse_merge_bulk_kernel(const void* __restrict__ part_O,
                                                                     const float* __restrict__ part_lse,
                                                                     void* __restrict__ out,
                                                                     float* __restrict__ out_lse, int P, int S, int H,
                                                                     long long rows, int rb) {
    constexpr int E = D / 32;
    constexpr int esz = PART_F32 ? 4 : 2;
    constexpr int kRowBytes = D * esz;
    extern __shared__ __align__(128) uint8_t smem[];  // [P][rb][D] partial rows, then the barrier
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + P * rb * kRowBytes);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long rid0 = static_cast<long long>(blockIdx.x) * rb;
    const int nr = static_cast<int>(rows - rid0 < rb ? rows - rid0 : rb);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dependency_wait();
    if (threadIdx.x == 0) {
        const uint32_t seg = static_cast<uint32_t>(nr) * kRowBytes;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(P) * seg);
        for (int p = 0; p < P; ++p)
            bulk_load(smem + p * rb * kRowBytes,
                      static_cast<const char*>(part_O) + (static_cast<long long>(p) * rows + rid0) * kRowBytes, seg,
                      bar);
    }
    const long long rid = rid0 + warp;
    long long lse_idx = 0;
    float L = -INFINITY;
    if (warp < nr) {
        const int h = static_cast<int>(rid % H);
        const long long bs = rid / H;
        const int s = static_cast<int>(bs % S);
        const long long b = bs / S;
        lse_idx = (b * H + h) * S + s;
        if (lane < P) L = part_lse[lane * rows + lse_idx];
    }
    if (!mbar_wait(bar, 0, abort_flag, g_merge_status, 0x31000000u | (blockIdx.x & 0xffffffu))) {
        if (threadIdx.x == 0) mbar_wait_landing(bar, 0);  // copies in flight land before the CTA exits
        return;
    }
    if (warp >= nr) return;
    float M = L;
#pragma unroll
    for (int sh = 16; sh; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
    const float myw = (L == -INFINITY) ? 0.f : expf(L - M);  // empty partial: weight 0
    float wsum = myw;
#pragma unroll
    for (int sh = 16; sh; sh >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, sh);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    const uint8_t* mine = smem + warp * kRowBytes + lane * E * esz;
    for (int p = 0; p < P; ++p) {
        const float w = __shfl_sync(0xffffffffu, myw, p);
        if (w != 0.f) {
            float x[E];
            Vec<E, PART_F32>::load(mine + p * rb * kRowBytes, x);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(w, x[e], acc[e]);
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= inv;
    Vec<E, OUT_F32>::store(static_cast<char*>(out) + (rid * D + lane * E) * (OUT_F32 ? 4 : 2), acc);
    if (out_lse && lane == 0) out_lse[lse_idx] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

template <int D, bool PART_F32, bool OUT_F32>
__global__ void __launch_bounds__(kWarps * 32) lse_merge_tiled_kernel(const void* __restrict__ part_O,
                                                                      const float* __restrict__ part_lse,
                                                                      void* __restrict__ out,
                                                                      float* __restrict__ out_lse, int P, int S,
                                                                      int H, long long rows) {
    constexpr int E = D / 32;
    extern __shared__ float wts[];             // [P][32] weights
    __shared__ float red[kWarps][32];
    __shared__ float Ms[32], inv_sum[32];
    grid_dependency_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_stiles = (S + 31) / 32;
    const long long bh = blockIdx.x / n_stiles;  // b*H + h
    const int s0 = (blockIdx.x % n_stiles) * 32;
    const int h = static_cast<int>(bh % H);
    const long long b = bh / H;
    const long long l_stride = rows;
    const long long lse_row = bh * S + s0;       // + lane
    const bool in_range = s0 + lane < S;

    float mloc = -INFINITY;
    for (int pp = warp; pp < P; pp += kWarps) {
        const float L = in_range ? part_lse[pp * l_stride + lse_row + lane] : -INFINITY;
        wts[pp * 32 + lane] = L;
        mloc = fmaxf(mloc, L);
    }
    red[warp][lane] = mloc;
    __syncthreads();
    if (warp == 0) {
        float M = red[0][lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red[w][lane]);
        Ms[lane] = M;
    }
    __syncthreads();
    const float M = Ms[lane];
    float ssum = 0.f;
    for (int pp = warp; pp < P; pp += kWarps) {
        const float L = wts[pp * 32 + lane];
        const float wgt = (L == -INFINITY) ? 0.f : expf(L - M);   // empty partial: weight 0
        wts[pp * 32 + lane] = wgt;
        ssum += wgt;
    }
    red[warp][lane] = ssum;
    __syncthreads();
    if (warp == 0) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t += red[w][lane];
        inv_sum[lane] = t > 0.f ? 1.f / t : 0.f;
        if (out_lse && in_range) out_lse[lse_row + lane] = t > 0.f ? M + logf(t) : -INFINITY;
    }
    __syncthreads();

    // Phase 2: a half-warp per row, lane l of the half owning D/16 consecutive
    // elements (16-byte loads for bf16); a warp merges two rows at a time.
    constexpr int E2 = D / 16;
    constexpr size_t esz = PART_F32 ? 4 : 2;
    const int half = lane >> 4, hl = lane & 15;
    const size_t o_step = static_cast<size_t>(rows) * D * esz;  // bytes between partials
    for (int r = 2 * warp + half; r < 32; r += 2 * kWarps) {
        const int s = s0 + r;
        const bool live = s < S;
        const long long rid = (b * S + (live ? s : s0)) * H + h;
        const char* ptr = static_cast<const char*>(part_O) + (rid * D + hl * E2) * esz;
        float acc[E2];
#pragma unroll
        for (int e = 0; e < E2; ++e) acc[e] = 0.f;
        for (int p0 = 0; p0 < P; p0 += 8) {
            float w[8];
            float x[8][E2];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                w[j] = (live && p0 + j < P) ? wts[(p0 + j) * 32 + r] : 0.f;
                if (w[j] != 0.f) {
                    load_elems<E2, PART_F32>(ptr + j * o_step, x[j]);
                } else {
#pragma unroll
                    for (int e = 0; e < E2; ++e) x[j][e] = 0.f;   // O of an empty partial is not read
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < E2; ++e) acc[e] = fmaf(w[j], x[j][e], acc[e]);
            ptr += 8 * o_step;
        }
        if (live) {
            const float inv = inv_sum[r];
#pragma unroll
            for (int e = 0; e < E2; ++e) acc[e] *= inv;
            store_elems<E2, OUT_F32>(static_cast<char*>(out) + (rid * D + hl * E2) * (OUT_F32 ? 4 : 2), acc);
        }
    }
}

// Head-block variant (H % 8 == 0, P <= 32, many rows): a block owns 8
// consecutive heads x 32 consecutive positions of one batch.  For a fixed
// position the 8 heads' rows of a partial are one contiguous segment (8 * D
// elements, 1 or 2 KB for bf16), so every load instruction of a warp reads 512
// contiguous bytes, where a block of one head reads D-element rows that lie
// H * D elements apart.  Phase 1: warp w reads lse of head h0 + w for the 32
// positions (lane = position, coalesced) for every partial and leaves the
// weights, the normalisers and a mask of the partials that are non-empty
// anywhere in the block in shared memory.  Phase 2: warp w merges positions
// w, w + 8, w + 16, w + 24; lane l holds the 16 bytes at l * 16 + j * 512 of
// the position's segment (j < kLoads), and the non-empty partials are walked
// a group at a time with the group's 16 loads per lane in flight.  A partial empty for a
// whole block (a causal shard after the rows' own) is never read.
constexpr int kHeadBlock = 8;
constexpr int kHeadBlockMaxP = 32;

template <int D, bool PART_F32, bool OUT_F32>
__global__ void __launch_bounds__(kWarps * 32, 2) lse_merge_headblock_kernel(const void* __restrict__ part_O,
                                                                          const float* __restrict__ part_lse,
                                                                          void* __restrict__ out,
                                                                          float* __restrict__ out_lse, int P,
                                                                          int B, int S, int H) {
    constexpr int esz = PART_F32 ? 4 : 2;
    constexpr int kSegBytes = kHeadBlock * D * esz;      // one position's 8-head segment of a partial
    constexpr int kLoads = kSegBytes / 512;              // 16-byte loads per lane per segment
    constexpr int kPer = 16 / esz;                       // elements per 16-byte load
    constexpr int kGroup = 16 / kLoads;                  // partials in flight per step (16 loads per lane)
    static_assert(kSegBytes % 512 == 0, "segment is a whole number of warp loads");
    __shared__ float wts[kHeadBlockMaxP][kHeadBlock][32];  // weight of partial p for (head, position)
    __shared__ float inv_sum[kHeadBlock][32];
    __shared__ unsigned live_mask;
    grid_dependency_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_stiles = (S + 31) / 32;
    const int n_htiles = H / kHeadBlock;
    const int s_tile = blockIdx.x % n_stiles;
    const int rest = blockIdx.x / n_stiles;
    const int h0 = (rest % n_htiles) * kHeadBlock;
    const long long b = rest / n_htiles;
    const int s0 = s_tile * 32;
    const long long rows = static_cast<long long>(B) * S * H;  // rows of one partial
    if (threadIdx.x == 0) live_mask = 0u;
    __syncthreads();

    // phase 1: weights of head h0 + warp at positions s0 + lane
    {
        const int h = h0 + warp;
        const bool in_range = s0 + lane < S;
        const float* lp = part_lse + (b * H + h) * S + s0 + lane;
        float L[kHeadBlockMaxP];
        float M = -INFINITY;
#pragma unroll
        for (int p = 0; p < kHeadBlockMaxP; ++p) {
            L[p] = (p < P && in_range) ? lp[p * rows] : -INFINITY;
            M = fmaxf(M, L[p]);
        }
        float sum = 0.f;
        unsigned mine = 0u;
#pragma unroll
        for (int p = 0; p < kHeadBlockMaxP; ++p) {
            const float wgt = (L[p] == -INFINITY) ? 0.f : expf(L[p] - M);  // empty partial: weight 0
            if (p < P) wts[p][warp][lane] = wgt;
            sum += wgt;
            if (wgt != 0.f) mine |= 1u << p;
        }
        inv_sum[warp][lane] = sum > 0.f ? 1.f / sum : 0.f;
        if (out_lse && in_range) out_lse[(b * H + h) * S + s0 + lane] = sum > 0.f ? M + logf(sum) : -INFINITY;
        mine = __reduce_or_sync(0xffffffffu, mine);
        if (lane == 0) atomicOr(&live_mask, mine);
    }
    __syncthreads();

    // phase 2: the non-empty partials, four at a time, for each of this warp's positions
    const unsigned live = live_mask;
    int hsel[kLoads], dsel[kLoads];  // head (within the block) and first dim of load j
#pragma unroll
    for (int j = 0; j < kLoads; ++j) {
        const int off = (j * 512 + lane * 16) / esz;  // element offset in the segment
        hsel[j] = off / D;
        dsel[j] = off % D;
    }
    const size_t p_stride = static_cast<size_t>(rows) * D * esz;  // bytes between partials
    for (int pos = warp; pos < 32; pos += kWarps) {
        const int s = s0 + pos;
        if (s >= S) break;
        const size_t seg = ((static_cast<size_t>(b) * S + s) * H + h0) * D * esz;
        const char* base = static_cast<const char*>(part_O) + seg + lane * 16;
        float acc[kLoads][kPer];
#pragma unroll
        for (int j = 0; j < kLoads; ++j)
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[j][e] = 0.f;
        unsigned todo = live;
        while (todo) {
            int pp[kGroup];
#pragma unroll
            for (int g = 0; g < kGroup; ++g) {
                pp[g] = todo ? __ffs(todo) - 1 : -1;
                if (todo) todo &= todo - 1;
            }
            // raw 16-byte words in flight (unpacked when accumulated)
            uint4 raw[kGroup][kLoads];
#pragma unroll
            for (int g = 0; g < kGroup; ++g)
#pragma unroll
                for (int j = 0; j < kLoads; ++j)
                    raw[g][j] = pp[g] >= 0 ? *reinterpret_cast<const uint4*>(base + pp[g] * p_stride + j * 512)
                                           : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int g = 0; g < kGroup; ++g) {
                if (pp[g] < 0) continue;
#pragma unroll
                for (int j = 0; j < kLoads; ++j) {
                    // a row of a non-empty partial may itself be empty: weight 0, O dropped
                    const float w = wts[pp[g]][hsel[j]][pos];
                    float x[kPer];
                    load_elems<kPer, PART_F32>(&raw[g][j], x);
#pragma unroll
                    for (int e = 0; e < kPer; ++e) acc[j][e] = w != 0.f ? fmaf(w, x[e], acc[j][e]) : acc[j][e];
                }
            }
        }
        char* dst = static_cast<char*>(out) + ((static_cast<size_t>(b) * S + s) * H + h0) * D * (OUT_F32 ? 4 : 2);
#pragma unroll
        for (int j = 0; j < kLoads; ++j) {
            const float inv = inv_sum[hsel[j]][pos];
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[j][e] *= inv;
            store_elems<kPer, OUT_F32>(dst + (static_cast<size_t>(hsel[j]) * D + dsel[j]) * (OUT_F32 ? 4 : 2),
                                       acc[j]);
        }
    }
}

// Split-partials variant, for few rows with many partials (the fan-out join):
// one block per row; warp w accumulates partials w, w + 8, ... and the eight
// warps' sums are combined in shared memory, so all of a row's partial loads
// are in flight at once.
template <int D, bool PART_F32, bool OUT_F32>
__global__ void __launch_bounds__(kWarps * 32) lse_merge_splitp_kernel(const void* __restrict__ part_O,
                                                                       const float* __restrict__ part_lse,
                                                                       void* __restrict__ out,
                                                                       float* __restrict__ out_lse, int P, int S,
                                                                       int H, long long rows) {
    constexpr int E = D / 32;
    __shared__ float part[kWarps][D];
    grid_dependency_wait();
    const long long rid = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = static_cast<int>(rid % H);
    const long long bs = rid / H;
    const int s = static_cast<int>(bs % S);
    const long long b = bs / S;
    const long long lse_idx = (b * H + h) * S + s;
    const long long l_stride = rows;
    const long long o_stride = rows * D;

    float M = -INFINITY;
    for (int g = 0; g < P; g += 32) {
        const int pp = g + lane;
        M = fmaxf(M, pp < P ? part_lse[pp * l_stride + lse_idx] : -INFINITY);
    }
#pragma unroll
    for (int x = 16; x; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    const size_t esz = PART_F32 ? 4 : 2;
    const char* base = static_cast<const char*>(part_O) + (rid * D + lane * E) * esz;
    if (M != -INFINITY) {
        for (int g = 0; g < P; g += 32) {
            const int pp = g + lane;
            const float L = pp < P ? part_lse[pp * l_stride + lse_idx] : -INFINITY;
            const float myw = (L == -INFINITY) ? 0.f : expf(L - M);   // empty partial: weight 0
            float ws = myw;
#pragma unroll
            for (int x = 16; x; x >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, x);
            wsum += ws;
            // this warp's partials in the group: g + warp, g + warp + 8, g + warp + 16, g + warp + 24
            float w[4];
            float x[4][E];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int q = warp + j * kWarps;
                w[j] = __shfl_sync(0xffffffffu, myw, q);
                if (w[j] != 0.f) {
                    Vec<E, PART_F32>::load(base + static_cast<long long>(g + q) * o_stride * esz, x[j]);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) x[j][e] = 0.f;   // O of an empty partial is not read
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(w[j], x[j][e], acc[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) part[warp][lane * E + e] = acc[e];
    __syncthreads();
    if (warp == 0) {
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        float o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            float t = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kWarps; ++w2) t += part[w2][lane * E + e];
            o[e] = t * inv;
        }
        Vec<E, OUT_F32>::store(static_cast<char*>(out) + (rid * D + lane * E) * (OUT_F32 ? 4 : 2), o);
        if (out_lse && lane == 0) out_lse[lse_idx] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
    }
}

int sm_count_cached() {
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            n = v;
        else
            n = 148;
    }
    return n;
}

// Launch with programmatic stream serialization: the merge may be scheduled
// while the kernel before it on the stream (the attention kernel producing
// the partials) is finishing; grid_dependency_wait() in the merge kernels
// waits for that kernel's completion and memory before any partial is read.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <int D, bool PF, bool OF>
cudaError_t run(const MergeArgs& a, long long rows, cudaStream_t stream) {
    const long long tiled_blocks = static_cast<long long>(a.B) * a.H * ((a.S + 31) / 32);
    const long long n_sm = sm_count_cached();
    if (a.H % kHeadBlock == 0 && a.P <= kHeadBlockMaxP && tiled_blocks / kHeadBlock >= 4 * n_sm) {
        const long long blocks = tiled_blocks / kHeadBlock;
        return launch_pdl(lse_merge_headblock_kernel<D, PF, OF>, static_cast<unsigned>(blocks), kWarps * 32, 0,
                          stream, a.part_O, a.part_lse, a.out, a.out_lse, a.P, a.B, a.S, a.H);
    }
    if (a.P <= kMaxTiledP && tiled_blocks >= 4 * n_sm) {
        const long long blocks = tiled_blocks;
        const size_t smem = static_cast<size_t>(a.P) * 32 * sizeof(float);
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(lse_merge_tiled_kernel<D, PF, OF>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        return launch_pdl(lse_merge_tiled_kernel<D, PF, OF>, static_cast<unsigned>(blocks), kWarps * 32, smem, stream,
                          a.part_O, a.part_lse, a.out, a.out_lse, a.P, a.S, a.H, rows);
    }
    if (a.P <= kBulkMaxP) {
        // rows per CTA: 8, halved while that leaves fewer than two CTAs per SM
        int rb = kWarps;
        while (rb > 1 && (rows + rb - 1) / rb < 2 * n_sm) rb >>= 1;
        const size_t smem = static_cast<size_t>(a.P) * rb * D * (PF ? 4 : 2) + 16;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(lse_merge_bulk_kernel<D, PF, OF>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        const long long blocks = (rows + rb - 1) / rb;
        return launch_pdl(lse_merge_bulk_kernel<D, PF, OF>, static_cast<unsigned>(blocks), kWarps * 32, smem, stream,
                          a.part_O, a.part_lse, a.out, a.out_lse, a.P, a.S, a.H, rows, rb);
    }
    if (a.P >= 8 && rows <= 64 * n_sm * kWarps) {
        return launch_pdl(lse_merge_splitp_kernel<D, PF, OF>, static_cast<unsigned>(rows), kWarps * 32, 0, stream,
                          a.part_O, a.part_lse, a.out, a.out_lse, a.P, a.S, a.H, rows);
    }
    const long long blocks = (rows + kWarps - 1) / kWarps;
    return launch_pdl(lse_merge_kernel<D, PF, OF>, static_cast<unsigned>(blocks), kWarps * 32, 0, stream, a.part_O,
                      a.part_lse, a.out, a.out_lse, a.P, a.S, a.H, rows);
}

}  // namespace

cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.B) * a.S * a.H;
    if (rows == 0) return cudaSuccess;
    const int key = (a.D == 128 ? 4 : 0) | (a.part_f32 ? 2 : 0) | (a.out_f32 ? 1 : 0);
    switch (key) {
        case 0: return run<64, false, false>(a, rows, stream);
        case 1: return run<64, false, true>(a, rows, stream);
        case 2: return run<64, true, false>(a, rows, stream);
        case 3: return run<64, true, true>(a, rows, stream);
        case 4: return run<128, false, false>(a, rows, stream);
        case 5: return run<128, false, true>(a, rows, stream);
        case 6: return run<128, true, false>(a, rows, stream);
        default: return run<128, true, true>(a, rows, stream);
    }
}

unsigned read_clear_status_merge(unsigned* where) {
    unsigned h[2] = {0, 0};
    cudaMemcpyFromSymbol(h, g_merge_status, sizeof h);
    if (h[0]) {
        const unsigned z[2] = {0, 0};
        cudaMemcpyToSymbol(g_merge_status, z, sizeof z);
    }
    if (where) *where = h[1];
    return h[0];
}

}  // namespace ra
