// attn_bwd.cu -- backward pass of blockwise ring attention on the sm_103a
// tensor cores: dQ, dK, dV for an upstream gradient dO.
//
// "RingAttention and Context Parallelism: Mathematical Foundations", section 7
// ("RingAttention backward pass logic"): the forward keeps Q and the
// log-sum-exp L = m + ln l of every row; the backward recomputes each block's
// scores from Q and the arriving K, accumulates dQ locally, and carries dK, dV
// with the K/V blocks as they rotate through the ring in reverse order.  With
// P = exp(S - L), dP = dO V^T, Delta = rowsum(dO * O) (= rowsum(P * dP)) and
// dS = P * (dP - Delta):
//
//   dV = P^T dO        dK = dS^T Q / sqrt(d)        dQ = dS K / sqrt(d)
//
// On one GPU the ring becomes two walks:
//   bwd_dq_kernel    one CTA per 128-row query tile of one head; KV tiles in
//                    the forward's ring order (shard k, k-1, ..., causal-empty
//                    shards skipped).  Per tile: S = Q K^T and dP = dO V^T
//                    (tcgen05, smem x smem -> TMEM), P and dS in the softmax
//                    warps (dS written back over S as packed bf16), then
//                    dQ += dS K (TMEM x smem -> TMEM).
//   bwd_dkdv_kernel  one CTA per 128-key tile of one KV head, holding its K
//                    and V tiles; the query tiles of every q head of the GQA
//                    group stream past in reverse ring order (query shard j,
//                    j-1, ..., the causal-empty ones skipped).  Per query tile:
//                    S^T = K Q^T and dP^T = V dO^T, P^T and dS^T in the softmax
//                    warps (thread = key row), then dV += P^T dO and
//                    dK += dS^T Q with P^T, dS^T read from TMEM.
// A preparation kernel computes Delta and L in log2 units first.  Neither walk
// needs atomics: each CTA owns its dQ rows or its dK / dV rows.
//
// Roles (384 threads): warp 0 lane 0 and warp 2 lane 0 stream the two TMA
// rings, warp 1 lane 0 issues the MMAs (and allocates TMEM), warps 4-7 and
// 8-11 handle columns 0-63 and 64-127 of each score tile (thread = TMEM lane =
// row).  Every mbarrier wait is bounded; a wait that runs out records
// RA_ERR_DEVICE_TIMEOUT and the CTA unwinds.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "ra_device.cuh"
#include "ra_internal.h"
#include "ra_walk.h"

namespace ra {

static __device__ unsigned g_bwd_status[2];

namespace {

constexpr int kT = 128;  // query rows and keys per tile
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
    static constexpr int kTileBytes = kT * D * 2;
    // dQ kernel: Q and dO resident; a K tile is held from S = Q K^T until
    // dQ += dS K two tiles later, so the K ring has one stage more than V's
    static constexpr int kDqK = D == 128 ? 3 : 4;
    static constexpr int kDqV = D == 128 ? 2 : 4;
    static constexpr int kDqBarOff = (2 + kDqK + kDqV) * kTileBytes;
    // dK/dV kernel: K and V resident; Q and dO rings, each Q stage with the
    // lse2 and delta of its 128 rows
    static constexpr int kKvS = D == 128 ? 2 : 4;
    static constexpr int kVecOff = (2 + 2 * kKvS) * kTileBytes;
    static constexpr int kInfoOff = kVecOff + kKvS * 1024;  // [kKvS] int2 per Q stage (layout walk)
    static constexpr int kKvBarOff = kInfoOff + 64;
    static constexpr int kNumBars = 24;
    static constexpr int kDqSmem = kDqBarOff + kNumBars * 8 + 16 + 1024;  // + alignment slack
    static constexpr int kKvSmem = kKvBarOff + kNumBars * 8 + 16 + 1024;
    static_assert(kDqSmem <= 232448 && kKvSmem <= 232448, "exceeds the 227 KB of shared memory a CTA may use");
    static_assert(1 + 2 * kDqK + 2 * kDqV + 5 <= kNumBars && 1 + 4 * kKvS + 5 <= kNumBars, "barrier slots");
};

struct BwdParams {
    int B, S, Hq, Hkv, n_shards, causal, G, n_tiles;
    int layout;        // shard layout of the rows (ra_walk.h); the LAY kernels run causal striped
    // causal zigzag in the contiguous kernels: the walk runs over sequence positions
    // (2 zz_n chunks of zz_half tokens as the shards) and every tile's rows are
    // addressed through the chunk map (zz_half = 0: rows are positions)
    int zz_n, zz_half;
    // causal striped in the SP kernels (N = st_n dividing 128): the contiguous walk over
    // positions, 128-position tiles gathered by 5-D boxes, lse2 / Delta in position order,
    // output row of position i at (i mod N) L + i / N
    int st_n;
    float scale_log2;  // log2(e) / sqrt(D)
    float scale;       // 1 / sqrt(D)
    const float* delta;
    const float* lse2;
    void *dq, *dk, *dv;
    int out_f32;
};

// ---------------------------------------------------------------------------
// preparation: Delta = rowsum(dO * O), lse2 = lse * log2(e)
// ---------------------------------------------------------------------------
// E consecutive elements of a row (E = D / 32: one 4-, 8- or 16-byte load per lane).
template <int E>
__device__ __forceinline__ void load_row(const float* src, float* v) {
    if constexpr (E == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
    } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        v[0] = x.x, v[1] = x.y;
    }
}
template <int E>
__device__ __forceinline__ void load_row(const __nv_bfloat16* src, float* v) {
    if constexpr (E == 4) {
        const uint2 x = *reinterpret_cast<const uint2*>(src);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
        v[0] = a.x, v[1] = a.y, v[2] = b.x, v[3] = b.y;
    } else {
        const uint32_t x = *reinterpret_cast<const uint32_t*>(src);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x));
        v[0] = a.x, v[1] = a.y;
    }
}

// One warp per row, rows in memory order ((b, i, h), h fastest: a block reads 8
// consecutive rows of [B, S, Hq, D]); lane l holds head dims [l E, l E + E).
// HBM-bound: reads O and dO once.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const T* out, const T* dout, const float* lse, float* delta,
                                                      float* lse2, long long rows, int S, int Hq, int st_n) {
    constexpr int E = D / 32;
    const long long w = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= rows) return;
    float o[E], g[E];
    load_row<E>(out + w * D + lane * E, o);
    load_row<E>(dout + w * D + lane * E, g);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc = fmaf(o[e], g[e], acc);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, x);
    if (lane == 0) {
        const int h = static_cast<int>(w % Hq);
        const long long bi = w / Hq;
        const int i = static_cast<int>(bi % S);
        const long long bh = (bi / S) * Hq + h;
        // striped rows walked over positions: Delta and lse2 stored at the row's position
        const int ip = st_n ? (i % (S / st_n)) * st_n + i / (S / st_n) : i;
        delta[bh * S + ip] = acc;
        lse2[bh * S + ip] = lse[bh * S + i] * kLog2e;
    }
}

// (a0, a1) *= (b0, b1), one packed fp32x2 multiply.
__device__ __forceinline__ void fmul2(float& a0, float& a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
}

// ---------------------------------------------------------------------------
// MMA issue helpers
// ---------------------------------------------------------------------------
// D = A B^T for two K-major 128 x D tiles in smem (the Q K^T form).
template <int D>
__device__ __forceinline__ void mma_kmajor(uint32_t tD, uint32_t a_lo, uint32_t b_lo) {
    constexpr uint32_t idesc = idesc_bf16_f32(kT, kT, false, false);
    asm volatile("" : "+r"(a_lo), "+r"(b_lo));
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * (16384 >> 4) + (kk & 3) * (32 >> 4);
        mma_ss(tD, sw128_desc(a_lo + off), sw128_desc(b_lo + off), idesc, kk > 0 ? 1u : 0u);
    }
}

// D (+)= A B: A a 128 x 128 bf16 operand packed in TMEM by the softmax warps
// (columns 0-63 of the tile at TMEM columns [0, 32), columns 64-127 at
// [64, 96)), B a 128 x D tile in smem read MN-major (b_lo: LBO 16 KB).
template <int D>
__device__ __forceinline__ void mma_tmem_a(uint32_t tD, uint32_t tA, uint32_t b_lo, bool acc_first) {
    constexpr uint32_t idesc = idesc_bf16_f32(kT, D, false, true);
    asm volatile("" : "+r"(tA), "+r"(b_lo));
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk)
        mma_ts(tD, tA + (kk >> 2) * 64 + (kk & 3) * 8, sw128_desc(b_lo + kk * (2048 >> 4)), idesc,
               (kk > 0 || acc_first) ? 1u : 0u);
}

template <int D>
__device__ __forceinline__ void load_tile(const CUtensorMap* map, uint64_t* bar, uint8_t* dst, int head, int row0,
                                          int b) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) tma_load_4d(map, bar, dst + c * 16384, c * 64, head, row0, b);
}

// The 128 positions [pos0, pos0 + 128) of a striped sequence of n shards (n
// dividing 128): rows pos0/n .. pos0/n + 128/n - 1 of every shard, one 5-D box per
// 64 columns with the shard the faster box dimension, so the rows land in position order.
template <int D>
__device__ __forceinline__ void load_tile_pos(const CUtensorMap* map, uint64_t* bar, uint8_t* dst, int head, int pos0,
                                              int b, int n) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) tma_load_5d(map, bar, dst + c * 16384, c * 64, head, 0, pos0 / n, b);
}

// Storage row of position i in a striped sequence of n shards of len rows.
__device__ __forceinline__ int striped_row(int i, int n, int len) { return (i % n) * len + i / n; }

struct Stage {
    int s = 0, ph = 0;
    __device__ __forceinline__ void next(int n) {
        if (++s == n) {
            s = 0;
            ph ^= 1;
        }
    }
};

// 32 fp32 values (one TMEM load) x `mul`, written to global row memory.
__device__ __forceinline__ void store32(void* base, long long off, const uint32_t* r, float mul, int f32) {
    if (f32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(r[4 * j]) * mul, __uint_as_float(r[4 * j + 1]) * mul,
                                 __uint_as_float(r[4 * j + 2]) * mul, __uint_as_float(r[4 * j + 3]) * mul);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float* f = reinterpret_cast<const float*>(r + 8 * j);
            dst[j] = make_uint4(pack_bf16x2(f[0] * mul, f[1] * mul), pack_bf16x2(f[2] * mul, f[3] * mul),
                                pack_bf16x2(f[4] * mul, f[5] * mul), pack_bf16x2(f[6] * mul, f[7] * mul));
        }
    }
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Lets the copies a producer issued land before its CTA exits (after an abort).
__device__ __forceinline__ void drain_ring(uint64_t* full, int issued, int n_stages) {
    Stage ls;
    for (int n = 0; n < issued; ++n) {
        if (n >= issued - n_stages) mbar_wait_landing(&full[ls.s], ls.ph);
        ls.next(n_stages);
    }
}

// ---------------------------------------------------------------------------
// dQ: query-tile outer, KV tiles in ring order
// ---------------------------------------------------------------------------
template <int D, bool LAY, bool SP>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const BwdParams p) {
    using C = BwdCfg<D>;
    constexpr int NK = C::kDqK, NV = C::kDqV;
    // (batch, KV head) outermost so the resident CTAs share K/V in L2; within
    // it the heaviest query tiles first, the heads of the group fastest
    const int per_kv = p.n_tiles * p.G;
    const int grp = blockIdx.x / per_kv;
    const int rem = blockIdx.x - grp * per_kv;
    const int qt_rev = rem / p.G;
    const int b = grp / p.Hkv, hk = grp - b * p.Hkv;
    const int h = hk * p.G + (rem - qt_rev * p.G);
    const int q0 = !p.causal ? qt_rev * kT
                   : LAY     ? heavy_tile_row0(p.layout, p.S, p.n_shards, kT, qt_rev)
                             : (p.n_tiles - 1 - qt_rev) * kT;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* q_smem = smem;
    uint8_t* do_smem = smem + C::kTileBytes;
    uint8_t* k_smem = smem + 2 * C::kTileBytes;
    uint8_t* v_smem = k_smem + NK * C::kTileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kDqBarOff);
    uint64_t* qd_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + NK;
    uint64_t* v_full = k_empty + NK;
    uint64_t* v_empty = v_full + NV;
    uint64_t* s_full = v_empty + NV;  // [2]: one per S buffer
    uint64_t* dp_full = s_full + 2;
    uint64_t* ds_ready = dp_full + 1;
    uint64_t* dq_done = ds_ready + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    unsigned* status = g_bwd_status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const RingWalk w = make_ring_walk(p.S, p.n_shards, kT, p.causal, q0, kT, LAY ? p.layout : kLayoutContiguous);
    const int total = w.total;
    const int q0s = zigzag_row(p.zz_n, p.zz_half, q0);  // storage row of the query tile

    if (threadIdx.x == 0) {
        mbar_init(qd_full, 1);
        for (int s = 0; s < NK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(dp_full, 1);
        mbar_init(ds_ready, 256);
        mbar_init(dq_done, 1);
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
    // TMEM columns: S buffer 0 [0, 128), dP [128, 256), dQ [256, 256 + D), S buffer 1 [384, 512)

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers
        if (lane == 0) {
            const bool is_k = warp == 0;
            const int ns = is_k ? NK : NV;
            const CUtensorMap* map = is_k ? &tm_k : &tm_v;
            uint64_t* full = is_k ? k_full : v_full;
            uint64_t* empty = is_k ? k_empty : v_empty;
            uint8_t* ring = is_k ? k_smem : v_smem;
            tma_prefetch_desc(map);
            if (is_k) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_do);
                mbar_arrive_expect_tx(qd_full, 2 * C::kTileBytes);
                if (SP) {
                    load_tile_pos<D>(&tm_q, qd_full, q_smem, h, q0, b, p.st_n);
                    load_tile_pos<D>(&tm_do, qd_full, do_smem, h, q0, b, p.st_n);
                } else {
                    load_tile<D>(&tm_q, qd_full, q_smem, h, q0s, b);
                    load_tile<D>(&tm_do, qd_full, do_smem, h, q0s, b);
                }
            }
            RingIterT<LAY> it;
            it.start(w);
            Stage st;
            int issued = 0;
            for (int i = 0; i < total; ++i, it.next()) {
                if (!mbar_wait(&empty[st.s], st.ph ^ 1, abort_flag, status, 0x11000000u | (2 * i + (is_k ? 0 : 1))))
                    break;
                mbar_arrive_expect_tx(&full[st.s], C::kTileBytes);
                if (SP)
                    load_tile_pos<D>(map, &full[st.s], ring + st.s * C::kTileBytes, hk, it.kb, b, p.st_n);
                else
                    load_tile<D>(map, &full[st.s], ring + st.s * C::kTileBytes, hk,
                                 zigzag_row(p.zz_n, p.zz_half, it.kb), b);
                st.next(ns);
                ++issued;
            }
            if (*abort_flag) {
                drain_ring(full, issued, ns);
                if (is_k) mbar_wait_landing(qd_full, 0);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Order: S(0) dP(0) S(1), then per tile i: dQ(i) dP(i+1) S(i+2).  S is
        // double-buffered, so the softmax warps turn S(i+1) into P while
        // dQ(i) and dP(i+1) run, and only the dS step waits for dP.
        if (lane == 0) {
            const uint32_t tSb0 = tmem_base, tSb1 = tmem_base + 384, tdP = tmem_base + 128, tdQ = tmem_base + 256;
            const uint32_t q_lo = sw128_desc_lo(smem_u32(q_smem), 16);
            const uint32_t do_lo = sw128_desc_lo(smem_u32(do_smem), 16);
            const uint32_t k_lo0 = sw128_desc_lo(smem_u32(k_smem), 16);       // K-major: S = Q K^T
            const uint32_t kmn_lo0 = sw128_desc_lo(smem_u32(k_smem), 16384);  // MN-major: dQ += dS K
            const uint32_t v_lo0 = sw128_desc_lo(smem_u32(v_smem), 16);
            constexpr uint32_t kStageLo = C::kTileBytes >> 4;
            bool ok = mbar_wait(qd_full, 0, abort_flag, status, 0x12000000u);
            Stage ck, cv, cq;  // next K tile for S, next V tile for dP, K tile of the next dQ
            auto issue_s = [&](int i) -> bool {
                if (!mbar_wait(&k_full[ck.s], ck.ph, abort_flag, status, 0x14000000u | i)) return false;
                tc_fence_after();
                mma_kmajor<D>((i & 1) ? tSb1 : tSb0, q_lo, k_lo0 + ck.s * kStageLo);
                mma_commit(&s_full[i & 1]);
                ck.next(NK);
                return true;
            };
            auto issue_dp = [&](int i) -> bool {
                if (!mbar_wait(&v_full[cv.s], cv.ph, abort_flag, status, 0x15000000u | i)) return false;
                tc_fence_after();
                mma_kmajor<D>(tdP, do_lo, v_lo0 + cv.s * kStageLo);
                mma_commit(dp_full);
                mma_commit(&v_empty[cv.s]);
                cv.next(NV);
                return true;
            };
            if (ok && total > 0) ok = issue_s(0) && issue_dp(0);
            if (ok && total > 1) ok = issue_s(1);
            for (int i = 0; ok && i < total; ++i) {
                // dS of tile i is in its S buffer: dQ += dS K, then K tile i is free
                if (!(ok = mbar_wait(ds_ready, i & 1, abort_flag, status, 0x13000000u | i))) break;
                tc_fence_after();
                mma_tmem_a<D>(tdQ, (i & 1) ? tSb1 : tSb0, kmn_lo0 + cq.s * kStageLo, i > 0);
                mma_commit(&k_empty[cq.s]);
                cq.next(NK);
                if (i + 1 < total && !(ok = issue_dp(i + 1))) break;
                if (i + 2 < total && !(ok = issue_s(i + 2))) break;
            }
            mma_commit(dq_done);
            mbar_wait(dq_done, 0, abort_flag, status, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax-backward + epilogue
        const int quad = warp & 3;
        const int hw = (warp - 4) >> 2;  // column half of the score tile
        const int lane_row = quad * 32 + lane;
        const int row = q0 + lane_row;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS0 = tmem_base + lane_off, tS1 = tS0 + 384, tdP = tS0 + 128, tdQ = tS0 + 256;
        const int srow = SP ? striped_row(row, p.st_n, p.S / p.st_n) : q0s + lane_row;  // storage row
        // lse2 / Delta: by storage row, or by position in the SP kernels
        const long long vrow = (static_cast<long long>(b) * p.Hq + h) * p.S + (SP ? row : srow);
        const float lse2_r = p.lse2[vrow];
        const float delta_r = p.delta[vrow];
        const float sl2 = p.scale_log2;
        // zigzag / striped: the row's sequence position; the tile's first row has the
        // smallest, so whole tiles of the keys it sees need no mask
        const int shard_len = p.S / p.n_shards;
        const int row_pos = LAY ? layout_pos(p.layout, shard_len, p.n_shards, row) : row;
        const int tile_minpos = LAY ? layout_pos(p.layout, shard_len, p.n_shards, q0) : 0;
        int lay_full = 0;
        RingIterT<LAY> it;
        it.start(w);
        bool ok = true;
        for (int i = 0; i < total; ++i) {
            if (i > 0) it.next();
            const uint32_t tS = (i & 1) ? tS1 : tS0;
            if (!(ok = mbar_wait(&s_full[i & 1], (i >> 1) & 1, abort_flag, status, 0x16000000u | i))) break;
            tc_fence_after();
            int lim = kT - 1;  // visible columns c <= lim
            if (LAY) {
                if (it.in == 0) lay_full = shard_visible(p.layout, shard_len, p.n_shards, it.j, tile_minpos) / kT;
                if (it.in >= lay_full)
                    lim = min(lim, shard_visible(p.layout, shard_len, p.n_shards, it.j, row_pos) -
                                       (it.kb - it.j * shard_len) - 1);
            } else if (p.causal) {
                lim = min(lim, row - it.kb);
            }
            // P = exp(S - L) for this thread's half of the columns
            // both 32-column chunks are loaded before one wait (one TMEM round trip)
            float pr[64];
            uint32_t sv[64];
            tmem_ld32(tS + hw * 64, sv);
            tmem_ld32(tS + hw * 64 + 32, sv + 32);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col0 = hw * 64 + c * 32;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float y0, y1;
                    ffma2(y0, y1, __uint_as_float(sv[c * 32 + 2 * j]), __uint_as_float(sv[c * 32 + 2 * j + 1]), sl2,
                          sl2, -lse2_r, -lse2_r);
                    pr[c * 32 + 2 * j] = ex2_approx(y0);
                    pr[c * 32 + 2 * j + 1] = ex2_approx(y1);
                }
                // masked columns (diagonal / partly visible tiles only) are zeroed
                // after the fact, so full tiles run no compare (values past lim may
                // be inf: they are replaced, never used)
                if (lim < col0 + 31) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j > lim) pr[c * 32 + j] = 0.f;
                }
            }
            // dS = P (dP - Delta), packed bf16 over this half's own S columns
            if (!(ok = mbar_wait(dp_full, i & 1, abort_flag, status, 0x18000000u | i))) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col0 = hw * 64 + c * 32;
                uint32_t dp[32], pk[16];
                tmem_ld32(tdP + col0, dp);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float d0 = __uint_as_float(dp[2 * j]), d1 = __uint_as_float(dp[2 * j + 1]);
                    fadd2(d0, d1, -delta_r, -delta_r);
                    fmul2(d0, d1, pr[c * 32 + 2 * j], pr[c * 32 + 2 * j + 1]);
                    pk[j] = pack_bf16x2(d0, d1);
                }
                tmem_st16(tS + hw * 64 + c * 16, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(ds_ready);
        }
        if (ok && mbar_wait(dq_done, 0, abort_flag, status, 0x17000000u)) {
            tc_fence_after();
            const long long off = ((static_cast<long long>(b) * p.S + srow) * p.Hq + h) * D + hw * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t r[32];
                tmem_ld32(tdQ + hw * (D / 2) + c * 32, r);
                tmem_wait_ld();
                store32(p.dq, off + c * 32, r, p.scale, p.out_f32);
            }
        }
        tc_fence_before();
    }
    // Launched as a programmatic dependent of the dK/dV kernel (it reads none of that
    // kernel's results, so its CTAs may fill SMs the dK/dV tail frees); a CTA does not
    // finish before that grid has, so work after this launch on the stream sees both.
    if (threadIdx.x == 0) grid_dependency_wait();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// dK, dV: KV-tile outer, query tiles of the GQA group in reverse ring order
// ---------------------------------------------------------------------------
// Query tiles that see a KV tile (key rows [k0, k0+128) of shard j): query
// shard j first, then j-1, j-2, ... (mod N); with the causal mask shard j from
// the diagonal tile on, and the shards before j skipped (they see nothing).
// The q heads of the group are the innermost loop.
struct QWalk {
    int N, tps, j, x0, G, causal;
    int a, qt, g;
    __device__ __forceinline__ void start(int n_shards, int tiles_per_shard, int shard, int x_in, int group,
                                          int is_causal) {
        N = n_shards;
        tps = tiles_per_shard;
        j = shard;
        x0 = x_in;
        G = group;
        causal = is_causal;
        a = j;
        qt = causal ? x0 : 0;
        g = 0;
    }
    __device__ __forceinline__ int total() const {
        return G * (causal ? (tps - x0) + (N - 1 - j) * tps : N * tps);
    }
    __device__ __forceinline__ void next() {
        if (++g < G) return;
        g = 0;
        if (++qt < tps) return;
        qt = 0;
        a = (causal && a == j) ? N - 1 : (a == 0 ? N - 1 : a - 1);
    }
    // first query column of the current tile that key row lane_row sees
    __device__ __forceinline__ int col_lo(int lane_row, int) const {
        return (causal && a == j && qt == x0) ? lane_row : 0;
    }
};

// The same walk over causal zigzag or striped shards (ra_walk.h).  Positions
// increase along a shard's rows, so the query rows of shard a that see the KV
// tile are a suffix of the shard: those whose position is at least the tile's
// first key's.  Shards with none are skipped.  Tiles from `full` on see every
// key of the tile; earlier ones mask per key row.
struct QWalkL {
    int N, L, tps, j, G, layout, minpos, maxpos;
    int t, a, qt, g, full;
    __device__ __forceinline__ void enter() {
        qt = shard_visible(layout, L, N, a, minpos - 1) / kT;                // rows before the first seeing row
        full = (shard_visible(layout, L, N, a, maxpos - 1) + kT - 1) / kT;
    }
    __device__ __forceinline__ void skip_empty() {
        while (qt >= tps && t + 1 < N) {
            ++t;
            a = (a == 0) ? N - 1 : a - 1;
            enter();
        }
    }
    __device__ __forceinline__ void start(int n_shards, int shard_len, int shard, int k0, int group, int lay) {
        N = n_shards;
        L = shard_len;
        tps = L / kT;
        j = shard;
        G = group;
        layout = lay;
        minpos = layout_pos(lay, L, N, k0);
        maxpos = layout_pos(lay, L, N, k0 + kT - 1);
        t = 0;
        a = j;
        g = 0;
        enter();
        skip_empty();
    }
    // units of the walk: O(N); computed by one thread
    __device__ int total() const {
        int n = 0;
        for (int tt = 0; tt < N; ++tt) {
            const int aa = (j - tt + N) % N;
            n += tps - min(tps, shard_visible(layout, L, N, aa, minpos - 1) / kT);
        }
        return G * n;
    }
    __device__ __forceinline__ void next() {
        if (++g < G) return;
        g = 0;
        if (++qt < tps) return;
        if (t + 1 < N) {
            ++t;
            a = (a == 0) ? N - 1 : a - 1;
            enter();
            skip_empty();
        }
    }
    // The query shard of a tile that masks per key row, or -1 where the tile sees
    // every key: key row at position kp sees the tile's columns from
    // max(0, shard_visible(.., shard, kp - 1) - qt * kT) on.
    __device__ __forceinline__ int col_lo_shard() const { return qt >= full ? -1 : a; }
};

template <int D, bool LAY, bool SP>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const BwdParams p) {
    using C = BwdCfg<D>;
    constexpr int NS = C::kKvS;
    // (batch, KV head) outermost (its CTAs share the group's Q / dO in L2);
    // within it the key tiles by sequence position, the earliest (seen by the
    // most queries) first
    const int grp = blockIdx.x / p.n_tiles;
    const int x = blockIdx.x - grp * p.n_tiles;
    const int b = grp / p.Hkv, hk = grp - b * p.Hkv;
    const int k0 = LAY ? heavy_tile_row0(p.layout, p.S, p.n_shards, kT, p.n_tiles - 1 - x) : x * kT;
    const int L = p.S / p.n_shards, tps = L / kT;
    const int j = k0 / L, x_in = (k0 - j * L) / kT;
    const int k0s = zigzag_row(p.zz_n, p.zz_half, k0);  // storage row of the key tile

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* k_smem = smem;
    uint8_t* v_smem = smem + C::kTileBytes;
    uint8_t* q_smem = smem + 2 * C::kTileBytes;
    uint8_t* do_smem = q_smem + NS * C::kTileBytes;
    float* vec = reinterpret_cast<float*>(smem + C::kVecOff);  // [NS][lse2 128 | delta 128]
    // LAY: per Q stage (query shard, first row of the tile), or shard -1 where the
    // tile sees every key; written by the Q producer before the stage's arrive
    int2* stage_info = reinterpret_cast<int2*>(smem + C::kInfoOff);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kKvBarOff);
    uint64_t* kv_full = bars;
    uint64_t* q_full = bars + 1;
    uint64_t* q_empty = q_full + NS;
    uint64_t* do_full = q_empty + NS;
    uint64_t* do_empty = do_full + NS;
    uint64_t* s_full = do_empty + NS;
    uint64_t* dp_full = s_full + 1;
    uint64_t* p_ready = dp_full + 1;
    uint64_t* ds_ready = p_ready + 1;
    uint64_t* done = ds_ready + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    unsigned* status = g_bwd_status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    using Walk = typename std::conditional<LAY, QWalkL, QWalk>::type;
    Walk qw;
    if constexpr (LAY)
        qw.start(p.n_shards, L, j, k0, p.G, p.layout);
    else
        qw.start(p.n_shards, tps, j, x_in, p.G, p.causal);
    int* total_smem = reinterpret_cast<int*>(bars + C::kNumBars) + 2;  // after tmem_slot and abort_flag
    if (threadIdx.x == 0) *total_smem = qw.total();

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 1);
            mbar_init(&do_full[s], 1);
            mbar_init(&do_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(dp_full, 1);
        mbar_init(p_ready, 256);
        mbar_init(ds_ready, 256);
        mbar_init(done, 1);
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
    const int total = *total_smem;
    if (threadIdx.x == 0) grid_launch_dependents();  // the dQ kernel may take SMs as this grid drains
    // TMEM columns: S^T [0, 128) (P^T packed over it), dP^T [128, 256) (dS^T
    // packed over it), dV [256, 256 + D), dK [256 + D, 256 + 2D)

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers
        if (lane == 0) {
            const bool is_q = warp == 0;
            const CUtensorMap* map = is_q ? &tm_q : &tm_do;
            uint64_t* full = is_q ? q_full : do_full;
            uint64_t* empty = is_q ? q_empty : do_empty;
            uint8_t* ring = is_q ? q_smem : do_smem;
            tma_prefetch_desc(map);
            if (is_q) {
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
                if (SP) {
                    load_tile_pos<D>(&tm_k, kv_full, k_smem, hk, k0, b, p.st_n);
                    load_tile_pos<D>(&tm_v, kv_full, v_smem, hk, k0, b, p.st_n);
                } else {
                    load_tile<D>(&tm_k, kv_full, k_smem, hk, k0s, b);
                    load_tile<D>(&tm_v, kv_full, v_smem, hk, k0s, b);
                }
            }
            Walk it = qw;
            Stage st;
            int issued = 0;
            for (int u = 0; u < total; ++u, it.next()) {
                if (!mbar_wait(&empty[st.s], st.ph ^ 1, abort_flag, status, 0x21000000u | (2 * u + (is_q ? 0 : 1))))
                    break;
                // first row of the query tile: its storage row, or its position in the SP kernels
                const int q0 = SP ? it.a * L + it.qt * kT : zigzag_row(p.zz_n, p.zz_half, it.a * L + it.qt * kT);
                const int h = hk * p.G + it.g;
                if constexpr (LAY) {
                    if (is_q) stage_info[st.s] = make_int2(it.col_lo_shard(), it.qt * kT);
                }
                mbar_arrive_expect_tx(&full[st.s], C::kTileBytes + (is_q ? 1024 : 0));
                if (SP)
                    load_tile_pos<D>(map, &full[st.s], ring + st.s * C::kTileBytes, h, q0, b, p.st_n);
                else
                    load_tile<D>(map, &full[st.s], ring + st.s * C::kTileBytes, h, q0, b);
                if (is_q) {
                    const long long vrow = (static_cast<long long>(b) * p.Hq + h) * p.S + q0;
                    bulk_load(vec + st.s * 256, p.lse2 + vrow, 512, &full[st.s]);
                    bulk_load(vec + st.s * 256 + 128, p.delta + vrow, 512, &full[st.s]);
                }
                st.next(NS);
                ++issued;
            }
            if (*abort_flag) {
                drain_ring(full, issued, NS);
                if (is_q) mbar_wait_landing(kv_full, 0);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Order: S^T(0) dP^T(0), then per unit u: dV(u) S^T(u+1) dK(u) dP^T(u+1).
        // The softmax warps hand over P^T (for dV) before dS^T (for dK) and keep
        // P in registers, so S^T(u+1) can overwrite P^T(u) once dV(u) is issued.
        if (lane == 0) {
            const uint32_t tS = tmem_base, tdP = tmem_base + 128, tdV = tmem_base + 256, tdK = tmem_base + 256 + D;
            const uint32_t k_lo = sw128_desc_lo(smem_u32(k_smem), 16);
            const uint32_t v_lo = sw128_desc_lo(smem_u32(v_smem), 16);
            const uint32_t q_lo0 = sw128_desc_lo(smem_u32(q_smem), 16);        // K-major: S^T = K Q^T
            const uint32_t qmn_lo0 = sw128_desc_lo(smem_u32(q_smem), 16384);   // MN-major: dK += dS^T Q
            const uint32_t do_lo0 = sw128_desc_lo(smem_u32(do_smem), 16);
            const uint32_t domn_lo0 = sw128_desc_lo(smem_u32(do_smem), 16384);
            constexpr uint32_t kStageLo = C::kTileBytes >> 4;
            bool ok = mbar_wait(kv_full, 0, abort_flag, status, 0x22000000u);
            Stage cs, cd;  // stage of the next S^T (Q ring), of the next dP^T (dO ring)
            auto issue_s = [&](int u) -> bool {
                if (!mbar_wait(&q_full[cs.s], cs.ph, abort_flag, status, 0x23000000u | u)) return false;
                tc_fence_after();
                mma_kmajor<D>(tS, k_lo, q_lo0 + cs.s * kStageLo);
                mma_commit(s_full);
                cs.next(NS);
                return true;
            };
            auto issue_dp = [&](int u) -> bool {
                if (!mbar_wait(&do_full[cd.s], cd.ph, abort_flag, status, 0x24000000u | u)) return false;
                tc_fence_after();
                mma_kmajor<D>(tdP, v_lo, do_lo0 + cd.s * kStageLo);
                mma_commit(dp_full);
                cd.next(NS);
                return true;
            };
            if (ok && total > 0) ok = issue_s(0) && issue_dp(0);
            Stage cu;  // stage of unit u
            for (int u = 0; ok && u < total; ++u) {
                const uint32_t so = cu.s * kStageLo;
                if (!(ok = mbar_wait(p_ready, u & 1, abort_flag, status, 0x25000000u | u))) break;
                tc_fence_after();
                mma_tmem_a<D>(tdV, tS, domn_lo0 + so, u > 0);
                mma_commit(&do_empty[cu.s]);
                if (u + 1 < total && !(ok = issue_s(u + 1))) break;
                if (!(ok = mbar_wait(ds_ready, u & 1, abort_flag, status, 0x29000000u | u))) break;
                tc_fence_after();
                mma_tmem_a<D>(tdK, tdP, qmn_lo0 + so, u > 0);
                mma_commit(&q_empty[cu.s]);
                if (u + 1 < total && !(ok = issue_dp(u + 1))) break;
                cu.next(NS);
            }
            mma_commit(done);
            mbar_wait(done, 0, abort_flag, status, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax-backward + epilogue
        const int quad = warp & 3;
        const int hw = (warp - 4) >> 2;
        const int lane_row = quad * 32 + lane;
        const int key = k0 + lane_row;
        const int key_pos = LAY ? layout_pos(p.layout, L, p.n_shards, key) : key;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem_base + lane_off, tdP = tS + 128, tdV = tS + 256, tdK = tS + 256 + D;
        const float sl2 = p.scale_log2;
        // the layout kernels read the walk's position from the stage (stage_info);
        // only the contiguous walk is stepped here
        Walk it = qw;
        Stage st;
        bool ok = true;
        for (int u = 0; u < total; ++u) {
            if (!(ok = mbar_wait(s_full, u & 1, abort_flag, status, 0x26000000u | u))) break;
            // the stage's lse2 / delta came with its Q tile (already landed: the MMA read it)
            if (!(ok = mbar_wait(&q_full[st.s], st.ph, abort_flag, status, 0x27000000u | u))) break;
            tc_fence_after();
            // key row `key` is visible to the query columns c >= lo of this tile
            int lo;
            if constexpr (LAY) {
                const int2 si = stage_info[st.s];
                lo = si.x < 0 ? 0 : max(0, shard_visible(p.layout, L, p.n_shards, si.x, key_pos - 1) - si.y);
            } else {
                lo = it.col_lo(lane_row, key_pos);
                it.next();
            }
            const float* lse2v = vec + st.s * 256;
            const float* dltv = lse2v + 128;
            // P^T = exp(S^T - L) for this thread's half of the columns, packed over its S^T columns
            // both 32-column chunks are loaded before one wait (one TMEM round trip),
            // the first chunk's lse2 read from shared memory meanwhile
            float pr[64];
            uint32_t sv[64];
            tmem_ld32(tS + hw * 64, sv);
            tmem_ld32(tS + hw * 64 + 32, sv + 32);
            float4 L0[8];
#pragma unroll
            for (int jq = 0; jq < 8; ++jq) L0[jq] = *reinterpret_cast<const float4*>(lse2v + hw * 64 + 4 * jq);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col0 = hw * 64 + c * 32;
                uint32_t pp[16];
#pragma unroll
                for (int jq = 0; jq < 8; ++jq) {
                    const int e = 4 * jq;
                    const float4 L4 = c == 0 ? L0[jq] : *reinterpret_cast<const float4*>(lse2v + col0 + e);
                    float y0, y1, y2, y3;
                    ffma2(y0, y1, __uint_as_float(sv[c * 32 + e]), __uint_as_float(sv[c * 32 + e + 1]), sl2, sl2,
                          -L4.x, -L4.y);
                    ffma2(y2, y3, __uint_as_float(sv[c * 32 + e + 2]), __uint_as_float(sv[c * 32 + e + 3]), sl2, sl2,
                          -L4.z, -L4.w);
                    pr[c * 32 + e] = ex2_approx(y0);
                    pr[c * 32 + e + 1] = ex2_approx(y1);
                    pr[c * 32 + e + 2] = ex2_approx(y2);
                    pr[c * 32 + e + 3] = ex2_approx(y3);
                }
                // masked columns (diagonal / partly visible tiles only) are zeroed
                // after the fact, so full tiles run no compare
                if (lo > col0) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (col0 + e < lo) pr[c * 32 + e] = 0.f;
                }
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) pp[jj] = pack_bf16x2(pr[c * 32 + 2 * jj], pr[c * 32 + 2 * jj + 1]);
                tmem_st16(tS + hw * 64 + c * 16, pp);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(p_ready);
            // dS^T = P^T (dP^T - Delta), packed over this half's own dP^T columns
            if (!(ok = mbar_wait(dp_full, u & 1, abort_flag, status, 0x2A000000u | u))) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col0 = hw * 64 + c * 32;
                uint32_t dp[32], pd[16];
                tmem_ld32(tdP + col0, dp);
                tmem_wait_ld();
#pragma unroll
                for (int jq = 0; jq < 8; ++jq) {
                    const int e = 4 * jq;
                    const float4 D4 = *reinterpret_cast<const float4*>(dltv + col0 + e);
                    float d0 = __uint_as_float(dp[e]), d1 = __uint_as_float(dp[e + 1]);
                    float d2 = __uint_as_float(dp[e + 2]), d3 = __uint_as_float(dp[e + 3]);
                    fadd2(d0, d1, -D4.x, -D4.y);
                    fadd2(d2, d3, -D4.z, -D4.w);
                    fmul2(d0, d1, pr[c * 32 + e], pr[c * 32 + e + 1]);
                    fmul2(d2, d3, pr[c * 32 + e + 2], pr[c * 32 + e + 3]);
                    pd[2 * jq] = pack_bf16x2(d0, d1);
                    pd[2 * jq + 1] = pack_bf16x2(d2, d3);
                }
                tmem_st16(tdP + hw * 64 + c * 16, pd);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(ds_ready);
            st.next(NS);
        }
        if (ok && mbar_wait(done, 0, abort_flag, status, 0x28000000u)) {
            tc_fence_after();
            const int krow = SP ? striped_row(key, p.st_n, L) : k0s + lane_row;  // storage row of the key
            const long long off = ((static_cast<long long>(b) * p.S + krow) * p.Hkv + hk) * D + hw * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t r[32];
                tmem_ld32(tdV + hw * (D / 2) + c * 32, r);
                tmem_wait_ld();
                store32(p.dv, off + c * 32, r, 1.f, p.out_f32);
                tmem_ld32(tdK + hw * (D / 2) + c * 32, r);
                tmem_wait_ld();
                store32(p.dk, off + c * 32, r, p.scale, p.out_f32);
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D, bool LAY, bool SP = false>
cudaError_t launch_tc(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
                      const CUtensorMap& tv, cudaStream_t stream) {
    using C = BwdCfg<D>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = set_smem(bwd_dkdv_kernel<D, LAY, SP>, C::kKvSmem);
        if (attr_err == cudaSuccess) attr_err = set_smem(bwd_dq_kernel<D, LAY, SP>, C::kDqSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    bwd_dkdv_kernel<D, LAY, SP><<<p.B * p.Hkv * p.n_tiles, kThreads, C::kKvSmem, stream>>>(tq, tdo, tk, tv, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B * p.Hq * p.n_tiles);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kDqSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bwd_dq_kernel<D, LAY, SP>, tq, tdo, tk, tv, p);
}

BwdParams make_params(const BwdArgs& a, int out_f32, int tile) {
    BwdParams p{};
    p.B = a.B;
    p.S = a.S;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.n_shards = a.n_shards;
    p.causal = a.causal;
    p.G = a.Hq / a.Hkv;
    p.n_tiles = a.S / tile;
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a.D)));
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.D)));
    p.delta = a.ws_delta;
    p.lse2 = a.ws_lse2;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dv = a.dv;
    p.out_f32 = out_f32;
    p.layout = a.causal ? a.layout : kLayoutContiguous;
    return p;
}

template <typename T>
cudaError_t launch_prep(const BwdArgs& a, cudaStream_t stream, int st_n = 0) {
    const long long rows = static_cast<long long>(a.B) * a.Hq * a.S;
    const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
    const T* o = static_cast<const T*>(a.out);
    const T* d = static_cast<const T*>(a.dout);
    if (a.D == 128)
        bwd_prep_kernel<T, 128><<<grid, 256, 0, stream>>>(o, d, a.lse, a.ws_delta, a.ws_lse2, rows, a.S, a.Hq, st_n);
    else
        bwd_prep_kernel<T, 64><<<grid, 256, 0, stream>>>(o, d, a.lse, a.ws_delta, a.ws_lse2, rows, a.S, a.Hq, st_n);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// exact fp32 path (CUDA-core FMA): the same two walks, 32 rows / keys per CTA
// ---------------------------------------------------------------------------
constexpr int kSimtRows = 32;

// dQ: a CTA owns 32 query rows of one head; thread `sub` of a row owns head
// dims sub, sub + D/32, ... (scores combine over the row's threads by xor
// shuffles).  KV shards in ring order, 32-key chunks staged in shared memory.
template <int D>
__global__ void __launch_bounds__(kSimtRows * (D / 32)) bwd_dq_simt_kernel(const BwdParams p, const float* q,
                                                                           const float* k, const float* v,
                                                                           const float* dout) {
    constexpr int TPR = D / 32;
    __shared__ __align__(16) float ks[kSimtRows][D];
    __shared__ __align__(16) float vs[kSimtRows][D];
    const int tid = threadIdx.x, r_local = tid / TPR, sub = tid % TPR;
    const int groups = p.B * p.Hq;
    const int qt_rev = blockIdx.x / groups, rem = blockIdx.x % groups;
    const int b = rem / p.Hq, h = rem % p.Hq, hk = h / p.G;
    const int r0 = p.causal ? heavy_tile_row0(p.layout, p.S, p.n_shards, kSimtRows, qt_rev) : qt_rev * kSimtRows;
    const int row = r0 + r_local;
    const int L = p.S / p.n_shards;
    const int row_pos = layout_pos(p.layout, L, p.n_shards, row);  // sequence position (causal mask)
    const long long qoff = ((static_cast<long long>(b) * p.S + row) * p.Hq + h) * D + sub;
    float qr[32], dor[32], dq[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        qr[e] = q[qoff + e * TPR];
        dor[e] = dout[qoff + e * TPR];
        dq[e] = 0.f;
    }
    const long long vrow = (static_cast<long long>(b) * p.Hq + h) * p.S + row;
    const float lse2_r = p.lse2[vrow];
    const float delta_r = p.delta[vrow];
    const RingWalk w = make_ring_walk(p.S, p.n_shards, kSimtRows, p.causal, r0, kSimtRows, p.layout);
    for (int t = 0; t < w.n_visited; ++t) {
        const int jsh = ring_shard_at(w, t);
        const int key_lo = jsh * L;
        // causal: the prefix of the shard the tile's last row can see
        const int key_hi = key_lo + (p.causal ? shard_visible(p.layout, L, p.n_shards, jsh, w.maxpos) : L);
        for (int c0 = key_lo; c0 < key_hi; c0 += kSimtRows) {
            __syncthreads();
            for (int e = tid; e < kSimtRows * (D / 4); e += blockDim.x) {
                const int kr = e / (D / 4), kc = (e % (D / 4)) * 4;
                const long long off = ((static_cast<long long>(b) * p.S + c0 + kr) * p.Hkv + hk) * D + kc;
                *reinterpret_cast<float4*>(&ks[kr][kc]) = *reinterpret_cast<const float4*>(k + off);
                *reinterpret_cast<float4*>(&vs[kr][kc]) = *reinterpret_cast<const float4*>(v + off);
            }
            __syncthreads();
#pragma unroll 4
            for (int c = 0; c < kSimtRows; ++c) {
                float s = 0.f, dp = 0.f;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    s = fmaf(qr[e], ks[c][e * TPR + sub], s);
                    dp = fmaf(dor[e], vs[c][e * TPR + sub], dp);
                }
#pragma unroll
                for (int x = 1; x < TPR; x <<= 1) {
                    s += __shfl_xor_sync(0xffffffffu, s, x);
                    dp += __shfl_xor_sync(0xffffffffu, dp, x);
                }
                const bool vis = !p.causal || layout_pos(p.layout, L, p.n_shards, c0 + c) <= row_pos;
                const float pc = vis ? exp2f(s * p.scale_log2 - lse2_r) : 0.f;
                const float ds = pc * (dp - delta_r);
#pragma unroll
                for (int e = 0; e < 32; ++e) dq[e] = fmaf(ds, ks[c][e * TPR + sub], dq[e]);
            }
        }
    }
    float* dst = static_cast<float*>(p.dq) + qoff;
#pragma unroll
    for (int e = 0; e < 32; ++e) dst[e * TPR] = dq[e] * p.scale;
}

// dK, dV: a CTA owns 32 key rows of one KV head; the query rows of every head
// of the group that see them stream past in 32-row chunks, query shards in
// reverse ring order (the key's shard first).
template <int D>
__global__ void __launch_bounds__(kSimtRows * (D / 32)) bwd_dkdv_simt_kernel(const BwdParams p, const float* q,
                                                                             const float* k, const float* v,
                                                                             const float* dout) {
    constexpr int TPR = D / 32;
    __shared__ __align__(16) float qs[kSimtRows][D];
    __shared__ __align__(16) float dos[kSimtRows][D];
    __shared__ float lse_s[kSimtRows], dlt_s[kSimtRows];
    const int tid = threadIdx.x, r_local = tid / TPR, sub = tid % TPR;
    const int groups = p.B * p.Hkv;
    const int x = blockIdx.x / groups, rem = blockIdx.x % groups;
    const int b = rem / p.Hkv, hk = rem % p.Hkv;
    // causal: the chunks by sequence position, the earliest (seen by the most queries) first
    const int k0 = p.causal ? heavy_tile_row0(p.layout, p.S, p.n_shards, kSimtRows, p.n_tiles - 1 - x) : x * kSimtRows;
    const int key = k0 + r_local;
    const int L = p.S / p.n_shards, N = p.n_shards, jsh = k0 / L;
    const int key_pos = layout_pos(p.layout, L, N, key);
    const int minpos = layout_pos(p.layout, L, N, k0);  // the chunk's first (smallest) key position
    const long long koff = ((static_cast<long long>(b) * p.S + key) * p.Hkv + hk) * D + sub;
    float kr[32], vr[32], dk[32], dv[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        kr[e] = k[koff + e * TPR];
        vr[e] = v[koff + e * TPR];
        dk[e] = dv[e] = 0.f;
    }
    for (int t = 0; t < N; ++t) {
        const int a = (jsh - t + N) % N;
        // causal: the rows of shard a whose position is at least the chunk's first key's
        // (a suffix of the shard), from a 32-row boundary
        const int row_lo = a * L + (p.causal ? shard_visible(p.layout, L, N, a, minpos - 1) / kSimtRows * kSimtRows : 0);
        const int row_hi = (a + 1) * L;
        if (row_lo >= row_hi) continue;
        for (int g = 0; g < p.G; ++g) {
            const int h = hk * p.G + g;
            for (int c0 = row_lo; c0 < row_hi; c0 += kSimtRows) {
                __syncthreads();
                for (int e = tid; e < kSimtRows * (D / 4); e += blockDim.x) {
                    const int qr_ = e / (D / 4), qc = (e % (D / 4)) * 4;
                    const long long off = ((static_cast<long long>(b) * p.S + c0 + qr_) * p.Hq + h) * D + qc;
                    *reinterpret_cast<float4*>(&qs[qr_][qc]) = *reinterpret_cast<const float4*>(q + off);
                    *reinterpret_cast<float4*>(&dos[qr_][qc]) = *reinterpret_cast<const float4*>(dout + off);
                }
                if (tid < kSimtRows) {
                    const long long vrow = (static_cast<long long>(b) * p.Hq + h) * p.S + c0 + tid;
                    lse_s[tid] = p.lse2[vrow];
                    dlt_s[tid] = p.delta[vrow];
                }
                __syncthreads();
#pragma unroll 4
                for (int c = 0; c < kSimtRows; ++c) {
                    float s = 0.f, dp = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        s = fmaf(kr[e], qs[c][e * TPR + sub], s);
                        dp = fmaf(vr[e], dos[c][e * TPR + sub], dp);
                    }
#pragma unroll
                    for (int xx = 1; xx < TPR; xx <<= 1) {
                        s += __shfl_xor_sync(0xffffffffu, s, xx);
                        dp += __shfl_xor_sync(0xffffffffu, dp, xx);
                    }
                    const bool vis = !p.causal || layout_pos(p.layout, L, N, c0 + c) >= key_pos;
                    const float pc = vis ? exp2f(s * p.scale_log2 - lse_s[c]) : 0.f;
                    const float dsc = pc * (dp - dlt_s[c]);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        dv[e] = fmaf(pc, dos[c][e * TPR + sub], dv[e]);
                        dk[e] = fmaf(dsc, qs[c][e * TPR + sub], dk[e]);
                    }
                }
            }
        }
    }
    float* dkp = static_cast<float*>(p.dk) + koff;
    float* dvp = static_cast<float*>(p.dv) + koff;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        dkp[e * TPR] = dk[e] * p.scale;
        dvp[e * TPR] = dv[e];
    }
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdArgs& a, cudaStream_t stream) {
    // causal striped with N dividing 128: the contiguous kernels over positions
    const int st_n = (a.causal && a.layout == kLayoutStriped && 128 % a.n_shards == 0) ? a.n_shards : 0;
    cudaError_t e = launch_prep<__nv_bfloat16>(a, stream, st_n);
    if (e != cudaSuccess) return e;
    BwdParams p = make_params(a, 0, kT);
    const unsigned long long D = a.D, esz = 2;
    const unsigned long long qd[4] = {D, (unsigned long long)a.Hq, (unsigned long long)a.S, (unsigned long long)a.B};
    const unsigned long long qs[3] = {D * esz, D * esz * a.Hq, D * esz * a.Hq * a.S};
    const unsigned long long kd[4] = {D, (unsigned long long)a.Hkv, (unsigned long long)a.S, (unsigned long long)a.B};
    const unsigned long long ks[3] = {D * esz, D * esz * a.Hkv, D * esz * a.Hkv * a.S};
    const unsigned box[4] = {64, 1, 128, 1};
    CUtensorMap tq, tdo, tk, tv;
    if (!make_map(&tq, a.q, qd, qs, box) || !make_map(&tdo, a.dout, qd, qs, box) || !make_map(&tk, a.k, kd, ks, box) ||
        !make_map(&tv, a.v, kd, ks, box))
        return cudaErrorInvalidValue;
    // A causal zigzag sequence is the contiguous causal problem on the 2N chunks of
    // its cut, each 128-row tile addressed through the chunk map: the contiguous
    // kernels walk the same tiles (in the ring over the 2N chunks; order changes
    // rounding only).
    if (a.causal && a.layout == kLayoutZigzag) {
        p.layout = kLayoutContiguous;
        p.n_shards = 2 * a.n_shards;
        p.zz_n = a.n_shards;
        p.zz_half = a.S / (2 * a.n_shards);
    }
    if (st_n) {
        // a tile of 128 consecutive positions holds 128/N rows of every shard: one 5-D box
        // [64 cols, 1 head, N shards, 128/N rows, 1 batch] per 64 columns lands it in position
        // order, and the contiguous kernels walk positions (N position-order shards)
        p.layout = kLayoutContiguous;
        p.st_n = st_n;
        const unsigned long long L = a.S / a.n_shards, N = a.n_shards, S = a.S, B = a.B;
        const unsigned long long qd5[5] = {D, (unsigned long long)a.Hq, N, L, B};
        const unsigned long long qs5[4] = {D * esz, L * a.Hq * D * esz, a.Hq * D * esz, S * a.Hq * D * esz};
        const unsigned long long kd5[5] = {D, (unsigned long long)a.Hkv, N, L, B};
        const unsigned long long ks5[4] = {D * esz, L * a.Hkv * D * esz, a.Hkv * D * esz, S * a.Hkv * D * esz};
        const unsigned box5[5] = {64, 1, (unsigned)N, (unsigned)(128 / N), 1};
        CUtensorMap tq5, tdo5, tk5, tv5;
        if (!make_map_5d(&tq5, a.q, qd5, qs5, box5) || !make_map_5d(&tdo5, a.dout, qd5, qs5, box5) ||
            !make_map_5d(&tk5, a.k, kd5, ks5, box5) || !make_map_5d(&tv5, a.v, kd5, ks5, box5))
            return cudaErrorInvalidValue;
        return a.D == 128 ? launch_tc<128, false, true>(p, tq5, tdo5, tk5, tv5, stream)
                          : launch_tc<64, false, true>(p, tq5, tdo5, tk5, tv5, stream);
    }
    // without a causal mask every layout is the same walk
    if (a.causal && p.layout != kLayoutContiguous)
        return a.D == 128 ? launch_tc<128, true>(p, tq, tdo, tk, tv, stream)
                          : launch_tc<64, true>(p, tq, tdo, tk, tv, stream);
    return a.D == 128 ? launch_tc<128, false>(p, tq, tdo, tk, tv, stream)
                      : launch_tc<64, false>(p, tq, tdo, tk, tv, stream);
}

cudaError_t launch_bwd_simt(const BwdArgs& a, cudaStream_t stream) {
    cudaError_t e = launch_prep<float>(a, stream);
    if (e != cudaSuccess) return e;
    const BwdParams p = make_params(a, 1, kSimtRows);
    const float* q = static_cast<const float*>(a.q);
    const float* k = static_cast<const float*>(a.k);
    const float* v = static_cast<const float*>(a.v);
    const float* d = static_cast<const float*>(a.dout);
    const unsigned gkv = static_cast<unsigned>(a.B * a.Hkv * p.n_tiles), gq = static_cast<unsigned>(a.B * a.Hq * p.n_tiles);
    if (a.D == 128) {
        bwd_dkdv_simt_kernel<128><<<gkv, kSimtRows * 4, 0, stream>>>(p, q, k, v, d);
        bwd_dq_simt_kernel<128><<<gq, kSimtRows * 4, 0, stream>>>(p, q, k, v, d);
    } else {
        bwd_dkdv_simt_kernel<64><<<gkv, kSimtRows * 2, 0, stream>>>(p, q, k, v, d);
        bwd_dq_simt_kernel<64><<<gq, kSimtRows * 2, 0, stream>>>(p, q, k, v, d);
    }
    return cudaGetLastError();
}

unsigned read_clear_status_bwd(unsigned* where) {
    unsigned h[2] = {0, 0};
    cudaMemcpyFromSymbol(h, g_bwd_status, sizeof h);
    if (h[0]) {
        const unsigned z[2] = {0, 0};
        cudaMemcpyToSymbol(g_bwd_status, z, sizeof z);
    }
    if (where) *where = h[1];
    return h[0];
}

}  // namespace ra
