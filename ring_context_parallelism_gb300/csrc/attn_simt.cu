// attn_simt.cu -- exact fp32 blockwise attention on the CUDA cores.
//
// The fp32 inputs are kept in fp32 end to end (no TF32 tensor-core rounding):
// scores and P~V are FFMA, exponentials use expf.  Same walk and the same
// online-softmax state transition as the tensor-core path ("RingAttention and
// Context Parallelism: Mathematical Foundations", sections 2-3, 5): a CTA owns
// 32 query rows of one head inside one shard and streams 32-key chunks of each
// KV block in ring order, staging them in shared memory.  A query row is split
// over D/32 threads (32 head dims each); a score is their partial dot products
// combined with xor shuffles.  Thread `sub` of a row owns head dims
// sub, sub + D/32, sub + 2*D/32, ... so that the threads of a row read
// consecutive shared-memory words.
#include <cmath>

#include "ra_device.cuh"
#include "ra_internal.h"
#include "ra_walk.h"

namespace ra {

static __device__ unsigned g_simt_status[2];

namespace {

constexpr int kRows = 32;   // query rows per CTA
constexpr int kChunk = 32;  // keys staged per step

struct SimtParams {
    const float *q, *k, *v;
    int B, S, Hq, Hkv, n_shards, block, causal, partials, n_qtiles, layout;
    float scale;
    OutDesc out;
};

template <int D>
__global__ void __launch_bounds__(kRows * (D / 32)) attn_simt_kernel(const SimtParams p) {
    constexpr int TPR = D / 32;  // threads per row
    __shared__ __align__(16) float ks[kChunk][D];
    __shared__ __align__(16) float vs[kChunk][D];

    const int tid = threadIdx.x;
    const int r_local = tid / TPR;
    const int sub = tid % TPR;  // which 32 dims
    const int idx = blockIdx.x;
    const int groups = p.B * p.Hq;
    const int qt_rev = idx / groups;
    const int rem = idx % groups;
    const int b = rem / p.Hq;
    const int h = rem % p.Hq;
    const int r0 = p.causal ? heavy_tile_row0(p.layout, p.S, p.n_shards, kRows, qt_rev) : qt_rev * kRows;
    const int row = r0 + r_local;
    const int hk = h / (p.Hq / p.Hkv);
    const int L = p.S / p.n_shards;
    const int row_pos = layout_pos(p.layout, L, p.n_shards, row);  // sequence position (causal mask)

    float q[32], o[32];
    const float* qp = p.q + ((static_cast<long long>(b) * p.S + row) * p.Hq + h) * D + sub;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        q[j] = qp[j * TPR];
        o[j] = 0.f;
    }
    float m = -INFINITY, l = 0.f;

    const OutDesc& out = p.out;
    const long long o_base = static_cast<long long>(b) * out.o_b + static_cast<long long>(row) * out.o_row +
                             static_cast<long long>(h) * out.o_h + sub;
    const long long lse_base = static_cast<long long>(b) * out.lse_b + static_cast<long long>(h) * out.lse_h + row;

    auto write = [&](int part) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float* dst = static_cast<float*>(out.o) + o_base + static_cast<long long>(part) * out.o_part;
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[j * TPR] = o[j] * inv;
        if (sub == 0 && out.lse)
            out.lse[lse_base + static_cast<long long>(part) * out.lse_part] = l > 0.f ? m + logf(l) : -INFINITY;
    };

    const RingWalk w = make_ring_walk(p.S, p.n_shards, kRows, p.causal, r0, kRows, p.layout);
    for (int t = 0; t < w.n_visited; ++t) {
        const int j = ring_shard_at(w, t);
        const int key_lo = j * L;
        // causal: the prefix of the shard the tile's last row can see
        const int key_hi = key_lo + (p.causal ? shard_visible(p.layout, L, p.n_shards, j, w.maxpos) : L);
        for (int blk = key_lo; blk < key_hi; blk += p.block) {
            const int blk_hi = min(blk + p.block, key_hi);
            for (int c0 = blk; c0 < blk_hi; c0 += kChunk) {
                const int n = min(kChunk, blk_hi - c0);
                __syncthreads();
                for (int e = tid; e < kChunk * (D / 4); e += blockDim.x) {
                    const int kr = e / (D / 4);
                    const int kc = (e % (D / 4)) * 4;
                    float4 kv4 = make_float4(0.f, 0.f, 0.f, 0.f), vv4 = kv4;
                    if (kr < n) {
                        const long long off = ((static_cast<long long>(b) * p.S + c0 + kr) * p.Hkv + hk) * D + kc;
                        kv4 = *reinterpret_cast<const float4*>(p.k + off);
                        vv4 = *reinterpret_cast<const float4*>(p.v + off);
                    }
                    *reinterpret_cast<float4*>(&ks[kr][kc]) = kv4;
                    *reinterpret_cast<float4*>(&vs[kr][kc]) = vv4;
                }
                __syncthreads();
                float s[kChunk];
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < kChunk; ++c) {
                    float acc = 0.f;
#pragma unroll
                    for (int d = 0; d < 32; ++d) acc = fmaf(q[d], ks[c][d * TPR + sub], acc);
#pragma unroll
                    for (int x = 1; x < TPR; x <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, x);
                    const bool vis = c < n && (!p.causal || layout_pos(p.layout, L, p.n_shards, c0 + c) <= row_pos);
                    s[c] = vis ? acc * p.scale : -INFINITY;
                    mx = fmaxf(mx, s[c]);
                }
                const float m_new = fmaxf(m, mx);
                if (m_new == -INFINITY) continue;  // nothing visible yet for this row
                const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
                float rs = 0.f;
#pragma unroll
                for (int d = 0; d < 32; ++d) o[d] *= alpha;
#pragma unroll
                for (int c = 0; c < kChunk; ++c) {
                    const float pc = expf(s[c] - m_new);
                    rs += pc;
#pragma unroll
                    for (int d = 0; d < 32; ++d) o[d] = fmaf(pc, vs[c][d * TPR + sub], o[d]);
                }
                l = l * alpha + rs;
                m = m_new;
            }
        }
        if (p.partials) {
            write(j);
            m = -INFINITY;
            l = 0.f;
#pragma unroll
            for (int d = 0; d < 32; ++d) o[d] = 0.f;
        }
    }
    if (!p.partials) {
        write(0);
    } else {
        for (int t = w.n_visited; t < p.n_shards; ++t) write(ring_shard_at(w, t));  // empty: O = 0, lse = -inf
    }
}

// Shared-prefix fan-out in exact fp32 ("AHBM Agentic Runtime Architecture",
// sections 1.3 and 3.2: the stacked query rows of all branches against one
// shared prefix; section 5.2: a branch never sees another branch's private
// KV).  A CTA owns up to 32 stacked (row, query head) pairs of one branch b and
// one KV head: the rows of b times the query heads of the KV head's group.  It
// walks the whole prefix, then b's suffix, with the ring kernel's online
// softmax, and writes O and lse directly (no partials, no merge).  The branch
// offsets live in device memory, so the grid covers every (branch, KV head)
// with as many row tiles as R allows; tiles past a branch's rows exit.
struct SimtFanParams {
    const float *q, *kp, *vp, *ks, *vs;  // q_rows [R,Hq,D]; prefix [Sp,Hkv,D]; suffix [nb,Ss,Hkv,D] (or page pools)
    const int* offsets;
    int R, nb, Sp, Ss, Hq, Hkv, G, tiles, suffix_causal;
    int paged, page_shift, n_pages, n_prefix_pages, n_suffix_pages;
    const int* prefix_pages;
    const int* suffix_pages;
    float scale;
    float* out;  // [R, Hq, D]
    float* lse;  // [Hq, R] (may be null)
};

template <int D>
__global__ void __launch_bounds__(kRows * (D / 32)) attn_simt_fanout_kernel(const SimtFanParams p) {
    constexpr int TPR = D / 32;
    __shared__ __align__(16) float ks[kChunk][D];
    __shared__ __align__(16) float vs[kChunk][D];
    const int tid = threadIdx.x;
    const int r_local = tid / TPR;
    const int sub = tid % TPR;
    const int tile = blockIdx.x % p.tiles;
    const int rest = blockIdx.x / p.tiles;
    const int hk = rest % p.Hkv;
    const int b = rest / p.Hkv;
    const int lo = p.offsets[b], hi = p.offsets[b + 1];
    if (lo < 0 || hi < lo || hi > p.R || (b == 0 && lo != 0) || (b == p.nb - 1 && hi != p.R)) {
        if (tid == 0) {
            atomicCAS(&g_simt_status[0], 0u, kDevInvalidArg);
            atomicCAS(&g_simt_status[1], 0u, 0x0F000000u | static_cast<unsigned>(b));
        }
        return;
    }
    const int n_rows = (hi - lo) * p.G;  // stacked (row, head) pairs of this branch and KV head
    if (tile * kRows >= n_rows) return;
    const int stacked = tile * kRows + r_local;
    const bool active = stacked < n_rows;
    const int row = lo + (active ? stacked / p.G : 0);
    const int h = hk * p.G + (active ? stacked % p.G : 0);
    // prefill: the branch's rows are the last tokens of its suffix, causal inside it
    const int last = p.suffix_causal ? p.Ss - (hi - lo) + (row - lo) : p.Ss - 1;

    float q[32], o[32];
    const float* qp = p.q + (static_cast<long long>(row) * p.Hq + h) * D + sub;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        q[j] = active ? qp[j * TPR] : 0.f;
        o[j] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int page_mask = (1 << p.page_shift) - 1;

    for (int seg = 0; seg < 2; ++seg) {
        const int n_keys = seg == 0 ? p.Sp : p.Ss;
        const float* kb = seg == 0 ? p.kp : p.ks;
        const float* vb = seg == 0 ? p.vp : p.vs;
        const int* table = seg == 0 ? p.prefix_pages : p.suffix_pages + static_cast<long long>(b) * p.n_suffix_pages;
        const int n_listed = seg == 0 ? p.n_prefix_pages : p.n_suffix_pages;
        for (int c0 = 0; c0 < n_keys; c0 += kChunk) {
            const int n = min(kChunk, n_keys - c0);
            __syncthreads();
            for (int e = tid; e < kChunk * (D / 4); e += blockDim.x) {
                const int kr = e / (D / 4);
                const int kc = (e % (D / 4)) * 4;
                float4 kv4 = make_float4(0.f, 0.f, 0.f, 0.f), vv4 = kv4;
                if (kr < n) {
                    const int key = c0 + kr;
                    long long r = -1;  // key's row in its tensor (or page pool)
                    if (p.paged) {
                        const int lp = key >> p.page_shift;
                        const int pg = lp < n_listed ? table[lp] : -1;
                        if (pg >= 0 && pg < p.n_pages) {
                            r = (static_cast<long long>(pg) << p.page_shift) + (key & page_mask);
                        } else {
                            atomicCAS(&g_simt_status[0], 0u, kDevInvalidArg);
                            atomicCAS(&g_simt_status[1], 0u, 0x0E000000u | static_cast<unsigned>(lp & 0xFFFFFF));
                        }
                    } else {
                        r = seg == 0 ? key : static_cast<long long>(b) * p.Ss + key;
                    }
                    if (r >= 0) {
                        const long long off = (r * p.Hkv + hk) * D + kc;
                        kv4 = *reinterpret_cast<const float4*>(kb + off);
                        vv4 = *reinterpret_cast<const float4*>(vb + off);
                    }
                }
                *reinterpret_cast<float4*>(&ks[kr][kc]) = kv4;
                *reinterpret_cast<float4*>(&vs[kr][kc]) = vv4;
            }
            __syncthreads();
            float s[kChunk];
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kChunk; ++c) {
                float acc = 0.f;
#pragma unroll
                for (int d = 0; d < 32; ++d) acc = fmaf(q[d], ks[c][d * TPR + sub], acc);
#pragma unroll
                for (int x = 1; x < TPR; x <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, x);
                const bool vis = c < n && (seg == 0 || c0 + c <= last);
                s[c] = vis ? acc * p.scale : -INFINITY;
                mx = fmaxf(mx, s[c]);
            }
            const float m_new = fmaxf(m, mx);
            if (m_new == -INFINITY) continue;  // nothing visible yet for this row
            const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
            float rs = 0.f;
#pragma unroll
            for (int d = 0; d < 32; ++d) o[d] *= alpha;
#pragma unroll
            for (int c = 0; c < kChunk; ++c) {
                const float pc = expf(s[c] - m_new);
                rs += pc;
#pragma unroll
                for (int d = 0; d < 32; ++d) o[d] = fmaf(pc, vs[c][d * TPR + sub], o[d]);
            }
            l = l * alpha + rs;
            m = m_new;
        }
    }
    if (!active) return;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* dst = p.out + (static_cast<long long>(row) * p.Hq + h) * D + sub;
#pragma unroll
    for (int j = 0; j < 32; ++j) dst[j * TPR] = o[j] * inv;
    if (sub == 0 && p.lse) p.lse[static_cast<long long>(h) * p.R + row] = l > 0.f ? m + logf(l) : -INFINITY;
}

}  // namespace

cudaError_t launch_fanout_simt(const FanoutSimtArgs& a, cudaStream_t stream) {
    if (a.R == 0) return cudaSuccess;
    SimtFanParams p{};
    p.q = a.q_rows;
    p.kp = a.k_prefix;
    p.vp = a.v_prefix;
    p.ks = a.k_suffix;
    p.vs = a.v_suffix;
    p.offsets = a.offsets;
    p.R = a.R;
    p.nb = a.n_branches;
    p.Sp = a.S_prefix;
    p.Ss = a.S_suffix;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.tiles = (a.R * p.G + kRows - 1) / kRows;  // at most every stacked row in one branch
    p.suffix_causal = a.suffix_causal;
    p.paged = a.paged;
    p.page_shift = a.page_shift;
    p.n_pages = a.n_pages;
    p.n_prefix_pages = a.n_prefix_pages;
    p.n_suffix_pages = a.n_suffix_pages;
    p.prefix_pages = a.prefix_pages;
    p.suffix_pages = a.suffix_pages;
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a.D)));
    p.out = a.out;
    p.lse = a.lse;
    const long long grid = static_cast<long long>(a.n_branches) * a.Hkv * p.tiles;
    if (grid > 0x7fffffffll) return cudaErrorInvalidValue;
    if (a.D == 128)
        attn_simt_fanout_kernel<128><<<static_cast<unsigned>(grid), kRows * 4, 0, stream>>>(p);
    else
        attn_simt_fanout_kernel<64><<<static_cast<unsigned>(grid), kRows * 2, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_ring_simt(const RingSimtArgs& a, cudaStream_t stream) {
    SimtParams p;
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.B = a.B;
    p.S = a.S;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.n_shards = a.n_shards;
    p.block = a.block;
    p.causal = a.causal;
    p.partials = a.partials;
    p.layout = a.layout;
    p.n_qtiles = a.S / kRows;
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a.D)));
    p.out = a.out;
    const int grid = p.n_qtiles * a.B * a.Hq;
    if (a.D == 128)
        attn_simt_kernel<128><<<grid, kRows * 4, 0, stream>>>(p);
    else
        attn_simt_kernel<64><<<grid, kRows * 2, 0, stream>>>(p);
    return cudaGetLastError();
}

unsigned read_clear_status_simt(unsigned* where) {
    unsigned h[2] = {0, 0};
    cudaMemcpyFromSymbol(h, g_simt_status, sizeof h);
    if (h[0]) {
        const unsigned z[2] = {0, 0};
        cudaMemcpyToSymbol(g_simt_status, z, sizeof z);
    }
    if (where) *where = h[1];
    return h[0];
}

}  // namespace ra
