// ra_internal.h -- launch interfaces between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

namespace ra {

// Where a kernel writes its per-row results.  Element offsets:
//   O   : part*o_part + b*o_b + row*o_row + head*o_h + d
//   lse : part*lse_part + b*lse_b + head*lse_h + row
struct OutDesc {
    void* o = nullptr;
    float* lse = nullptr;
    long long o_b = 0, o_row = 0, o_h = 0, o_part = 0;
    long long lse_b = 0, lse_h = 0, lse_part = 0;
    int o_f32 = 0;  // 1: fp32 O, 0: bf16 O
};

// Ring-order prefill on the tensor cores (bf16).  partials=1 flushes one
// normalised partial per KV shard.
struct RingTcArgs {
    const void *q, *k, *v;
    int B, S, Hq, Hkv, D, n_shards, causal, partials;
    OutDesc out;
    int layout = 0;  // shard layout of the rows (ra_walk.h kLayout*)
};
cudaError_t launch_ring_tc(const RingTcArgs& a, cudaStream_t stream);

// Shared-prefix fan-out on the tensor cores (bf16): prefix chunks + per-branch
// suffix, each writing an fp32 partial into the workspace.
struct FanoutTcArgs {
    const void* q_rows;
    const int* offsets;
    int n_branches, R;
    const void *k_prefix, *v_prefix;
    int S_prefix;
    const void *k_suffix, *v_suffix;
    int S_suffix;
    int Hq, Hkv, D;
    int n_chunks;               // prefix split
    int chunk_start[65];        // prefix tile where chunk c starts (n_chunks + 1 entries)
    OutDesc part;               // fp32 partials [P][R][Hq][D], lse [P][Hq][R]
    int suffix_causal = 0;      // prefill: causal inside each branch's suffix
    // paged KV (k_prefix / v_prefix then point at the page pools [n_pages, page_size, Hkv, D])
    int paged = 0, page_shift = 0, n_pages = 0, n_prefix_pages = 0, n_suffix_pages = 0;
    const int* prefix_pages = nullptr;
    const int* suffix_pages = nullptr;
};
cudaError_t launch_fanout_tc(const FanoutTcArgs& a, cudaStream_t stream);

// Partial slots of a fan-out call: one per prefix chunk (each branch's suffix
// is folded into the chunk b % n_chunks), or one for the suffix units when
// there is no prefix.  *split_prefix: the stacked rows fit one row tile, so
// each prefix unit splits its KV tiles over its two softmax slots and combines
// them before writing.  Returns the slot count P.
int fanout_slots(int R, int Hq, int Hkv, int n_chunks, int S_prefix, int S_suffix, int* split_prefix,
                 int* suffix_slot0);

// Prefix split of a fan-out call (fanout_plan.cu): the chunk count (at most
// 64) and the n_chunks + 1 prefix-tile boundaries, from a simulation of the
// block scheduler; cached per shape.  `paged`: the KV comes from a page pool
// (rows in one row tile then still spread over every SM).
void fanout_plan(int R, int S_prefix, int S_suffix, int n_branches, int Hq, int Hkv, int n_sm, int* n_chunks,
                 int* chunk_start, bool paged = false);

// Equal-work boundaries for a given chunk count (the no-alloc entry point's
// fallback when the planned partials do not fit its scratch).
void fanout_split_equal(int n_chunks, int R, int S_prefix, int S_suffix, int n_branches, int Hq, int Hkv,
                        int* chunk_start);

// Exact fp32 path (CUDA-core FMA).
struct RingSimtArgs {
    const float *q, *k, *v;
    int B, S, Hq, Hkv, D, n_shards, block, causal, partials;
    OutDesc out;
    int layout = 0;
};
cudaError_t launch_ring_simt(const RingSimtArgs& a, cudaStream_t stream);

// Shared-prefix fan-out in exact fp32 on the CUDA cores: O [R, Hq, D] and lse
// [Hq, R] written directly (no partials, no workspace).
struct FanoutSimtArgs {
    const float* q_rows;
    const int* offsets;
    int n_branches, R;
    const float *k_prefix, *v_prefix;
    int S_prefix;
    const float *k_suffix, *v_suffix;
    int S_suffix;
    int Hq, Hkv, D;
    float* out;
    float* lse;
    int suffix_causal = 0;
    int paged = 0, page_shift = 0, n_pages = 0, n_prefix_pages = 0, n_suffix_pages = 0;
    const int* prefix_pages = nullptr;
    const int* suffix_pages = nullptr;
};
cudaError_t launch_fanout_simt(const FanoutSimtArgs& a, cudaStream_t stream);

// Row-indexed LSE merge.  part_f32 / out_f32 select fp32 or bf16 storage.
struct MergeArgs {
    const void* part_O;
    const float* part_lse;
    void* out;
    float* out_lse;
    int P, B, S, H, D;
    int part_f32, out_f32;
};
cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t stream);

// 4-D bf16 tensor map (dims innermost first, byte strides of dims 1..3, box
// (64, b1, b2, b3), 128-byte swizzle) for the TMA loads of the tensor-core
// kernels.  Returns false if the driver entry point or the encode fails.
bool make_map(CUtensorMap* m, const void* base, const unsigned long long dims[4], const unsigned long long strides[3],
              const unsigned box[4]);
// The same for 5 dims (strides for dims 1..4, box of 5).
bool make_map_5d(CUtensorMap* m, const void* base, const unsigned long long dims[5],
                 const unsigned long long strides[4], const unsigned box[5]);

// Backward pass (dQ, dK, dV) for an upstream gradient dO.  ws_delta / ws_lse2:
// workspace [B, Hq, S] fp32 each (rowsum(dO * O), lse * log2 e).
struct BwdArgs {
    const void *q, *k, *v, *out, *dout;
    const float* lse;
    void *dq, *dk, *dv;
    float *ws_delta, *ws_lse2;
    int B, S, Hq, Hkv, D, n_shards, causal;
    int layout = 0;  // shard layout of the rows (ra_walk.h kLayout*)
};
cudaError_t launch_bwd_tc(const BwdArgs& a, cudaStream_t stream);    // bf16
cudaError_t launch_bwd_simt(const BwdArgs& a, cudaStream_t stream);  // fp32

// Status words of each translation unit: read (after the caller synchronised)
// and clear.  Returns the first non-zero code, 0 if none.
unsigned read_clear_status_tc(unsigned* where);
unsigned read_clear_status_simt(unsigned* where);
unsigned read_clear_status_merge(unsigned* where);
unsigned read_clear_status_bwd(unsigned* where);
unsigned read_clear_status_selftest(unsigned* where);

// Failure-detection health check: a bounded wait that is never satisfied.
cudaError_t launch_selftest_wait_timeout(unsigned long long limit_ns, cudaStream_t stream);

}  // namespace ra
