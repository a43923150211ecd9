// ra_api.cu -- the C ABI declared in include/ra.h: host-side validation,
// output layout descriptors, dispatch to the kernels, device status.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/ra.h"
#include "ra_internal.h"
#include "ra_walk.h"

namespace {

thread_local char g_err[256] = "";

ra_status fail(ra_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

ra_status ok() {
    g_err[0] = '\0';
    return RA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ra_status cuda_fail(cudaError_t e, const char* what) {
    return fail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

// Checks shared by the fused and partial ring entry points.
ra_status check_ring(const void* q, const void* k, const void* v, const void* out, int B, int S, int Hq, int Hkv,
                     int D, int n_shards, int block, int causal, ra_dtype dt, int layout) {
    if (!q || !k || !v || !out) return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(RA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1) return fail(RA_ERR_INVALID_ARG, "B, S, Hq, Hkv must be >= 1");
    if (Hq % Hkv) return fail(RA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
    if (D != 64 && D != 128) return fail(RA_ERR_INVALID_ARG, "D must be 64 or 128 (got %d)", D);
    if (n_shards < 1 || S % n_shards) return fail(RA_ERR_INVALID_ARG, "S (%d) %% n_shards (%d) != 0", S, n_shards);
    const int L = S / n_shards;
    if (block < 1 || L % block) return fail(RA_ERR_INVALID_ARG, "shard length %d %% block %d != 0", L, block);
    if (causal != 0 && causal != 1) return fail(RA_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG && layout != RA_LAYOUT_STRIPED)
        return fail(RA_ERR_INVALID_ARG, "unknown layout %d", layout);
    if (layout == RA_LAYOUT_ZIGZAG && L % 2)
        return fail(RA_ERR_INVALID_ARG, "zigzag layout needs an even shard length (got %d)", L);
    const int tile = dt == RA_BF16 ? 128 : 32;  // query rows / keys per tile of the kernels
    if (layout == RA_LAYOUT_ZIGZAG && (L / 2) % tile)
        return fail(RA_ERR_UNSUPPORTED, "zigzag layout needs (shard length / 2) %% %d == 0 (got %d)", tile, L / 2);
    if (dt == RA_BF16) {
        if (L % 128) return fail(RA_ERR_UNSUPPORTED, "bf16 path needs shard length %% 128 == 0 (got %d)", L);
        if (block != 64 && block % 128)
            return fail(RA_ERR_UNSUPPORTED, "bf16 path walks 128-key tiles: block must be 64 or a multiple of 128");
    } else if (dt == RA_F32) {
        if (L % 32) return fail(RA_ERR_UNSUPPORTED, "fp32 path needs shard length %% 32 == 0 (got %d)", L);
    } else {
        return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dt));
    }
    const long long elems = static_cast<long long>(B) * S * Hq * D;
    if (elems > (1ll << 40)) return fail(RA_ERR_INVALID_ARG, "tensor too large");
    return RA_OK;
}

ra_status ring_common(const void* q, const void* k, const void* v, void* out, float* lse, int B, int S, int Hq,
                      int Hkv, int D, int n_shards, int block, int causal, ra_dtype dt, void* stream, int partials,
                      int layout) {
    ra_status st = check_ring(q, k, v, out, B, S, Hq, Hkv, D, n_shards, block, causal, dt, layout);
    if (st != RA_OK) return st;
    if (lse && !aligned16(lse)) return fail(RA_ERR_INVALID_ARG, "lse must be 16-byte aligned");
    ra::OutDesc od;
    od.o = out;
    od.lse = lse;
    od.o_row = static_cast<long long>(Hq) * D;
    od.o_h = D;
    od.o_b = static_cast<long long>(S) * Hq * D;
    od.o_part = static_cast<long long>(B) * S * Hq * D;
    od.lse_h = S;
    od.lse_b = static_cast<long long>(Hq) * S;
    od.lse_part = static_cast<long long>(B) * Hq * S;
    od.o_f32 = (dt == RA_F32);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dt == RA_BF16) {
        ra::RingTcArgs a{q, k, v, B, S, Hq, Hkv, D, n_shards, causal, partials, od};
        a.layout = layout;
        e = ra::launch_ring_tc(a, s);
    } else {
        ra::RingSimtArgs a{static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
                           B, S, Hq, Hkv, D, n_shards, block, causal, partials, od};
        a.layout = layout;
        e = ra::launch_ring_simt(a, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, partials ? "ring partials launch" : "ring attention launch");
    return ok();
}

struct FanoutPlan {
    int n_chunks, P;
    int chunk_start[65];
    size_t part_o_bytes, part_lse_bytes, total;
};

// Slots and workspace bytes of a plan whose chunk count and boundaries are set.
FanoutPlan finish_plan(FanoutPlan f, int R, int S_prefix, int S_suffix, int Hq, int Hkv, int D) {
    f.P = ra::fanout_slots(R, Hq, Hkv, f.n_chunks, S_prefix, S_suffix, nullptr, nullptr);
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    f.part_o_bytes = up(static_cast<size_t>(f.P) * R * Hq * D * sizeof(float));
    f.part_lse_bytes = up(static_cast<size_t>(f.P) * Hq * R * sizeof(float));
    f.total = f.part_o_bytes + f.part_lse_bytes;
    return f;
}

// A plan with a given prefix chunk count and equal-work chunks.
FanoutPlan plan_with_chunks(int n_chunks, int R, int n_branches, int S_prefix, int S_suffix, int Hq, int Hkv,
                            int D) {
    FanoutPlan f{};
    f.n_chunks = S_prefix > 0 ? n_chunks : 0;
    if (f.n_chunks > 0) ra::fanout_split_equal(f.n_chunks, R, S_prefix, S_suffix, n_branches, Hq, Hkv, f.chunk_start);
    return finish_plan(f, R, S_prefix, S_suffix, Hq, Hkv, D);
}

// The planned split (chunk count and boundaries from the scheduler simulation).
FanoutPlan plan_fanout(int R, int n_branches, int S_prefix, int S_suffix, int Hq, int Hkv, int D,
                       bool paged = false) {
    FanoutPlan f{};
    f.n_chunks = 0;
    if (S_prefix > 0)
        ra::fanout_plan(R, S_prefix, S_suffix, n_branches, Hq, Hkv, sm_count(), &f.n_chunks, f.chunk_start, paged);
    return finish_plan(f, R, S_prefix, S_suffix, Hq, Hkv, D);
}

ra_status check_fanout(const void* q_rows, const int* offsets, int n_branches, int R, const void* k_prefix,
                       const void* v_prefix, int S_prefix, const void* k_suffix, const void* v_suffix, int S_suffix,
                       const void* out, int Hq, int Hkv, int D, ra_dtype dt) {
    if (dt != RA_BF16 && dt != RA_F32) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dt));
    if (R < 0 || n_branches < 1 || S_prefix < 0 || S_suffix < 0)
        return fail(RA_ERR_INVALID_ARG, "R >= 0, n_branches >= 1, S_prefix >= 0, S_suffix >= 0 required");
    if (Hq < 1 || Hkv < 1 || Hq % Hkv) return fail(RA_ERR_INVALID_ARG, "Hq must be a positive multiple of Hkv");
    if (128 % (Hq / Hkv)) return fail(RA_ERR_UNSUPPORTED, "128 %% (Hq / Hkv) != 0");
    if (D != 64 && D != 128) return fail(RA_ERR_INVALID_ARG, "D must be 64 or 128 (got %d)", D);
    if (S_prefix + S_suffix < 1) return fail(RA_ERR_INVALID_ARG, "no keys: S_prefix + S_suffix must be >= 1");
    if (R > 0 && (!q_rows || !out || !offsets)) return fail(RA_ERR_INVALID_ARG, "null pointer");
    if (S_prefix > 0 && (!k_prefix || !v_prefix)) return fail(RA_ERR_INVALID_ARG, "null prefix pointer");
    if (S_suffix > 0 && (!k_suffix || !v_suffix)) return fail(RA_ERR_INVALID_ARG, "null suffix pointer");
    const void* ptrs[6] = {q_rows, k_prefix, v_prefix, k_suffix, v_suffix, out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(RA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    if (offsets && (reinterpret_cast<uintptr_t>(offsets) & 3u)) return fail(RA_ERR_INVALID_ARG, "offsets misaligned");
    return RA_OK;
}

}  // namespace

// Scratch of ra_prefix_fanout_attn_noalloc: the fan-out partials of callers
// that cannot allocate a workspace.  Shared by every such call on a device.
static __device__ __align__(256) unsigned char g_fanout_scratch[RA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
    unsigned long long ctx_id;  // context the address belongs to (0: not looked up)
    void* addr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

// Unique id of the calling thread's current context (0 if it cannot be read).
// A device reset gives the device a new primary context, where the module and
// its scratch array are loaded again, possibly at another address.
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_fanout_scratch on the current device (host code only
// sees a stand-in for the array's name).  Looked up once per device and
// context: again after a device reset has replaced the context.
ra_status scratch_address(void** addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(RA_ERR_UNSUPPORTED, "device index %d out of range", dev);
    const unsigned long long ctx = current_context_id();  // 0 before the device's first runtime call
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr& c = g_scratch_addr[dev];
    if (!c.addr || ctx == 0 || c.ctx_id != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fanout_scratch);  // sets up the device's context if needed
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(fan-out scratch)");
        c.addr = p;
        c.ctx_id = current_context_id();
    }
    *addr = c.addr;
    return RA_OK;
}

// The usual plan if its partials fit in the scratch array, else the largest
// chunk count that does; total == 0 if none fits.
FanoutPlan plan_fanout_bounded(int R, int n_branches, int S_prefix, int S_suffix, int Hq, int Hkv, int D,
                               size_t cap) {
    FanoutPlan f = plan_fanout(R, n_branches, S_prefix, S_suffix, Hq, Hkv, D);
    if (f.total <= cap) return f;
    for (int c = f.n_chunks - 1; c >= 1; --c) {
        FanoutPlan g = plan_with_chunks(c, R, n_branches, S_prefix, S_suffix, Hq, Hkv, D);
        if (g.total <= cap) return g;
    }
    FanoutPlan none{};
    return none;
}

}  // namespace

extern "C" {

ra_status ra_blockwise_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int S,
                                int Hq, int Hkv, int D, int n_shards, int block, int causal, ra_dtype dt,
                                void* stream) {
    return ring_common(q, k, v, out, lse, B, S, Hq, Hkv, D, n_shards, block, causal, dt, stream, 0,
                       RA_LAYOUT_CONTIGUOUS);
}

ra_status ra_blockwise_attn_fwd_layout(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                                       int S, int Hq, int Hkv, int D, int n_shards, int block, int causal,
                                       int layout, ra_dtype dt, void* stream) {
    return ring_common(q, k, v, out, lse, B, S, Hq, Hkv, D, n_shards, block, causal, dt, stream, 0, layout);
}

ra_status ra_ring_partials_fwd(const void* q, const void* k, const void* v, void* partials_O, float* partials_lse,
                               int B, int S, int Hq, int Hkv, int D, int n_shards, int block, int causal,
                               ra_dtype dt, void* stream) {
    if (!partials_lse) return fail(RA_ERR_INVALID_ARG, "partials_lse must not be NULL");
    return ring_common(q, k, v, partials_O, partials_lse, B, S, Hq, Hkv, D, n_shards, block, causal, dt, stream, 1,
                       RA_LAYOUT_CONTIGUOUS);
}

ra_status ra_ring_partials_fwd_layout(const void* q, const void* k, const void* v, void* partials_O,
                                      float* partials_lse, int B, int S, int Hq, int Hkv, int D, int n_shards,
                                      int block, int causal, int layout, ra_dtype dt, void* stream) {
    if (!partials_lse) return fail(RA_ERR_INVALID_ARG, "partials_lse must not be NULL");
    return ring_common(q, k, v, partials_O, partials_lse, B, S, Hq, Hkv, D, n_shards, block, causal, dt, stream, 1,
                       layout);
}

ra_status ra_lse_merge(const void* partials_O, const float* partials_lse, void* out, float* out_lse, int P, int B,
                       int S, int H, int D, ra_dtype dt, void* stream) {
    if (!partials_O || !partials_lse || !out) return fail(RA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(partials_O) || !aligned16(out) || !aligned16(partials_lse) || (out_lse && !aligned16(out_lse)))
        return fail(RA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (P < 1 || B < 1 || S < 1 || H < 1) return fail(RA_ERR_INVALID_ARG, "P, B, S, H must be >= 1");
    if (D != 64 && D != 128) return fail(RA_ERR_INVALID_ARG, "D must be 64 or 128 (got %d)", D);
    if (dt != RA_BF16 && dt != RA_F32) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dt));
    if (static_cast<long long>(P) * B * S * H * D > (1ll << 42)) return fail(RA_ERR_INVALID_ARG, "too large");
    ra::MergeArgs a{partials_O, partials_lse, out, out_lse, P, B, S, H, D, dt == RA_F32, dt == RA_F32};
    cudaError_t e = ra::launch_lse_merge(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "lse merge launch");
    return ok();
}

size_t ra_prefix_fanout_workspace_size(int R, int n_branches, int S_prefix, int S_suffix, int Hq, int Hkv, int D,
                                       ra_dtype dt) {
    if (R < 0 || n_branches < 1 || S_prefix < 0 || S_suffix < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv ||
        (D != 64 && D != 128) || (dt != RA_BF16 && dt != RA_F32) || 128 % (Hq / Hkv) || S_prefix + S_suffix < 1)
        return 0;
    if (dt == RA_F32) return 0;  // the fp32 path writes its rows directly
    // one size for the contiguous and the paged entry points (their splits may differ)
    const size_t a = plan_fanout(R, n_branches, S_prefix, S_suffix, Hq, Hkv, D, false).total;
    const size_t b = plan_fanout(R, n_branches, S_prefix, S_suffix, Hq, Hkv, D, true).total;
    return a > b ? a : b;
}

// Paged KV of a fan-out call (all zero: contiguous prefix / suffix tensors).
struct PagedKv {
    int paged = 0, page_shift = 0, n_pages = 0;
    const int* prefix_pages = nullptr;
    const int* suffix_pages = nullptr;
};

// Launches a fan-out call on a checked plan: the attention kernel writes the
// plan's chunk partials to part_o / part_lse (laid out as finish_plan sizes
// them), the merge joins them into out / lse.  Both the workspace entry points
// and the no-allocation one go through here.
static ra_status launch_fanout(const FanoutPlan& f, float* part_o, float* part_lse, const void* q_rows,
                               const int* branch_offsets, int n_branches, int R, const void* k_prefix,
                               const void* v_prefix, int S_prefix, const void* k_suffix, const void* v_suffix,
                               int S_suffix, void* out, float* lse, int Hq, int Hkv, int D, void* stream,
                               int suffix_causal, const PagedKv& pg) {
    ra::FanoutTcArgs a{};
    a.q_rows = q_rows;
    a.offsets = branch_offsets;
    a.n_branches = n_branches;
    a.R = R;
    a.k_prefix = k_prefix;
    a.v_prefix = v_prefix;
    a.S_prefix = S_prefix;
    a.k_suffix = k_suffix;
    a.v_suffix = v_suffix;
    a.S_suffix = S_suffix;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.n_chunks = f.n_chunks;
    for (int c = 0; c <= f.n_chunks; ++c) a.chunk_start[c] = f.chunk_start[c];
    a.part.o = part_o;
    a.part.lse = part_lse;
    a.part.o_row = static_cast<long long>(Hq) * D;
    a.part.o_h = D;
    a.part.o_part = static_cast<long long>(R) * Hq * D;
    a.part.lse_h = R;
    a.part.lse_part = static_cast<long long>(Hq) * R;
    a.part.o_f32 = 1;
    a.suffix_causal = suffix_causal;
    if (pg.paged) {
        const int page_size = 1 << pg.page_shift;
        a.paged = 1;
        a.page_shift = pg.page_shift;
        a.n_pages = pg.n_pages;
        a.n_prefix_pages = (S_prefix + page_size - 1) / page_size;
        a.n_suffix_pages = (S_suffix + page_size - 1) / page_size;
        a.prefix_pages = pg.prefix_pages;
        a.suffix_pages = pg.suffix_pages;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = ra::launch_fanout_tc(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "fan-out attention launch");
    ra::MergeArgs m{part_o, part_lse, out, lse, f.P, 1, R, Hq, D, 1, 0};
    e = ra::launch_lse_merge(m, s);
    if (e != cudaSuccess) return cuda_fail(e, "fan-out merge launch");
    return ok();
}

// fp32 fan-out: the CUDA-core kernel writes O and lse itself (no workspace).
static ra_status launch_fanout_f32(const void* q_rows, const int* branch_offsets, int n_branches, int R,
                                   const void* k_prefix, const void* v_prefix, int S_prefix, const void* k_suffix,
                                   const void* v_suffix, int S_suffix, void* out, float* lse, int Hq, int Hkv, int D,
                                   void* stream, int suffix_causal, const PagedKv& pg) {
    ra::FanoutSimtArgs a{};
    a.q_rows = static_cast<const float*>(q_rows);
    a.offsets = branch_offsets;
    a.n_branches = n_branches;
    a.R = R;
    a.k_prefix = static_cast<const float*>(k_prefix);
    a.v_prefix = static_cast<const float*>(v_prefix);
    a.S_prefix = S_prefix;
    a.k_suffix = static_cast<const float*>(k_suffix);
    a.v_suffix = static_cast<const float*>(v_suffix);
    a.S_suffix = S_suffix;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.out = static_cast<float*>(out);
    a.lse = lse;
    a.suffix_causal = suffix_causal;
    if (pg.paged) {
        const int page_size = 1 << pg.page_shift;
        a.paged = 1;
        a.page_shift = pg.page_shift;
        a.n_pages = pg.n_pages;
        a.n_prefix_pages = (S_prefix + page_size - 1) / page_size;
        a.n_suffix_pages = (S_suffix + page_size - 1) / page_size;
        a.prefix_pages = pg.prefix_pages;
        a.suffix_pages = pg.suffix_pages;
    }
    const cudaError_t e = ra::launch_fanout_simt(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fp32 fan-out launch");
    return ok();
}

static ra_status fanout_common(const void* q_rows, const int* branch_offsets, int n_branches, int R,
                               const void* k_prefix, const void* v_prefix, int S_prefix, const void* k_suffix,
                               const void* v_suffix, int S_suffix, void* out, float* lse, int Hq, int Hkv, int D,
                               ra_dtype dt, void* workspace, size_t workspace_bytes, void* stream,
                               int suffix_causal, const PagedKv& pg = PagedKv()) {
    ra_status st = check_fanout(q_rows, branch_offsets, n_branches, R, k_prefix, v_prefix, S_prefix, k_suffix,
                                v_suffix, S_suffix, out, Hq, Hkv, D, dt);
    if (st != RA_OK) return st;
    if (lse && !aligned16(lse)) return fail(RA_ERR_INVALID_ARG, "lse must be 16-byte aligned");
    if (R == 0) return ok();
    if (dt == RA_F32)
        return launch_fanout_f32(q_rows, branch_offsets, n_branches, R, k_prefix, v_prefix, S_prefix, k_suffix,
                                 v_suffix, S_suffix, out, lse, Hq, Hkv, D, stream, suffix_causal, pg);
    const FanoutPlan f = plan_fanout(R, n_branches, S_prefix, S_suffix, Hq, Hkv, D, pg.paged != 0);
    if (!workspace || workspace_bytes < f.total)
        return fail(RA_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", f.total, workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(RA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    float* part_o = static_cast<float*>(workspace);
    float* part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + f.part_o_bytes);
    return launch_fanout(f, part_o, part_lse, q_rows, branch_offsets, n_branches, R, k_prefix, v_prefix, S_prefix,
                         k_suffix, v_suffix, S_suffix, out, lse, Hq, Hkv, D, stream, suffix_causal, pg);
}

ra_status ra_prefix_fanout_attn(const void* q_rows, const int* branch_offsets, int n_branches, int R,
                                const void* k_prefix, const void* v_prefix, int S_prefix, const void* k_suffix,
                                const void* v_suffix, int S_suffix, void* out, float* lse, int Hq, int Hkv, int D,
                                ra_dtype dt, void* workspace, size_t workspace_bytes, void* stream) {
    return fanout_common(q_rows, branch_offsets, n_branches, R, k_prefix, v_prefix, S_prefix, k_suffix, v_suffix,
                         S_suffix, out, lse, Hq, Hkv, D, dt, workspace, workspace_bytes, stream, 0);
}

ra_status ra_prefix_fanout_prefill(const void* q_rows, const int* branch_offsets, int n_branches, int R,
                                   const void* k_prefix, const void* v_prefix, int S_prefix, const void* k_suffix,
                                   const void* v_suffix, int S_suffix, void* out, float* lse, int Hq, int Hkv,
                                   int D, ra_dtype dt, void* workspace, size_t workspace_bytes, void* stream) {
    return fanout_common(q_rows, branch_offsets, n_branches, R, k_prefix, v_prefix, S_prefix, k_suffix, v_suffix,
                         S_suffix, out, lse, Hq, Hkv, D, dt, workspace, workspace_bytes, stream, 1);
}

ra_status ra_prefix_fanout_attn_paged(const void* q_rows, const int* branch_offsets, int n_branches, int R,
                                      const void* k_pages, const void* v_pages, int n_pages, int page_size,
                                      const int* prefix_pages, int S_prefix, const int* suffix_pages, int S_suffix,
                                      void* out, float* lse, int Hq, int Hkv, int D, ra_dtype dt, int prefill,
                                      void* workspace, size_t workspace_bytes, void* stream) {
    if (page_size < 8 || (page_size & (page_size - 1)) || page_size > (1 << 20))
        return fail(RA_ERR_INVALID_ARG, "page_size must be a power of two in [8, 2^20] (got %d)", page_size);
    if (n_pages < 1 || static_cast<long long>(n_pages) * page_size > (1ll << 31) - 1)
        return fail(RA_ERR_INVALID_ARG, "n_pages must be >= 1 and n_pages * page_size < 2^31");
    if (prefill != 0 && prefill != 1) return fail(RA_ERR_INVALID_ARG, "prefill must be 0 or 1");
    if ((S_prefix > 0 && !prefix_pages) || (S_suffix > 0 && !suffix_pages))
        return fail(RA_ERR_INVALID_ARG, "null page table");
    if ((reinterpret_cast<uintptr_t>(prefix_pages) & 3u) || (reinterpret_cast<uintptr_t>(suffix_pages) & 3u))
        return fail(RA_ERR_INVALID_ARG, "page tables misaligned");
    PagedKv pg;
    pg.paged = 1;
    while ((1 << pg.page_shift) < page_size) ++pg.page_shift;
    pg.n_pages = n_pages;
    pg.prefix_pages = prefix_pages;
    pg.suffix_pages = suffix_pages;
    // the pools stand in for both the prefix and the suffix tensors
    return fanout_common(q_rows, branch_offsets, n_branches, R, k_pages, v_pages, S_prefix, k_pages, v_pages,
                         S_suffix, out, lse, Hq, Hkv, D, dt, workspace, workspace_bytes, stream, prefill, pg);
}

ra_status ra_prefix_fanout_attn_noalloc(const void* q_rows, const int* branch_offsets, int n_branches, int R,
                                        const void* k_prefix, const void* v_prefix, int S_prefix,
                                        const void* k_suffix, const void* v_suffix, int S_suffix, void* out,
                                        float* lse, int Hq, int Hkv, int D, ra_dtype dt, void* stream) {
    ra_status st = check_fanout(q_rows, branch_offsets, n_branches, R, k_prefix, v_prefix, S_prefix, k_suffix,
                                v_suffix, S_suffix, out, Hq, Hkv, D, dt);
    if (st != RA_OK) return st;
    if (lse && !aligned16(lse)) return fail(RA_ERR_INVALID_ARG, "lse must be 16-byte aligned");
    if (R == 0) return ok();
    if (dt == RA_F32)  // the fp32 path has no partials: the scratch array is not used
        return launch_fanout_f32(q_rows, branch_offsets, n_branches, R, k_prefix, v_prefix, S_prefix, k_suffix,
                                 v_suffix, S_suffix, out, lse, Hq, Hkv, D, stream, 0, PagedKv());
    const size_t cap = RA_NOALLOC_SCRATCH_BYTES;
    const FanoutPlan f = plan_fanout_bounded(R, n_branches, S_prefix, S_suffix, Hq, Hkv, D, cap);
    if (f.total == 0)
        return fail(RA_ERR_WORKSPACE,
                    "fan-out partials for R=%d, Hq=%d, D=%d do not fit the %zu-byte static scratch; "
                    "use ra_prefix_fanout_attn with a workspace", R, Hq, D, cap);
    void* scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != RA_OK) return st;
    float* part_o = static_cast<float*>(scratch);
    float* part_lse = reinterpret_cast<float*>(static_cast<char*>(scratch) + f.part_o_bytes);
    return launch_fanout(f, part_o, part_lse, q_rows, branch_offsets, n_branches, R, k_prefix, v_prefix, S_prefix,
                         k_suffix, v_suffix, S_suffix, out, lse, Hq, Hkv, D, stream, 0, PagedKv());
}

int ra_ring_shard_order(int S, int n_shards, int causal, int q_row0, int* shard_order) {
    if (S < 1 || n_shards < 1 || S % n_shards || q_row0 < 0 || q_row0 >= S || !shard_order) return -1;
    const ra::RingWalk w = ra::make_ring_walk(S, n_shards, 1, causal ? 1 : 0, q_row0, 1);
    for (int t = 0; t < w.n_visited; ++t) shard_order[t] = ra::ring_shard_at(w, t);
    return w.n_visited;
}

size_t ra_blockwise_attn_bwd_workspace_size(int B, int S, int Hq, int D, ra_dtype dt) {
    if (B < 1 || S < 1 || Hq < 1 || (D != 64 && D != 128) || (dt != RA_BF16 && dt != RA_F32)) return 0;
    const size_t vec = (static_cast<size_t>(B) * Hq * S * sizeof(float) + 255) & ~size_t(255);
    return 2 * vec;  // Delta, then lse in log2 units
}

static ra_status bwd_common(const void* q, const void* k, const void* v, const void* out, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int B, int S, int Hq, int Hkv, int D,
                            int n_shards, int block, int causal, int layout, ra_dtype dt, void* workspace,
                            size_t workspace_bytes, void* stream) {
    ra_status st = check_ring(q, k, v, out, B, S, Hq, Hkv, D, n_shards, block, causal, dt, layout);
    if (st != RA_OK) return st;
    if (!lse || !dout || !dq || !dk || !dv) return fail(RA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(lse) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return fail(RA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    const size_t need = ra_blockwise_attn_bwd_workspace_size(B, S, Hq, D, dt);
    if (!workspace || workspace_bytes < need)
        return fail(RA_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", need, workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(RA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    ra::BwdArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.ws_delta = static_cast<float*>(workspace);
    a.ws_lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + need / 2);
    a.B = B;
    a.S = S;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.n_shards = n_shards;
    a.causal = causal;
    a.layout = layout;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = dt == RA_BF16 ? ra::launch_bwd_tc(a, s) : ra::launch_bwd_simt(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "attention backward launch");
    return ok();
}

ra_status ra_blockwise_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                                const void* dout, void* dq, void* dk, void* dv, int B, int S, int Hq, int Hkv,
                                int D, int n_shards, int block, int causal, ra_dtype dt, void* workspace,
                                size_t workspace_bytes, void* stream) {
    return bwd_common(q, k, v, out, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D, n_shards, block, causal,
                      RA_LAYOUT_CONTIGUOUS, dt, workspace, workspace_bytes, stream);
}

ra_status ra_blockwise_attn_bwd_layout(const void* q, const void* k, const void* v, const void* out,
                                       const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                                       int S, int Hq, int Hkv, int D, int n_shards, int block, int causal,
                                       int layout, ra_dtype dt, void* workspace, size_t workspace_bytes,
                                       void* stream) {
    return bwd_common(q, k, v, out, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D, n_shards, block, causal, layout, dt,
                      workspace, workspace_bytes, stream);
}

int ra_prefix_fanout_plan(int R, int n_branches, int S_prefix, int S_suffix, int Hq, int Hkv, int n_sm,
                          int* chunk_start) {
    if (R < 1 || n_branches < 1 || S_prefix < 1 || S_suffix < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv ||
        128 % (Hq / Hkv) || n_sm < 1 || !chunk_start)
        return -1;
    int n = 0;
    ra::fanout_plan(R, S_prefix, S_suffix, n_branches, Hq, Hkv, n_sm, &n, chunk_start);
    return n;
}

int ra_layout_positions(int S, int n_shards, int layout, int* pos) {
    if (S < 1 || n_shards < 1 || S % n_shards || !pos) return -1;
    if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG && layout != RA_LAYOUT_STRIPED) return -1;
    const int L = S / n_shards;
    if (layout == RA_LAYOUT_ZIGZAG && L % 2) return -1;
    for (int p = 0; p < S; ++p) pos[p] = ra::layout_pos(layout, L, n_shards, p);
    return 0;
}

int ra_tile_launch_order(int S, int n_shards, int layout, int tile_rows, int* row0) {
    if (S < 1 || n_shards < 1 || S % n_shards || tile_rows < 1 || !row0) return -1;
    if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG && layout != RA_LAYOUT_STRIPED) return -1;
    const int L = S / n_shards;
    const int span = layout == RA_LAYOUT_ZIGZAG ? L / 2 : L;  // a tile stays inside one span
    if ((layout == RA_LAYOUT_ZIGZAG && L % 2) || span % tile_rows) return -1;
    for (int r = 0; r < S / tile_rows; ++r) row0[r] = ra::heavy_tile_row0(layout, S, n_shards, tile_rows, r);
    return 0;
}

int ra_ring_walk_layout(int S, int n_shards, int causal, int layout, int q_row0, int q_rows, int tile,
                        int* shard_order, int* visible_keys, int* total_tiles) {
    if (S < 1 || n_shards < 1 || S % n_shards || !shard_order || !visible_keys || !total_tiles) return -1;
    if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG && layout != RA_LAYOUT_STRIPED) return -1;
    const int L = S / n_shards;
    const int span = layout == RA_LAYOUT_ZIGZAG ? L / 2 : L;  // a query tile stays inside one span
    if (layout == RA_LAYOUT_ZIGZAG && L % 2) return -1;
    if (tile < 1 || span % tile || q_rows < 1 || q_row0 < 0 || q_row0 + q_rows > S) return -1;
    if (q_row0 / span != (q_row0 + q_rows - 1) / span) return -1;
    const ra::RingWalk w = ra::make_ring_walk(S, n_shards, tile, causal ? 1 : 0, q_row0, q_rows, layout);
    ra::RingIter it;
    it.start(w);
    for (int t = 0; t < w.n_visited; ++t) {
        // the iterator's shard sequence, and the keys of each shard the last query row sees
        shard_order[t] = it.j;
        visible_keys[t] = causal ? ra::shard_visible(layout, L, n_shards, it.j, w.maxpos) : L;
        const int n = it.count;
        for (int i = 0; i < n; ++i) it.next();
    }
    *total_tiles = w.total;
    return w.n_visited;
}

ra_status ra_device_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    unsigned where = 0, code = ra::read_clear_status_tc(&where);
    const char* who = "tensor-core attention";
    if (!code) {
        code = ra::read_clear_status_simt(&where);
        who = "fp32 attention";
    }
    if (!code) {
        code = ra::read_clear_status_merge(&where);
        who = "lse merge";
    }
    if (!code) {
        code = ra::read_clear_status_bwd(&where);
        who = "attention backward";
    }
    if (!code) {
        code = ra::read_clear_status_selftest(&where);
        who = "wait self-test";
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "device status");
    if (code == RA_ERR_DEVICE_TIMEOUT)
        return fail(RA_ERR_DEVICE_TIMEOUT, "%s: bounded device wait ran out (site 0x%08x)", who, where);
    if (code == RA_ERR_INVALID_ARG && (where >> 24) == 0x0E)
        return fail(RA_ERR_INVALID_ARG, "%s: page table entry %u is outside the page pool", who, where & 0xFFFFFFu);
    if (code == RA_ERR_INVALID_ARG)
        return fail(RA_ERR_INVALID_ARG, "%s: device-side argument check failed (0x%08x)", who, where);
    if (code) return fail(static_cast<ra_status>(code), "%s: device status %u", who, code);
    return ok();
}

ra_status ra_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
    if (limit_ns == 0 || limit_ns > 2000000000ull) return fail(RA_ERR_INVALID_ARG, "limit_ns must be in (0, 2e9]");
    const cudaError_t e = ra::launch_selftest_wait_timeout(limit_ns, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "wait self-test launch");
    return ok();
}

const char* ra_last_error(void) { return g_err; }

}  // extern "C"
