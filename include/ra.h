/*
 * ra.h -- C ABI of libra.so: blockwise exact attention walked in ring order,
 * per-shard partials, the row-indexed log-sum-exp merge, and shared-prefix
 * fan-out attention, on one NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers, owned and allocated by the
 *    caller.  The library never allocates or frees memory and never
 *    synchronises, except ra_device_status().  Inputs are read-only; outputs
 *    are fully overwritten.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *    the legacy default stream) of the current CUDA device.
 *  - Layouts are dense row-major.  q/k/v/out are [B, S, H, D] (token-major,
 *    head, then head dimension); lse is [B, Hq, S] fp32.
 *  - Scores are q.k / sqrt(D) (the softmax scale of the attention definition
 *    in "RingAttention and Context Parallelism: Mathematical Foundations",
 *    section 1).  lse is the natural-log log-sum-exp of the scaled scores,
 *    L = m + ln(l) (same page, section 7 figure).
 *  - Grouped-query attention: q head h reads kv head h / (Hq / Hkv).
 *  - Causal masking uses global positions: query i sees keys j <= i (same page,
 *    section 5).
 *  - Arguments are validated on the host before any launch.  A rejected call
 *    returns a non-OK status and launches nothing; ra_last_error() then holds a
 *    one-line message for the calling thread.  A failed launch returns
 *    RA_ERR_CUDA.  Device-side waits are bounded: a wait that runs out records
 *    RA_ERR_DEVICE_TIMEOUT in a device status word that ra_device_status()
 *    reports (the kernel returns instead of hanging).
 *  - Pointers must be 16-byte aligned (bulk tensor copies start on 16-byte
 *    boundaries).
 *  - dtype RA_BF16 runs the tensor-core path (tcgen05 MMA, TMEM accumulators,
 *    TMA-staged tiles); RA_F32 runs an exact fp32 FMA path.  There is no CPU
 *    fallback.
 */
#ifndef RA_H_
#define RA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = 1,    /* bad pointer, size, alignment or divisibility */
    RA_ERR_UNSUPPORTED = 2,    /* valid request the kernels do not implement */
    RA_ERR_CUDA = 3,           /* a CUDA runtime/driver call or launch failed */
    RA_ERR_DEVICE_TIMEOUT = 4, /* a bounded device-side wait ran out */
    RA_ERR_WORKSPACE = 5       /* workspace missing or smaller than required */
} ra_status;

typedef enum { RA_F32 = 0, RA_BF16 = 1 } ra_dtype;

/*
 * Shard layouts: how the rows of q/k/v/out are arranged over the n_shards ring
 * shards ("RingAttention and Context Parallelism: Mathematical Foundations",
 * section 5).  Shard s holds storage rows [s*L, (s+1)*L), L = S / n_shards; the
 * layout fixes the sequence position of each row, which is what the causal mask
 * compares (query at position i sees keys at positions j <= i):
 *   RA_LAYOUT_CONTIGUOUS  shard s holds tokens [s*L, (s+1)*L) in order.
 *   RA_LAYOUT_ZIGZAG      the sequence is cut into 2N chunks c_0..c_{2N-1} of
 *                         L/2 tokens; shard s holds c_s then c_{2N-1-s}
 *                         (zigzag ring attention: one early and one late chunk
 *                         per shard, which balances the causal work).
 *   RA_LAYOUT_STRIPED     shard s holds the tokens i with i mod N = s, in
 *                         increasing order (striped attention).
 * Without a causal mask the layout changes nothing: output row p is the
 * attention of query row p over every key row.
 */
typedef enum { RA_LAYOUT_CONTIGUOUS = 0, RA_LAYOUT_ZIGZAG = 1, RA_LAYOUT_STRIPED = 2 } ra_layout;

/*
 * Blockwise exact attention with online softmax, KV walked in ring order.
 *
 * Defined by "RingAttention and Context Parallelism: Mathematical Foundations":
 * section 2 (online softmax state (m, l, O), its five-step transition and the
 * final A = O / l), section 3 (the sequence cut into n_shards contiguous shards
 * of S/n_shards tokens; the query block of shard k visits KV shards
 * k, k-1, ..., 0, N-1, ..., k+1, i.e. (k - t) mod N at step t) and section 5
 * (causal: KV shards after the query's shard are skipped without loads).
 *
 *   q    [B, S, Hq, D]  dtype dt          k, v [B, S, Hkv, D] dtype dt
 *   out  [B, S, Hq, D]  dtype dt          lse  [B, Hq, S] fp32 (may be NULL)
 *   n_shards : shards of the ring; S % n_shards == 0.
 *   block    : KV block walked within a shard; (S / n_shards) % block == 0.
 *              The bf16 path consumes keys in 128-key tiles (a block of 64 is
 *              walked as consecutive pairs, the same key order) and needs
 *              (S / n_shards) % 128 == 0.
 *   causal   : 0 or 1.
 *   D        : 64 or 128.   Hq % Hkv == 0.
 * Errors: RA_ERR_INVALID_ARG for any violated rule above, RA_ERR_UNSUPPORTED
 * for a valid shape outside what the kernels implement, RA_ERR_CUDA if the
 * launch fails.
 */
ra_status ra_blockwise_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                                int B, int S, int Hq, int Hkv, int D, int n_shards, int block,
                                int causal, ra_dtype dt, void* stream);

/*
 * ra_blockwise_attn_fwd for rows stored in a zigzag or striped shard layout
 * (ra_layout above; same page, section 5).  q/k/v/out/lse are indexed by
 * storage row; the causal mask compares the rows' sequence positions.
 * Striped: each query tile walks the KV shards in the same ring order, taking
 * from each shard the prefix of its rows that the tile can see (positions
 * increase along a shard's rows in every layout); when n_shards divides 128
 * the causal walk runs over positions instead (tiles of 128 consecutive
 * positions, 128 / n_shards rows of every shard).  Zigzag: the causal walk
 * runs in sequence-position order over the 2 n_shards chunks of the zigzag
 * cut (the query's own chunk, then the earlier ones: the contiguous ring over
 * those chunks), each tile of rows addressed through the layout; it visits the
 * same keys, and the order changes rounding only.
 *   layout : an ra_layout value.  RA_LAYOUT_ZIGZAG needs an even shard length,
 *            and (S / n_shards / 2) % 128 == 0 on the bf16 path, % 32 == 0 on
 *            the fp32 path.
 * Other arguments and errors as ra_blockwise_attn_fwd; layout = RA_LAYOUT_CONTIGUOUS
 * is that call.
 */
ra_status ra_blockwise_attn_fwd_layout(const void* q, const void* k, const void* v, void* out, float* lse,
                                       int B, int S, int Hq, int Hkv, int D, int n_shards, int block,
                                       int causal, int layout, ra_dtype dt, void* stream);

/*
 * Per-shard partial states: the same ring walk, but the state is normalised and
 * written out after every KV shard instead of being carried across shards --
 * the per-shard partials that the "AHBM Agentic Runtime Architecture" page
 * (section 3.3) has each sequence shard produce before the row-indexed merge.
 *
 *   partials_O   [n_shards, B, S, Hq, D] dtype dt : O_j / l_j for KV shard j
 *   partials_lse [n_shards, B, Hq, S] fp32        : m_j + ln(l_j)
 * A (query, KV shard) pair that the causal mask empties entirely is written as
 * O = 0, lse = -inf without any compute.  Other arguments and errors as
 * ra_blockwise_attn_fwd.  Merging the partials with ra_lse_merge gives
 * ra_blockwise_attn_fwd's result up to rounding.
 */
ra_status ra_ring_partials_fwd(const void* q, const void* k, const void* v, void* partials_O,
                               float* partials_lse, int B, int S, int Hq, int Hkv, int D,
                               int n_shards, int block, int causal, ra_dtype dt, void* stream);

/*
 * ra_ring_partials_fwd for a zigzag or striped shard layout: partial j holds
 * the attention of every query row over the key rows of storage shard j under
 * the layout's causal mask; a row that sees none of them gets O = 0,
 * lse = -inf.  Arguments as ra_blockwise_attn_fwd_layout.
 */
ra_status ra_ring_partials_fwd_layout(const void* q, const void* k, const void* v, void* partials_O,
                                      float* partials_lse, int B, int S, int Hq, int Hkv, int D,
                                      int n_shards, int block, int causal, int layout, ra_dtype dt,
                                      void* stream);

/*
 * Backward pass of ra_blockwise_attn_fwd: dQ, dK, dV for an upstream gradient
 * dO ("RingAttention and Context Parallelism: Mathematical Foundations",
 * section 7, "RingAttention backward pass logic": the forward keeps Q and the
 * log-sum-exp L = m + ln l of every row; the backward recomputes the scores of
 * each block from Q and K, accumulates dQ locally and carries dK, dV with the
 * K/V blocks as they rotate through the ring in reverse order).  With
 * P = exp(q.k/sqrt(D) - L), Delta = rowsum(dO * O) and dS = P (dO.v - Delta):
 *   dV = P^T dO,   dK = dS^T Q / sqrt(D),   dQ = dS K / sqrt(D);
 * the q heads of a GQA group add into their kv head's dK and dV.
 *
 * Two walks, no atomics: every 128-row query tile walks the KV tiles in the
 * forward's ring order for dQ; every 128-key KV tile walks the query tiles of
 * its group's q heads, query shard j, j-1, ... (mod N, causal-empty shards
 * skipped), for dK and dV.
 *
 *   q, out, dout, dq [B, S, Hq, D] dtype dt     k, v, dk, dv [B, S, Hkv, D] dtype dt
 *   lse [B, Hq, S] fp32: the forward's lse for these q, k, v.  out: its O.
 *   workspace: device scratch of ra_blockwise_attn_bwd_workspace_size(...)
 *              bytes, 256-byte aligned, owned by the caller (contents ignored).
 * Other arguments, shape rules and errors as ra_blockwise_attn_fwd (contiguous
 * shards); RA_ERR_WORKSPACE if the workspace is missing or too small.
 * dq, dk, dv are fully overwritten.
 */
ra_status ra_blockwise_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                                const void* dout, void* dq, void* dk, void* dv, int B, int S, int Hq, int Hkv,
                                int D, int n_shards, int block, int causal, ra_dtype dt, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * ra_blockwise_attn_bwd for rows stored in a zigzag or striped shard layout
 * (ra_layout; the forward is ra_blockwise_attn_fwd_layout).  All tensors are
 * indexed by storage row; the causal mask compares the rows' sequence
 * positions.  The dQ walk takes from each KV shard the prefix of its rows a
 * query tile can see (as the forward); the dK/dV walk takes from each query
 * shard the suffix of its rows that can see a KV tile (positions increase
 * along a shard's rows in every layout).  A causal zigzag sequence is walked,
 * as in the forward, over the 2 n_shards chunks of its cut in sequence-position
 * order, and a causal striped one with n_shards dividing 128 over positions
 * (tiles of 128 consecutive positions; rounding differs only).  Other
 * arguments, rules and errors
 * as ra_blockwise_attn_bwd and ra_blockwise_attn_fwd_layout.
 */
ra_status ra_blockwise_attn_bwd_layout(const void* q, const void* k, const void* v, const void* out,
                                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                       int B, int S, int Hq, int Hkv, int D, int n_shards, int block,
                                       int causal, int layout, ra_dtype dt, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* Bytes of workspace ra_blockwise_attn_bwd (and _layout) needs (0 if the sizes are invalid). */
size_t ra_blockwise_attn_bwd_workspace_size(int B, int S, int Hq, int D, ra_dtype dt);

/*
 * Row-indexed log-sum-exp merge of P partial states computed over disjoint key
 * sets ("AHBM Agentic Runtime Architecture", sections 3.4-3.5: the same row
 * index is merged across sequence shards, never different rows).  Per
 * (b, s, h):  M = max_p lse_p;  w_p = exp(lse_p - M);  O = sum_p w_p O_p / sum_p w_p;
 * lse = M + ln(sum_p w_p).  A partial with lse_p = -inf has weight 0 and its
 * O_p does not enter the result, whatever it holds (NaN included; the memory
 * must still lie inside the partials_O buffer); if every partial is empty the
 * result is O = 0, lse = -inf.
 *
 *   partials_O   [P, B, S, H, D] dtype dt     partials_lse [P, B, H, S] fp32
 *   out          [B, S, H, D]    dtype dt     out_lse      [B, H, S] fp32 (may be NULL)
 *   D : 64 or 128.  P >= 1.
 */
ra_status ra_lse_merge(const void* partials_O, const float* partials_lse, void* out, float* out_lse,
                       int P, int B, int S, int H, int D, ra_dtype dt, void* stream);

/*
 * Shared-prefix fan-out attention ("AHBM Agentic Runtime Architecture",
 * sections 1.1-1.3, 3.2-3.4 and 5.2; "Supporting Agentic Workloads",
 * stationary-KV policy).  The new query rows of n_branches branches are stacked
 * into one tall Q; every row attends to the one shared prefix KV plus its own
 * branch's private suffix KV (never another branch's).  The prefix is split into
 * chunks processed in parallel; each prefix K/V tile is read from HBM once per
 * KV head for all stacked rows; the prefix partials and the suffix partial are
 * joined with the row-indexed log-sum-exp merge.  No causal mask.
 *
 *   q_rows         [R, Hq, D] dtype dt
 *   branch_offsets int32 device array [n_branches + 1], CSR over the stacked
 *                  rows: branch b owns rows [off[b], off[b+1]); off[0] = 0,
 *                  off[n_branches] = R, non-decreasing (checked on device: a
 *                  violation records RA_ERR_INVALID_ARG in the device status).
 *   k_prefix, v_prefix [S_prefix, Hkv, D] dtype dt, shared by all branches.
 *   k_suffix, v_suffix [n_branches, S_suffix, Hkv, D] dtype dt.
 *   out            [R, Hq, D] dtype dt;   lse [Hq, R] fp32 (may be NULL).
 *   workspace      device scratch of at least
 *                  ra_prefix_fanout_workspace_size(...) bytes, 256-byte aligned,
 *                  owned by the caller; contents on entry are ignored.  Not
 *                  used (may be NULL) for dt = RA_F32.
 *   dt = RA_BF16: tensor cores, prefix split into chunks joined by the merge.
 *   dt = RA_F32: exact fp32 on the CUDA cores (FFMA, expf), each branch's rows
 *   walking the whole prefix and their suffix; no partials.
 *   D = 64 or 128; Hq % Hkv == 0 and 128 % (Hq / Hkv) == 0; S_prefix >= 0,
 *   S_suffix >= 0, R >= 0.
 * Errors: RA_ERR_WORKSPACE if a bf16 call's workspace is NULL or too small,
 * otherwise as above.
 */
ra_status ra_prefix_fanout_attn(const void* q_rows, const int* branch_offsets, int n_branches, int R,
                                const void* k_prefix, const void* v_prefix, int S_prefix,
                                const void* k_suffix, const void* v_suffix, int S_suffix, void* out,
                                float* lse, int Hq, int Hkv, int D, ra_dtype dt, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Shared-prefix fan-out PREFILL ("AHBM Agentic Runtime Architecture", section
 * 3.6: the new tokens of all branches -- e.g. 8 sub-agents x 20 tokens -- are
 * processed together against the shared prefix; section 3.1: each branch's
 * private pages follow the shared ones).  Same arguments, layouts, workspace
 * and errors as ra_prefix_fanout_attn; the difference is the mask inside a
 * private suffix: the n_b new rows of branch b are the last n_b tokens of its
 * suffix, so its row t (t = 0 .. n_b-1) sits at suffix position
 * S_suffix - n_b + t and sees the suffix keys at positions <= that one, plus
 * the whole prefix.  (A branch with n_b > S_suffix has rows that see no suffix
 * key.)  The last row of each branch gets the ra_prefix_fanout_attn result.
 */
ra_status ra_prefix_fanout_prefill(const void* q_rows, const int* branch_offsets, int n_branches, int R,
                                   const void* k_prefix, const void* v_prefix, int S_prefix,
                                   const void* k_suffix, const void* v_suffix, int S_suffix, void* out,
                                   float* lse, int Hq, int Hkv, int D, ra_dtype dt, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * Fan-out over a PAGED KV cache ("AHBM Agentic Runtime Architecture", section
 * 3.1: the branches' page tables list the shared prefix pages, referenced by
 * every branch without copying, followed by each branch's private pages).
 *
 *   k_pages, v_pages [n_pages, page_size, Hkv, D] dtype dt: the page pools.
 *   page_size      power of two, 8 <= page_size <= 2^20.
 *   prefix_pages   int32 device array [ceil(S_prefix / page_size)]: the shared
 *                  prefix's pages in order (key k is row k % page_size of page
 *                  prefix_pages[k / page_size]).
 *   suffix_pages   int32 device array [n_branches][ceil(S_suffix / page_size)]:
 *                  each branch's private pages in order.
 *   prefill        0: ra_prefix_fanout_attn semantics; 1: ra_prefix_fanout_prefill.
 * Page indices are checked on the device: one outside [0, n_pages) records
 * RA_ERR_INVALID_ARG (reported by ra_device_status) and its keys read as zeros.
 * The rows of a sequence's last page past S_prefix / S_suffix are read and
 * given weight zero: they must hold finite values (zeros, or stale keys).
 * Each prefix tile is still read from HBM once per KV head for all rows.
 * Other arguments, the workspace (ra_prefix_fanout_workspace_size with the
 * same R, n_branches, S_prefix, S_suffix) and errors as ra_prefix_fanout_attn.
 */
ra_status ra_prefix_fanout_attn_paged(const void* q_rows, const int* branch_offsets, int n_branches, int R,
                                      const void* k_pages, const void* v_pages, int n_pages, int page_size,
                                      const int* prefix_pages, int S_prefix, const int* suffix_pages,
                                      int S_suffix, void* out, float* lse, int Hq, int Hkv, int D, ra_dtype dt,
                                      int prefill, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace ra_prefix_fanout_attn (and ra_prefix_fanout_prefill,
 * ra_prefix_fanout_attn_paged) needs for these sizes on the current device (0
 * if the sizes are invalid, and for dt = RA_F32, which needs none). */
size_t ra_prefix_fanout_workspace_size(int R, int n_branches, int S_prefix, int S_suffix, int Hq,
                                       int Hkv, int D, ra_dtype dt);

/*
 * Size of the device scratch array behind ra_prefix_fanout_attn_noalloc:
 * 32 MiB, held on every GPU that loads libra.so until the process exits.
 */
#define RA_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * ra_prefix_fanout_attn without a workspace argument, for callers that cannot
 * allocate device memory themselves -- for example a plugin inside a host
 * framework that owns every allocation and hands it only fixed input/output
 * buffers, or a latency-critical decode loop where a cudaMalloc (which can
 * synchronise the device) is not allowed.  The pages have no counterpart: this
 * is a packaging variant of the fan-out entry point above, not a step of the
 * method.
 *
 * Same arguments, layouts, semantics and errors as ra_prefix_fanout_attn, minus
 * the workspace.  The partials live instead in one file-scope device array of
 * RA_NOALLOC_SCRATCH_BYTES inside the library; the prefix is split into as
 * many chunks as fit in it.  A call whose partials cannot fit even with one
 * prefix chunk (roughly R * Hq * D * 8 bytes > RA_NOALLOC_SCRATCH_BYTES) is
 * rejected with RA_ERR_WORKSPACE before anything is launched.  Nothing is
 * allocated or freed: no cudaMalloc, no cudaFree, no allocating library call.
 *
 * The first call on a device (with that device current) looks up the array's
 * device address with cudaGetSymbolAddress; make that first call before any
 * stream capture.  The address is kept per device and context: after a device
 * reset (cudaDeviceReset) the next call looks it up again in the new context,
 * so that call, too, belongs before any capture.  Every call, on every stream, shares the one array, and it
 * keeps the previous call's contents (nothing in it needs to start at zero):
 * calls that can overlap on the GPU race on it, so serialise them, e.g. on
 * one stream.
 */
ra_status ra_prefix_fanout_attn_noalloc(const void* q_rows, const int* branch_offsets, int n_branches, int R,
                                        const void* k_prefix, const void* v_prefix, int S_prefix,
                                        const void* k_suffix, const void* v_suffix, int S_suffix, void* out,
                                        float* lse, int Hq, int Hkv, int D, ra_dtype dt, void* stream);

/*
 * Host-side view of the ring walk the kernels take (no GPU needed): for the
 * 128-row query tile starting at q_row0, writes to shard_order[] the KV shards
 * in the order they are visited ((k - t) mod n_shards, causal-empty shards
 * skipped) and returns how many there are, or -1 on invalid arguments.
 * shard_order must hold n_shards ints.
 */
int ra_ring_shard_order(int S, int n_shards, int causal, int q_row0, int* shard_order);

/*
 * Host-side view of how a fan-out call splits the shared prefix (no GPU): for
 * these sizes on n_sm SMs, writes the n_chunks + 1 prefix-tile boundaries
 * (128-key tiles; chunk c covers tiles [chunk_start[c], chunk_start[c+1]))
 * and returns n_chunks (<= 64), or -1 on invalid arguments.  chunk_start
 * holds 65 ints.  The split is chosen by simulating the block scheduler over
 * the launch's units (prefix chunk x KV head x row pair) and minimising the
 * makespan; it may make chunks unequal.  Calls whose stacked rows fit one
 * 128-row tile per KV head are bound by HBM bandwidth: their units take at
 * most 4/5 of the SMs (fewer chunks, fewer partials to merge).  This is the
 * split of the contiguous entry points; ra_prefix_fanout_attn_paged spreads
 * such units over every SM.
 */
int ra_prefix_fanout_plan(int R, int n_branches, int S_prefix, int S_suffix, int Hq, int Hkv, int n_sm,
                          int* chunk_start);

/*
 * Host-side (no GPU): pos[p] = sequence position of storage row p under
 * `layout` (ra_layout) for S rows in n_shards shards.  pos holds S ints.
 * Returns 0, or -1 on invalid arguments (zigzag needs an even shard length).
 */
int ra_layout_positions(int S, int n_shards, int layout, int* pos);

/*
 * Host-side (no GPU): the order in which the causal kernels launch the tiles of
 * `tile_rows` storage rows.  Under the causal mask a query's work grows with its
 * position (the load imbalance of "RingAttention and Context Parallelism:
 * Mathematical Foundations ...", section 5); the kernels launch the tiles
 * heaviest first, which keeps the last wave of the grid short.  row0[r] = first
 * storage row of the r-th query tile launched; the
 * backward's key tiles are launched in the reverse order (a key's work shrinks
 * with its position).  row0 holds S / tile_rows ints.  Returns 0, or -1 on
 * invalid arguments (S % n_shards, the shard length -- half of it for zigzag --
 * % tile_rows, zigzag with an odd shard length).
 */
int ra_tile_launch_order(int S, int n_shards, int layout, int tile_rows, int* row0);

/*
 * Host-side view of the walk of one query tile under a layout: the query rows
 * [q_row0, q_row0 + q_rows) (inside one shard; for zigzag inside one half of
 * it), KV tiles of `tile` keys.  Writes, for each visited shard in ring order,
 * shard_order[t] and visible_keys[t] (the keys of that shard the tile's last
 * row can see, a prefix of the shard's rows; the shard length when not
 * causal), and *total_tiles = the KV tiles the layout's own ring walk takes
 * for this tile (the per-shard partials, and striped with n_shards not
 * dividing 128).  The single-output zigzag kernels take the same keys in the
 * order of the 2 n_shards chunks (this call with RA_LAYOUT_CONTIGUOUS and
 * 2 n_shards shards on sequence positions); the striped ones with n_shards
 * dividing 128 walk sequence positions (RA_LAYOUT_CONTIGUOUS, n_shards shards).
 * Shards after the returned count see nothing.  Arrays hold n_shards ints.
 * Returns the number of visited shards, or -1 on invalid arguments.
 */
int ra_ring_walk_layout(int S, int n_shards, int causal, int layout, int q_row0, int q_rows, int tile,
                        int* shard_order, int* visible_keys, int* total_tiles);

/* Synchronises `stream`, then returns and clears the device status word:
 * RA_OK, RA_ERR_DEVICE_TIMEOUT or RA_ERR_INVALID_ARG (device-side check), or
 * RA_ERR_CUDA if the stream reports an error. */
ra_status ra_device_status(void* stream);

/*
 * Health check of the device-side failure detection (not a step of the method):
 * launches one thread that waits, for at most limit_ns nanoseconds of the GPU
 * timer, on an mbarrier that nothing completes -- the bounded wait that guards
 * every pipeline stage of the attention kernels.  The wait runs out, the
 * kernel records RA_ERR_DEVICE_TIMEOUT and returns, so the next
 * ra_device_status(stream) reports RA_ERR_DEVICE_TIMEOUT and the context stays
 * usable.  limit_ns in (0, 2e9]; RA_ERR_INVALID_ARG otherwise.
 */
ra_status ra_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/* Thread-local one-line description of the last non-OK status ("" if none). */
const char* ra_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* RA_H_ */
