/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for blockwise ring attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the package smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code with the CUDA kernels.
 *
 * What it computes is the plain definition of the result the blockwise method
 * reaches exactly, written out with no blocking, no shards and no online
 * recurrence:
 *
 *   - Scaled dot-product softmax attention, A = softmax(q K^T / sqrt(d_k) + M) V
 *     with M the optional causal mask ("RingAttention and Context Parallelism:
 *     Mathematical Foundations ...", section 1, the attention equation), and the
 *     statement in section 2 that the blockwise recurrence equals softmax over
 *     the concatenated sequence (the exactness identity after the online-softmax
 *     equations).
 *   - Causal masking on global positions: token i sees keys j <= i (same page,
 *     section 5, first paragraph).  Rows may be stored out of sequence order
 *     (the striped and zigzag shard layouts of section 5): then pos[r] gives the
 *     sequence position of stored row r and the mask compares positions.
 *   - The log-sum-exp statistic L = m + ln(l) kept for the backward pass (same
 *     page, section 7, "RingAttention backward pass logic" figure), which is the
 *     natural log of sum_j exp(s_j).
 *   - Shared-prefix fan-out: a branch row sees the shared prefix keys plus its
 *     own private suffix keys and never another branch's suffix ("AHBM Agentic
 *     Runtime Architecture", sections 1.1, 3.2 and 5.2; "Supporting Agentic
 *     Workloads", the context_i equation in the motivation subsection).
 *   - The row-indexed merge of partial states over disjoint key sets ("AHBM
 *     Agentic Runtime Architecture", sections 3.4-3.5), written as the
 *     log-sum-exp combination that the exactness identity implies.
 *
 * Readings where the pages are silent:
 *   - grouped-query heads: q head h reads kv head h / (Hq / Hkv);
 *   - a query with no visible key has O = 0 and lse = -inf;
 *   - layouts: q/k/v/out are [B, S, H, D] row-major, lse is [B, Hq, S].
 *
 * Every input element is widened to double exactly (fp32 or bf16 storage) and
 * all arithmetic is double.  Parallelised over queries with OpenMP; each query
 * materialises its full score row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };

/* Widen one stored element to double.  bf16 is the upper half of an IEEE
 * binary32, so the widening is exact. */
static double load_elem(const void* base, int dtype, int64_t idx) {
    if (dtype == OR_F64) return ((const double*)base)[idx];
    if (dtype == OR_F32) return (double)((const float*)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Softmax-weighted sum over an explicit list of key rows.
 *   q_row      : D doubles
 *   key_ptrs   : for each visible key, (tensor, element offset of its row)
 * Writes D doubles to out and returns lse (or -inf with out = 0 when n == 0). */
typedef struct {
    const void* k;
    const void* v;
    int64_t off;
} key_ref;

static double softmax_row(const double* q_row, const key_ref* keys, int64_t n, int D,
                          int dtype, double scale, double* s, double* out) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n == 0) return -INFINITY;
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q_row[d] * load_elem(keys[j].k, dtype, keys[j].off + d);
        s[j] = acc * scale;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(s[j] - m);
        l += p;
        for (int d = 0; d < D; ++d) out[d] += p * load_elem(keys[j].v, dtype, keys[j].off + d);
    }
    for (int d = 0; d < D; ++d) out[d] /= l;
    return m + log(l);
}

/*
 * Attention for the queries listed in `sel` (or every query when sel == NULL).
 *   q [B,S,Hq,D], k/v [B,S,Hkv,D] in `dtype`.
 *   Visible keys of query (b,i,h): j in [kv_begin, kv_end) and, if causal,
 *   pos[j] <= pos[i] (pos == NULL: the stored order is the sequence order,
 *   pos[r] = r).
 *   sel ids encode (b,i,h) as (b*S + i)*Hq + h.
 *   sel == NULL: out [B,S,Hq,D], lse [B,Hq,S].  Otherwise out [n_sel,D], lse [n_sel].
 * Returns 0, or -1 on bad arguments.
 */
int oracle_attention(const void* q, const void* k, const void* v, int dtype,
                     int B, int S, int Hq, int Hkv, int D, int causal, const int32_t* pos,
                     int kv_begin, int kv_end, const int64_t* sel, int64_t n_sel,
                     double* out, double* lse) {
    if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv) return -1;
    if (kv_begin < 0 || kv_end > S || kv_begin > kv_end) return -1;
    const int64_t n_q = sel ? n_sel : (int64_t)B * S * Hq;
    const int group = Hq / Hkv;
    const double scale = 1.0 / sqrt((double)D);
    int bad = 0;
#pragma omp parallel
    {
        double* q_row = (double*)malloc(sizeof(double) * D);
        double* s = (double*)malloc(sizeof(double) * (size_t)S);
        key_ref* keys = (key_ref*)malloc(sizeof(key_ref) * (size_t)S);
        double tmp_out[512];
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < n_q; ++t) {
            const int64_t id = sel ? sel[t] : t;
            if (id < 0 || id >= (int64_t)B * S * Hq) { bad = 1; continue; }
            const int h = (int)(id % Hq);
            const int64_t bi = id / Hq;
            const int i = (int)(bi % S);
            const int b = (int)(bi / S);
            const int hk = h / group;
            for (int d = 0; d < D; ++d) q_row[d] = load_elem(q, dtype, id * D + d);
            int64_t n = 0;
            int hi = kv_end;
            if (causal && i + 1 < hi) hi = i + 1;
            for (int j = kv_begin; j < (pos ? kv_end : hi); ++j) {
                if (pos && causal && pos[j] > pos[i]) continue;
                keys[n].k = k;
                keys[n].v = v;
                keys[n].off = (((int64_t)b * S + j) * Hkv + hk) * D;
                ++n;
            }
            double* o = D <= 512 ? tmp_out : NULL;
            if (!o) { bad = 1; continue; }
            const double L = softmax_row(q_row, keys, n, D, dtype, scale, s, o);
            if (sel) {
                memcpy(out + t * D, o, sizeof(double) * D);
                lse[t] = L;
            } else {
                memcpy(out + id * D, o, sizeof(double) * D);
                lse[((int64_t)b * Hq + h) * S + i] = L;
            }
        }
        free(q_row);
        free(s);
        free(keys);
    }
    return bad ? -1 : 0;
}

/*
 * Shared-prefix fan-out attention.
 *   q_rows [R,Hq,D]; branch b owns stacked rows [off[b], off[b+1]).
 *   k/v_prefix [Sp,Hkv,D] shared by every branch; k/v_suffix [nb,Ss,Hkv,D].
 *   Row r of branch b sees all Sp prefix keys and all Ss keys of suffix b.
 *   suffix_causal (fan-out prefill, "AHBM Agentic Runtime Architecture" 3.6:
 *   the branches' new tokens are prefilled together): the n_b new rows of
 *   branch b are the last n_b tokens of its suffix, so its row t (t = 0 ..
 *   n_b-1) sits at suffix position Ss - n_b + t and sees the suffix keys at
 *   positions <= that one (and the whole prefix).
 *   sel ids encode (r,h) as r*Hq + h.  sel == NULL: out [R,Hq,D], lse [Hq,R];
 *   otherwise out [n_sel,D], lse [n_sel].
 */
int oracle_fanout(const void* q_rows, const int32_t* off, int nb, int R,
                  const void* k_prefix, const void* v_prefix, int Sp,
                  const void* k_suffix, const void* v_suffix, int Ss,
                  int Hq, int Hkv, int D, int dtype, int suffix_causal, const int64_t* sel, int64_t n_sel,
                  double* out, double* lse) {
    if (R < 0 || nb <= 0 || Sp < 0 || Ss < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || D > 512)
        return -1;
    if (off[0] != 0 || off[nb] != R) return -1;
    for (int b = 0; b < nb; ++b)
        if (off[b + 1] < off[b]) return -1;
    const int64_t n_q = sel ? n_sel : (int64_t)R * Hq;
    const int group = Hq / Hkv;
    const double scale = 1.0 / sqrt((double)D);
    const int64_t n_keys = (int64_t)Sp + Ss;
    int bad = 0;
#pragma omp parallel
    {
        double q_row[512], o[512];
        double* s = (double*)malloc(sizeof(double) * (size_t)(n_keys ? n_keys : 1));
        key_ref* keys = (key_ref*)malloc(sizeof(key_ref) * (size_t)(n_keys ? n_keys : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < n_q; ++t) {
            const int64_t id = sel ? sel[t] : t;
            if (id < 0 || id >= (int64_t)R * Hq) { bad = 1; continue; }
            const int h = (int)(id % Hq);
            const int r = (int)(id / Hq);
            int b = 0;
            while (!(off[b] <= r && r < off[b + 1])) ++b;
            const int hk = h / group;
            for (int d = 0; d < D; ++d) q_row[d] = load_elem(q_rows, dtype, id * D + d);
            int64_t n = 0;
            for (int j = 0; j < Sp; ++j) {
                keys[n].k = k_prefix;
                keys[n].v = v_prefix;
                keys[n].off = ((int64_t)j * Hkv + hk) * D;
                ++n;
            }
            /* suffix keys this row sees: all, or up to its own suffix position */
            const int last = suffix_causal ? Ss - (off[b + 1] - off[b]) + (r - off[b]) : Ss - 1;
            for (int j = 0; j < Ss && j <= last; ++j) {
                keys[n].k = k_suffix;
                keys[n].v = v_suffix;
                keys[n].off = (((int64_t)b * Ss + j) * Hkv + hk) * D;
                ++n;
            }
            const double L = softmax_row(q_row, keys, n, D, dtype, scale, s, o);
            if (sel) {
                memcpy(out + t * D, o, sizeof(double) * D);
                lse[t] = L;
            } else {
                memcpy(out + id * D, o, sizeof(double) * D);
                lse[(int64_t)h * R + r] = L;
            }
        }
        free(s);
        free(keys);
    }
    return bad ? -1 : 0;
}

/*
 * Row-indexed merge of P partial states computed over disjoint key sets.
 *   part_O [P,B,S,H,D] (normalised partial outputs), part_lse [P,B,H,S].
 *   For each (b,s,h): M = max_p lse_p; w_p = exp(lse_p - M) (0 when lse_p = -inf);
 *   O = sum_p w_p O_p / sum_p w_p; lse = M + ln(sum_p w_p).
 *   All partials empty: O = 0, lse = -inf.
 *   out [B,S,H,D], out_lse [B,H,S].
 */
int oracle_lse_merge(const double* part_O, const double* part_lse, int P, int B, int S, int H,
                     int D, double* out, double* out_lse) {
    if (P <= 0 || B <= 0 || S <= 0 || H <= 0 || D <= 0) return -1;
    const int64_t rows = (int64_t)B * S * H;
    const int64_t o_stride = rows * D;
    const int64_t l_stride = rows;
#pragma omp parallel for schedule(static)
    for (int64_t id = 0; id < rows; ++id) {
        const int h = (int)(id % H);
        const int64_t bs = id / H;
        const int s = (int)(bs % S);
        const int b = (int)(bs / S);
        const int64_t lidx = ((int64_t)b * H + h) * S + s;
        double M = -INFINITY;
        for (int p = 0; p < P; ++p)
            if (part_lse[p * l_stride + lidx] > M) M = part_lse[p * l_stride + lidx];
        double* o = out + id * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (M == -INFINITY) {
            out_lse[lidx] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int p = 0; p < P; ++p) {
            const double L = part_lse[p * l_stride + lidx];
            if (L == -INFINITY) continue;
            const double w = exp(L - M);
            wsum += w;
            for (int d = 0; d < D; ++d) o[d] += w * part_O[p * o_stride + id * D + d];
        }
        for (int d = 0; d < D; ++d) o[d] /= wsum;
        out_lse[lidx] = M + log(wsum);
    }
    return 0;
}

/*
 * Backward pass: gradients of the attention output with respect to q, k and v,
 * given the upstream gradient dO ("RingAttention and Context Parallelism:
 * Mathematical Foundations", section 7, "RingAttention backward pass logic":
 * the scores of every block are recomputed and dQ, dK, dV accumulated).  The
 * oracle does not recompute blockwise: it materialises each query's full
 * softmax row and applies the chain rule to A = softmax(s) V, s = q K^T / sqrt(d):
 *
 *   P_j   = exp(s_j) / sum_j' exp(s_j')          (visible keys j only)
 *   dV_j += P_j dO_i                             (every query i that sees j)
 *   dP_j  = dO_i . v_j
 *   dS_j  = P_j (dP_j - sum_j' P_j' dP_j')       (softmax Jacobian)
 *   dQ_i  = scale sum_j dS_j k_j
 *   dK_j += scale dS_j q_i
 *
 * GQA: the q heads of a group add into their kv head's dK and dV.
 */

/* One query row's softmax-backward terms over its visible keys: fills P[j]
 * and dS[j] for the n keys listed (n == 0: nothing to fill). */
static void backward_row(const double* q_row, const double* do_row, const key_ref* keys, int64_t n, int D,
                         int dtype, double scale, double* P, double* dS) {
    if (n == 0) return;
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q_row[d] * load_elem(keys[j].k, dtype, keys[j].off + d);
        P[j] = acc * scale;
        if (P[j] > m) m = P[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        P[j] = exp(P[j] - m);
        l += P[j];
    }
    double delta = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        P[j] /= l;
        double dp = 0.0;
        for (int d = 0; d < D; ++d) dp += do_row[d] * load_elem(keys[j].v, dtype, keys[j].off + d);
        dS[j] = dp;
        delta += P[j] * dp;
    }
    for (int64_t j = 0; j < n; ++j) {
        dS[j] = P[j] * (dS[j] - delta);
    }
}

/* Visible keys of query (b, i) with kv head hk: all, or pos[j] <= pos[i] when
 * causal (pos == NULL: stored order = sequence order).  Returns the count. */
static int64_t visible_keys(const void* k, const void* v, int b, int i, int hk, int S, int Hkv, int D,
                            int causal, const int32_t* pos, key_ref* keys) {
    int64_t n = 0;
    for (int j = 0; j < S; ++j) {
        if (causal && (pos ? pos[j] > pos[i] : j > i)) continue;
        keys[n].k = k;
        keys[n].v = v;
        keys[n].off = (((int64_t)b * S + j) * Hkv + hk) * D;
        ++n;
    }
    return n;
}

/*
 * Full gradients.  q, dout [B,S,Hq,D]; k, v [B,S,Hkv,D] in `dtype` (dout in the
 * same storage type).  dq [B,S,Hq,D], dk / dv [B,S,Hkv,D] double.
 * Parallel over (b, kv head): each thread owns its group's dK and dV.
 */
int oracle_attention_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype,
                         int B, int S, int Hq, int Hkv, int D, int causal, const int32_t* pos,
                         double* dq, double* dk, double* dv) {
    if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || D > 512 || Hq % Hkv) return -1;
    const int group = Hq / Hkv;
    const double scale = 1.0 / sqrt((double)D);
    memset(dk, 0, sizeof(double) * (size_t)B * S * Hkv * D);
    memset(dv, 0, sizeof(double) * (size_t)B * S * Hkv * D);
#pragma omp parallel
    {
        double q_row[512], do_row[512];
        double* P = (double*)malloc(sizeof(double) * (size_t)S);
        double* dS = (double*)malloc(sizeof(double) * (size_t)S);
        key_ref* keys = (key_ref*)malloc(sizeof(key_ref) * (size_t)S);
#pragma omp for schedule(dynamic, 1)
        for (int64_t g = 0; g < (int64_t)B * Hkv; ++g) {
            const int b = (int)(g / Hkv), hk = (int)(g % Hkv);
            for (int h = hk * group; h < (hk + 1) * group; ++h) {
                for (int i = 0; i < S; ++i) {
                    const int64_t qoff = (((int64_t)b * S + i) * Hq + h) * D;
                    for (int d = 0; d < D; ++d) {
                        q_row[d] = load_elem(q, dtype, qoff + d);
                        do_row[d] = load_elem(dout, dtype, qoff + d);
                    }
                    const int64_t n = visible_keys(k, v, b, i, hk, S, Hkv, D, causal, pos, keys);
                    backward_row(q_row, do_row, keys, n, D, dtype, scale, P, dS);
                    double* dqi = dq + qoff;
                    for (int d = 0; d < D; ++d) dqi[d] = 0.0;
                    for (int64_t jj = 0; jj < n; ++jj) {
                        const int64_t koff = keys[jj].off;  /* the key's row in k, v, dk, dv */
                        for (int d = 0; d < D; ++d) {
                            dqi[d] += scale * dS[jj] * load_elem(k, dtype, koff + d);
                            dk[koff + d] += scale * dS[jj] * q_row[d];
                            dv[koff + d] += P[jj] * do_row[d];
                        }
                    }
                }
            }
        }
        free(P);
        free(dS);
        free(keys);
    }
    return 0;
}

/*
 * Selected rows of the same gradients, each computed on its own:
 *   qsel ids (b*S + i)*Hq + h   -> dq_rows [n_q, D]
 *   ksel ids (b*S + j)*Hkv + hk -> dk_rows, dv_rows [n_k, D]; a key's gradient
 *   sums over every query (of every q head of the group) that sees it, each
 *   with its full softmax row.
 */
int oracle_attention_bwd_rows(const void* q, const void* k, const void* v, const void* dout, int dtype,
                              int B, int S, int Hq, int Hkv, int D, int causal, const int32_t* pos,
                              const int64_t* qsel, int64_t n_q, double* dq_rows,
                              const int64_t* ksel, int64_t n_k, double* dk_rows, double* dv_rows) {
    if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || D > 512 || Hq % Hkv) return -1;
    const int group = Hq / Hkv;
    const double scale = 1.0 / sqrt((double)D);
    int bad = 0;
#pragma omp parallel
    {
        double q_row[512], do_row[512];
        double* P = (double*)malloc(sizeof(double) * (size_t)S);
        double* dS = (double*)malloc(sizeof(double) * (size_t)S);
        key_ref* keys = (key_ref*)malloc(sizeof(key_ref) * (size_t)S);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < n_q + n_k; ++t) {
            if (t < n_q) {
                const int64_t id = qsel[t];
                if (id < 0 || id >= (int64_t)B * S * Hq) { bad = 1; continue; }
                const int h = (int)(id % Hq);
                const int i = (int)((id / Hq) % S), b = (int)(id / Hq / S);
                for (int d = 0; d < D; ++d) {
                    q_row[d] = load_elem(q, dtype, id * D + d);
                    do_row[d] = load_elem(dout, dtype, id * D + d);
                }
                const int64_t n = visible_keys(k, v, b, i, h / group, S, Hkv, D, causal, pos, keys);
                backward_row(q_row, do_row, keys, n, D, dtype, scale, P, dS);
                double* o = dq_rows + t * D;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (int64_t jj = 0; jj < n; ++jj)
                    for (int d = 0; d < D; ++d) o[d] += scale * dS[jj] * load_elem(k, dtype, keys[jj].off + d);
            } else {
                const int64_t u = t - n_q, id = ksel[u];
                if (id < 0 || id >= (int64_t)B * S * Hkv) { bad = 1; continue; }
                const int hk = (int)(id % Hkv);
                const int j = (int)((id / Hkv) % S), b = (int)(id / Hkv / S);
                double* ok = dk_rows + u * D;
                double* ov = dv_rows + u * D;
                for (int d = 0; d < D; ++d) ok[d] = ov[d] = 0.0;
                for (int h = hk * group; h < (hk + 1) * group; ++h) {
                    for (int i = 0; i < S; ++i) {
                        if (causal && (pos ? pos[j] > pos[i] : j > i)) continue;
                        const int64_t qoff = (((int64_t)b * S + i) * Hq + h) * D;
                        for (int d = 0; d < D; ++d) {
                            q_row[d] = load_elem(q, dtype, qoff + d);
                            do_row[d] = load_elem(dout, dtype, qoff + d);
                        }
                        const int64_t n = visible_keys(k, v, b, i, hk, S, Hkv, D, causal, pos, keys);
                        backward_row(q_row, do_row, keys, n, D, dtype, scale, P, dS);
                        int64_t jj = 0;  /* the listed index of key j */
                        const int64_t koff = (((int64_t)b * S + j) * Hkv + hk) * D;
                        while (keys[jj].off != koff) ++jj;
                        for (int d = 0; d < D; ++d) {
                            ok[d] += scale * dS[jj] * q_row[d];
                            ov[d] += P[jj] * do_row[d];
                        }
                    }
                }
            }
        }
        free(P);
        free(dS);
        free(keys);
    }
    return bad ? -1 : 0;
}
