/*
 * oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, float64 CPU statement of the mixed-batch multi-adapter LoRA
 * linear layer and its LoRA backward.  Only tests/, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA library; it is written from the definitions below
 * and nothing else.
 *
 * What it computes (row-vector notation; tokens are rows):
 *
 *   x  [T,K]  layer input              Wt [N,K]  frozen weight, stored as W^T
 *   A_a       adapter a's down factor, stored as an [r_a,K] row-major block
 *   B_a       adapter a's up factor,   stored as an [r_a,N] row-major block
 *   s_a       adapter a's scale
 *
 *   LoRA linear layer -- "DeltaServe: Host-Agnostic Co-Serving of Inference
 *   and Fine-Tuning for LLMs", section 2.2 (W_eff = W + BA, only A and B are
 *   trained) and "MOLT: A Fine-Grained GPU Memory Sharing System for LLM
 *   Serving with Opportunistic Fine-Tuning", section 2.1 (h(x) = Wx + BAx):
 *
 *     u[t,j] = sum_k x[t,k] * A_a[j,k]                 (the shrink, "xA")
 *     y[t,n] = sum_k x[t,k] * Wt[n,k] + s_a * sum_j u[t,j] * B_a[j,n]
 *
 *   Multi-LoRA batching -- DeltaServe section 2.2: every token in one batch
 *   uses the adapter of the segment that holds it; adapter id -1 means the
 *   base projection alone.  A fine-tuning sample is an ordinary batch entry
 *   routed to its adapter -- DeltaServe section 3.2 ("Mixed forward batch").
 *
 *   LoRA backward for the fine-tuning segments -- DeltaServe section 3.2
 *   ("Backward subprocess": the loss and LoRA gradients are computed from the
 *   captured activations, unsaved intermediates recomputed).  The pages print
 *   no gradient formula; the ones below are the chain rule for a loss whose
 *   gradient with respect to y is dY, with W frozen:
 *
 *     v[t,j]     = sum_n dY[t,n] * B_a[j,n]                      (dY B^T)
 *     dX[t,k]    = sum_n dY[t,n] * Wt[n,k] + s_a * sum_j v[t,j] * A_a[j,k]
 *     dB_a[j,n] += s_a * u[t,j] * dY[t,n]       summed over t in a's segments
 *     dA_a[j,k] += s_a * v[t,j] * x[t,k]        summed over t in a's segments
 *
 *   dA_a and dB_a are laid out like A_a and B_a (same element offsets).
 *   Several fine-tuning segments on one adapter add their contributions (the
 *   gradient of the summed loss), in increasing segment-start order.
 *
 * Inputs arrive as float32 arrays whose values are exact in the layer's
 * element type (bf16-rounded for bf16 layers); every product and sum here is
 * carried out in double.  Loops run in the order of the sums above; OpenMP
 * only splits independent output elements between threads.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAX_RANK 128

/* segment table entries: {start, len, adapter_id, is_train}, 4 x int32 each */
#define SEG_START(s, i) ((s)[4 * (i) + 0])
#define SEG_LEN(s, i) ((s)[4 * (i) + 1])
#define SEG_ADAPTER(s, i) ((s)[4 * (i) + 2])
#define SEG_TRAIN(s, i) ((s)[4 * (i) + 3])

/* Which segment holds token t (or -1).  Linear scan: slow and obvious. */
static int32_t segment_of(const int32_t* segs, int32_t n_segs, int64_t t) {
    for (int32_t i = 0; i < n_segs; ++i) {
        if (t >= SEG_START(segs, i) && t < (int64_t)SEG_START(segs, i) + SEG_LEN(segs, i)) return i;
    }
    return -1;
}

/* u[j] = sum_k x[t,k] * A_a[j,k], j < r_a */
static void shrink_row(int64_t K, const float* xrow, const float* Aa, int32_t r, double* u) {
    for (int32_t j = 0; j < r; ++j) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += (double)xrow[k] * (double)Aa[(int64_t)j * K + k];
        u[j] = acc;
    }
}

/*
 * Forward over the tokens listed in rows[0..n_rows) (rows == NULL: all T
 * tokens in order).  y is [n_rows, N]; u (optional) is [n_rows, 128] and gets
 * the shrink values of each row (zero past r_a, and all zero for id -1).
 * Returns 0, or -1 if a token lies in no segment or an adapter id is out of
 * range.
 */
int oracle_forward(int64_t T, int64_t K, int64_t N, const float* x, const float* Wt, const float* A,
                   const float* B, const int64_t* a_off, const int64_t* b_off, const int32_t* rank,
                   const double* scale, int32_t n_adapters, const int32_t* segs, int32_t n_segs,
                   const int64_t* rows, int64_t n_rows, double* y, double* u) {
    if (rows == NULL) n_rows = T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < n_rows; ++i) {
        int64_t t = rows ? rows[i] : i;
        int32_t g = (t >= 0 && t < T) ? segment_of(segs, n_segs, t) : -1;
        if (g < 0) { bad = 1; continue; }
        int32_t a = SEG_ADAPTER(segs, g);
        if (a < -1 || a >= n_adapters) { bad = 1; continue; }
        const float* xrow = x + t * K;
        double ut[ORACLE_MAX_RANK];
        int32_t r = 0;
        if (a >= 0) {
            r = rank[a];
            shrink_row(K, xrow, A + a_off[a], r, ut);
        }
        if (u) {
            for (int32_t j = 0; j < ORACLE_MAX_RANK; ++j) u[i * ORACLE_MAX_RANK + j] = (j < r) ? ut[j] : 0.0;
        }
        for (int64_t n = 0; n < N; ++n) {
            double base = 0.0;
            for (int64_t k = 0; k < K; ++k) base += (double)xrow[k] * (double)Wt[n * K + k];
            double lora = 0.0;
            if (a >= 0) {
                const float* Ba = B + b_off[a];
                for (int32_t j = 0; j < r; ++j) lora += ut[j] * (double)Ba[(int64_t)j * N + n];
                lora *= scale[a];
            }
            y[i * N + n] = base + lora;
        }
    }
    return bad ? -1 : 0;
}

/* index of training segments in increasing start order */
static int32_t train_segments_sorted(const int32_t* segs, int32_t n_segs, int32_t* out) {
    int32_t m = 0;
    for (int32_t i = 0; i < n_segs; ++i)
        if (SEG_TRAIN(segs, i) && SEG_LEN(segs, i) > 0) out[m++] = i;
    for (int32_t p = 1; p < m; ++p) { /* insertion sort by start */
        int32_t v = out[p], q = p - 1;
        while (q >= 0 && SEG_START(segs, out[q]) > SEG_START(segs, v)) { out[q + 1] = out[q]; --q; }
        out[q + 1] = v;
    }
    return m;
}

/*
 * Backward for the fine-tuning segments.
 *   dX    [n_dx_rows, K]: dX rows of the listed tokens (dx_rows == NULL: every
 *         training token, in increasing segment-start order); may be NULL.
 *   dA,dB pool-shaped (same sizes and offsets as A and B).  For every adapter
 *         with a training segment, its block is overwritten (accumulate == 0)
 *         or added to (accumulate != 0); other blocks are left untouched.
 *   cols_b / cols_a (optional): compute only the listed columns n of dB_a
 *         (entries dB_a[j, n], all j) and columns k of dA_a; the other
 *         entries keep their initial values.  NULL = every column.
 *   u_saved (optional): the shrink activations u = xA captured by a forward
 *         pass, used for dB in place of recomputing them -- DeltaServe
 *         section 3.2 ("Backward subprocess": the LoRA gradients come from
 *         the activations captured during the mixed forward; only what was
 *         not captured is recomputed) and MOLT section 4.3 (flexible
 *         activation checkpointing: a saved activation is read back, an
 *         unsaved one recomputed).  Layout: for every training segment in
 *         increasing start order, a [len, r_a] row-major block (row p =
 *         token start + p).  Only dB reads u; v = dY B^T, dX and dA do not
 *         depend on it.  NULL = recompute u from x and A.
 * Returns 0, or -1 on a malformed table (a training segment on id -1 or out
 * of range, or a dX row that is not a training token).
 */
int oracle_backward(int64_t T, int64_t K, int64_t N, const float* x, const float* Wt, const float* A,
                    const float* B, const int64_t* a_off, const int64_t* b_off, const int32_t* rank,
                    const double* scale, int32_t n_adapters, const int32_t* segs, int32_t n_segs,
                    const float* dY, const int64_t* dx_rows, int64_t n_dx_rows, double* dX, double* dA,
                    double* dB, int accumulate, const int64_t* cols_b, int64_t n_cols_b, const int64_t* cols_a,
                    int64_t n_cols_a, const double* u_saved) {
    int32_t* tsegs = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_segs > 0 ? n_segs : 1));
    int32_t n_train = train_segments_sorted(segs, n_segs, tsegs);
    for (int32_t q = 0; q < n_train; ++q) {
        int32_t a = SEG_ADAPTER(segs, tsegs[q]);
        if (a < 0 || a >= n_adapters) { free(tsegs); return -1; }
    }

    /* ---- dX for the requested training rows ---- */
    int64_t n_all = 0;
    for (int32_t q = 0; q < n_train; ++q) n_all += SEG_LEN(segs, tsegs[q]);
    if (dX) {
        int64_t nr = dx_rows ? n_dx_rows : n_all;
        int64_t* rowlist = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nr > 0 ? nr : 1));
        if (dx_rows) {
            memcpy(rowlist, dx_rows, sizeof(int64_t) * (size_t)nr);
        } else {
            int64_t p = 0;
            for (int32_t q = 0; q < n_train; ++q)
                for (int32_t i = 0; i < SEG_LEN(segs, tsegs[q]); ++i) rowlist[p++] = SEG_START(segs, tsegs[q]) + i;
        }
        int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
        for (int64_t i = 0; i < nr; ++i) {
            int64_t t = rowlist[i];
            int32_t g = (t >= 0 && t < T) ? segment_of(segs, n_segs, t) : -1;
            if (g < 0 || !SEG_TRAIN(segs, g)) { bad = 1; continue; }
            int32_t a = SEG_ADAPTER(segs, g);
            int32_t r = rank[a];
            const float* dyrow = dY + t * N;
            const float* Ba = B + b_off[a];
            const float* Aa = A + a_off[a];
            double v[ORACLE_MAX_RANK];
            for (int32_t j = 0; j < r; ++j) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) acc += (double)dyrow[n] * (double)Ba[(int64_t)j * N + n];
                v[j] = acc;
            }
            for (int64_t k = 0; k < K; ++k) {
                double base = 0.0;
                for (int64_t n = 0; n < N; ++n) base += (double)dyrow[n] * (double)Wt[n * K + k];
                double lora = 0.0;
                for (int32_t j = 0; j < r; ++j) lora += v[j] * (double)Aa[(int64_t)j * K + k];
                dX[i * K + k] = base + scale[a] * lora;
            }
        }
        free(rowlist);
        if (bad) { free(tsegs); return -1; }
    }

    /* ---- dA, dB per training adapter ---- */
    if (dA || dB) {
        /* u and v of every training token, in increasing segment-start order */
        double* uu = (double*)calloc((size_t)(n_all > 0 ? n_all : 1) * ORACLE_MAX_RANK, sizeof(double));
        double* vv = (double*)calloc((size_t)(n_all > 0 ? n_all : 1) * ORACLE_MAX_RANK, sizeof(double));
        int64_t* tok = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_all > 0 ? n_all : 1));
        int32_t* tad = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_all > 0 ? n_all : 1));
        int64_t* uoff = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_all > 0 ? n_all : 1));
        int64_t p = 0, blk = 0;
        for (int32_t q = 0; q < n_train; ++q) {
            int32_t r_q = rank[SEG_ADAPTER(segs, tsegs[q])];
            for (int32_t i = 0; i < SEG_LEN(segs, tsegs[q]); ++i) {
                tok[p] = SEG_START(segs, tsegs[q]) + i;
                tad[p] = SEG_ADAPTER(segs, tsegs[q]);
                uoff[p] = blk + (int64_t)i * r_q;      /* row i of segment q's block of u_saved */
                ++p;
            }
            blk += (int64_t)SEG_LEN(segs, tsegs[q]) * r_q;
        }
#pragma omp parallel for schedule(dynamic, 4)
        for (int64_t i = 0; i < n_all; ++i) {
            int32_t a = tad[i];
            int32_t r = rank[a];
            if (u_saved) {
                for (int32_t j = 0; j < r; ++j) uu[i * ORACLE_MAX_RANK + j] = u_saved[uoff[i] + j];
            } else {
                shrink_row(K, x + tok[i] * K, A + a_off[a], r, uu + i * ORACLE_MAX_RANK);
            }
            const float* dyrow = dY + tok[i] * N;
            const float* Ba = B + b_off[a];
            for (int32_t j = 0; j < r; ++j) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) acc += (double)dyrow[n] * (double)Ba[(int64_t)j * N + n];
                vv[i * ORACLE_MAX_RANK + j] = acc;
            }
        }
        for (int32_t a = 0; a < n_adapters; ++a) {
            int used = 0;
            for (int64_t i = 0; i < n_all; ++i) used |= (tad[i] == a);
            if (!used) continue;
            int32_t r = rank[a];
            double s = scale[a];
            if (dB) {
                double* dBa = dB + b_off[a];
                int64_t nn = cols_b ? n_cols_b : N;
#pragma omp parallel for schedule(static)
                for (int64_t c = 0; c < nn; ++c) {
                    int64_t n = cols_b ? cols_b[c] : c;
                    for (int32_t j = 0; j < r; ++j) {
                        double acc = 0.0;
                        for (int64_t i = 0; i < n_all; ++i)
                            if (tad[i] == a) acc += s * uu[i * ORACLE_MAX_RANK + j] * (double)dY[tok[i] * N + n];
                        dBa[(int64_t)j * N + n] = (accumulate ? dBa[(int64_t)j * N + n] : 0.0) + acc;
                    }
                }
            }
            if (dA) {
                double* dAa = dA + a_off[a];
                int64_t nk = cols_a ? n_cols_a : K;
#pragma omp parallel for schedule(static)
                for (int64_t c = 0; c < nk; ++c) {
                    int64_t k = cols_a ? cols_a[c] : c;
                    for (int32_t j = 0; j < r; ++j) {
                        double acc = 0.0;
                        for (int64_t i = 0; i < n_all; ++i)
                            if (tad[i] == a) acc += s * vv[i * ORACLE_MAX_RANK + j] * (double)x[tok[i] * K + k];
                        dAa[(int64_t)j * K + k] = (accumulate ? dAa[(int64_t)j * K + k] : 0.0) + acc;
                    }
                }
            }
        }
        free(uu); free(vv); free(tok); free(tad); free(uoff);
    }
    free(tsegs);
    return 0;
}
