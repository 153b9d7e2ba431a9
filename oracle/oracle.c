/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the DLRM
 * embedding lookup + dot interaction path and its training backward.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares nothing with the
 * CUDA library: no headers, no helpers, no tables.
 *
 * Everything follows the page "DLRM For PyTorch":
 *   - §Model architecture: one embedding table per categorical feature; the
 *     bottom-MLP output and the embedding vectors enter the "dot interaction",
 *     whose output is concatenated with the bottom-MLP output.
 *   - §Command-line options: --embedding_type joint* (all tables in one joint
 *     buffer), --hash_indices (the index is reduced modulo the table size),
 *     --interaction_op cuda_dot|dot.
 *   - §Training process: embedding tables are stored in FP32.
 * Readings where the page is silent (all taken as the plainest choice):
 *   - pooling is a plain sum over the bag; an empty bag pools to zero;
 *   - the interaction keeps the strictly-lower triangle of Z Z^T, row-major,
 *     with vector 0 = dense features, vector t+1 = table t; output row is
 *     [dense (D) | triangle (F(F+1)/2) | zeros up to out_cols];
 *   - an out-of-range index with hashing off contributes nothing and sets
 *     status bit 1; with hashing on, idx := ((idx % N) + N) % N;
 *   - the optimizer is plain SGD, w := w - lr * g, g summed over every
 *     occurrence of the row in the batch (duplicates count each time).
 *
 *   - §Model architecture / --bottom_mlp_sizes 512,256,128: the bottom MLP is
 *     a chain of linear layers, each followed by a ReLU (the last included);
 *     under mixed precision (--amp, §Mixed precision training) its tensors
 *     are fp16 while the bias and the accumulation stay fp32 or wider.
 *
 * Arithmetic: every sum is accumulated in double and rounded once to the
 * output type (fp16 by round-to-nearest-even, converter below).  Build with
 * -ffp-contract=off so that x86 and Arm hosts give identical doubles.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_F16 1
#define OR_F64 2

#define OR_FLAG_HASH 1u
#define OR_STATUS_OOB 1u

#define OR_OK 0
#define OR_EINVAL 1

#define OR_SKIP_KEY 0xFFFFFFFFu

/* ---------------------------------------------------------------------- */
/* IEEE binary16 <-> binary64, written from the format's definition:        */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.                 */
/* ---------------------------------------------------------------------- */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* zero / subnormal */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) 2^(e-15) */
    return sign ? -v : v;
}

uint16_t oracle_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x))
        return (uint16_t)(sign | 0x7E00u);
    if (isinf(x))
        return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: units of 2^-24, ties to even (rint, default mode) */
        double q = rint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q);    /* q == 1024 is the smallest normal */
    }
    int e2;
    double m = frexp(a, &e2);                     /* a = m 2^e2, m in [0.5, 1) */
    double q = rint(ldexp(m, 11));                /* 11 significant bits: [1024, 2048] */
    int E = e2 - 1 + 15;
    if (q == 2048.0) {
        q = 1024.0;
        E += 1;
    }
    if (E >= 31)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)(E << 10) | (uint16_t)((int)q - 1024));
}

static double load_val(const void* base, int dt, int64_t i)
{
    if (dt == OR_F32) return (double)((const float*)base)[i];
    if (dt == OR_F16) return oracle_f16_to_f64(((const uint16_t*)base)[i]);
    return ((const double*)base)[i];
}

static void store_val(void* base, int dt, int64_t i, double v)
{
    if (dt == OR_F32) ((float*)base)[i] = (float)v;
    else if (dt == OR_F16) ((uint16_t*)base)[i] = oracle_f64_to_f16(v);
    else ((double*)base)[i] = v;
}

static int check_offsets(const int32_t* off, int64_t nbags, int64_t nnz)
{
    if (off[0] != 0 || (int64_t)off[nbags] != nnz) return 0;
    for (int64_t g = 0; g < nbags; ++g)
        if (off[g + 1] < off[g]) return 0;
    return 1;
}

/* Row of table t addressed by idx, after the hashing rule; -1 if skipped. */
static int64_t resolve_row(const int64_t* row_base, int t, int64_t idx, unsigned flags,
                           uint32_t* status)
{
    int64_t n = row_base[t + 1] - row_base[t];
    if (flags & OR_FLAG_HASH) {
        if (n <= 0) { *status |= OR_STATUS_OOB; return -1; }
        idx = ((idx % n) + n) % n;           /* non-negative remainder by the table size */
    } else if (idx < 0 || idx >= n) {
        *status |= OR_STATUS_OOB;
        return -1;
    }
    return row_base[t] + idx;
}

/* ---------------------------------------------------------------------- */
/* Embedding lookup with sum pooling ("DLRM For PyTorch", §Model            */
/* architecture; joint table layout per --embedding_type joint*).           */
/*   pooled[b][t][:] = sum over p in bag (t,b) of table[row(t, idx[p])][:]  */
/* ---------------------------------------------------------------------- */
int oracle_emb_fwd(const void* tables, int dt, const int64_t* row_base, int F, int D, int B,
                   const int32_t* indices, const int32_t* offsets, int64_t nnz,
                   void* pooled, unsigned flags, uint32_t* status)
{
    if (F < 1 || D < 1 || B < 0 || !row_base || !offsets || !status) return OR_EINVAL;
    if (!check_offsets(offsets, (int64_t)F * B, nnz)) return OR_EINVAL;
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    for (int t = 0; t < F; ++t) {
        for (int b = 0; b < B; ++b) {
            for (int k = 0; k < D; ++k) acc[k] = 0.0;
            int64_t g = (int64_t)t * B + b;
            for (int64_t p = offsets[g]; p < offsets[g + 1]; ++p) {
                int64_t row = resolve_row(row_base, t, indices[p], flags, status);
                if (row < 0) continue;
                for (int k = 0; k < D; ++k) acc[k] += load_val(tables, dt, row * D + k);
            }
            int64_t o = ((int64_t)b * F + t) * D;
            for (int k = 0; k < D; ++k) store_val(pooled, dt, o + k, acc[k]);
        }
    }
    free(acc);
    return OR_OK;
}

/* Vector i of sample b's Z: 0 = dense[b], t+1 = pooled[b][t]. */
static double z_at(const void* dense, const void* pooled, int dt, int F, int D, int b, int i, int k)
{
    if (i == 0) return load_val(dense, dt, (int64_t)b * D + k);
    return load_val(pooled, dt, ((int64_t)b * F + (i - 1)) * D + k);
}

/* Full Gram matrix Z Z^T of one sample, (F+1)^2 doubles (symmetry pin). */
int oracle_gram(const void* dense, const void* pooled, int dt, int F, int D, int b, double* gram)
{
    for (int i = 0; i <= F; ++i)
        for (int j = 0; j <= F; ++j) {
            double s = 0.0;
            for (int k = 0; k < D; ++k)
                s += z_at(dense, pooled, dt, F, D, b, i, k) * z_at(dense, pooled, dt, F, D, b, j, k);
            gram[i * (F + 1) + j] = s;
        }
    return OR_OK;
}

/* ---------------------------------------------------------------------- */
/* Dot interaction ("DLRM For PyTorch", §Model architecture and             */
/* --interaction_op): pairwise dot products among the F+1 vectors, strict   */
/* lower triangle in row-major order, concatenated after the dense vector.  */
/*   out[b] = [ z_0 | z_i . z_j for i = 1..F, j = 0..i-1 | 0 ... ]          */
/* ---------------------------------------------------------------------- */
int oracle_interact_fwd(const void* dense, const void* pooled, int dt, int F, int D, int B,
                        void* out, int out_cols)
{
    int W = D + F * (F + 1) / 2;
    if (F < 1 || D < 1 || B < 0 || out_cols < W) return OR_EINVAL;
    for (int b = 0; b < B; ++b) {
        int64_t o = (int64_t)b * out_cols;
        for (int k = 0; k < D; ++k)
            store_val(out, dt, o + k, z_at(dense, pooled, dt, F, D, b, 0, k));
        int col = D;
        for (int i = 1; i <= F; ++i)
            for (int j = 0; j < i; ++j) {
                double s = 0.0;
                for (int k = 0; k < D; ++k)
                    s += z_at(dense, pooled, dt, F, D, b, i, k) * z_at(dense, pooled, dt, F, D, b, j, k);
                store_val(out, dt, o + col, s);
                ++col;
            }
        for (; col < out_cols; ++col) store_val(out, dt, o + col, 0.0);
    }
    return OR_OK;
}

/* ---------------------------------------------------------------------- */
/* Interaction backward.  With G the upstream gradient of one output row,   */
/* out[D + i(i-1)/2 + j] = z_i . z_j (i > j) gives                          */
/*   dL/dz_i = sum_{j<i} G[D + i(i-1)/2 + j] z_j + sum_{j>i} G[D + j(j-1)/2 + i] z_j */
/* and the copied dense block adds G[0..D) to dL/dz_0.  Pad columns carry   */
/* no dependence and are ignored.                                          */
/* grad arrays are float unless dt == F64, in which case they are double.   */
/* ---------------------------------------------------------------------- */
int oracle_interact_bwd(const void* grad_out, const void* dense, const void* pooled, int dt,
                        int F, int D, int B, int out_cols, void* grad_dense, void* grad_pooled)
{
    int W = D + F * (F + 1) / 2;
    if (F < 1 || D < 1 || B < 0 || out_cols < W) return OR_EINVAL;
    int gdt = (dt == OR_F64) ? OR_F64 : OR_F32;
    for (int b = 0; b < B; ++b) {
        int64_t o = (int64_t)b * out_cols;
        for (int i = 0; i <= F; ++i) {
            for (int k = 0; k < D; ++k) {
                double s = 0.0;
                for (int j = 0; j <= F; ++j) {
                    if (j == i) continue;
                    int hi = i > j ? i : j, lo = i > j ? j : i;
                    double g = load_val(grad_out, gdt, o + D + hi * (hi - 1) / 2 + lo);
                    s += g * z_at(dense, pooled, dt, F, D, b, j, k);
                }
                if (i == 0) {
                    s += load_val(grad_out, gdt, o + k);
                    store_val(grad_dense, gdt, (int64_t)b * D + k, s);
                } else {
                    store_val(grad_pooled, gdt, ((int64_t)b * F + (i - 1)) * D + k, s);
                }
            }
        }
    }
    return OR_OK;
}

/* Stable merge sort of (key, val) pairs by key. */
static void merge_sort_pairs(uint32_t* k, uint32_t* v, uint32_t* tk, uint32_t* tv, int64_t n)
{
    for (int64_t width = 1; width < n; width *= 2) {
        for (int64_t lo = 0; lo < n; lo += 2 * width) {
            int64_t mid = lo + width < n ? lo + width : n;
            int64_t hi = lo + 2 * width < n ? lo + 2 * width : n;
            int64_t a = lo, b = mid, o = lo;
            while (a < mid && b < hi) {
                if (k[b] < k[a]) { tk[o] = k[b]; tv[o] = v[b]; ++b; }
                else { tk[o] = k[a]; tv[o] = v[a]; ++a; }    /* ties keep the left one first */
                ++o;
            }
            while (a < mid) { tk[o] = k[a]; tv[o] = v[a]; ++a; ++o; }
            while (b < hi) { tk[o] = k[b]; tv[o] = v[b]; ++b; ++o; }
        }
        memcpy(k, tk, sizeof(uint32_t) * (size_t)n);
        memcpy(v, tv, sizeof(uint32_t) * (size_t)n);
    }
}

/* ---------------------------------------------------------------------- */
/* Sparse embedding gradient + SGD (the gradient of the sum pooling above,  */
/* applied with plain SGD to the FP32 tables of §Training process).         */
/* For each position p of bag (t,b): key = global row, val = b*F + t (the  */
/* row of grad_pooled).  Pairs are stably sorted by key, then each run of   */
/* equal keys is summed in double in ascending position order and applied: */
/*   w := (float)((double)w - (double)lr * g)                               */
/* Skipped indices get key 0xFFFFFFFF and sort last.  If sorted_keys /       */
/* sorted_vals are non-null they receive the sorted pairs.                  */
/* ---------------------------------------------------------------------- */
int oracle_emb_bwd_sgd(float* tables, const int64_t* row_base, int F, int D, int B,
                       const int32_t* indices, const int32_t* offsets, int64_t nnz,
                       const float* grad_pooled, float lr, unsigned flags, uint32_t* status,
                       uint32_t* sorted_keys, uint32_t* sorted_vals)
{
    if (F < 1 || D < 1 || B < 0 || !row_base || !offsets || !status) return OR_EINVAL;
    if (!check_offsets(offsets, (int64_t)F * B, nnz)) return OR_EINVAL;
    size_t n = (size_t)nnz;
    uint32_t* key = (uint32_t*)malloc(sizeof(uint32_t) * (n + 1));
    uint32_t* val = (uint32_t*)malloc(sizeof(uint32_t) * (n + 1));
    uint32_t* tk = (uint32_t*)malloc(sizeof(uint32_t) * (n + 1));
    uint32_t* tv = (uint32_t*)malloc(sizeof(uint32_t) * (n + 1));
    double* g = (double*)malloc(sizeof(double) * (size_t)D);
    for (int t = 0; t < F; ++t)
        for (int b = 0; b < B; ++b) {
            int64_t bag = (int64_t)t * B + b;
            for (int64_t p = offsets[bag]; p < offsets[bag + 1]; ++p) {
                int64_t row = resolve_row(row_base, t, indices[p], flags, status);
                key[p] = row < 0 ? OR_SKIP_KEY : (uint32_t)row;
                val[p] = (uint32_t)((int64_t)b * F + t);
            }
        }
    merge_sort_pairs(key, val, tk, tv, nnz);
    if (sorted_keys) memcpy(sorted_keys, key, sizeof(uint32_t) * n);
    if (sorted_vals) memcpy(sorted_vals, val, sizeof(uint32_t) * n);
    int64_t p = 0;
    while (p < nnz && key[p] != OR_SKIP_KEY) {
        int64_t q = p;
        for (int k = 0; k < D; ++k) g[k] = 0.0;
        while (q < nnz && key[q] == key[p]) {
            for (int k = 0; k < D; ++k) g[k] += (double)grad_pooled[(int64_t)val[q] * D + k];
            ++q;
        }
        float* w = tables + (int64_t)key[p] * D;
        for (int k = 0; k < D; ++k) w[k] = (float)((double)w[k] - (double)lr * g[k]);
        p = q;
    }
    free(key); free(val); free(tk); free(tv); free(g);
    return OR_OK;
}

/* Bottom MLP forward ("DLRM For PyTorch", §Model architecture): for layers
 * l = 0..L-1, h_{l+1}[j] = max(0, sum_k W_l[j][k] h_l[k] + b_l[j]), h_0 = x.
 * dims[0..L] are the widths; W_all holds the layers' [dims[l+1]][dims[l]]
 * weights one after another, b_all their biases.  Sums in double.  With
 * half_io, x, the weights and every layer's output are rounded to binary16
 * (the tensors of the mixed-precision recipe; bias and accumulation wider).
 * out: double [B][dims[L]]. */
int oracle_mlp_fwd(const float* x, int B, int L, const int* dims, const float* W_all, const float* b_all,
                   int half_io, double* out)
{
    if (B < 0 || L < 1) return OR_EINVAL;
    int wmax = 0;
    for (int l = 0; l <= L; ++l) {
        if (dims[l] < 1) return OR_EINVAL;
        if (dims[l] > wmax) wmax = dims[l];
    }
    double* h = (double*)malloc(sizeof(double) * wmax);
    double* nh = (double*)malloc(sizeof(double) * wmax);
    if (!h || !nh) { free(h); free(nh); return OR_EINVAL; }
    for (int b = 0; b < B; ++b) {
        for (int k = 0; k < dims[0]; ++k) {
            double v = (double)x[(int64_t)b * dims[0] + k];
            h[k] = half_io ? oracle_f16_to_f64(oracle_f64_to_f16(v)) : v;
        }
        int64_t woff = 0, boff = 0;
        for (int l = 0; l < L; ++l) {
            const int K = dims[l], N = dims[l + 1];
            for (int j = 0; j < N; ++j) {
                double acc = 0.0;
                for (int k = 0; k < K; ++k) {
                    double w = (double)W_all[woff + (int64_t)j * K + k];
                    if (half_io) w = oracle_f16_to_f64(oracle_f64_to_f16(w));
                    acc += w * h[k];
                }
                acc += (double)b_all[boff + j];
                if (acc < 0.0) acc = 0.0;
                nh[j] = half_io ? oracle_f16_to_f64(oracle_f64_to_f16(acc)) : acc;
            }
            for (int j = 0; j < N; ++j) h[j] = nh[j];
            woff += (int64_t)N * K;
            boff += N;
        }
        for (int j = 0; j < dims[L]; ++j) out[(int64_t)b * dims[L] + j] = h[j];
    }
    free(h);
    free(nh);
    return OR_OK;
}

/* Rounds n doubles to binary16 (round to nearest, ties to even) with the
 * converter above: the single rounding of the mixed-precision tensors
 * ("DLRM For PyTorch", §Mixed precision training). */
void oracle_round_f16(const double* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_f16(x[i]);
}
