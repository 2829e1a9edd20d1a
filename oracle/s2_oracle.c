/*
 * CPU oracle for the S2 Reducer encode -> reduce -> decode path.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * statement of what the hot path computes. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the product path
 * never does. It shares no code with the CUDA library: the hash, the bitmap
 * rule, the sketch insertion and the median are written out again here.
 *
 * Source: "S2 Reducer: High-Performance Sparse Communication to Accelerate
 * Distributed Deep Learning" (Ge et al.), Section 3.1 (paragraphs
 * "Compressing Sparse Gradient", "Collecting Sparse-Sketch with AllReduce",
 * "Decompressing Sparse Gradient") and Algorithm 1 (Sparse-Sketch Reducer).
 *
 * Notation. The paper writes the gradient length as d, the number of sketch
 * rows as r and the buckets per row as c (or m). Here: n = gradient length,
 * d = rows, w = buckets per row, W = workers.
 *
 * Arithmetic: sketch buckets and decoded estimates are accumulated in double;
 * gradient values are read exactly (fp32 or bf16 widened to double). The
 * decoded value is rounded to float once, at the end.
 *
 * Readings of points the paper leaves open (each one a choice, not a quote):
 *  - bitmap unit: one bit per element (the paper sets one bit per block; an
 *    element is a block of size one); bit i is bit (i mod 32) of 32-bit word
 *    i/32, least significant bit first; bits at positions >= n are zero;
 *  - nonzero test: on the bit pattern with the sign bit cleared, so -0.0 is
 *    zero and subnormals are nonzero;
 *  - aggregation of bitmaps: bitwise OR (a bit of the aggregate is set iff it
 *    is set in some worker, which is how the paper reads the aggregated
 *    bitmap: the union of the workers' nonzero positions);
 *  - hash family (unspecified in the paper): the 32-bit MurmurHash3
 *    finalizer; row keys from the seed; bucket by multiply-shift; sign from
 *    the top bit;
 *  - median of an even number of estimates: mean of the two middle values;
 *  - the decoded quantity is the estimate of the SUM of the W gradients,
 *    times a caller-given scale.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- hash family ------------------------------------------------------- */

/* MurmurHash3 32-bit finalizer (Austin Appleby, public domain), mod 2^32. */
uint32_t s2o_fmix32(uint32_t x)
{
    x ^= x >> 16;
    x *= 0x85ebca6bu;
    x ^= x >> 13;
    x *= 0xc2b2ae35u;
    x ^= x >> 16;
    return x;
}

/* Per-row keys: bucket key kh_j and sign key ks_j, derived from the seed. */
void s2o_row_keys(uint32_t seed, uint32_t j, uint32_t *kh, uint32_t *ks)
{
    const uint32_t golden = 0x9E3779B9u;
    *kh = s2o_fmix32(seed ^ (uint32_t)(golden * (2u * j + 1u)));
    *ks = s2o_fmix32(seed ^ (uint32_t)(golden * (2u * j + 2u)));
}

/* Bucket hash h_j(i) in [0, w): the high 32 bits of fmix32(i ^ kh_j) * w. */
uint32_t s2o_bucket(uint32_t i, uint32_t kh, uint32_t w)
{
    uint64_t prod = (uint64_t)s2o_fmix32(i ^ kh) * (uint64_t)w;
    return (uint32_t)(prod >> 32);
}

/* Sign hash s_j(i) in {-1, +1}: -1 iff the top bit of fmix32(i ^ ks_j) is set. */
int s2o_sign(uint32_t i, uint32_t ks)
{
    return (s2o_fmix32(i ^ ks) >> 31) ? -1 : +1;
}

/* Buckets and signs of m given indices for rows 0..d-1: bucket[j*m + t], sign[j*m + t]. */
void s2o_hash(const uint32_t *idx, uint64_t m, uint32_t d, uint32_t w, uint32_t seed,
              uint32_t *bucket, int8_t *sign)
{
    for (uint32_t j = 0; j < d; ++j) {
        uint32_t kh, ks;
        s2o_row_keys(seed, j, &kh, &ks);
        for (uint64_t t = 0; t < m; ++t) {
            bucket[(uint64_t)j * m + t] = s2o_bucket(idx[t], kh, w);
            sign[(uint64_t)j * m + t] = (int8_t)s2o_sign(idx[t], ks);
        }
    }
}

/* ---- gradient element access ------------------------------------------- */

/* dtype codes: 0 = fp32, 1 = bf16 (raw 16-bit patterns). */
static int elem_is_nonzero(const void *g, int dt, uint64_t i)
{
    if (dt == 0) {
        uint32_t bits;
        memcpy(&bits, (const char *)g + 4 * i, 4);
        return (bits & 0x7fffffffu) != 0;
    } else {
        uint16_t bits;
        memcpy(&bits, (const char *)g + 2 * i, 2);
        return (bits & 0x7fffu) != 0;
    }
}

static double elem_value(const void *g, int dt, uint64_t i)
{
    if (dt == 0) {
        float v;
        memcpy(&v, (const char *)g + 4 * i, 4);
        return (double)v;
    } else {
        uint16_t bits;
        memcpy(&bits, (const char *)g + 2 * i, 2);
        uint32_t wide = (uint32_t)bits << 16;
        float v;
        memcpy(&v, &wide, 4);
        return (double)v;
    }
}

static int bit_is_set(const uint32_t *bitmap, uint64_t i)
{
    return (bitmap[i >> 5] >> (i & 31)) & 1u;
}

/* ---- compression (one worker) ------------------------------------------ */

/*
 * Section 3.1 "Compressing Sparse Gradient" and Algorithm 1, compression
 * phase, for one worker's gradient g of length n:
 *   first the bitmap: C[x] <- 1 if element x is nonzero;
 *   then for every i in Sparse(g) and every row j:
 *       S[j][h_j(i)] += s_j(i) * g(i).
 * Zeros are never inserted. A[j][b] accumulates |g(i)| over the same
 * insertions: it is not part of the method, it is the size of the bucket's
 * contributions, from which the tests derive their fp32 tolerance.
 * bitmap: ceil(n/32) words. S, A: d*w doubles, row-major [j][b].
 */
void s2o_encode(const void *grad, int dt, uint64_t n, uint32_t d, uint32_t w, uint32_t seed,
                uint32_t *bitmap, double *S, double *A)
{
    uint64_t nw = (n + 31) / 32;
    memset(bitmap, 0, nw * sizeof(uint32_t));
    memset(S, 0, (uint64_t)d * w * sizeof(double));
    if (A)
        memset(A, 0, (uint64_t)d * w * sizeof(double));

    for (uint64_t x = 0; x < n; ++x)
        if (elem_is_nonzero(grad, dt, x))
            bitmap[x >> 5] |= 1u << (x & 31);

    for (uint64_t i = 0; i < n; ++i) {
        if (!bit_is_set(bitmap, i))
            continue; /* i is not in Sparse(g) */
        double g = elem_value(grad, dt, i);
        for (uint32_t j = 0; j < d; ++j) {
            uint32_t kh, ks;
            s2o_row_keys(seed, j, &kh, &ks);
            uint32_t b = s2o_bucket((uint32_t)i, kh, w);
            int s = s2o_sign((uint32_t)i, ks);
            S[(uint64_t)j * w + b] += (double)s * g;
            if (A)
                A[(uint64_t)j * w + b] += g < 0 ? -g : g;
        }
    }
}

/* ---- aggregation (the AllReduce of S and C) ---------------------------- */

/*
 * Section 3.1 "Collecting Sparse-Sketch with AllReduce" and Algorithm 1,
 * AllReduce(S, C): the sketches of the W workers add element by element
 * (the sketch is linear: A^T sum_k g_k = sum_k A^T g_k); the bitmaps
 * aggregate so that a position is marked iff some worker marked it.
 * bitmaps: W x nw words, S_in/A_in: W x dw doubles, worker-major.
 */
void s2o_reduce(uint32_t W, uint64_t nw, uint64_t dw, const uint32_t *bitmaps, const double *S_in,
                const double *A_in, uint32_t *bitmap_out, double *S_out, double *A_out)
{
    for (uint64_t q = 0; q < nw; ++q) {
        uint32_t acc = 0;
        for (uint32_t k = 0; k < W; ++k)
            acc |= bitmaps[(uint64_t)k * nw + q];
        bitmap_out[q] = acc;
    }
    for (uint64_t x = 0; x < dw; ++x) {
        double s = 0.0, a = 0.0;
        for (uint32_t k = 0; k < W; ++k) {
            s += S_in[(uint64_t)k * dw + x];
            if (A_in)
                a += A_in[(uint64_t)k * dw + x];
        }
        S_out[x] = s;
        if (A_out)
            A_out[x] = a;
    }
}

/* ---- decompression ----------------------------------------------------- */

/* Median of e[0..d-1] (sorts e in place): the middle value for odd d, the
 * mean of the two middle values for even d. */
static double median_of(double *e, uint32_t d)
{
    for (uint32_t a = 1; a < d; ++a) { /* insertion sort */
        double v = e[a];
        uint32_t b = a;
        while (b > 0 && e[b - 1] > v) {
            e[b] = e[b - 1];
            --b;
        }
        e[b] = v;
    }
    if (d & 1u)
        return e[d / 2];
    return 0.5 * (e[d / 2 - 1] + e[d / 2]);
}

/*
 * Section 3.1 "Decompressing Sparse Gradient" and Algorithm 1, decompression
 * phase, for one recovered index i: estimates[j] = s_j(i) * S[j][h_j(i)] for
 * every row j, g^(i) = median(estimates). Also returns the tolerance scale
 * max_j A[j][h_j(i)] through *amax (0 if A is NULL).
 */
static double query(const double *S, const double *A, uint32_t i, uint32_t d, uint32_t w,
                    uint32_t seed, double *amax)
{
    double e[64];
    double am = 0.0;
    for (uint32_t j = 0; j < d; ++j) {
        uint32_t kh, ks;
        s2o_row_keys(seed, j, &kh, &ks);
        uint32_t b = s2o_bucket(i, kh, w);
        int s = s2o_sign(i, ks);
        e[j] = (double)s * S[(uint64_t)j * w + b];
        if (A && A[(uint64_t)j * w + b] > am)
            am = A[(uint64_t)j * w + b];
    }
    if (amax)
        *amax = am;
    return median_of(e, d);
}

/*
 * Dense output: recover Sparse(g) from the aggregated bitmap, query every
 * recovered index, and write +0.0f at every other position.
 * out: n floats. amax (optional): n doubles, 0 at unset positions.
 */
void s2o_decode_dense(const uint32_t *bitmap, const double *S, const double *A, uint64_t n,
                      uint32_t d, uint32_t w, uint32_t seed, double scale, float *out, double *amax)
{
    for (uint64_t i = 0; i < n; ++i) {
        if (!bit_is_set(bitmap, i)) {
            out[i] = 0.0f;
            if (amax)
                amax[i] = 0.0;
            continue;
        }
        double am;
        double med = query(S, A, (uint32_t)i, d, w, seed, &am);
        out[i] = (float)(scale * med);
        if (amax)
            amax[i] = am;
    }
}

/*
 * Compacted output: the recovered indices in ascending order with their
 * estimates. Entry t of the output is the t-th set bit of the bitmap.
 * Entries at t >= capacity are not written. Returns the number of set bits.
 */
uint64_t s2o_decode_compact(const uint32_t *bitmap, const double *S, const double *A, uint64_t n,
                            uint32_t d, uint32_t w, uint32_t seed, double scale, uint32_t *idx_out,
                            float *val_out, double *amax_out, uint64_t capacity)
{
    uint64_t t = 0;
    for (uint64_t i = 0; i < n; ++i) {
        if (!bit_is_set(bitmap, i))
            continue;
        if (t < capacity) {
            double am;
            double med = query(S, A, (uint32_t)i, d, w, seed, &am);
            idx_out[t] = (uint32_t)i;
            val_out[t] = (float)(scale * med);
            if (amax_out)
                amax_out[t] = am;
        }
        ++t;
    }
    return t;
}

/* ---- block-granular bitmap ----------------------------------------------- */

/*
 * Section 3.1 "Compressing Sparse Gradient" in the paper's own granularity:
 * one bitmap bit per block of `block` consecutive positions (an embedding
 * row, a gradient block); block x is marked iff it holds a nonzero. The
 * sketch is the same as s2o_encode's: only nonzero positions are inserted.
 * bitmap: ceil(ceil(n/block)/32) words.
 */
void s2o_encode_blocks(const void *grad, int dt, uint64_t n, uint64_t block, uint32_t d, uint32_t w,
                       uint32_t seed, uint32_t *bitmap, double *S, double *A)
{
    uint64_t nb = (n + block - 1) / block;
    uint64_t nw = (n + 31) / 32;
    uint32_t *elem = (uint32_t *)calloc(nw ? nw : 1, sizeof(uint32_t));
    s2o_encode(grad, dt, n, d, w, seed, elem, S, A);
    memset(bitmap, 0, ((nb + 31) / 32) * sizeof(uint32_t));
    for (uint64_t x = 0; x < n; ++x)
        if (bit_is_set(elem, x))
            bitmap[(x / block) >> 5] |= 1u << ((x / block) & 31);
    free(elem);
}

/*
 * Decompression with a block bitmap: Sparse(g) is every position of every
 * marked block (zeros inside a marked block included); each is queried as in
 * s2o_decode_dense, every other position gets +0.0f.
 */
void s2o_decode_dense_blocks(const uint32_t *bitmap, const double *S, const double *A, uint64_t n,
                             uint64_t block, uint32_t d, uint32_t w, uint32_t seed, double scale,
                             float *out, double *amax)
{
    for (uint64_t i = 0; i < n; ++i) {
        if (!bit_is_set(bitmap, i / block)) {
            out[i] = 0.0f;
            if (amax)
                amax[i] = 0.0;
            continue;
        }
        double am;
        double med = query(S, A, (uint32_t)i, d, w, seed, &am);
        out[i] = (float)(scale * med);
        if (amax)
            amax[i] = am;
    }
}

/* ---- block-wise Top-K sparsification with error feedback ------------------ */

/*
 * Squared l2 norm of one block, as defined: the sum of the squares of its
 * elements, accumulated in double precision in index order (each square of
 * a float is exact in double). The pages fix no precision for the norm, so
 * the plain definition is taken.
 */
static double block_norm2(const float *a, uint64_t len)
{
    double s = 0.0;
    for (uint64_t j = 0; j < len; ++j)
        s += (double)a[j] * (double)a[j];
    return s;
}

/*
 * The split of the error-feedback step for one worker, given which blocks
 * are kept ("S2 Reducer", Appendix A.2, proof of Theorem 2: U(g) is what is
 * sent and e_{t+1} = g_t - U(g_t) is carried):
 *   acc = grad + residual (one float addition per element);
 *   sparse = acc on kept blocks, 0 elsewhere; residual = acc on the other
 *   blocks, 0 on kept ones. keep: nb bytes, nonzero = kept.
 */
void s2o_block_split(const float *grad, float *residual, uint64_t n, uint64_t block, const uint8_t *keep,
                     float *sparse)
{
    for (uint64_t i = 0; i < n; ++i) {
        float acc = grad[i] + residual[i];
        int kept = keep[i / block] != 0;
        sparse[i] = kept ? acc : 0.0f;
        residual[i] = kept ? 0.0f : acc;
    }
}

/*
 * Block-wise Top-K with error feedback for one worker ("S2 Reducer", Section
 * 2.2 "Sparse Gradient & AllGather" for the sparsifier; Appendix A.2 for the
 * error sequence):
 *   acc = grad + residual (float additions);
 *   view acc as blocks of `block` elements (the last one may be shorter) and
 *   take each block's squared l2 norm (block_norm2, double precision);
 *   keep the K blocks with the largest norms, ties to the lower block index;
 *   split acc into the sent part and the new residual (s2o_block_split).
 * norms (optional): nb doubles. keep (optional): nb bytes, 1 for kept blocks.
 */
void s2o_block_topk(const float *grad, float *residual, uint64_t n, uint64_t block, uint64_t K, float *sparse,
                    double *norms_out, uint8_t *keep_out)
{
    uint64_t nb = (n + block - 1) / block;
    double *nrm = (double *)malloc((nb ? nb : 1) * sizeof(double));
    uint8_t *keep = (uint8_t *)calloc(nb ? nb : 1, 1);
    float *acc = (float *)malloc((block ? block : 1) * sizeof(float));
    for (uint64_t x = 0; x < nb; ++x) {
        uint64_t len = (x + 1) * block <= n ? block : n - x * block;
        for (uint64_t j = 0; j < len; ++j)
            acc[j] = grad[x * block + j] + residual[x * block + j];
        nrm[x] = block_norm2(acc, len);
    }
    /* K rounds of "largest remaining norm, lowest index among equals" */
    for (uint64_t r = 0; r < K && r < nb; ++r) {
        uint64_t best = nb;
        for (uint64_t x = 0; x < nb; ++x)
            if (!keep[x] && (best == nb || nrm[x] > nrm[best]))
                best = x;
        keep[best] = 1;
    }
    s2o_block_split(grad, residual, n, block, keep, sparse);
    if (norms_out)
        memcpy(norms_out, nrm, nb * sizeof(double));
    if (keep_out)
        memcpy(keep_out, keep, nb);
    free(acc);
    free(nrm);
    free(keep);
}

/* ---- sparse AllGather baseline -------------------------------------------- */

/*
 * Section 2.2 "Sparse Gradient & AllGather" / Figure 1(b): a worker's message
 * is the list of its nonzero indices and values (ascending); entries at
 * t >= capacity are not written. Returns the number of nonzeros.
 */
uint64_t s2o_sparse_list(const float *grad, uint64_t n, uint32_t *idx, float *val, uint64_t capacity)
{
    uint64_t t = 0;
    for (uint64_t i = 0; i < n; ++i) {
        if (!elem_is_nonzero(grad, 0, i))
            continue;
        if (t < capacity) {
            idx[t] = (uint32_t)i;
            val[t] = grad[i];
        }
        ++t;
    }
    return t;
}

/* The gathered lists added up: out[i] = sum over workers of their value at i
 * (double accumulation, rounded once). grads: W x n. */
void s2o_exact_sum(const float *grads, uint32_t W, uint64_t n, float *out)
{
    for (uint64_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (uint32_t k = 0; k < W; ++k)
            s += (double)grads[(uint64_t)k * n + i];
        out[i] = (float)s;
    }
}
