/*
 * s2.h -- C ABI of libs2, the GB300 (sm_103a) S2 Reducer hot path.
 *
 * The operations follow "S2 Reducer: High-Performance Sparse Communication
 * to Accelerate Distributed Deep Learning" (Ge et al.), Section 3.1 and
 * Algorithm 1 (Sparse-Sketch Reducer):
 *   encode  -- each worker marks its nonzero positions in a bitmap and adds
 *              every nonzero into a d x w count-sketch (the compression phase);
 *   reduce  -- the workers' sketches are summed and their bitmaps OR-ed (the
 *              AllReduce(S, C) step; here all workers live on one GPU);
 *   decode  -- every position set in the aggregated bitmap is queried as the
 *              median over the rows of its signed buckets (the decompression
 *              phase), giving a dense vector or an (index, value) list.
 *
 * Notation: n = gradient length, d = sketch rows, w = buckets per row,
 * W = workers. (The paper writes d for the length, r for the rows and c or m
 * for the buckets.)
 *
 * Common conventions
 *  - Every pointer argument is DEVICE memory owned by the caller, except the
 *    host_* arguments of s2_pipeline_dense_host. The library allocates
 *    nothing and keeps no pointer after a call returns.
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream) and never synchronises the host. Validation errors are returned
 *    before anything is launched; a failed launch returns S2_ERR_CUDA.
 *  - Outputs are overwritten, never accumulated into. Outputs must not
 *    overlap inputs (S2_ERR_INVALID_ARG).
 *  - Gradient, bitmap, sketch and dense-output base pointers must be 16-byte
 *    aligned (S2_ERR_ALIGNMENT). Other arrays need their natural alignment.
 *  - Positions are 32-bit: n must be below 2^32 (S2_ERR_UNSUPPORTED).
 *  - Bitmap layout: position i is bit (i % 32) of 32-bit word i / 32, least
 *    significant bit first; nw = ceil(n / 32) words; bits at positions >= n
 *    are written as 0.
 *  - Sketch layout: float32, row-major [d][w]; batched arrays are
 *    worker-major: grad[W][n], bitmaps[W][nw], sketches[W][d][w].
 *  - A position is nonzero iff its bit pattern without the sign bit is not
 *    zero: -0.0 counts as zero, subnormals count as nonzero. NaN and Inf
 *    inputs are outside the contract.
 *  - Hash family (the paper leaves it open): with fmix32 the 32-bit
 *    MurmurHash3 finalizer and G = 0x9E3779B9, row j has keys
 *    kh_j = fmix32(seed ^ G*(2j+1)) and ks_j = fmix32(seed ^ G*(2j+2))
 *    (mod 2^32); bucket h_j(i) = (fmix32(i ^ kh_j) * w) >> 32 computed in
 *    64 bits; sign s_j(i) = -1 if fmix32(i ^ ks_j) >= 2^31, else +1.
 *  - The library is stateless and thread-safe; no exception crosses the ABI.
 */
#ifndef S2_H
#define S2_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define S2_API __attribute__((visibility("default")))
#else
#define S2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL selects the legacy default stream. */
typedef struct CUstream_st *s2_stream_t;

typedef enum {
    S2_OK = 0,
    S2_ERR_INVALID_ARG = 1, /* null pointer, bad d/w/W, overlapping buffers, small workspace */
    S2_ERR_ALIGNMENT = 2,   /* a pointer misses its required alignment */
    S2_ERR_UNSUPPORTED = 3, /* n >= 2^32 or another size the library does not handle */
    S2_ERR_CUDA = 4         /* a CUDA runtime call or kernel launch failed */
} s2_status;

typedef enum {
    S2_F32 = 0, /* IEEE float32 gradient */
    S2_BF16 = 1 /* bfloat16 gradient (the sketch and the decoded values stay float32) */
} s2_dtype;

#define S2_MAX_ROWS 16u

/* Sketch shape and hash seed. d in [1, S2_MAX_ROWS]; w in [1, 2^31]. */
typedef struct {
    uint32_t d;
    uint32_t w;
    uint32_t seed;
} s2_params;

/*
 * s2_encode -- compression phase for ONE worker (Section 3.1 "Compressing
 * Sparse Gradient"; Algorithm 1, compression loop).
 *   grad   [n] elements of type dt (16-byte aligned).
 *   bitmap [nw] uint32 out: bit i set iff grad[i] is nonzero.
 *   sketch [d][w] float32 out: zeroed, then sketch[j][h_j(i)] += s_j(i)*grad[i]
 *          for every nonzero i and row j. float32 adds in an unspecified order.
 * n = 0 is valid (the sketch is zeroed, no bitmap word is written).
 */
S2_API s2_status s2_encode(const void *grad, s2_dtype dt, uint64_t n, s2_params p, uint32_t *bitmap,
                    float *sketch, s2_stream_t stream);

/*
 * s2_encode_batched -- s2_encode on W workers at once.
 *   grad     [W][n] (worker k starts at element k*n), 16-byte aligned base.
 *   bitmaps  [W][nw] uint32 out.   sketches [W][d][w] float32 out.
 * W = 0 is valid and does nothing. When n*sizeof(dt) is not a multiple of 16
 * the workers' rows are not 16-byte aligned and a scalar-load kernel is used.
 */
S2_API s2_status s2_encode_batched(const void *grad, s2_dtype dt, uint32_t W, uint64_t n, s2_params p,
                            uint32_t *bitmaps, float *sketches, s2_stream_t stream);

/* Where the count-sketch inserts of an encode accumulate. */
typedef enum {
    S2_PATH_AUTO = 0, /* the library picks one of the two below */
    S2_PATH_L2 = 1,   /* float reductions straight into the sketch in global memory (resolved in L2) */
    S2_PATH_SMEM = 2  /* a private copy of the sketch per thread block in shared memory, added into the
                         global sketch once at the end; only for 4*d*w <= S2_SMEM_SKETCH_MAX_BYTES */
} s2_encode_path;

#define S2_SMEM_SKETCH_MAX_BYTES (192u * 1024u)

/*
 * s2_encode_batched_path -- s2_encode_batched with the accumulation path
 * chosen by the caller (s2_encode_batched is this call with S2_PATH_AUTO).
 * The results are the same on both paths up to the order of the float32
 * adds: identical bitmaps, sketches within float32 rounding of each other.
 * S2_PATH_SMEM: each thread block owns a contiguous range of one worker's
 * positions and adds its inserts into a d x w copy in shared memory (lanes of
 * a warp that hit the same bucket in one step are merged first), then adds
 * the copy into the worker's sketch (stores it when one block covers the
 * worker). A sketch larger than S2_SMEM_SKETCH_MAX_BYTES returns
 * S2_ERR_UNSUPPORTED. S2_PATH_AUTO takes the shared-memory path when the
 * sketch fits, n >= 4096*w (many positions per bucket, so that the adds of a
 * moderately dense gradient pile up on each bucket) and the blocks' final
 * additions cost at most half as many L2 sector operations as reading the
 * gradient; otherwise the L2 path.
 */
S2_API s2_status s2_encode_batched_path(const void *grad, s2_dtype dt, uint32_t W, uint64_t n, s2_params p,
                                        s2_encode_path path, uint32_t *bitmaps, float *sketches,
                                        s2_stream_t stream);

/*
 * s2_encode_batched_blocks -- s2_encode_batched with the paper's block-granular
 * bitmap (Section 3.1 "Compressing Sparse Gradient": one bit per word vector
 * or gradient block, set iff the block contains a nonzero).
 *   block: positions per block, a multiple of 32 (S2_ERR_UNSUPPORTED
 *   otherwise); nb = ceil(n / block) blocks, nbw = ceil(nb / 32) words.
 *   block_bitmaps [W][nbw] uint32 out: bit x of worker k set iff positions
 *   [x*block, (x+1)*block) of worker k hold a nonzero (same bit layout as the
 *   element bitmap, over blocks).
 *   sketches: exactly as s2_encode_batched (only nonzero positions are
 *   inserted). Aggregate the block bitmaps with s2_reduce passing nb as n.
 */
S2_API s2_status s2_encode_batched_blocks(const void *grad, s2_dtype dt, uint32_t W, uint64_t n, uint32_t block,
                                          s2_params p, uint32_t *block_bitmaps, float *sketches,
                                          s2_stream_t stream);

/*
 * s2_block_topk -- block-wise Top-K sparsification with error feedback, the
 * step before encode in the paper's second setting (Section 2.2 "Sparse
 * Gradient & AllGather": keep the K blocks of largest l2 norm; Appendix A.2:
 * the residual e_{t+1} = g_t - U(g_t) joins the next step's gradient).
 *   grad [W][n] float32 in; residual [W][n] float32 in/out (zeros at the
 *   first step); sparse_out [W][n] float32 out. Per worker: acc = grad +
 *   residual (float32 additions); the K blocks of `block` elements (the last
 *   one may be shorter) with the largest l2 norm are kept, ties going to the
 *   lower block index; sparse_out = acc on kept blocks and 0 elsewhere,
 *   residual = acc elsewhere and 0 on kept blocks.
 *   The squared norms are summed in float32 in a fixed order, so the result
 *   is deterministic; against the exact norms, each square passes through at
 *   most ceil(block/32) + 5 roundings, and blocks whose exact norms differ by
 *   less than that relative rounding may be ranked either way. Blocks with
 *   identical contents always tie, and the lower index wins.
 *   block: a multiple of 32 (S2_ERR_UNSUPPORTED otherwise); K <= ceil(n/block)
 *   (S2_ERR_INVALID_ARG otherwise). workspace: s2_block_topk_workspace_size
 *   bytes, 16-byte aligned, contents on entry irrelevant.
 */
S2_API s2_status s2_block_topk_workspace_size(uint32_t W, uint64_t n, uint32_t block, size_t *bytes);
S2_API s2_status s2_block_topk(const float *grad, float *residual, uint32_t W, uint64_t n, uint32_t block,
                               uint64_t K, float *sparse_out, void *workspace, size_t workspace_bytes,
                               s2_stream_t stream);

/*
 * s2_sparse_pack / s2_sparse_sum -- the sparse AllGather baseline the paper
 * compares S2 Reducer with (Section 2.2 "Sparse Gradient & AllGather" and
 * Figure 1(b)): each worker sends the indices and values of its nonzeros,
 * every worker gathers all the lists and adds them up. Here, on one GPU:
 *   s2_sparse_pack: grad [W][n] float32 in; idx_out [W][capacity] uint32 and
 *   val_out [W][capacity] float32 out, worker k's nonzeros (bit pattern test
 *   as in s2_encode) in ascending index order; counts_out [W] uint64 (device)
 *   receives each worker's true count (entries past capacity are not
 *   written). workspace: s2_sparse_pack_workspace_size bytes, 16-byte aligned.
 *   s2_sparse_sum: out [n] float32 = the sum of all W lists, added in worker
 *   order 0..W-1 (the exact aggregate the sketch approximates; bit-identical
 *   to a sequential float32 sum over workers). Indices >= n are skipped.
 */
S2_API s2_status s2_sparse_pack_workspace_size(uint32_t W, uint64_t n, size_t *bytes);
S2_API s2_status s2_sparse_pack(const float *grad, uint32_t W, uint64_t n, uint32_t *idx_out, float *val_out,
                                uint64_t capacity, uint64_t *counts_out, void *workspace, size_t workspace_bytes,
                                s2_stream_t stream);
S2_API s2_status s2_sparse_sum(const uint32_t *idx, const float *val, const uint64_t *counts, uint32_t W,
                               uint64_t capacity, uint64_t n, float *out, s2_stream_t stream);

/*
 * s2_reduce -- the AllReduce(S, C) of Algorithm 1 (Section 3.1 "Collecting
 * Sparse-Sketch with AllReduce"), with all W workers resident on this GPU.
 *   bitmaps [W][nw], sketches [W][d][w]  in.
 *   bitmap_out [nw] = OR over k of bitmaps[k];
 *   sketch_out [d][w] = sum over k of sketches[k], added in the fixed order
 *   k = 0, 1, ..., W-1 (deterministic). W = 0 writes zeros.
 */
S2_API s2_status s2_reduce(const uint32_t *bitmaps, const float *sketches, uint32_t W, uint64_t n,
                    s2_params p, uint32_t *bitmap_out, float *sketch_out, s2_stream_t stream);

/*
 * s2_encode_reduce_fused -- s2_encode_batched followed by s2_reduce in one
 * pass, for workers that all live on this GPU (Section 3.1 "Collecting
 * Sparse-Sketch with AllReduce": because the sketch is linear, the sum of the
 * workers' sketches is the sketch of the summed gradient).
 *   grad [W][n] in (16-byte aligned base, any n);
 *   bitmap_out [nw] = OR over k of the workers' nonzero bitmaps (identical to
 *   s2_reduce's output); sketch_out [d][w] = the summed sketch: the workers'
 *   values are added per position (order k = 0..W-1) and each union position
 *   is inserted once, so the result equals s2_reduce's up to float32
 *   rounding order.
 * The per-worker bitmaps and sketches (what each worker of a real
 * distributed run would send into the AllReduce) are never formed, so this
 * is a same-GPU shortcut, measured separately from the per-worker path.
 * W = 0 writes a zero bitmap and sketch.
 */
S2_API s2_status s2_encode_reduce_fused(const void *grad, s2_dtype dt, uint32_t W, uint64_t n, s2_params p,
                                        uint32_t *bitmap_out, float *sketch_out, s2_stream_t stream);

/*
 * s2_decode_dense -- decompression phase with a dense output (Section 3.1
 * "Decompressing Sparse Gradient"; Algorithm 1, decompression loop).
 *   bitmap [nw], sketch [d][w] in; out [n] float32 (16-byte aligned).
 *   For every set bit i: out[i] = scale * median_j( s_j(i) * sketch[j][h_j(i)] );
 *   the median of an even number of rows is the mean of the two middle values.
 *   Every unset position receives exactly +0.0f.
 */
S2_API s2_status s2_decode_dense(const uint32_t *bitmap, const float *sketch, uint64_t n, s2_params p,
                          float scale, float *out, s2_stream_t stream);

/*
 * s2_decode_dense_blocks -- s2_decode_dense under a block bitmap (Section 3.1
 * "Decompressing Sparse Gradient": the recovered indices are every position
 * of every marked block, zeros inside a marked block included).
 *   block_bitmap [nbw] (from s2_reduce over block bitmaps), block as in
 *   s2_encode_batched_blocks; out [n]: the median estimate at every position
 *   of a marked block, +0.0f elsewhere.
 */
S2_API s2_status s2_decode_dense_blocks(const uint32_t *block_bitmap, const float *sketch, uint64_t n,
                                        uint32_t block, s2_params p, float scale, float *out,
                                        s2_stream_t stream);

/*
 * s2_decode_dense_ws -- s2_decode_dense with a workspace, for summed sketches
 * too large to stay in the L2 cache under random reads (Section 3.1
 * "Decompressing Sparse Gradient"; the median query of Algorithm 1).
 *   Arguments, results and errors as s2_decode_dense, plus
 *   workspace: device scratch of at least s2_decode_dense_workspace_size(n, p)
 *   bytes (about 8n for d = 5 and 4n for d = 3, plus 4 bytes per 512
 *   positions; 0 for other d), 16-byte aligned, not overlapping the other
 *   arrays; its contents on entry do not matter (S2_ERR_INVALID_ARG if it is
 *   too small).
 * When the sketch (4*d*w bytes) is larger than 2/5 of this device's L2 cache
 * and d is 3 or 5, the median is taken in passes over groups of whole rows
 * that fit in 2/5 of L2, the smallest group first: a first launch writes the zeros of every
 * 512-position stretch without a set bit and lists the others; each pass then
 * reads only its rows for every set position of the listed stretches and
 * carries the candidates for the median that remain (at most 2 for d = 3, 3
 * for d = 5) to the next pass in `out` and the workspace. A sketch of at most
 * 96 MB whose set positions reach at least half of the stretches is decoded
 * in one launch over all rows instead (the device picks, from the count of
 * listed stretches). The
 * decoded values are the same as s2_decode_dense's (the median selects one
 * of the row values, or averages none); an estimate of zero may come out as
 * +0.0 or -0.0 as with s2_decode_dense. Otherwise the call launches exactly
 * what s2_decode_dense launches and does not touch the workspace.
 */
S2_API s2_status s2_decode_dense_workspace_size(uint64_t n, s2_params p, size_t *bytes);
S2_API s2_status s2_decode_dense_ws(const uint32_t *bitmap, const float *sketch, uint64_t n, s2_params p,
                                    float scale, float *out, void *workspace, size_t workspace_bytes,
                                    s2_stream_t stream);

/* Device workspace bytes that s2_decode_compact needs for length n. */
S2_API s2_status s2_decode_workspace_size(uint64_t n, size_t *bytes);

/*
 * s2_decode_compact -- decompression phase with a compacted output: the set
 * positions of the bitmap in ascending order and their estimates.
 *   idx_out [capacity] uint32, val_out [capacity] float32: entry t holds the
 *   t-th set position and its estimate (same value as s2_decode_dense).
 *   count_out: ONE uint64 in device memory, receives the number of set bits
 *   (always the true count, even when it exceeds capacity; entries at
 *   t >= capacity are not written).
 *   workspace: device scratch of at least s2_decode_workspace_size(n) bytes,
 *   16-byte aligned; its contents on entry do not matter.
 * Compaction is exact and deterministic: no inter-block waiting is involved.
 */
S2_API s2_status s2_decode_compact(const uint32_t *bitmap, const float *sketch, uint64_t n, s2_params p,
                            float scale, uint32_t *idx_out, float *val_out, uint64_t capacity,
                            uint64_t *count_out, void *workspace, size_t workspace_bytes,
                            s2_stream_t stream);

/*
 * s2_decode_compact_noalloc -- s2_decode_compact without a workspace argument.
 *
 * The paper has no counterpart to this call; it exists for callers that
 * cannot allocate device memory for a workspace: code running where a
 * framework owns every byte of device memory through its own pool and
 * forbids side allocations, code on a latency-critical path where a
 * cudaMalloc (which may synchronise the device) is not acceptable, and code
 * that keeps no state between calls in which a workspace could live.
 *
 * Same arguments, results and errors as s2_decode_compact, minus the
 * workspace. The scratch it needs (per-tile counts and offsets, per-task
 * prefixes) is a fixed 5 MiB array inside the library, allocated once per
 * GPU when the library's device code is first loaded there and held until
 * the process exits; the call itself allocates nothing. It accepts n up to 2^30 positions and
 * returns S2_ERR_UNSUPPORTED beyond that.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and caches it; make that first call before any
 *     stream capture. A lookup that fails (S2_ERR_CUDA) is not cached: the
 *     next call on that device tries again. The cached address belongs to
 *     the device's current context: after cudaDeviceReset on that device,
 *     do not call this function again in the same process.
 *   - Every call on a device shares the one array: calls whose kernels can
 *     overlap on the GPU (different streams without ordering between them)
 *     race and corrupt each other's results. Order such calls, or use
 *     s2_decode_compact with one workspace per stream.
 *   - Nothing in the array needs clearing between calls: each call writes
 *     every entry it later reads.
 */
S2_API s2_status s2_decode_compact_noalloc(const uint32_t *bitmap, const float *sketch, uint64_t n,
                                           s2_params p, float scale, uint32_t *idx_out, float *val_out,
                                           uint64_t capacity, uint64_t *count_out, s2_stream_t stream);

/*
 * s2_hash -- the bucket and sign hashes of m given positions, for checking.
 *   idx [m] uint32 in; bucket_out [d][m] uint32 and sign_out [d][m] int8
 *   (+1 or -1) out, row-major by row j.
 */
S2_API s2_status s2_hash(const uint32_t *idx, uint64_t m, s2_params p, uint32_t *bucket_out,
                  int8_t *sign_out, s2_stream_t stream);

/* Device workspace bytes that s2_pipeline_dense_host needs. */
S2_API s2_status s2_pipeline_workspace_size(s2_dtype dt, uint32_t W, uint64_t n, s2_params p,
                                     size_t *bytes);

/*
 * s2_pipeline_dense_host -- the whole path from HOST memory to HOST memory:
 * grad [W][n] to the device, s2_encode_batched, s2_reduce, s2_decode_dense,
 * and the decoded [n] float32 vector back to the host.
 *   host_grad / host_out: host memory. Page-locked memory that the device can
 *   address (cudaHostAlloc, cudaHostRegister, torch pin_memory), 16-byte
 *   aligned, is accessed in place by the kernels: the encode reads the
 *   gradient from it and the decode writes the output to it, with no copy
 *   (the gradient is still staged when the sketch is larger than 3/4 of the
 *   L2 cache, where the encode reads it more than once). Other host memory
 *   is staged through the workspace with copies, which are synchronous for
 *   pageable memory.
 *   workspace: device scratch of s2_pipeline_workspace_size bytes, 16-byte
 *   aligned. The call returns once the work is queued on `stream`; host_out
 *   is valid after the stream is synchronised.
 */
S2_API s2_status s2_pipeline_dense_host(const void *host_grad, s2_dtype dt, uint32_t W, uint64_t n,
                                 s2_params p, float scale, float *host_out, void *workspace,
                                 size_t workspace_bytes, s2_stream_t stream);

/* Human-readable name of a status code (static string). */
S2_API const char *s2_status_string(s2_status st);

/* Library version string (static). */
S2_API const char *s2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* S2_H */
