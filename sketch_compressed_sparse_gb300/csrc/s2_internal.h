// Host-side launchers shared between the translation units of libs2.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "s2_device.cuh"

namespace s2 {

// A warp task covers 512 consecutive positions of one worker: 16 bitmap
// words. Each lane owns 16 of the positions ("slots").
constexpr int kTaskElems = 512;
constexpr int kTaskWords = 16;
constexpr int kThreads = 256;

struct DeviceInfo {
    int sms;
    int l2_bytes;
};
cudaError_t device_info(DeviceInfo* out);

// Keys of rows 0..d-1 for a seed (rows >= d are zero).
RowKeys make_keys(uint32_t seed, uint32_t d);

// ---- encode ----------------------------------------------------------------
struct EncodeArgs {
    const void* grad;   // first worker of the group
    uint32_t* bitmaps;  // first worker of the group, [G][nw]
    float* sketches;    // first worker of the group, [G][d*w]
    uint64_t n;         // positions per worker
    uint64_t nw;        // bitmap words per worker
    uint64_t dw;        // d * w
    uint32_t workers;   // G, workers in this launch
    uint32_t tasks_per_worker;
    uint32_t d;
    uint32_t w;
    RowKeys keys;
    uint32_t block_words;  // 0: element bitmap; else one bit per block of this many bitmap words
    uint64_t nbw;          // block bitmap words per worker (block mode)
    uint64_t x_lo;         // slice of the flattened sketch (j*w + b) this launch updates:
    uint64_t x_span;       //   [x_lo, x_lo + x_span); [0, d*w) in a single pass
};

// dtype: 0 = f32, 1 = bf16. vec: rows are 16-byte aligned (vector loads).
cudaError_t launch_encode(const EncodeArgs& a, int dtype, bool vec, cudaStream_t s);
cudaError_t launch_zero(float* p, uint64_t count, cudaStream_t s);

// Shared-memory privatised sketches (4*d*w <= kPrivMaxBytes), all a.workers
// workers in one pass; zeroes the sketches itself when it needs to. With
// only_if_preferred the launch is skipped (*launched = false) when the
// blocks' final additions would cost more than half of the gradient read.
constexpr size_t kPrivMaxBytes = 192 * 1024;
cudaError_t launch_encode_smem(const EncodeArgs& a, int dtype, bool vec, bool only_if_preferred, bool* launched,
                               cudaStream_t s);

// ---- fused encode + reduce (single sketch) ----------------------------------
struct FusedArgs {
    const void* grad;  // [W][n]
    uint32_t* bitmap;  // [nw] aggregate (OR) bitmap
    float* sketch;     // [d*w] summed sketch
    uint64_t n;
    uint64_t nw;
    uint32_t workers;
    uint32_t d;
    uint32_t w;
    RowKeys keys;
};
// Zero-fills the sketch, then one pass over all workers (dtype: 0 f32, 1 bf16).
cudaError_t launch_fused(const FusedArgs& a, int dtype, cudaStream_t s);

// ---- block-wise Top-K with error feedback (upstream of encode) -------------
size_t topk_workspace_bytes(uint32_t W, uint64_t n, uint32_t block);
cudaError_t launch_block_topk(const float* grad, float* resid, uint32_t W, uint64_t n, uint32_t block, uint64_t K,
                              float* sparse, void* workspace, cudaStream_t s);

// ---- reduce ----------------------------------------------------------------
cudaError_t launch_reduce(const uint32_t* bitmaps, const float* sketches, uint32_t W, uint64_t nw,
                          uint64_t dw, uint32_t* bitmap_out, float* sketch_out, cudaStream_t s);

// ---- decode ----------------------------------------------------------------
struct DecodeArgs {
    const uint32_t* bitmap;
    const float* sketch;
    uint64_t n;
    uint64_t nw;
    uint32_t d;
    uint32_t w;
    float scale;
    RowKeys keys;
    uint32_t block;  // 0: element bitmap; else a block bitmap, one bit per `block` positions
};
cudaError_t launch_decode_dense(const DecodeArgs& a, float* out, cudaStream_t s);

// Dense decode that takes the median in passes over groups of rows when the
// summed sketch is larger than 2/5 of L2 (d = 3 or 5, element bitmap);
// otherwise the same launches as launch_decode_dense. ws: dense_workspace_bytes.
struct DenseWsLayout {
    uint64_t cand1, cand2, count, list, total;  // byte offsets
};
DenseWsLayout dense_ws_layout(uint64_t n, uint32_t d);
size_t dense_workspace_bytes(uint64_t n, uint32_t d);
uint32_t dense_decode_passes(const DecodeArgs& a, uint64_t l2_bytes);
cudaError_t launch_decode_dense_ws(const DecodeArgs& a, float* out, float* ws, cudaStream_t s);

constexpr int kCompactTileWords = 256;  // 8192 positions per tile
uint64_t compact_tiles(uint64_t nw);
size_t compact_workspace_bytes(uint64_t n);
cudaError_t launch_decode_compact(const DecodeArgs& a, uint32_t* idx_out, float* val_out,
                                  uint64_t capacity, unsigned long long* count_out,
                                  uint32_t* tile_counts, uint32_t* tile_offsets, cudaStream_t s);

// Exclusive scan of `tiles` 32-bit counts by one block; *total gets the sum.
cudaError_t launch_tile_scan(const uint32_t* counts, uint64_t tiles, uint32_t* offsets, unsigned long long* total,
                             cudaStream_t s);

// ---- sparse AllGather baseline ---------------------------------------------
size_t pack_workspace_bytes(uint32_t W, uint64_t n);
cudaError_t launch_sparse_pack(const float* grad, uint32_t W, uint64_t n, uint32_t* idx, float* val,
                               uint64_t capacity, unsigned long long* counts, void* workspace, cudaStream_t s);
cudaError_t launch_sparse_sum(const uint32_t* idx, const float* val, const unsigned long long* counts, uint32_t W,
                              uint64_t capacity, uint64_t n, float* out, cudaStream_t s);

// Library-owned scratch of s2_decode_compact_noalloc (see s2_decode.cu).
uint64_t noalloc_compact_max_n();
cudaError_t noalloc_compact_scratch(uint32_t** counts, uint32_t** offsets);

cudaError_t launch_hash(const uint32_t* idx, uint64_t m, uint32_t d, uint32_t w, RowKeys keys,
                        uint32_t* bucket_out, int8_t* sign_out, cudaStream_t s);

// Resident blocks per SM of kernel `fn` (occupancy calculator, cached per
// device, kernel, block size and dynamic shared memory); at least 1.
int blocks_per_sm(const void* fn, int threads, size_t smem);

// Blocks to launch for a grid-stride kernel: a multiple of the SM count
// (resident blocks per SM from the occupancy calculator), capped by the work.
template <typename Kernel>
int grid_for(Kernel k, uint64_t work_blocks, size_t smem = 0) {
    const int per_sm = blocks_per_sm(reinterpret_cast<const void*>(k), kThreads, smem);
    DeviceInfo di{};
    if (device_info(&di) != cudaSuccess) di.sms = 1;
    uint64_t full = (uint64_t)di.sms * (uint64_t)per_sm;
    if (work_blocks < 1) work_blocks = 1;
    return (int)(work_blocks < full ? work_blocks : full);
}

}  // namespace s2
