// The sparse AllGather baseline the paper compares against ("S2 Reducer",
// Section 2.2 and Figure 1(b): every worker sends the indices and values of
// its nonzeros, every worker gathers all lists and adds them up), on one GPU:
//   pack: per worker, the ascending (index, value) list of its nonzeros --
//         the message it would contribute to the AllGather;
//   sum:  the gathered lists added into a dense vector in worker order
//         0..W-1, the exact aggregate that the sketch approximates.
// Pack = per-tile nonzero counts, one-block scans of the tile counts, and a
// writer that keeps each warp's 1024 positions in registers; sum = one
// scatter pass per worker (the indices of one list are distinct, so no
// atomics are needed and the order of additions is fixed).
#include "s2_internal.h"

namespace s2 {
namespace {

constexpr uint32_t kPackTile = 8192;  // positions per tile (8 warps x 1024)

__device__ __forceinline__ bool nonzero_f32(uint32_t bits) { return (bits & 0x7fffffffu) != 0; }

// counts[k * tiles + t] = nonzeros of tile t of worker k.
__global__ void __launch_bounds__(kThreads)
    pack_count_kernel(const float* __restrict__ grad, uint32_t W, uint64_t n, uint64_t tiles,
                      uint32_t* __restrict__ counts) {
    __shared__ uint32_t s_warp[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (uint64_t bt = blockIdx.x; bt < (uint64_t)W * tiles; bt += gridDim.x) {
        const uint64_t k = bt / tiles, t = bt - k * tiles;
        const uint64_t base = t * kPackTile + (uint64_t)warp * 1024;
        const float* g = grad + k * n;
        uint32_t c = 0;
#pragma unroll 8
        for (int r = 0; r < 32; ++r) {
            const uint64_t i = base + r * 32 + lane;
            const bool nz = i < n && nonzero_f32(ld_stream_u32(g + i));
            c += __popc(__ballot_sync(kFull, nz));
        }
        if (lane == 0) s_warp[warp] = c;
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t tot = 0;
            for (int q = 0; q < kThreads / 32; ++q) tot += s_warp[q];
            counts[bt] = tot;
        }
        __syncthreads();
    }
}

// Writes worker k's nonzeros of tile t at offsets[k * tiles + t] onwards.
__global__ void __launch_bounds__(kThreads)
    pack_write_kernel(const float* __restrict__ grad, uint32_t W, uint64_t n, uint64_t tiles,
                      const uint32_t* __restrict__ offsets, uint32_t* __restrict__ idx, float* __restrict__ val,
                      uint64_t capacity) {
    __shared__ uint32_t s_warp[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (uint64_t bt = blockIdx.x; bt < (uint64_t)W * tiles; bt += gridDim.x) {
        const uint64_t k = bt / tiles, t = bt - k * tiles;
        const uint64_t base = t * kPackTile + (uint64_t)warp * 1024;
        const float* g = grad + k * n;
        uint32_t v[32];
        uint32_t c = 0;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const uint64_t i = base + r * 32 + lane;
            v[r] = i < n ? ld_stream_u32(g + i) : 0u;
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) c += __popc(__ballot_sync(kFull, nonzero_f32(v[r])));
        if (lane == 0) s_warp[warp] = c;
        __syncthreads();
        uint64_t at = offsets[bt];
        for (int q = 0; q < warp; ++q) at += s_warp[q];
        uint32_t* ik = idx + k * capacity;
        float* vk = val + k * capacity;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const bool nz = nonzero_f32(v[r]);
            const uint32_t bal = __ballot_sync(kFull, nz);
            const uint64_t o = at + __popc(bal & ((1u << lane) - 1u));
            if (nz && o < capacity) {
                ik[o] = (uint32_t)(base + r * 32 + lane);
                vk[o] = __uint_as_float(v[r]);
            }
            at += __popc(bal);
        }
        __syncthreads();  // s_warp is rewritten by the next tile
    }
}

// out[idx[t]] += val[t] for the first min(count, capacity) entries of worker
// k; indices at or beyond n are skipped.
__global__ void __launch_bounds__(kThreads)
    sum_list_kernel(const uint32_t* __restrict__ idx, const float* __restrict__ val,
                    const unsigned long long* __restrict__ count, uint64_t capacity, uint64_t n,
                    float* __restrict__ out) {
    const uint64_t m = *count < capacity ? *count : capacity;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; t < m; t += stride) {
        const uint32_t i = idx[t];
        if (i < n) out[i] += val[t];
    }
}

}  // namespace

size_t pack_workspace_bytes(uint32_t W, uint64_t n) {
    const uint64_t tiles = (n + kPackTile - 1) / kPackTile;
    const uint64_t one = ((uint64_t)W * tiles * 4 + 255) / 256 * 256;
    return (size_t)(2 * one);
}

cudaError_t launch_sparse_pack(const float* grad, uint32_t W, uint64_t n, uint32_t* idx, float* val,
                               uint64_t capacity, unsigned long long* counts, void* workspace, cudaStream_t s) {
    const uint64_t tiles = (n + kPackTile - 1) / kPackTile;
    uint32_t* tcount = static_cast<uint32_t*>(workspace);
    uint32_t* toff = tcount + ((uint64_t)W * tiles * 4 + 255) / 256 * 256 / 4;
    if (tiles > 0) {
        pack_count_kernel<<<grid_for(pack_count_kernel, (uint64_t)W * tiles), kThreads, 0, s>>>(grad, W, n, tiles,
                                                                                               tcount);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    for (uint32_t k = 0; k < W; ++k) {
        cudaError_t e = launch_tile_scan(tcount + (uint64_t)k * tiles, tiles, toff + (uint64_t)k * tiles, counts + k, s);
        if (e != cudaSuccess) return e;
    }
    if (tiles == 0) return cudaSuccess;
    pack_write_kernel<<<grid_for(pack_write_kernel, (uint64_t)W * tiles), kThreads, 0, s>>>(grad, W, n, tiles, toff,
                                                                                           idx, val, capacity);
    return cudaGetLastError();
}

cudaError_t launch_sparse_sum(const uint32_t* idx, const float* val, const unsigned long long* counts, uint32_t W,
                              uint64_t capacity, uint64_t n, float* out, cudaStream_t s) {
    cudaError_t e = launch_zero(out, n, s);
    if (e != cudaSuccess) return e;
    const uint64_t blocks = (capacity + kThreads - 1) / kThreads;
    for (uint32_t k = 0; k < W && capacity > 0; ++k) {
        sum_list_kernel<<<grid_for(sum_list_kernel, blocks), kThreads, 0, s>>>(idx + (uint64_t)k * capacity,
                                                                               val + (uint64_t)k * capacity,
                                                                               counts + k, capacity, n, out);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace s2
