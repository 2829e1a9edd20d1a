// Block-wise Top-K sparsification with error feedback, upstream of encode
// ("S2 Reducer", Section 2.2 "Sparse Gradient & AllGather": keep the K blocks
// of largest l2 norm; Appendix A.2: the residual e_{t+1} = g_t - U(g_t) is
// carried into the next step's gradient).
//
// Per worker: acc = grad + residual; the squared norm of every block of
// `block` elements in float32, one warp per block (each lane accumulates
// fmaf(a, a, s) over its block/32 elements in a fixed order, then an XOR
// butterfly): a fixed order, so that which blocks are kept -- an integer
// decision -- is the same on every run; the K-th largest norm by a 4-pass
// 8-bit radix select over the norms' bit patterns (non-negative floats order
// like their bits), ties broken towards the lower block index; finally
// sparse = acc on kept blocks and residual = acc elsewhere. Against the
// exact norm, each square passes through at most ceil(block/32) + 5
// roundings, so blocks whose exact norms differ by less than that relative
// rounding may be ranked either way.
//
// The select runs on many thread blocks per worker: each radix pass is one
// launch that adds the digit counts of its slice of the norms into a global
// 256-bin histogram per worker (every block first replays the earlier
// passes' histograms, one thread per digit and a scan per pass, to find the
// prefix it must match); a counting launch
// and a marking launch then keep every norm above the final threshold and,
// of the norms equal to it, the first ones in index order (each block starts
// its rank after the equal norms of the blocks before it). No launch waits on
// another block.
#include "s2_internal.h"

namespace s2 {
namespace {

// Squared norm of block x of worker k, one warp per (k, x) task. acc =
// grad + residual is written back into the residual array (each element by
// the thread that reads it): it is the new residual of every block that is
// not kept, so the apply step only touches kept blocks' values. Plain loads
// for both arrays: with the residual stored in the same kernel, evict-first
// (.cs) loads measured 2-12 times slower on this GPU (8 x 25.6 M floats:
// 0.54 ms with plain loads, 1.21 ms with an evict-first gradient load, 3.57
// ms with both).
// VEC (worker rows 16-byte aligned, block a multiple of 128): lane l takes
// the 16-byte vectors at elements 4l + 128i, i = 0, 1, ..., adding their four
// squares in order into one sum, so each lane still sums block/32 squares
// (the rounding bound above holds as it is); otherwise lane l takes elements
// l, l + 32, ... one at a time.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
    topk_norms_kernel(const float* __restrict__ grad, float* __restrict__ resid, uint64_t n, uint32_t block,
                      uint64_t nb, uint32_t W, float* __restrict__ norms) {
    const int lane = threadIdx.x & 31;
    const uint64_t tasks = (uint64_t)W * nb;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t t = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < tasks; t += nwarps) {
        const uint64_t k = t / nb, x = t - k * nb;
        const uint64_t base = k * n + x * block;
        const uint64_t len = (x + 1) * block <= n ? block : n - x * block;
        float s = 0.f;
        if (VEC) {  // len is a multiple of 4 (n % 4 == 0, block % 128 == 0)
            const float4* g4 = reinterpret_cast<const float4*>(grad + base);
            float4* r4 = reinterpret_cast<float4*>(resid + base);
#pragma unroll 4
            for (uint64_t j = lane; j < len / 4; j += 32) {
                const float4 g = g4[j], r = r4[j];
                const float4 a = make_float4(__fadd_rn(g.x, r.x), __fadd_rn(g.y, r.y), __fadd_rn(g.z, r.z),
                                             __fadd_rn(g.w, r.w));
                r4[j] = a;
                s = __fmaf_rn(a.x, a.x, s);
                s = __fmaf_rn(a.y, a.y, s);
                s = __fmaf_rn(a.z, a.z, s);
                s = __fmaf_rn(a.w, a.w, s);
            }
        } else {
#pragma unroll 8
            for (uint64_t j = lane; j < len; j += 32) {
                const float a = __fadd_rn(grad[base + j], resid[base + j]);
                resid[base + j] = a;
                s = __fmaf_rn(a, a, s);
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(kFull, s, off));
        if (lane == 0) norms[t] = s;
    }
}

constexpr int kSelThreads = 256;
constexpr int kSelPerThread = 16;                       // norms per thread and launch
constexpr uint64_t kSelSlice = (uint64_t)kSelThreads * kSelPerThread;  // norms per block
static_assert(kSelThreads == 256, "one thread per histogram bin");

// The radix state after `passes` passes of worker k: the digits fixed so far
// (prefix under pmask) and how many norms equal to that prefix are still to
// be kept. hist: [4][W][256] digit counts of the passes (pass-major). Run by
// all kSelThreads threads of the block, one per digit: per pass an inclusive
// scan of the counts from digit 255 down finds the first digit at which the
// count of norms at or above it reaches the number still to keep. The result
// is left in *s_prefix, *s_pmask, *s_rest (shared); the call ends with a
// __syncthreads.
__device__ void select_state(const uint32_t* __restrict__ hist, uint32_t W, uint32_t k, int passes, uint64_t K,
                             uint32_t* s_prefix, uint32_t* s_pmask, unsigned long long* s_rest) {
    __shared__ uint32_t s_wsum[kSelThreads / 32];
    __shared__ uint32_t s_first;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    if (t == 0) {
        *s_prefix = 0u;
        *s_pmask = 0u;
        *s_rest = K;
    }
    __syncthreads();
    for (int p = 0; p < passes; ++p) {
        const uint32_t dg = 255u - (uint32_t)t;  // thread t holds digit 255 - t
        const uint32_t c = hist[((uint64_t)p * W + k) * 256 + dg];
        uint32_t incl = c;  // norms (matching the prefix) with digit in [dg, 255]
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_wsum[warp] = incl;
        if (t == 0) s_first = kSelThreads - 1;  // no digit reaches it: digit 0
        __syncthreads();
        for (int w = 0; w < warp; ++w) incl += s_wsum[w];
        const unsigned long long r = *s_rest;
        const unsigned hit = __ballot_sync(kFull, incl >= r);
        if (hit && lane == __ffs(hit) - 1) atomicMin(&s_first, (uint32_t)t);
        __syncthreads();
        if (t == (int)s_first) {  // above = the norms with a digit above dg
            const int shift = 24 - 8 * p;
            *s_prefix |= dg << shift;
            *s_pmask |= 255u << shift;
            *s_rest = r - (incl - c);
        }
        __syncthreads();
    }
}

// Pass `pass` of the radix select: digit counts of the norms that match the
// prefix fixed by the earlier passes. Grid: (W, slices).
__global__ void __launch_bounds__(kSelThreads)
    topk_hist_kernel(const float* __restrict__ norms, uint64_t nb, uint64_t K, uint32_t W, int pass,
                     uint32_t* __restrict__ hist) {
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_prefix, s_pmask;
    __shared__ unsigned long long s_rest;
    const uint32_t k = blockIdx.x;
    s_hist[threadIdx.x] = 0;  // kSelThreads == 256 bins
    select_state(hist, W, k, pass, K, &s_prefix, &s_pmask, &s_rest);  // ends with __syncthreads
    const uint32_t prefix = s_prefix, pmask = s_pmask;
    const int shift = 24 - 8 * pass;
    const uint32_t* key = reinterpret_cast<const uint32_t*>(norms) + (uint64_t)k * nb;
    const uint64_t x0 = (uint64_t)blockIdx.y * kSelSlice;
    uint32_t v[kSelPerThread];
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {  // independent loads first
        const uint64_t x = x0 + (uint64_t)q * kSelThreads + threadIdx.x;
        v[q] = x < nb ? __ldg(key + x) : 0u;
    }
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
        const uint64_t x = x0 + (uint64_t)q * kSelThreads + threadIdx.x;
        if (x < nb && (v[q] & pmask) == prefix) atomicAdd(&s_hist[(v[q] >> shift) & 255u], 1u);
    }
    __syncthreads();
    const uint32_t c = s_hist[threadIdx.x];
    if (c) atomicAdd(hist + ((uint64_t)pass * W + k) * 256 + threadIdx.x, c);
}

// Norms equal to the final threshold in each slice. Grid: (W, slices).
__global__ void __launch_bounds__(kSelThreads)
    topk_eq_kernel(const float* __restrict__ norms, uint64_t nb, uint64_t K, uint32_t W,
                   const uint32_t* __restrict__ hist, uint32_t* __restrict__ eq_counts) {
    __shared__ uint32_t s_thr, s_pm;
    __shared__ unsigned long long s_rest;
    __shared__ uint32_t s_warp[kSelThreads / 32];
    const uint32_t k = blockIdx.x;
    select_state(hist, W, k, 4, K, &s_thr, &s_pm, &s_rest);  // ends with __syncthreads
    const uint32_t thr = s_thr;
    const uint32_t* key = reinterpret_cast<const uint32_t*>(norms) + (uint64_t)k * nb;
    const uint64_t x0 = (uint64_t)blockIdx.y * kSelSlice;
    uint32_t c = 0;
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
        const uint64_t x = x0 + (uint64_t)q * kSelThreads + threadIdx.x;
        c += (x < nb && __ldg(key + x) == thr) ? 1u : 0u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
    if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int w = 0; w < kSelThreads / 32; ++w) t += s_warp[w];
        eq_counts[(uint64_t)k * gridDim.y + blockIdx.y] = t;
    }
}

// keep[k][x] = 1 for the K blocks of largest norm (ties: lower index).
// Grid: (W, slices).
__global__ void __launch_bounds__(kSelThreads)
    topk_keep_kernel(const float* __restrict__ norms, uint64_t nb, uint64_t K, uint32_t W,
                     const uint32_t* __restrict__ hist, const uint32_t* __restrict__ eq_counts,
                     uint8_t* __restrict__ keep) {
    __shared__ uint32_t s_thr, s_pm;
    __shared__ unsigned long long s_rest, s_base;
    __shared__ uint32_t s_scan[kSelThreads / 32];
    __shared__ unsigned long long s_part[kSelThreads / 32];
    const uint32_t k = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t x0 = (uint64_t)blockIdx.y * kSelSlice;
    uint8_t* kp = keep + (uint64_t)k * nb;
    if (K == 0 || K >= nb) {
        for (int q = 0; q < kSelPerThread; ++q) {
            const uint64_t x = x0 + (uint64_t)q * kSelThreads + threadIdx.x;
            if (x < nb) kp[x] = K == 0 ? 0 : 1;
        }
        return;
    }
    // equal norms in the slices before this one, summed by the whole block
    unsigned long long part = 0;
    for (uint32_t b = threadIdx.x; b < blockIdx.y; b += kSelThreads) part += eq_counts[(uint64_t)k * gridDim.y + b];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
    if (lane == 0) s_part[warp] = part;
    select_state(hist, W, k, 4, K, &s_thr, &s_pm, &s_rest);  // ends with __syncthreads
    if (threadIdx.x == 0) {
        unsigned long long base = 0;
        for (int w = 0; w < kSelThreads / 32; ++w) base += s_part[w];
        s_base = base;
    }
    __syncthreads();
    const uint32_t thr = s_thr;
    const uint64_t rest = s_rest;
    uint64_t taken = s_base;  // equal norms before the current chunk (uniform across the block)
    const uint32_t* key = reinterpret_cast<const uint32_t*>(norms) + (uint64_t)k * nb;
    for (int q = 0; q < kSelPerThread; ++q) {  // chunks of kSelThreads norms in index order
        const uint64_t x = x0 + (uint64_t)q * kSelThreads + threadIdx.x;
        const uint32_t v = x < nb ? __ldg(key + x) : 0u;
        const bool eq = x < nb && v == thr;
        const unsigned bal = __ballot_sync(kFull, eq);
        if (lane == 0) s_scan[warp] = __popc(bal);
        __syncthreads();
        uint64_t before = taken;
        for (int w = 0; w < warp; ++w) before += s_scan[w];
        before += __popc(bal & ((1u << lane) - 1u));
        if (x < nb) kp[x] = (v > thr || (eq && before < rest)) ? 1 : 0;
        uint32_t chunk = 0;
        for (int w = 0; w < kSelThreads / 32; ++w) chunk += s_scan[w];
        __syncthreads();
        taken += chunk;
    }
}

// sparse = acc on kept blocks, 0 elsewhere; residual = acc elsewhere, 0 on
// kept blocks, where acc is already in the residual array (written by
// topk_norms_kernel): a kept block moves its values from the residual to
// sparse and zeroes them in the residual; any other block writes zeros to
// sparse and leaves its residual as it is. VEC: worker rows are 16-byte
// aligned (n % 4 == 0), so every block (a multiple of 32 elements) starts
// on a 16-byte boundary.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
    topk_apply_kernel(float* __restrict__ resid, const uint8_t* __restrict__ keep, uint64_t n, uint32_t block,
                      uint64_t nb, uint32_t W, float* __restrict__ sparse) {
    const int lane = threadIdx.x & 31;
    const uint64_t tasks = (uint64_t)W * nb;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t t = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < tasks; t += nwarps) {
        const uint64_t k = t / nb, x = t - k * nb;
        const uint64_t base = k * n + x * block;
        const uint64_t len = (x + 1) * block <= n ? block : n - x * block;
        const bool kept = keep[t] != 0;  // warp-uniform
        uint64_t j0 = 0;
        if (VEC) {
            const uint64_t len4 = len / 4;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (uint64_t j = lane; j < len4; j += 32) {
                if (kept) {
                    float4* r4 = reinterpret_cast<float4*>(resid + base) + j;
                    st_stream_f4(reinterpret_cast<float4*>(sparse + base) + j, *r4);
                    st_stream_f4(r4, z);
                } else {
                    st_stream_f4(reinterpret_cast<float4*>(sparse + base) + j, z);
                }
            }
            j0 = len4 * 4;
        }
        for (uint64_t j = j0 + lane; j < len; j += 32) {
            if (kept) {
                sparse[base + j] = resid[base + j];
                resid[base + j] = 0.f;
            } else {
                sparse[base + j] = 0.f;
            }
        }
    }
}

}  // namespace

// Workspace: norms [W][nb] float, keep [W][nb] bytes, the radix histograms
// [4][W][256] and the per-slice equal counts [W][slices], each region
// rounded to 256 bytes.
namespace {
struct TopkLayout {
    uint64_t norms, keep, hist, eq, total, slices;
};
TopkLayout topk_layout(uint32_t W, uint64_t n, uint32_t block) {
    const uint64_t nb = (n + block - 1) / block;
    auto r256 = [](uint64_t x) { return (x + 255) / 256 * 256; };
    TopkLayout L{};
    L.slices = (nb + kSelSlice - 1) / kSelSlice;
    L.norms = 0;
    L.keep = r256((uint64_t)W * nb * 4);
    L.hist = L.keep + r256((uint64_t)W * nb);
    L.eq = L.hist + r256(4ull * W * 256 * 4);
    L.total = L.eq + r256((uint64_t)W * L.slices * 4);
    return L;
}
}  // namespace

size_t topk_workspace_bytes(uint32_t W, uint64_t n, uint32_t block) { return (size_t)topk_layout(W, n, block).total; }

cudaError_t launch_block_topk(const float* grad, float* resid, uint32_t W, uint64_t n, uint32_t block, uint64_t K,
                              float* sparse, void* workspace, cudaStream_t s) {
    const uint64_t nb = (n + block - 1) / block;
    if ((uint64_t)W * nb == 0) return cudaSuccess;
    const TopkLayout L = topk_layout(W, n, block);
    char* ws = static_cast<char*>(workspace);
    float* norms = reinterpret_cast<float*>(ws + L.norms);
    uint8_t* keep = reinterpret_cast<uint8_t*>(ws + L.keep);
    uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
    uint32_t* eq = reinterpret_cast<uint32_t*>(ws + L.eq);
    const uint64_t blocks = ((uint64_t)W * nb + (kThreads / 32) - 1) / (kThreads / 32);
    if (n % 4 == 0 && block % 128 == 0)
        topk_norms_kernel<true><<<grid_for(topk_norms_kernel<true>, blocks), kThreads, 0, s>>>(grad, resid, n, block,
                                                                                               nb, W, norms);
    else
        topk_norms_kernel<false><<<grid_for(topk_norms_kernel<false>, blocks), kThreads, 0, s>>>(grad, resid, n, block,
                                                                                                 nb, W, norms);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const dim3 grid(W, (unsigned)L.slices);  // slices <= 65535: nb < 2^28 for n < 2^32
    if (K > 0 && K < nb) {
        e = launch_zero(reinterpret_cast<float*>(hist), 4ull * W * 256, s);
        if (e != cudaSuccess) return e;
        for (int pass = 0; pass < 4; ++pass) {
            topk_hist_kernel<<<grid, kSelThreads, 0, s>>>(norms, nb, K, W, pass, hist);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        topk_eq_kernel<<<grid, kSelThreads, 0, s>>>(norms, nb, K, W, hist, eq);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    topk_keep_kernel<<<grid, kSelThreads, 0, s>>>(norms, nb, K, W, hist, eq, keep);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (n % 4 == 0)
        topk_apply_kernel<true><<<grid_for(topk_apply_kernel<true>, blocks), kThreads, 0, s>>>(resid, keep, n, block, nb,
                                                                                               W, sparse);
    else
        topk_apply_kernel<false><<<grid_for(topk_apply_kernel<false>, blocks), kThreads, 0, s>>>(resid, keep, n, block,
                                                                                                 nb, W, sparse);
    return cudaGetLastError();
}

}  // namespace s2
