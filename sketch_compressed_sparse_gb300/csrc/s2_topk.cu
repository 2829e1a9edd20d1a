// Block-wise Top-K sparsification with error feedback, upstream of encode
// ("S2 Reducer", Section 2.2 "Sparse Gradient & AllGather": keep the K blocks
// of largest l2 norm; Appendix A.2: the residual e_{t+1} = g_t - U(g_t) is
// carried into the next step's gradient).
//
// Per worker: acc = grad + residual; the squared norm of every block of
// `block` elements in float32, one warp per block (lane l accumulates
// fmaf(a, a, s) over elements l, l+32, ... of the block, then an XOR
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
// passes' histograms to find the prefix it must match); a counting launch
// and a marking launch then keep every norm above the final threshold and,
// of the norms equal to it, the first ones in index order (each block starts
// its rank after the equal norms of the blocks before it). No launch waits on
// another block.
#include "s2_internal.h"

namespace s2 {
namespace {

// Squared norm of block x of worker k, one warp per (k, x) task.
__global__ void __launch_bounds__(kThreads)
    topk_norms_kernel(const float* __restrict__ grad, const float* __restrict__ resid, uint64_t n, uint32_t block,
                      uint64_t nb, uint32_t W, float* __restrict__ norms) {
    const int lane = threadIdx.x & 31;
    const uint64_t tasks = (uint64_t)W * nb;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t t = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < tasks; t += nwarps) {
        const uint64_t k = t / nb, x = t - k * nb;
        const uint64_t base = k * n + x * block;
        const uint64_t len = (x + 1) * block <= n ? block : n - x * block;
        float s = 0.f;
#pragma unroll 8
        for (uint64_t j = lane; j < len; j += 32) {
            const float a = __fadd_rn(ld_stream_f32(grad + base + j), __ldg(resid + base + j));
            s = __fmaf_rn(a, a, s);
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
// be kept. hist: [4][W][256] digit counts of the passes (pass-major).
__device__ void select_state(const uint32_t* __restrict__ hist, uint32_t W, uint32_t k, int passes, uint64_t K,
                             uint32_t* prefix, uint32_t* pmask, uint64_t* rest) {
    uint32_t pf = 0, pm = 0;
    uint64_t r = K;
    for (int p = 0; p < passes; ++p) {
        const uint32_t* h = hist + ((uint64_t)p * W + k) * 256;
        const int shift = 24 - 8 * p;
        uint64_t above = 0;
        int dg = 255;
        for (; dg > 0; --dg) {
            if (above + h[dg] >= r) break;
            above += h[dg];
        }
        pf |= (uint32_t)dg << shift;
        pm |= 255u << shift;
        r -= above;
    }
    *prefix = pf;
    *pmask = pm;
    *rest = r;
}

// Pass `pass` of the radix select: digit counts of the norms that match the
// prefix fixed by the earlier passes. Grid: (W, slices).
__global__ void __launch_bounds__(kSelThreads)
    topk_hist_kernel(const float* __restrict__ norms, uint64_t nb, uint64_t K, uint32_t W, int pass,
                     uint32_t* __restrict__ hist) {
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_prefix, s_pmask;
    const uint32_t k = blockIdx.x;
    if (threadIdx.x == 0) {
        uint64_t rest;
        select_state(hist, W, k, pass, K, &s_prefix, &s_pmask, &rest);
    }
    s_hist[threadIdx.x] = 0;  // kSelThreads == 256 bins
    __syncthreads();
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
    __shared__ uint32_t s_thr;
    __shared__ uint32_t s_warp[kSelThreads / 32];
    const uint32_t k = blockIdx.x;
    if (threadIdx.x == 0) {
        uint32_t pm;
        uint64_t rest;
        select_state(hist, W, k, 4, K, &s_thr, &pm, &rest);
    }
    __syncthreads();
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
    __shared__ uint32_t s_thr;
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
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t pm;
        uint64_t rest;
        select_state(hist, W, k, 4, K, &s_thr, &pm, &rest);
        s_rest = rest;
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
// kept blocks. VEC: worker rows are 16-byte aligned (n % 4 == 0), so every
// block (a multiple of 32 elements) starts on a 16-byte boundary.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
    topk_apply_kernel(const float* __restrict__ grad, float* __restrict__ resid, const uint8_t* __restrict__ keep,
                      uint64_t n, uint32_t block, uint64_t nb, uint32_t W, float* __restrict__ sparse) {
    const int lane = threadIdx.x & 31;
    const uint64_t tasks = (uint64_t)W * nb;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t t = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < tasks; t += nwarps) {
        const uint64_t k = t / nb, x = t - k * nb;
        const uint64_t base = k * n + x * block;
        const uint64_t len = (x + 1) * block <= n ? block : n - x * block;
        const bool kept = keep[t] != 0;
        uint64_t j0 = 0;
        if (VEC) {
            const uint64_t len4 = len / 4;
#pragma unroll 4
            for (uint64_t j = lane; j < len4; j += 32) {
                const uint4 g = ld_stream_u4(grad + base + 4 * j);
                const float4 r = reinterpret_cast<const float4*>(resid + base)[j];
                const float4 a = make_float4(__fadd_rn(__uint_as_float(g.x), r.x), __fadd_rn(__uint_as_float(g.y), r.y),
                                             __fadd_rn(__uint_as_float(g.z), r.z), __fadd_rn(__uint_as_float(g.w), r.w));
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4*>(sparse + base)[j] = kept ? a : z;
                reinterpret_cast<float4*>(resid + base)[j] = kept ? z : a;
            }
            j0 = len4 * 4;
        }
        for (uint64_t j = j0 + lane; j < len; j += 32) {
            const float a = __fadd_rn(ld_stream_f32(grad + base + j), resid[base + j]);
            sparse[base + j] = kept ? a : 0.f;
            resid[base + j] = kept ? 0.f : a;
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
    topk_norms_kernel<<<grid_for(topk_norms_kernel, blocks), kThreads, 0, s>>>(grad, resid, n, block, nb, W, norms);
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
        topk_apply_kernel<true><<<grid_for(topk_apply_kernel<true>, blocks), kThreads, 0, s>>>(grad, resid, keep, n, block,
                                                                                               nb, W, sparse);
    else
        topk_apply_kernel<false><<<grid_for(topk_apply_kernel<false>, blocks), kThreads, 0, s>>>(grad, resid, keep, n,
                                                                                                 block, nb, W, sparse);
    return cudaGetLastError();
}

}  // namespace s2
