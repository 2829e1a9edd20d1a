// Block-wise Top-K sparsification with error feedback, upstream of encode
// ("S2 Reducer", Section 2.2 "Sparse Gradient & AllGather": keep the K blocks
// of largest l2 norm; Appendix A.2: the residual e_{t+1} = g_t - U(g_t) is
// carried into the next step's gradient).
//
// Per worker: acc = grad + residual; the squared norm of every block of
// `block` elements in one fixed fp32 order (lane l of a warp accumulates
// fmaf(a, a, s) over elements l, l+32, ... of the block, then a fixed XOR
// butterfly), so that which blocks are kept -- an integer decision -- does
// not depend on scheduling; the K-th largest norm by a 4-pass 8-bit radix
// select over the norms' bit patterns (non-negative floats order like their
// bits), ties broken towards the lower block index by an ordered block-wide
// scan; finally sparse = acc on kept blocks and residual = acc elsewhere.
// Three kernels, no inter-block waiting.
#include "s2_internal.h"

namespace s2 {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelUnroll = 8;

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

// One block of kSelThreads threads per worker: keep[k][x] = 1 for the K
// blocks of largest norm (ties: lower index).
__global__ void __launch_bounds__(kSelThreads)
    topk_select_kernel(const float* __restrict__ norms, uint64_t nb, uint64_t K, uint8_t* __restrict__ keep) {
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_digit, s_rest;
    __shared__ uint32_t s_scan[kSelThreads / 32];
    const uint32_t k = blockIdx.x;
    const uint32_t* key = reinterpret_cast<const uint32_t*>(norms) + (uint64_t)k * nb;
    uint8_t* kp = keep + (uint64_t)k * nb;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (K == 0 || K >= nb) {
        for (uint64_t x = threadIdx.x; x < nb; x += kSelThreads) kp[x] = K == 0 ? 0 : 1;
        return;
    }
    // radix select of the K-th largest key: prefix/mask narrow down, `rest`
    // counts how many keys equal to the final prefix are to be kept
    uint32_t prefix = 0, pmask = 0;
    uint64_t rest = K;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += kSelThreads) s_hist[b] = 0;
        __syncthreads();
        for (uint64_t x0 = 0; x0 < nb; x0 += kSelUnroll * kSelThreads) {
            uint32_t v[kSelUnroll];
#pragma unroll
            for (int q = 0; q < kSelUnroll; ++q) {  // independent loads first
                const uint64_t x = x0 + q * kSelThreads + threadIdx.x;
                v[q] = x < nb ? key[x] : 0u;
            }
#pragma unroll
            for (int q = 0; q < kSelUnroll; ++q) {
                const uint64_t x = x0 + q * kSelThreads + threadIdx.x;
                const bool in = x < nb && (v[q] & pmask) == prefix;
                const uint32_t dg = in ? (v[q] >> shift) & 255u : 256u;  // 256: no vote
                const unsigned grp = __match_any_sync(kFull, dg);
                if (in && __ffs(grp) - 1 == lane) atomicAdd(&s_hist[dg], (uint32_t)__popc(grp));
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            uint64_t above = 0;
            int dg = 255;
            for (; dg > 0; --dg) {
                if (above + s_hist[dg] >= rest) break;
                above += s_hist[dg];
            }
            s_digit = (uint32_t)dg;
            s_rest = (uint32_t)(rest - above);
        }
        __syncthreads();
        prefix |= s_digit << shift;
        pmask |= 255u << shift;
        rest = s_rest;
        __syncthreads();
    }
    // keep every key above the threshold and the first `rest` keys equal to
    // it in index order
    const uint32_t thr = prefix;
    uint32_t taken = 0;  // equal keys already kept (uniform across the block)
    for (uint64_t x0 = 0; x0 < nb; x0 += kSelThreads) {
        const uint64_t x = x0 + threadIdx.x;
        const uint32_t v = x < nb ? key[x] : 0u;
        const bool eq = x < nb && v == thr;
        const unsigned bal = __ballot_sync(kFull, eq);
        if (lane == 0) s_scan[warp] = __popc(bal);
        __syncthreads();
        uint32_t before = taken;
        for (int q = 0; q < warp; ++q) before += s_scan[q];
        before += __popc(bal & ((1u << lane) - 1u));
        if (x < nb) kp[x] = (v > thr || (eq && before < rest)) ? 1 : 0;
        uint32_t chunk = 0;
        for (int q = 0; q < kSelThreads / 32; ++q) chunk += s_scan[q];
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

size_t topk_workspace_bytes(uint32_t W, uint64_t n, uint32_t block) {
    const uint64_t nb = (n + block - 1) / block;
    const uint64_t norms = ((uint64_t)W * nb * 4 + 255) / 256 * 256;
    return (size_t)(norms + ((uint64_t)W * nb + 255) / 256 * 256);
}

cudaError_t launch_block_topk(const float* grad, float* resid, uint32_t W, uint64_t n, uint32_t block, uint64_t K,
                              float* sparse, void* workspace, cudaStream_t s) {
    const uint64_t nb = (n + block - 1) / block;
    if ((uint64_t)W * nb == 0) return cudaSuccess;
    float* norms = static_cast<float*>(workspace);
    uint8_t* keep = static_cast<uint8_t*>(workspace) + ((uint64_t)W * nb * 4 + 255) / 256 * 256;
    const uint64_t blocks = ((uint64_t)W * nb + (kThreads / 32) - 1) / (kThreads / 32);
    topk_norms_kernel<<<grid_for(topk_norms_kernel, blocks), kThreads, 0, s>>>(grad, resid, n, block, nb, W, norms);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    topk_select_kernel<<<W, kSelThreads, 0, s>>>(norms, nb, K, keep);
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
