// Fused single-sketch mode: encode and reduce in one pass for W workers that
// live on the same GPU ("S2 Reducer", Section 3.1 "Collecting Sparse-Sketch
// with AllReduce": the sketch is linear, so the sum of the workers' sketches
// equals the sketch of the summed gradient, and the aggregated bitmap marks
// every position some worker marked).
//
// A warp owns 512 consecutive positions and walks the W workers' rows for
// them: it ORs the workers' nonzero bits and sums their values per position
// in registers (fixed worker order 0..W-1), writes the aggregate bitmap words
// from one ballot per 32 positions, and issues d sketch reductions per
// position of the union whose summed value is not zero. Compared with
// encode_batched + reduce it skips the W per-worker sketches (their zero
// fill, reductions, write-back and re-read) and issues d reductions per
// union position instead of per worker nonzero. The per-worker structures a
// real distributed run would transmit are never formed, which is why this is
// a separate entry point and not the simulated data-parallel path.
//
// The reductions carry no L2 policy: the zero fill stored the sketch's lines
// evict-last (large LM, 84 MB sketch: 1.323 ms per step with evict-last
// reductions, 1.277 without; embedding and top-k within 0.5 %).
//
// Two layouts: fp32 rows that are 16-byte aligned go through 16-byte vector
// loads; every other case (bf16, unaligned rows) has lane l load position
// u*32 + l of the task (u = 0..15) with plain 4- or 2-byte loads.
#include "s2_internal.h"

namespace s2 {
namespace {

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads) fused_encode_reduce(FusedArgs a) {
    __shared__ uint32_t s_kh[kMaxRows], s_ks[kMaxRows];
    if (threadIdx.x < kMaxRows) {
        s_kh[threadIdx.x] = a.keys.kh[threadIdx.x];
        s_ks[threadIdx.x] = a.keys.ks[threadIdx.x];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const uint64_t ntasks = (a.n + kTaskElems - 1) / kTaskElems;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t t = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < ntasks; t += nwarps) {
        const uint64_t e0 = t * kTaskElems;
        float acc[16];
        uint32_t nzmask = 0;
#pragma unroll
        for (int u = 0; u < 16; ++u) acc[u] = 0.f;
#pragma unroll 2
        for (uint32_t k = 0; k < a.workers; ++k) {
            uint32_t x[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const uint64_t e = e0 + u * 32 + lane;
                x[u] = 0;
                if (e < a.n) {
                    if (BF16)
                        x[u] = (uint32_t)ld_stream_u16(static_cast<const uint16_t*>(a.grad) + (uint64_t)k * a.n + e)
                               << 16;
                    else
                        x[u] = ld_stream_u32(static_cast<const float*>(a.grad) + (uint64_t)k * a.n + e);
                }
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                nzmask |= (uint32_t)((x[u] & 0x7fffffffu) != 0) << u;
                acc[u] += __uint_as_float(x[u]);
            }
        }
        uint32_t my_word = 0;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const uint32_t word = __ballot_sync(kFull, (nzmask >> u) & 1u);
            if (lane == u) my_word = word;
        }
        if (lane < kTaskWords) {
            const uint64_t wi = t * kTaskWords + lane;
            if (wi < a.nw) a.bitmap[wi] = my_word;
        }
        for (uint32_t m = nzmask; m; m &= m - 1) {
            const int u = __ffs(m) - 1;
            float v = acc[0];
#pragma unroll
            for (int s = 1; s < 16; ++s) v = (u == s) ? acc[s] : v;
            if (v == 0.f) continue;  // the workers' values cancel: nothing to add
            const uint32_t i = (uint32_t)(e0 + u * 32 + lane);
            const int rows = D > 0 ? D : a.d;
#pragma unroll
            for (int j = 0; j < (D > 0 ? D : kMaxRows); ++j) {
                if (D > 0 || j < rows) {
                    const uint32_t b = bucket_of(i, s_kh[j], a.w);
                    red_add_f32(a.sketch + (uint64_t)j * a.w + b, apply_sign(v, signbit_of(i, s_ks[j])));
                }
            }
        }
    }
}

// fp32 rows that are 16-byte aligned: lane l holds positions u*128 + 4l + c
// of the task in 16-byte vectors (u = 0..3), the next worker's vectors are
// loaded before the current ones are added, and the bitmap words are
// assembled from the lanes' nibbles with shuffles (word q of chunk u is made
// of lanes 8q..8q+7).
__device__ __forceinline__ void load_vec4(uint4 (&v)[4], const float* g, uint64_t e0, uint64_t n, int lane) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint64_t e = e0 + u * 128 + lane * 4;
        if (e + 4 <= n) {
            v[u] = ld_stream_u4(g + e);
        } else {
            v[u] = make_uint4(0, 0, 0, 0);
            if (e + 0 < n) v[u].x = ld_stream_u32(g + e + 0);
            if (e + 1 < n) v[u].y = ld_stream_u32(g + e + 1);
            if (e + 2 < n) v[u].z = ld_stream_u32(g + e + 2);
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads) fused_f32_vec(FusedArgs a) {
    __shared__ uint32_t s_kh[kMaxRows], s_ks[kMaxRows];
    if (threadIdx.x < kMaxRows) {
        s_kh[threadIdx.x] = a.keys.kh[threadIdx.x];
        s_ks[threadIdx.x] = a.keys.ks[threadIdx.x];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const uint64_t ntasks = (a.n + kTaskElems - 1) / kTaskElems;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    const float* grad = static_cast<const float*>(a.grad);
    for (uint64_t t = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < ntasks; t += nwarps) {
        const uint64_t e0 = t * kTaskElems;
        float acc[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) acc[s] = 0.f;
        uint32_t mask = 0;
        uint4 v[4];
        if (a.workers > 0) load_vec4(v, grad, e0, a.n, lane);
        for (uint32_t k = 0; k < a.workers; ++k) {
            uint4 nv[4];
            if (k + 1 < a.workers) load_vec4(nv, grad + (uint64_t)(k + 1) * a.n, e0, a.n, lane);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t q[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    mask |= (uint32_t)((q[c] & 0x7fffffffu) != 0) << (4 * u + c);
                    acc[4 * u + c] += __uint_as_float(q[c]);
                }
            }
            if (k + 1 < a.workers) {
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = nv[u];
            }
        }
        uint32_t my_word = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t part = ((mask >> (4 * u)) & 0xfu) << (4 * (lane & 7));
            part |= __shfl_xor_sync(kFull, part, 1);
            part |= __shfl_xor_sync(kFull, part, 2);
            part |= __shfl_xor_sync(kFull, part, 4);
            const uint32_t got = __shfl_sync(kFull, part, (lane & 3) * 8);
            if ((lane >> 2) == u) my_word = got;
        }
        if (lane < kTaskWords) {
            const uint64_t wi = t * kTaskWords + lane;
            if (wi < a.nw) a.bitmap[wi] = my_word;
        }
        for (uint32_t m = mask; m; m &= m - 1) {
            const int slot = __ffs(m) - 1;
            float val = acc[0];
#pragma unroll
            for (int s = 1; s < 16; ++s) val = (slot == s) ? acc[s] : val;
            if (val == 0.f) continue;  // the workers' values cancel: nothing to add
            const uint32_t i = (uint32_t)(e0 + (slot >> 2) * 128 + lane * 4 + (slot & 3));
            const int rows = D > 0 ? D : a.d;
#pragma unroll
            for (int j = 0; j < (D > 0 ? D : kMaxRows); ++j) {
                if (D > 0 || j < rows) {
                    const uint32_t b = bucket_of(i, s_kh[j], a.w);
                    red_add_f32(a.sketch + (uint64_t)j * a.w + b, apply_sign(val, signbit_of(i, s_ks[j])));
                }
            }
        }
    }
}

template <int D, bool BF16>
cudaError_t launch_fused_t(const FusedArgs& a, cudaStream_t s) {
    const uint64_t tasks = (a.n + kTaskElems - 1) / kTaskElems;
    const uint64_t blocks = (tasks + (kThreads / 32) - 1) / (kThreads / 32);
    fused_encode_reduce<D, BF16><<<grid_for(fused_encode_reduce<D, BF16>, blocks), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_fused_d(const FusedArgs& a, int dtype, cudaStream_t s) {
    // 16-byte vectors need every worker row aligned (the base is checked by the API)
    if (dtype == 0 && ((a.n * 4) % 16 == 0 || a.workers == 1)) {
        const uint64_t tasks = (a.n + kTaskElems - 1) / kTaskElems;
        const uint64_t blocks = (tasks + (kThreads / 32) - 1) / (kThreads / 32);
        fused_f32_vec<D><<<grid_for(fused_f32_vec<D>, blocks), kThreads, 0, s>>>(a);
        return cudaGetLastError();
    }
    return dtype == 0 ? launch_fused_t<D, false>(a, s) : launch_fused_t<D, true>(a, s);
}

}  // namespace

cudaError_t launch_fused(const FusedArgs& a, int dtype, cudaStream_t s) {
    cudaError_t e = launch_zero(a.sketch, (uint64_t)a.d * a.w, s);
    if (e != cudaSuccess || a.n == 0) return e;
    switch (a.d) {
        case 3: return launch_fused_d<3>(a, dtype, s);
        case 5: return launch_fused_d<5>(a, dtype, s);
        case 1: return launch_fused_d<1>(a, dtype, s);
        default: return launch_fused_d<0>(a, dtype, s);
    }
}

}  // namespace s2
