// Compression phase of S2 Reducer ("S2 Reducer", Section 3.1 "Compressing
// Sparse Gradient"; Algorithm 1, compression loop), one fused pass per worker:
//   bitmap: bit i set iff g(i) is nonzero;
//   sketch: for every nonzero i and row j, S[j][h_j(i)] += s_j(i) * g(i).
//
// Design (sm_103a): the gradient is the only large input and is read exactly
// once with streaming (evict-first) loads, so the sketch being built stays in
// L2. A warp owns a task of 512 consecutive positions: it loads them, forms
// the 16 bitmap words with warp shuffles (or ballots), stores them with one
// 64-byte store, and then each lane walks only its own nonzero slots, issuing
// d fire-and-forget float reductions (red.global.add.f32) that resolve in L2.
// Work is proportional to the nonzeros, whatever their pattern (whole rows or
// scattered entries). Tasks are handed out worker-major so that the sketches
// being written at any moment are those of one or two workers.
#include "s2_internal.h"

namespace s2 {
namespace {

// Pick 32-bit lane-slot `slot` (0..15) out of four 16-byte vectors.
__device__ __forceinline__ uint32_t pick16(const uint4 (&v)[4], int slot) {
    uint4 q = (slot < 8) ? ((slot < 4) ? v[0] : v[1]) : ((slot < 12) ? v[2] : v[3]);
    int c = slot & 3;
    return c == 0 ? q.x : (c == 1 ? q.y : (c == 2 ? q.z : q.w));
}

// Insert value `val` of position `i` into every row of the sketch.
template <int D>
__device__ __forceinline__ void insert(float* __restrict__ sk, uint32_t i, float val, int d, uint32_t w,
                                       const uint32_t* s_kh, const uint32_t* s_ks) {
    const int rows = D > 0 ? D : d;
#pragma unroll
    for (int j = 0; j < (D > 0 ? D : kMaxRows); ++j) {
        if (D > 0 || j < rows) {
            uint32_t b = bucket_of(i, s_kh[j], w);
            uint32_t sb = signbit_of(i, s_ks[j]);
            red_add_f32(sk + (uint64_t)j * w + b, apply_sign(val, sb));
        }
    }
}

__device__ __forceinline__ void load_keys(const RowKeys& k, uint32_t* s_kh, uint32_t* s_ks) {
    if (threadIdx.x < kMaxRows) {
        s_kh[threadIdx.x] = k.kh[threadIdx.x];
        s_ks[threadIdx.x] = k.ks[threadIdx.x];
    }
    __syncthreads();
}

// ---- fp32, 16-byte vector loads --------------------------------------------
// Lane l loads positions u*128 + 4l .. +3 of the task for u = 0..3; slot
// 4u + c is position u*128 + 4l + c. Word q of chunk u is made of the
// nibbles of lanes 8q .. 8q+7.
template <int D>
__global__ void __launch_bounds__(kThreads) encode_f32_vec(EncodeArgs a) {
    __shared__ uint32_t s_kh[kMaxRows], s_ks[kMaxRows];
    load_keys(a.keys, s_kh, s_ks);
    const int lane = threadIdx.x & 31;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    uint32_t k = 0;
    uint32_t local = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    while (local >= a.tasks_per_worker && k < a.workers) {
        local -= a.tasks_per_worker;
        ++k;
    }
    for (; k < a.workers;) {
        const uint64_t e0 = (uint64_t)local * kTaskElems;
        const float* g = reinterpret_cast<const float*>(a.grad) + (uint64_t)k * a.n;
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint64_t e = e0 + u * 128 + lane * 4;
            if (e + 4 <= a.n) {
                v[u] = ld_stream_u4(g + e);
            } else {
                v[u] = make_uint4(0, 0, 0, 0);
                if (e + 0 < a.n) v[u].x = ld_stream_u32(g + e + 0);
                if (e + 1 < a.n) v[u].y = ld_stream_u32(g + e + 1);
                if (e + 2 < a.n) v[u].z = ld_stream_u32(g + e + 2);
            }
        }
        uint32_t mask = 0;
        uint32_t my_word = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t nib = ((v[u].x & 0x7fffffffu) != 0) | (((v[u].y & 0x7fffffffu) != 0) << 1) |
                           (((v[u].z & 0x7fffffffu) != 0) << 2) | (((v[u].w & 0x7fffffffu) != 0) << 3);
            mask |= nib << (4 * u);
            uint32_t part = nib << (4 * (lane & 7));
            part |= __shfl_xor_sync(kFull, part, 1);
            part |= __shfl_xor_sync(kFull, part, 2);
            part |= __shfl_xor_sync(kFull, part, 4);
            uint32_t got = __shfl_sync(kFull, part, (lane & 3) * 8);
            if ((lane >> 2) == u) my_word = got;
        }
        if (lane < kTaskWords) {
            const uint64_t wi = (uint64_t)local * kTaskWords + lane;
            if (wi < a.nw) a.bitmaps[(uint64_t)k * a.nw + wi] = my_word;
        }
        float* sk = a.sketches + (uint64_t)k * a.dw;
        while (mask) {
            const int slot = __ffs(mask) - 1;
            mask &= mask - 1;
            const uint32_t i = (uint32_t)(e0 + (slot >> 2) * 128 + lane * 4 + (slot & 3));
            insert<D>(sk, i, __uint_as_float(pick16(v, slot)), a.d, a.w, s_kh, s_ks);
        }
        local += nwarps;
        while (local >= a.tasks_per_worker && k < a.workers) {
            local -= a.tasks_per_worker;
            ++k;
        }
    }
}

// ---- bf16, 16-byte vector loads --------------------------------------------
// Lane l loads positions u*256 + 8l .. +7 for u = 0..1; slot 8u + c is
// position u*256 + 8l + c. Word q of chunk u is made of the bytes of lanes
// 4q .. 4q+3.
template <int D>
__global__ void __launch_bounds__(kThreads) encode_bf16_vec(EncodeArgs a) {
    __shared__ uint32_t s_kh[kMaxRows], s_ks[kMaxRows];
    load_keys(a.keys, s_kh, s_ks);
    const int lane = threadIdx.x & 31;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    uint32_t k = 0;
    uint32_t local = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    while (local >= a.tasks_per_worker && k < a.workers) {
        local -= a.tasks_per_worker;
        ++k;
    }
    for (; k < a.workers;) {
        const uint64_t e0 = (uint64_t)local * kTaskElems;
        const uint16_t* g = reinterpret_cast<const uint16_t*>(a.grad) + (uint64_t)k * a.n;
        uint4 v[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const uint64_t e = e0 + u * 256 + lane * 8;
            if (e + 8 <= a.n) {
                v[u] = ld_stream_u4(g + e);
            } else {
                uint32_t h[4] = {0, 0, 0, 0};
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (e + c < a.n) h[c >> 1] |= (uint32_t)ld_stream_u16(g + e + c) << (16 * (c & 1));
                v[u] = make_uint4(h[0], h[1], h[2], h[3]);
            }
        }
        uint32_t mask = 0;
        uint32_t my_word = 0;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const uint32_t q[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            uint32_t byte = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                byte |= ((q[c] & 0x7fffu) != 0) << (2 * c);
                byte |= ((q[c] & 0x7fff0000u) != 0) << (2 * c + 1);
            }
            mask |= byte << (8 * u);
            uint32_t part = byte << (8 * (lane & 3));
            part |= __shfl_xor_sync(kFull, part, 1);
            part |= __shfl_xor_sync(kFull, part, 2);
            uint32_t got = __shfl_sync(kFull, part, (lane & 7) * 4);
            if ((lane >> 3) == u) my_word = got;
        }
        if (lane < kTaskWords) {
            const uint64_t wi = (uint64_t)local * kTaskWords + lane;
            if (wi < a.nw) a.bitmaps[(uint64_t)k * a.nw + wi] = my_word;
        }
        float* sk = a.sketches + (uint64_t)k * a.dw;
        while (mask) {
            const int slot = __ffs(mask) - 1;
            mask &= mask - 1;
            const uint4 q = (slot < 8) ? v[0] : v[1];
            const int c = slot & 7;
            const uint32_t word = (c >> 1) == 0 ? q.x : ((c >> 1) == 1 ? q.y : ((c >> 1) == 2 ? q.z : q.w));
            const uint32_t bits = (c & 1) ? (word & 0xffff0000u) : (word << 16);
            const uint32_t i = (uint32_t)(e0 + (slot >> 3) * 256 + lane * 8 + c);
            insert<D>(sk, i, __uint_as_float(bits), a.d, a.w, s_kh, s_ks);
        }
        local += nwarps;
        while (local >= a.tasks_per_worker && k < a.workers) {
            local -= a.tasks_per_worker;
            ++k;
        }
    }
}

// ---- any alignment: one element per lane and load -------------------------
// Lane l loads position u*32 + l for u = 0..15; a ballot gives word u
// directly; slot u is position u*32 + l.
template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads) encode_scalar(EncodeArgs a) {
    __shared__ uint32_t s_kh[kMaxRows], s_ks[kMaxRows];
    load_keys(a.keys, s_kh, s_ks);
    const int lane = threadIdx.x & 31;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    uint32_t k = 0;
    uint32_t local = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    while (local >= a.tasks_per_worker && k < a.workers) {
        local -= a.tasks_per_worker;
        ++k;
    }
    for (; k < a.workers;) {
        const uint64_t e0 = (uint64_t)local * kTaskElems;
        uint32_t x[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const uint64_t e = e0 + u * 32 + lane;
            x[u] = 0;
            if (e < a.n) {
                if (BF16)
                    x[u] = (uint32_t)ld_stream_u16(reinterpret_cast<const uint16_t*>(a.grad) +
                                                   (uint64_t)k * a.n + e)
                           << 16;
                else
                    x[u] = ld_stream_u32(reinterpret_cast<const float*>(a.grad) + (uint64_t)k * a.n + e);
            }
        }
        uint32_t mask = 0;
        uint32_t my_word = 0;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const bool nz = (x[u] & 0x7fffffffu) != 0;
            const uint32_t word = __ballot_sync(kFull, nz);
            mask |= (uint32_t)nz << u;
            if (lane == u) my_word = word;
        }
        if (lane < kTaskWords) {
            const uint64_t wi = (uint64_t)local * kTaskWords + lane;
            if (wi < a.nw) a.bitmaps[(uint64_t)k * a.nw + wi] = my_word;
        }
        float* sk = a.sketches + (uint64_t)k * a.dw;
        while (mask) {
            const int slot = __ffs(mask) - 1;
            mask &= mask - 1;
            uint32_t bits = x[0];
#pragma unroll
            for (int s = 1; s < 16; ++s) bits = (slot == s) ? x[s] : bits;
            const uint32_t i = (uint32_t)(e0 + slot * 32 + lane);
            insert<D>(sk, i, __uint_as_float(bits), a.d, a.w, s_kh, s_ks);
        }
        local += nwarps;
        while (local >= a.tasks_per_worker && k < a.workers) {
            local -= a.tasks_per_worker;
            ++k;
        }
    }
}

// Zero `count` floats from any 4-byte-aligned address: a scalar head up to
// the first 16-byte boundary, 16-byte stores, a scalar tail.
__global__ void __launch_bounds__(kThreads) zero_f32(float* __restrict__ p, uint64_t count) {
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    uint64_t head = ((16u - (reinterpret_cast<uintptr_t>(p) & 15u)) & 15u) / 4u;
    if (head > count) head = count;
    if (tid < head) p[tid] = 0.f;
    float* body = p + head;
    const uint64_t n4 = (count - head) / 4;
    float4* p4 = reinterpret_cast<float4*>(body);
    for (uint64_t x = tid; x < n4; x += stride) p4[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (uint64_t x = head + n4 * 4 + tid; x < count; x += stride) p[x] = 0.f;
}

template <int D>
cudaError_t launch_encode_d(const EncodeArgs& a, int dtype, bool vec, cudaStream_t s) {
    const uint64_t tasks = (uint64_t)a.workers * a.tasks_per_worker;
    const uint64_t blocks = (tasks + (kThreads / 32) - 1) / (kThreads / 32);
    if (vec && dtype == 0) {
        encode_f32_vec<D><<<grid_for(encode_f32_vec<D>, blocks), kThreads, 0, s>>>(a);
    } else if (vec && dtype == 1) {
        encode_bf16_vec<D><<<grid_for(encode_bf16_vec<D>, blocks), kThreads, 0, s>>>(a);
    } else if (dtype == 0) {
        encode_scalar<D, false><<<grid_for(encode_scalar<D, false>, blocks), kThreads, 0, s>>>(a);
    } else {
        encode_scalar<D, true><<<grid_for(encode_scalar<D, true>, blocks), kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_encode(const EncodeArgs& a, int dtype, bool vec, cudaStream_t s) {
    if (a.workers == 0 || a.tasks_per_worker == 0) return cudaSuccess;
    switch (a.d) {
        case 3: return launch_encode_d<3>(a, dtype, vec, s);
        case 5: return launch_encode_d<5>(a, dtype, vec, s);
        case 1: return launch_encode_d<1>(a, dtype, vec, s);
        default: return launch_encode_d<0>(a, dtype, vec, s);
    }
}

cudaError_t launch_zero(float* p, uint64_t count, cudaStream_t s) {
    if (count == 0) return cudaSuccess;
    const uint64_t blocks = (count / 4 + kThreads - 1) / kThreads + 1;
    zero_f32<<<grid_for(zero_f32, blocks), kThreads, 0, s>>>(p, count);
    return cudaGetLastError();
}

}  // namespace s2
