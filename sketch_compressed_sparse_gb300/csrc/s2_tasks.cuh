// Device helpers shared by the encode kernels: loading a warp task of 512
// consecutive positions of one worker into registers, forming its bitmap
// words, and picking out a lane's nonzero slots.
//
// The task registers of every load layout fit in four 16-byte vectors:
//   L = 0: fp32, vector loads: slot 4u+c is position u*128 + 4*lane + c;
//   L = 1: bf16, vector loads: slot 8u+c is position u*256 + 8*lane + c;
//   L = 2: fp32, 4-byte loads: slot u is position u*32 + lane;
//   L = 3: bf16, 2-byte loads: as L = 2, the value in the word's upper half.
#pragma once

#include "s2_internal.h"

namespace s2 {

// Pick 32-bit lane-slot `slot` (0..15) out of four 16-byte vectors.
__device__ __forceinline__ uint32_t pick16(const uint4 (&v)[4], int slot) {
    uint4 q = (slot < 8) ? ((slot < 4) ? v[0] : v[1]) : ((slot < 12) ? v[2] : v[3]);
    int c = slot & 3;
    return c == 0 ? q.x : (c == 1 ? q.y : (c == 2 ? q.z : q.w));
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
// Load the 4 vectors of lane `lane` for the fp32 task at e0 of row g.
__device__ __forceinline__ void load_f32_task(uint4 (&v)[4], const float* g, uint64_t e0, uint64_t n, int lane) {
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

template <int L>
__device__ __forceinline__ void load_task(uint4 (&v)[4], const void* row, uint64_t e0, uint64_t n, int lane) {
    if constexpr (L == 0) {
        load_f32_task(v, static_cast<const float*>(row), e0, n, lane);
    } else if constexpr (L == 1) {
        const uint16_t* g = static_cast<const uint16_t*>(row);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const uint64_t e = e0 + u * 256 + lane * 8;
            if (e + 8 <= n) {
                v[u] = ld_stream_u4(g + e);
            } else {
                uint32_t h[4] = {0, 0, 0, 0};
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (e + c < n) h[c >> 1] |= (uint32_t)ld_stream_u16(g + e + c) << (16 * (c & 1));
                v[u] = make_uint4(h[0], h[1], h[2], h[3]);
            }
        }
        v[2] = v[3] = make_uint4(0, 0, 0, 0);
    } else {
        uint32_t x[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const uint64_t e = e0 + u * 32 + lane;
            x[u] = 0;
            if (e < n) {
                if constexpr (L == 2)
                    x[u] = ld_stream_u32(static_cast<const float*>(row) + e);
                else
                    x[u] = (uint32_t)ld_stream_u16(static_cast<const uint16_t*>(row) + e) << 16;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = make_uint4(x[4 * u], x[4 * u + 1], x[4 * u + 2], x[4 * u + 3]);
    }
}

// Nonzero mask of the lane's 16 slots; *word gets bitmap word `lane` of the
// task (meaningful on lanes 0..15).
template <int L>
__device__ __forceinline__ uint32_t task_bits(const uint4 (&v)[4], int lane, uint32_t* word) {
    uint32_t mask = 0, my_word = 0;
    if constexpr (L == 0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t nib = ((v[u].x & 0x7fffffffu) != 0) | (((v[u].y & 0x7fffffffu) != 0) << 1) |
                                 (((v[u].z & 0x7fffffffu) != 0) << 2) | (((v[u].w & 0x7fffffffu) != 0) << 3);
            mask |= nib << (4 * u);
            uint32_t part = nib << (4 * (lane & 7));
            part |= __shfl_xor_sync(kFull, part, 1);
            part |= __shfl_xor_sync(kFull, part, 2);
            part |= __shfl_xor_sync(kFull, part, 4);
            const uint32_t got = __shfl_sync(kFull, part, (lane & 3) * 8);
            if ((lane >> 2) == u) my_word = got;
        }
    } else if constexpr (L == 1) {
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
            const uint32_t got = __shfl_sync(kFull, part, (lane & 7) * 4);
            if ((lane >> 3) == u) my_word = got;
        }
    } else {
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const uint4 q = v[u >> 2];
            const uint32_t x = (u & 3) == 0 ? q.x : ((u & 3) == 1 ? q.y : ((u & 3) == 2 ? q.z : q.w));
            const bool nz = (x & 0x7fffffffu) != 0;
            const uint32_t b = __ballot_sync(kFull, nz);
            mask |= (uint32_t)nz << u;
            if (lane == u) my_word = b;
        }
    }
    *word = my_word;
    return mask;
}

template <int L>
__device__ __forceinline__ uint32_t slot_bits(const uint4 (&v)[4], int slot) {
    if constexpr (L == 1) {
        const uint4 q = (slot < 8) ? v[0] : v[1];
        const int c = slot & 7;
        const uint32_t word = (c >> 1) == 0 ? q.x : ((c >> 1) == 1 ? q.y : ((c >> 1) == 2 ? q.z : q.w));
        return (c & 1) ? (word & 0xffff0000u) : (word << 16);
    } else {
        return pick16(v, slot);
    }
}

template <int L>
__device__ __forceinline__ uint32_t slot_position(uint64_t e0, int slot, int lane) {
    if constexpr (L == 0) return (uint32_t)(e0 + (slot >> 2) * 128 + lane * 4 + (slot & 3));
    if constexpr (L == 1) return (uint32_t)(e0 + (slot >> 3) * 256 + lane * 8 + (slot & 7));
    return (uint32_t)(e0 + slot * 32 + lane);
}

}  // namespace s2
