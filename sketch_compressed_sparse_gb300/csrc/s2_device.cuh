// Device-side building blocks of the S2 Reducer kernels (sm_103a).
//
// Hash family: 32-bit MurmurHash3 finalizer (fmix32), per-row keys derived
// from the seed on the host, bucket by multiply-shift (high half of a
// 32x32-bit product), sign from the top bit. The paper ("S2 Reducer",
// Section 3.1) asks for a random bucket map h and random signs s per row and
// leaves the family open; this fixes one.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace s2 {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxRows = 16;

// Row keys travel as a kernel parameter (host-computed from the seed).
struct RowKeys {
    uint32_t kh[kMaxRows];  // bucket keys
    uint32_t ks[kMaxRows];  // sign keys
};

__device__ __forceinline__ uint32_t fmix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x85ebca6bu;
    x ^= x >> 13;
    x *= 0xc2b2ae35u;
    x ^= x >> 16;
    return x;
}

// h_j(i): high 32 bits of fmix32(i ^ kh) * w (w <= 2^31 fits the 32x32 product).
__device__ __forceinline__ uint32_t bucket_of(uint32_t i, uint32_t kh, uint32_t w) {
    return __umulhi(fmix32(i ^ kh), w);
}

// s_j(i) as a float sign bit: 0x80000000 when the sign is -1, else 0.
__device__ __forceinline__ uint32_t signbit_of(uint32_t i, uint32_t ks) {
    return fmix32(i ^ ks) & 0x80000000u;
}

__device__ __forceinline__ float apply_sign(float v, uint32_t sbit) {
    return __uint_as_float(__float_as_uint(v) ^ sbit);
}

// ---- memory access with cache policy -------------------------------------

// Streaming 16-byte load: read once, evict first (keeps L2 for the sketch).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 r;
    asm("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t r;
    asm("ld.global.cs.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ float ld_stream_f32(const float* p) { return __uint_as_float(ld_stream_u32(p)); }

__device__ __forceinline__ uint16_t ld_stream_u16(const void* p) {
    uint16_t r;
    asm("ld.global.cs.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ void st_stream_f4(void* p, float4 v) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

// Fire-and-forget float add into global memory (resolved in L2).
__device__ __forceinline__ void red_add_f32(float* p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Four float reductions into 16 consecutive bytes (p 16-byte aligned).
__device__ __forceinline__ void red_add_f32x4(float* p, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// L2 eviction-priority policies (createpolicy); "last" keeps a line in L2
// ahead of normal and evict-first lines, "first" lets a line go first.
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void red_add_f32_hint(float* p, float v, uint64_t pol) {
    asm volatile("red.global.add.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

// Read-only 4-byte gather with an L2 eviction policy.
__device__ __forceinline__ float ld_gather_f32(const float* p, uint64_t pol) {
    float r;
    asm("ld.global.nc.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(r) : "l"(p), "l"(pol));
    return r;
}

__device__ __forceinline__ void st_f4_hint(void* p, float4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w), "l"(pol)
                 : "memory");
}

// Exclusive prefix sum over the warp; *total receives the warp-wide sum.
__device__ __forceinline__ uint32_t warp_exclusive_scan(uint32_t v, int lane, uint32_t* total) {
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    *total = __shfl_sync(kFull, incl, 31);
    return incl - v;
}

// ---- median of the row estimates ------------------------------------------

__device__ __forceinline__ float med3(float a, float b, float c) {
    return fmaxf(fminf(a, b), fminf(fmaxf(a, b), c));
}

// Median of d values held in e[0..D-1] (D known at compile time, 1..5), or of
// the first d of kMaxRows values when D == 0. Even counts: mean of the two
// middle values.
template <int D>
__device__ __forceinline__ float median_rows(const float (&e)[(D > 0 ? D : kMaxRows)], int d) {
    if constexpr (D == 1) {
        return e[0];
    } else if constexpr (D == 2) {
        return 0.5f * (e[0] + e[1]);
    } else if constexpr (D == 3) {
        return med3(e[0], e[1], e[2]);
    } else if constexpr (D == 4) {
        float lo = fmaxf(fminf(e[0], e[1]), fminf(e[2], e[3]));
        float hi = fminf(fmaxf(e[0], e[1]), fmaxf(e[2], e[3]));
        return 0.5f * (lo + hi);
    } else if constexpr (D == 5) {
        // Of the first four, the smallest and the largest cannot be the median
        // of five; the median is the median of the two middle ones and e[4].
        float t0 = fminf(e[0], e[1]), t1 = fmaxf(e[0], e[1]);
        float t2 = fminf(e[2], e[3]), t3 = fmaxf(e[2], e[3]);
        return med3(fmaxf(t0, t2), fminf(t1, t3), e[4]);
    } else {
        // General d <= 16: rank selection with a stable tie order; all indices
        // are compile-time constants so the values stay in registers.
        const int lo_rank = (d - 1) >> 1;
        const int hi_rank = d >> 1;
        float lo = 0.f, hi = 0.f;
#pragma unroll
        for (int a = 0; a < kMaxRows; ++a) {
            if (a < d) {
                int rank = 0;
#pragma unroll
                for (int b = 0; b < kMaxRows; ++b) {
                    if (b < d && b != a) {
                        rank += (e[b] < e[a]) || (e[b] == e[a] && b < a);
                    }
                }
                if (rank == lo_rank) lo = e[a];
                if (rank == hi_rank) hi = e[a];
            }
        }
        return (d & 1) ? lo : 0.5f * (lo + hi);
    }
}

}  // namespace s2
