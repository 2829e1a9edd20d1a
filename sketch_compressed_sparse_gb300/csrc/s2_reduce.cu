// The AllReduce(S, C) step of S2 Reducer ("S2 Reducer", Section 3.1
// "Collecting Sparse-Sketch with AllReduce"; Algorithm 1) for W workers that
// all live on this GPU: the sketch is linear, so the aggregate sketch is the
// element-wise sum of the workers' sketches; the aggregate bitmap marks a
// position iff some worker marked it (bitwise OR).
//
// Design: a pure streaming kernel. Each thread owns one 16-byte vector of
// the output and reads the W inputs at that offset with streaming loads
// (they are read once), summing in the fixed order k = 0..W-1, so the result
// is deterministic. The summed sketch is stored with an evict-last L2 policy
// so that the decode that follows finds it in L2. The sketch part and the bitmap part are two
// index ranges of one grid.
#include "s2_internal.h"

namespace s2 {
namespace {

__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
    uint4 r = ld_stream_u4(p);
    return make_float4(__uint_as_float(r.x), __uint_as_float(r.y), __uint_as_float(r.z), __uint_as_float(r.w));
}

// SVEC: dw % 4 == 0 (every worker's sketch is 16-byte aligned), 16-byte
// vectors; else one float per item. BVEC likewise for the bitmaps (nw % 4).
template <bool SVEC, bool BVEC>
__global__ void __launch_bounds__(kThreads)
    reduce_kernel(const uint32_t* __restrict__ bitmaps, const float* __restrict__ sketches, uint32_t W,
                  uint64_t nw, uint64_t dw, uint32_t* __restrict__ bitmap_out, float* __restrict__ sketch_out) {
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t s_items = SVEC ? dw / 4 : dw;
    const uint64_t b_items = BVEC ? nw / 4 : nw;
    const uint64_t keep = policy_evict_last();  // the decode gathers from this sketch next
    for (uint64_t x = tid; x < s_items + b_items; x += stride) {
        if (x < s_items) {
            if (SVEC) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                uint32_t k = 0;
                for (; k + 4 <= W; k += 4) {
                    float4 t[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) t[q] = ld_stream_f4(sketches + (uint64_t)(k + q) * dw + x * 4);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc.x += t[q].x;
                        acc.y += t[q].y;
                        acc.z += t[q].z;
                        acc.w += t[q].w;
                    }
                }
                for (; k < W; ++k) {
                    float4 t = ld_stream_f4(sketches + (uint64_t)k * dw + x * 4);
                    acc.x += t.x;
                    acc.y += t.y;
                    acc.z += t.z;
                    acc.w += t.w;
                }
                st_f4_hint(reinterpret_cast<float4*>(sketch_out) + x, acc, keep);
            } else {
                float acc = 0.f;
                for (uint32_t k = 0; k < W; ++k)
                    acc += __uint_as_float(ld_stream_u32(sketches + (uint64_t)k * dw + x));
                sketch_out[x] = acc;
            }
        } else {
            const uint64_t y = x - s_items;
            if (BVEC) {
                uint4 acc = make_uint4(0, 0, 0, 0);
                for (uint32_t k = 0; k < W; ++k) {
                    uint4 t = ld_stream_u4(bitmaps + (uint64_t)k * nw + y * 4);
                    acc.x |= t.x;
                    acc.y |= t.y;
                    acc.z |= t.z;
                    acc.w |= t.w;
                }
                reinterpret_cast<uint4*>(bitmap_out)[y] = acc;
            } else {
                uint32_t acc = 0;
                for (uint32_t k = 0; k < W; ++k) acc |= ld_stream_u32(bitmaps + (uint64_t)k * nw + y);
                bitmap_out[y] = acc;
            }
        }
    }
}

template <bool SVEC, bool BVEC>
cudaError_t launch_reduce_t(const uint32_t* bitmaps, const float* sketches, uint32_t W, uint64_t nw,
                            uint64_t dw, uint32_t* bitmap_out, float* sketch_out, cudaStream_t s) {
    const uint64_t items = (SVEC ? dw / 4 : dw) + (BVEC ? nw / 4 : nw);
    const uint64_t blocks = (items + kThreads - 1) / kThreads;
    reduce_kernel<SVEC, BVEC><<<grid_for(reduce_kernel<SVEC, BVEC>, blocks), kThreads, 0, s>>>(
        bitmaps, sketches, W, nw, dw, bitmap_out, sketch_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reduce(const uint32_t* bitmaps, const float* sketches, uint32_t W, uint64_t nw,
                          uint64_t dw, uint32_t* bitmap_out, float* sketch_out, cudaStream_t s) {
    if (dw + nw == 0) return cudaSuccess;
    const bool sv = dw % 4 == 0, bv = nw % 4 == 0;
    if (sv && bv) return launch_reduce_t<true, true>(bitmaps, sketches, W, nw, dw, bitmap_out, sketch_out, s);
    if (sv) return launch_reduce_t<true, false>(bitmaps, sketches, W, nw, dw, bitmap_out, sketch_out, s);
    if (bv) return launch_reduce_t<false, true>(bitmaps, sketches, W, nw, dw, bitmap_out, sketch_out, s);
    return launch_reduce_t<false, false>(bitmaps, sketches, W, nw, dw, bitmap_out, sketch_out, s);
}

}  // namespace s2
