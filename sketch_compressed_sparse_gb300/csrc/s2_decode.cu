// Decompression phase of S2 Reducer ("S2 Reducer", Section 3.1
// "Decompressing Sparse Gradient"; Algorithm 1, decompression loop): recover
// the set positions from the aggregated bitmap and, for each, take the median
// over the d rows of s_j(i) * S[j][h_j(i)].
//
// Design: a warp owns 512 consecutive positions (16 bitmap words). Lanes
// 0..15 load the words; every lane then owns 16 positions (4 chunks of 4
// consecutive positions, so the dense output leaves as 16-byte streaming
// stores). A lane walks only its set positions, two per step so that 2*d
// independent gathers are in flight, and keeps the results in registers.
// Unset positions are written as +0.0f with the same stores. The summed
// sketch is gathered with an evict-last L2 policy so that the output stream
// does not push it out of L2 (for a sketch of tens of MB this decides
// between L2 hits and scattered DRAM reads).
//
// The compacted output uses three kernels and no inter-block waiting:
// per-tile popcounts, one block that scans the tile totals (and writes the
// final count), and a writer with one warp per task that recomputes its rank
// inside the tile from the bitmap and writes (index, value) pairs in
// ascending order.
#include <mutex>

#include "s2_internal.h"

namespace s2 {
namespace {

__device__ __forceinline__ void load_keys(const RowKeys& k, uint32_t* s_kh, uint32_t* s_ks) {
    if (threadIdx.x < kMaxRows) {
        s_kh[threadIdx.x] = k.kh[threadIdx.x];
        s_ks[threadIdx.x] = k.ks[threadIdx.x];
    }
    __syncthreads();
}

// Bitmap word wi, with the bits at positions >= n cleared (0 past the end).
__device__ __forceinline__ uint32_t load_word(const uint32_t* __restrict__ bm, uint64_t wi, uint64_t nw, uint64_t n) {
    if (wi >= nw) return 0u;
    uint32_t v = __ldg(bm + wi);
    if (wi == nw - 1 && (n & 31)) v &= (1u << (n & 31)) - 1u;
    return v;
}

// Position of slot `slot` of this lane inside a 512-position task.
__device__ __forceinline__ uint32_t slot_pos(int slot, int lane) {
    return (uint32_t)((slot >> 2) * 128 + lane * 4 + (slot & 3));
}

// This lane's 16 slots of a task as a bit mask (slot 4u + c is bit c of the
// nibble of word 4u + lane/8 at nibble position lane%8). `my_word` is the
// word held by lane L = word L of the task (lanes 0..15).
__device__ __forceinline__ uint32_t lane_mask(uint32_t my_word, int lane) {
    uint32_t mask = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint32_t wv = __shfl_sync(kFull, my_word, u * 4 + (lane >> 3));
        mask |= ((wv >> (4 * (lane & 7))) & 0xfu) << (4 * u);
    }
    return mask;
}

// Load the d signed estimates of position i with an L2 policy for the sketch.
template <int D>
__device__ __forceinline__ void gather_hint(float (&e)[(D > 0 ? D : kMaxRows)], const float* __restrict__ sk,
                                            uint32_t i, int d, uint32_t w, const uint32_t* s_kh,
                                            const uint32_t* s_ks, uint64_t pol) {
#pragma unroll
    for (int j = 0; j < (D > 0 ? D : kMaxRows); ++j) {
        if (D > 0 || j < d) {
            const uint32_t b = bucket_of(i, s_kh[j], w);
            e[j] = apply_sign(ld_gather_f32(sk + (uint64_t)j * w + b, pol), signbit_of(i, s_ks[j]));
        } else {
            e[j] = 0.f;
        }
    }
}

// Dense decode, one warp per task of 512 positions. Lanes 0..15 load the 16
// bitmap words; every lane then owns 16 positions (4 chunks of 4 consecutive
// positions) and walks only its set ones, kPop per step, so that kPop * d
// independent gathers from the L2-resident sketch (evict-last policy) are in
// flight; results stay in registers and the 16 positions leave as four
// 16-byte streaming stores, +0.0f at unset positions.
constexpr int kPop = 2;

// This lane's 16 slots of a task under a block bitmap: position p is set iff
// block p / a.block is marked. A lane's 4 consecutive positions never
// straddle a block (blocks are multiples of 32 positions).
__device__ __forceinline__ uint32_t lane_mask_blocks(const DecodeArgs& a, uint64_t e0, int lane) {
    uint32_t mask = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint64_t p = e0 + u * 128 + lane * 4;
        if (p < a.n) {
            const uint32_t blk = (uint32_t)p / a.block;  // positions are below 2^32
            if ((__ldg(a.bitmap + (blk >> 5)) >> (blk & 31)) & 1u) {
                const uint64_t left = a.n - p;
                mask |= (left >= 4 ? 0xfu : ((1u << left) - 1u)) << (4 * u);
            }
        }
    }
    return mask;
}

// PHASED: the launch handles only the tasks without a set position (their
// 512 zeros; set_tasks = 0) or only the tasks with one (set_tasks = 1). An
// output larger than L2 is written in these two launches, zeros first, so
// that the zero stream does not evict the summed sketch while the gathers
// need it. Without PHASED every task is handled (and the kernel carries no
// phase test).
// guard (optional): the launch works only if *guard >= guard_at (a count
// written by an earlier launch; the same for every thread).
template <int D, bool BLK, bool PHASED>
__global__ void __launch_bounds__(kThreads)
    decode_dense_kernel(DecodeArgs a, float* __restrict__ out, int set_tasks,
                        const unsigned int* __restrict__ guard = nullptr, uint32_t guard_at = 0) {
    if (guard && *guard < guard_at) return;
    __shared__ uint32_t s_kh[kMaxRows], s_ks[kMaxRows];
    load_keys(a.keys, s_kh, s_ks);
    const int lane = threadIdx.x & 31;
    const uint64_t keep = policy_evict_last();
    const uint64_t ntasks = (a.n + kTaskElems - 1) / kTaskElems;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t t = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < ntasks; t += nwarps) {
        const uint64_t e0 = t * kTaskElems;
        const uint64_t wi = t * kTaskWords + lane;
        uint32_t mask;
        if (BLK) {
            mask = lane_mask_blocks(a, e0, lane);
        } else {
            const uint32_t my_word = lane < kTaskWords ? load_word(a.bitmap, wi, a.nw, a.n) : 0u;
            mask = lane_mask(my_word, lane);
        }
        if (PHASED) {
            const bool any = __any_sync(kFull, mask != 0);  // warp-uniform
            if (any != (set_tasks != 0)) continue;
        }
        float r[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) r[s] = 0.f;
        while (mask) {
            int sl[kPop];
            bool ok[kPop];
#pragma unroll
            for (int q = 0; q < kPop; ++q) {
                ok[q] = mask != 0;
                sl[q] = ok[q] ? __ffs(mask) - 1 : (q ? sl[0] : 0);
                if (ok[q]) mask &= mask - 1;
            }
            float ev[kPop][(D > 0 ? D : kMaxRows)];
#pragma unroll
            for (int q = 0; q < kPop; ++q)
                gather_hint<D>(ev[q], a.sketch, (uint32_t)e0 + slot_pos(sl[q], lane), a.d, a.w, s_kh, s_ks, keep);
#pragma unroll
            for (int q = 0; q < kPop; ++q) {
                const float v = a.scale * median_rows<D>(ev[q], a.d);
#pragma unroll
                for (int s = 0; s < 16; ++s) r[s] = (ok[q] && s == sl[q]) ? v : r[s];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint64_t e = e0 + u * 128 + lane * 4;
            if (e + 4 <= a.n) {
                st_stream_f4(out + e, make_float4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]));
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (e + c < a.n) out[e + c] = r[4 * u + c];
            }
        }
    }
}

// ---- dense decode in passes over groups of rows -------------------------------
// A summed sketch much larger than 2/5 of L2 does not stay in L2 under
// random gathers (84 MB of large-LM sketch: 44 % hits), so the median is
// taken in passes: each pass gathers only its group of rows, which L2 holds,
// for every set position, and carries to the next pass the candidates of the
// median that remain after the rows seen so far. Of 3 rows at most 2
// candidates remain (after 2 rows: their min and max); of 5 rows at most 3
// (after 2 rows: min and max; after 3: all three, sorted; after 4: the middle
// two of the four, since the smallest and the largest of four cannot be the
// third of five). The candidates live at the position's own index in the
// output (the first) and in up to two workspace arrays of n floats, so each
// pass reads and writes them with coalesced 16-byte accesses. Tasks without
// a set position are written (zeros) by one launch before the passes, which
// skip them; the last pass writes every position of the other tasks.

// Median candidates left after r of D rows.
__host__ __device__ constexpr int kept_after(int D, int r) {
    return D == 3 ? (r == 0 ? 0 : (r == 1 ? 1 : (r == 2 ? 2 : 1)))
                  : (r == 0 ? 0 : (r == 1 ? 1 : (r == 2 ? 2 : (r == 3 ? 3 : (r == 4 ? 2 : 1)))));
}

// Fold the value e of row r (rows counted from 0) into the candidates c.
template <int D>
__device__ __forceinline__ void fold_row(float (&c)[3], int r, float e) {
    if (r == 0) {
        c[0] = e;
    } else if (r == 1) {
        const float lo = fminf(c[0], e), hi = fmaxf(c[0], e);
        c[0] = lo;
        c[1] = hi;
    } else if (D == 3 || r == 4) {  // the median: of lo <= hi and e
        c[0] = fmaxf(c[0], fminf(c[1], e));
    } else if (r == 2) {  // three sorted values
        const float x = fminf(c[0], e), y = fmaxf(c[0], fminf(c[1], e)), z = fmaxf(c[1], e);
        c[0] = x;
        c[1] = y;
        c[2] = z;
    } else {  // r == 3: the middle two of four
        const float p = fmaxf(c[0], fminf(c[1], e)), q = fminf(c[2], fmaxf(c[1], e));
        c[0] = p;
        c[1] = q;
    }
}

// Four consecutive floats at e (16-byte aligned when e + 4 <= n), streamed.
__device__ __forceinline__ float4 ld_stream_f4_tail(const float* p, uint64_t e, uint64_t n) {
    if (e + 4 <= n) {
        const uint4 v = ld_stream_u4(p + e);
        return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
    }
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e + 0 < n) v.x = ld_stream_f32(p + e + 0);
    if (e + 1 < n) v.y = ld_stream_f32(p + e + 1);
    if (e + 2 < n) v.z = ld_stream_f32(p + e + 2);
    return v;
}

__device__ __forceinline__ void st_stream_f4_tail(float* p, uint64_t e, uint64_t n, float4 v) {
    if (e + 4 <= n) {
        st_stream_f4(p + e, v);
    } else {
        if (e + 0 < n) p[e + 0] = v.x;
        if (e + 1 < n) p[e + 1] = v.y;
        if (e + 2 < n) p[e + 2] = v.z;
    }
}

__device__ __forceinline__ float f4_at(const float4& v, int q) {
    return q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w));
}

// Bitmap word wi of a task, read once per pass (evict-first), bits >= n cleared.
__device__ __forceinline__ uint32_t task_word(const DecodeArgs& a, uint64_t wi, int lane) {
    uint32_t v = 0;
    if (lane < kTaskWords && wi < a.nw) {
        v = ld_stream_u32(a.bitmap + wi);
        if (wi == a.nw - 1 && (a.n & 31)) v &= (1u << (a.n & 31)) - 1u;
    }
    return v;
}

// The launch before the passes: writes the 512 zeros of every task without a
// set position and lists the others (task ids in any order, their number in
// *count, which starts at zero) for the passes to work through. A warp keeps
// up to 32 ids in its lanes and appends them with one atomic.
__global__ void __launch_bounds__(kThreads)
    decode_zero_list_kernel(DecodeArgs a, float* __restrict__ out, uint32_t* __restrict__ list,
                            unsigned int* __restrict__ count) {
    const int lane = threadIdx.x & 31;
    const uint64_t ntasks = (a.n + kTaskElems - 1) / kTaskElems;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    uint32_t held = 0;  // task ids held by the lanes (lane q holds the q-th), warp-uniform
    uint32_t mine = 0;
    auto flush = [&]() {
        unsigned int base = 0;
        if (lane == 0) base = atomicAdd(count, held);
        base = __shfl_sync(kFull, base, 0);
        if ((uint32_t)lane < held) list[base + lane] = mine;
        held = 0;
    };
    // the bitmap words of a warp's next kAhead tasks are loaded together, so
    // the zero stores of one task do not wait for the next task's word
    constexpr int kAhead = 4;
    for (uint64_t t0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t0 < ntasks; t0 += kAhead * nwarps) {
        uint32_t words[kAhead];
#pragma unroll
        for (int q = 0; q < kAhead; ++q) {
            const uint64_t t = t0 + q * nwarps;
            words[q] = t < ntasks ? task_word(a, t * kTaskWords + lane, lane) : 0u;
        }
#pragma unroll
        for (int q = 0; q < kAhead; ++q) {
            const uint64_t t = t0 + q * nwarps;
            if (t >= ntasks) break;  // warp-uniform
            const uint32_t mask = lane_mask(words[q], lane);
            if (__any_sync(kFull, mask != 0)) {
                if ((uint32_t)lane == held) mine = (uint32_t)t;
                if (++held == 32) flush();
                continue;
            }
            const uint64_t e0 = t * kTaskElems;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                st_stream_f4_tail(out, e0 + u * 128 + lane * 4, a.n, make_float4(0.f, 0.f, 0.f, 0.f));
        }
    }
    if (held) flush();
}

// One pass over rows [j0, j1) of the median (D = 3 or 5), one warp per listed
// task of 512 positions; a lane owns 4 chunks of 4 consecutive positions,
// like decode_dense_kernel. The launch works only if fewer than dense_at
// tasks are listed (otherwise the one-launch decode has done the work).
// Four resident blocks per SM (58 registers instead of 78, no spills):
// large-LM decode 0.382 -> 0.377 ms; five (48 registers) spill and gain less.
template <int D>
__global__ void __launch_bounds__(kThreads, 4)
    decode_rows_kernel(DecodeArgs a, float* __restrict__ out, float* __restrict__ cand1,
                       float* __restrict__ cand2, const uint32_t* __restrict__ list,
                       const unsigned int* __restrict__ count, int j0, int j1, uint32_t dense_at) {
    static_assert(D == 3 || D == 5, "row passes are specialised for 3 and 5 rows");
    const uint32_t listed = *count;
    if (listed >= dense_at) return;  // the same for every thread of the launch
    __shared__ uint32_t s_kh[kMaxRows], s_ks[kMaxRows];
    load_keys(a.keys, s_kh, s_ks);
    const int lane = threadIdx.x & 31;
    const uint64_t keep = policy_evict_last();
    const int k_in = kept_after(D, j0), k_out = kept_after(D, j1);
    const bool last = j1 == D;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    for (uint32_t x = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; x < listed; x += nwarps) {
        const uint64_t t = list[x];
        const uint64_t e0 = t * kTaskElems;
        const uint32_t mask = lane_mask(task_word(a, t * kTaskWords + lane, lane), lane);
#pragma unroll 1
        for (int u = 0; u < 4; ++u) {
            const uint32_t nib = (mask >> (4 * u)) & 0xfu;
            const uint64_t e = e0 + u * 128 + lane * 4;
            if (!nib && !last) continue;
            float c[4][3] = {};
            if (nib) {
                if (k_in >= 1) {
                    const float4 v = ld_stream_f4_tail(out, e, a.n);
#pragma unroll
                    for (int q = 0; q < 4; ++q) c[q][0] = f4_at(v, q);
                }
                if (k_in >= 2) {
                    const float4 v = ld_stream_f4_tail(cand1, e, a.n);
#pragma unroll
                    for (int q = 0; q < 4; ++q) c[q][1] = f4_at(v, q);
                }
                if (k_in >= 3) {
                    const float4 v = ld_stream_f4_tail(cand2, e, a.n);
#pragma unroll
                    for (int q = 0; q < 4; ++q) c[q][2] = f4_at(v, q);
                }
                // every gather of the pass first, then the folds
                float ev[4][D];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t i = (uint32_t)(e + q);
#pragma unroll
                    for (int j = 0; j < D; ++j) {
                        ev[q][j] = 0.f;
                        if (j >= j0 && j < j1 && ((nib >> q) & 1u)) {
                            const uint32_t b = bucket_of(i, s_kh[j], a.w);
                            ev[q][j] = apply_sign(ld_gather_f32(a.sketch + (uint64_t)j * a.w + b, keep),
                                                  signbit_of(i, s_ks[j]));
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int j = 0; j < D; ++j)
                        if (j >= j0 && j < j1) fold_row<D>(c[q], j, ev[q][j]);
                }
            }
            if (last) {
                float r[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) r[q] = ((nib >> q) & 1u) ? a.scale * c[q][0] : 0.f;
                st_stream_f4_tail(out, e, a.n, make_float4(r[0], r[1], r[2], r[3]));
            } else {
                st_stream_f4_tail(out, e, a.n, make_float4(c[0][0], c[1][0], c[2][0], c[3][0]));
                if (k_out >= 2) st_stream_f4_tail(cand1, e, a.n, make_float4(c[0][1], c[1][1], c[2][1], c[3][1]));
                if (k_out >= 3) st_stream_f4_tail(cand2, e, a.n, make_float4(c[0][2], c[1][2], c[2][2], c[3][2]));
            }
        }
    }
}

// ---- compacted output -------------------------------------------------------

// Set bits per tile of kCompactTileWords words (one word per thread), and the
// set bits of the tile's tasks before each task (its in-tile prefix).
static_assert(kCompactTileWords == kThreads, "one thread per word of a tile");
__global__ void __launch_bounds__(kThreads)
    compact_count_kernel(const uint32_t* __restrict__ bitmap, uint64_t nw, uint64_t n, uint64_t tiles,
                         uint32_t* __restrict__ counts, uint16_t* __restrict__ task_prefix) {
    constexpr int kTasksPerTile = kCompactTileWords / kTaskWords;
    __shared__ uint32_t s_task[kTasksPerTile];
    for (uint64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const uint64_t wi = t * kCompactTileWords + threadIdx.x;
        uint32_t c = __popc(load_word(bitmap, wi, nw, n));
        // the 16 words of a task are a half warp
#pragma unroll
        for (int o = kTaskWords / 2; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
        if ((threadIdx.x & (kTaskWords - 1)) == 0) s_task[threadIdx.x / kTaskWords] = c;
        __syncthreads();
        if (threadIdx.x < kTasksPerTile) {
            uint32_t before = 0;
            for (int q = 0; q < (int)threadIdx.x; ++q) before += s_task[q];
            task_prefix[t * kTasksPerTile + threadIdx.x] = (uint16_t)before;  // at most 15 * 512
            if (threadIdx.x == kTasksPerTile - 1) counts[t] = before + s_task[kTasksPerTile - 1];
        }
        __syncthreads();  // s_task is rewritten by the next tile
    }
}

// Exclusive scan of the tile counts by one block; writes the total count.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads)
    compact_scan_kernel(const uint32_t* __restrict__ counts, uint64_t tiles, uint32_t* __restrict__ offsets,
                        unsigned long long* __restrict__ count_out) {
    __shared__ unsigned long long s_warp[kScanThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t per = (tiles + kScanThreads - 1) / kScanThreads;
    const uint64_t lo = threadIdx.x * per;
    const uint64_t hi = lo + per < tiles ? lo + per : tiles;
    unsigned long long local = 0;
    for (uint64_t x = lo; x < hi; ++x) local += counts[x];
    // inclusive warp scan of the per-thread sums
    unsigned long long incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned long long y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        unsigned long long v = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            unsigned long long y = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += y;
        }
        s_warp[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    unsigned long long run = (warp > 0 ? s_warp[warp - 1] : 0ull) + incl - local;
    for (uint64_t x = lo; x < hi; ++x) {
        offsets[x] = (uint32_t)run;
        run += counts[x];
    }
    if (threadIdx.x == kScanThreads - 1) *count_out = s_warp[31];
}

// Writer, one warp per task of 512 positions (grid-stride, like the dense
// decode), no block-wide synchronisation. Tiles without a set position are
// skipped from their count alone; a task's first rank is its tile's offset
// plus the in-tile prefix the count kernel stored for it. Within a task each
// lane walks its set slots kPop at a time, writing (index, value) at the
// position's rank: task prefix + earlier words of the task + earlier bits of
// the word.
template <int D>
__device__ __forceinline__ void compact_task(const DecodeArgs& a, uint64_t t, uint32_t my_word, uint64_t tbase,
                                             int lane, const uint32_t* s_kh, const uint32_t* s_ks, uint64_t keep,
                                             uint32_t* __restrict__ idx_out, float* __restrict__ val_out,
                                             uint64_t capacity) {
    const uint32_t cnt = __popc(my_word);
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - cnt;
    uint32_t wv[4], wo[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        wv[u] = __shfl_sync(kFull, my_word, u * 4 + (lane >> 3));
        wo[u] = __shfl_sync(kFull, excl, u * 4 + (lane >> 3));
    }
    const uint64_t e0 = t * kTaskElems;
    uint32_t mask = lane_mask(my_word, lane);
    while (mask) {
        int sl[kPop];
        bool ok[kPop];
#pragma unroll
        for (int q = 0; q < kPop; ++q) {
            ok[q] = mask != 0;
            sl[q] = ok[q] ? __ffs(mask) - 1 : (q ? sl[0] : 0);
            if (ok[q]) mask &= mask - 1;
        }
        float ev[kPop][(D > 0 ? D : kMaxRows)];
#pragma unroll
        for (int q = 0; q < kPop; ++q)
            gather_hint<D>(ev[q], a.sketch, (uint32_t)e0 + slot_pos(sl[q], lane), a.d, a.w, s_kh, s_ks, keep);
#pragma unroll
        for (int q = 0; q < kPop; ++q) {
            if (!ok[q]) continue;
            const int u = sl[q] >> 2;
            const uint32_t bitpos = 4 * (lane & 7) + (sl[q] & 3);
            const uint32_t word = u == 0 ? wv[0] : (u == 1 ? wv[1] : (u == 2 ? wv[2] : wv[3]));
            const uint32_t woff = u == 0 ? wo[0] : (u == 1 ? wo[1] : (u == 2 ? wo[2] : wo[3]));
            const uint64_t off = tbase + woff + __popc(word & ((1u << bitpos) - 1u));
            if (off < capacity) {
                idx_out[off] = (uint32_t)e0 + slot_pos(sl[q], lane);
                val_out[off] = a.scale * median_rows<D>(ev[q], a.d);
            }
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    compact_write_kernel(DecodeArgs a, const uint32_t* __restrict__ tile_counts,
                         const uint32_t* __restrict__ offsets, const uint16_t* __restrict__ task_prefix,
                         uint32_t* __restrict__ idx_out, float* __restrict__ val_out, uint64_t capacity) {
    __shared__ uint32_t s_kh[kMaxRows], s_ks[kMaxRows];
    load_keys(a.keys, s_kh, s_ks);
    constexpr uint32_t kTasksPerTile = kCompactTileWords / kTaskWords;
    const int lane = threadIdx.x & 31;
    const uint64_t keep = policy_evict_last();
    const uint64_t ntasks = (a.n + kTaskElems - 1) / kTaskElems;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t t = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < ntasks; t += nwarps) {
        const uint64_t tile = t / kTasksPerTile;
        if (__ldg(tile_counts + tile) == 0) continue;
        const uint32_t my_word = lane < kTaskWords ? load_word(a.bitmap, t * kTaskWords + lane, a.nw, a.n) : 0u;
        if (!__any_sync(kFull, my_word != 0)) continue;
        compact_task<D>(a, t, my_word, (uint64_t)offsets[tile] + __ldg(task_prefix + t), lane, s_kh, s_ks, keep,
                        idx_out, val_out, capacity);
    }
}

template <int D, bool BLK>
cudaError_t launch_dense_db(const DecodeArgs& a, float* out, cudaStream_t s) {
    const uint64_t tasks = (a.n + kTaskElems - 1) / kTaskElems;
    const uint64_t blocks = (tasks + (kThreads / 32) - 1) / (kThreads / 32);
    DeviceInfo di{};
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    if (a.n * 4 <= (uint64_t)di.l2_bytes) {
        decode_dense_kernel<D, BLK, false>
            <<<grid_for(decode_dense_kernel<D, BLK, false>, blocks), kThreads, 0, s>>>(a, out, 0);
        return cudaGetLastError();
    }
    const int grid = grid_for(decode_dense_kernel<D, BLK, true>, blocks);
    decode_dense_kernel<D, BLK, true><<<grid, kThreads, 0, s>>>(a, out, 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_dense_kernel<D, BLK, true><<<grid, kThreads, 0, s>>>(a, out, 1);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_dense_d(const DecodeArgs& a, float* out, cudaStream_t s) {
    return a.block ? launch_dense_db<D, true>(a, out, s) : launch_dense_db<D, false>(a, out, s);
}

// Rows of the summed sketch that one pass of the sliced dense decode gathers
// from: as many whole rows as fit in 2/5 of L2 (at least one). Measured on
// the large-LM sketch (5 rows of 16.8 MB): 3 rows a pass 0.382 ms, 2 rows
// 0.395 ms, 4 rows 0.398 ms.
uint64_t pass_budget(uint64_t l2_bytes) { return l2_bytes * 2 / 5; }

// Largest summed sketch for which a decode with most tasks set runs in one
// launch over all rows instead of in passes (see launch_dense_rows).
constexpr uint64_t kOneLaunchMax = 96ull << 20;

uint32_t rows_per_pass(uint64_t w, uint64_t l2_bytes) {
    const uint64_t budget = pass_budget(l2_bytes), row = 4 * w;
    return row >= budget ? 1u : (uint32_t)(budget / row);
}

template <int D>
cudaError_t launch_dense_rows(const DecodeArgs& a, float* out, float* ws, uint32_t rpp, cudaStream_t s) {
    const uint64_t tasks = (a.n + kTaskElems - 1) / kTaskElems;
    const uint64_t blocks = (tasks + (kThreads / 32) - 1) / (kThreads / 32);
    const DenseWsLayout L = dense_ws_layout(a.n, a.d);
    float* cand1 = ws + L.cand1 / 4;
    float* cand2 = ws + L.cand2 / 4;
    unsigned int* count = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(ws) + L.count);
    uint32_t* list = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(ws) + L.list);
    cudaError_t e = cudaMemsetAsync(count, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    // zeros of the tasks without a set position; the list of the others
    decode_zero_list_kernel<<<grid_for(decode_zero_list_kernel, blocks), kThreads, 0, s>>>(a, out, list, count);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // A sketch up to kOneLaunchMax whose set positions reach at least half of
    // the tasks is decoded faster in one launch over all rows (the set-task
    // launch of the two-launch decode) than in passes, which would then carry
    // candidates for nearly every position (measured on 8 workers of 2^26
    // positions at 10 % density, d = 5, an 84 MB sketch: 0.76 ms in one
    // launch, 1.12 ms in passes; with 3 % of the tasks set, as in the large-LM
    // workload with the same sketch, the passes win, 0.38 against 0.50 ms).
    // Both forms are queued; the count of listed tasks picks one on the device.
    uint32_t dense_at = 0xffffffffu;
    if ((uint64_t)a.d * a.w * 4 <= kOneLaunchMax) {
        dense_at = (uint32_t)((tasks + 1) / 2);
        decode_dense_kernel<D, false, true>
            <<<grid_for(decode_dense_kernel<D, false, true>, blocks), kThreads, 0, s>>>(a, out, 1, count, dense_at);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int grid = grid_for(decode_rows_kernel<D>, blocks);
    // The smallest group of rows goes first: fewer candidates are carried
    // after it (d = 5 in groups of 3: rows {0, 1} then {2, 3, 4}, two
    // candidates instead of three).
    const uint32_t passes = ((uint32_t)D + rpp - 1) / rpp;
    for (uint32_t p = 0, j0 = 0; p < passes; ++p) {
        const uint32_t j1 = j0 + (p == 0 ? (uint32_t)D - rpp * (passes - 1) : rpp);
        decode_rows_kernel<D><<<grid, kThreads, 0, s>>>(a, out, cand1, cand2, list, count, (int)j0, (int)j1,
                                                         dense_at);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        j0 = j1;
    }
    return cudaSuccess;
}

template <int D>
cudaError_t launch_compact_write_d(const DecodeArgs& a, const uint32_t* tile_counts, const uint32_t* offsets,
                                   const uint16_t* task_prefix, uint32_t* idx_out, float* val_out,
                                   uint64_t capacity, cudaStream_t s) {
    const uint64_t tasks = (a.n + kTaskElems - 1) / kTaskElems;
    const uint64_t blocks = (tasks + (kThreads / 32) - 1) / (kThreads / 32);
    compact_write_kernel<D><<<grid_for(compact_write_kernel<D>, blocks), kThreads, 0, s>>>(
        a, tile_counts, offsets, task_prefix, idx_out, val_out, capacity);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_dense(const DecodeArgs& a, float* out, cudaStream_t s) {
    if (a.n == 0) return cudaSuccess;
    switch (a.d) {
        case 3: return launch_dense_d<3>(a, out, s);
        case 5: return launch_dense_d<5>(a, out, s);
        case 1: return launch_dense_d<1>(a, out, s);
        default: return launch_dense_d<0>(a, out, s);
    }
}

// Workspace of the row-pass dense decode: the candidate arrays (n floats
// each, rounded to 64), the listed-task count (256 bytes), the task list
// (one 32-bit id per task of 512 positions). Empty for other d.
DenseWsLayout dense_ws_layout(uint64_t n, uint32_t d) {
    DenseWsLayout L{};
    if (d != 3 && d != 5) return L;
    const uint64_t arr = (n + 63) / 64 * 64 * 4;
    const uint64_t tasks = (n + kTaskElems - 1) / kTaskElems;
    L.cand1 = 0;
    L.cand2 = arr;
    L.count = (d == 5 ? 2 : 1) * arr;
    L.list = L.count + 256;
    L.total = L.list + (tasks * 4 + 255) / 256 * 256;
    return L;
}

size_t dense_workspace_bytes(uint64_t n, uint32_t d) { return (size_t)dense_ws_layout(n, d).total; }

uint32_t dense_decode_passes(const DecodeArgs& a, uint64_t l2_bytes) {
    if (a.block || (a.d != 3 && a.d != 5) || (uint64_t)a.d * a.w * 4 <= pass_budget(l2_bytes)) return 1;
    const uint32_t rpp = rows_per_pass(a.w, l2_bytes);
    return (a.d + rpp - 1) / rpp;
}

cudaError_t launch_decode_dense_ws(const DecodeArgs& a, float* out, float* ws, cudaStream_t s) {
    if (a.n == 0) return cudaSuccess;
    DeviceInfo di{};
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    if (dense_decode_passes(a, (uint64_t)di.l2_bytes) == 1) return launch_decode_dense(a, out, s);
    const uint32_t rpp = rows_per_pass(a.w, (uint64_t)di.l2_bytes);
    return a.d == 3 ? launch_dense_rows<3>(a, out, ws, rpp, s) : launch_dense_rows<5>(a, out, ws, rpp, s);
}

cudaError_t launch_tile_scan(const uint32_t* counts, uint64_t tiles, uint32_t* offsets, unsigned long long* total,
                             cudaStream_t s) {
    compact_scan_kernel<<<1, kScanThreads, 0, s>>>(counts, tiles, offsets, total);
    return cudaGetLastError();
}

uint64_t compact_tiles(uint64_t nw) { return (nw + kCompactTileWords - 1) / kCompactTileWords; }

// Workspace of the compacted decode: tile counts, tile offsets (each rounded
// to 256 bytes), then the in-tile prefix of every task (16-bit).
size_t compact_workspace_bytes(uint64_t n) {
    const uint64_t tiles = compact_tiles((n + 31) / 32);
    const uint64_t one = (tiles * sizeof(uint32_t) + 255) / 256 * 256;
    const uint64_t prefix = (tiles * (kCompactTileWords / kTaskWords) * sizeof(uint16_t) + 255) / 256 * 256;
    return (size_t)(2 * one + prefix);
}

cudaError_t launch_decode_compact(const DecodeArgs& a, uint32_t* idx_out, float* val_out, uint64_t capacity,
                                  unsigned long long* count_out, uint32_t* tile_counts, uint32_t* tile_offsets,
                                  cudaStream_t s) {
    const uint64_t tiles = compact_tiles(a.nw);
    // the task prefixes follow the tile offsets (see compact_workspace_bytes)
    uint16_t* task_prefix = reinterpret_cast<uint16_t*>(tile_offsets + (tiles * sizeof(uint32_t) + 255) / 256 * 64);
    if (tiles > 0) {
        compact_count_kernel<<<grid_for(compact_count_kernel, tiles), kThreads, 0, s>>>(a.bitmap, a.nw, a.n,
                                                                                        tiles, tile_counts, task_prefix);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    compact_scan_kernel<<<1, kScanThreads, 0, s>>>(tile_counts, tiles, tile_offsets, count_out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || tiles == 0) return e;
    switch (a.d) {
        case 3: return launch_compact_write_d<3>(a, tile_counts, tile_offsets, task_prefix, idx_out, val_out, capacity, s);
        case 5: return launch_compact_write_d<5>(a, tile_counts, tile_offsets, task_prefix, idx_out, val_out, capacity, s);
        case 1: return launch_compact_write_d<1>(a, tile_counts, tile_offsets, task_prefix, idx_out, val_out, capacity, s);
        default: return launch_compact_write_d<0>(a, tile_counts, tile_offsets, task_prefix, idx_out, val_out, capacity, s);
    }
}

// ---- compaction with library-owned scratch -----------------------------------
// s2_decode_compact_noalloc runs the same three kernels as s2_decode_compact,
// but its tile counts, tile offsets and task prefixes live in this
// file-scope device array instead of a caller workspace. It covers n up to
// kNoAllocMaxN positions (2^30: 131,072 tiles; 1 MiB of counts and offsets,
// 4 MiB of 16-bit task prefixes); every GPU that loads the library holds the
// array until the process exits. Nothing in it has to start at zero: a call
// writes every count it later scans and every offset or prefix it later
// reads. The prefixes of a call start right after its own tile offsets.
constexpr uint64_t kNoAllocMaxN = 1ull << 30;
constexpr uint64_t kNoAllocMaxTiles = (kNoAllocMaxN / 32) / kCompactTileWords;
static __device__ __align__(256) uint32_t
    g_noalloc_compact_scratch[2 * kNoAllocMaxTiles + (kNoAllocMaxTiles * (kCompactTileWords / kTaskWords)) / 2 + 64];

uint64_t noalloc_compact_max_n() { return kNoAllocMaxN; }

// Device address of the scratch for the current device. The address is looked
// up with cudaGetSymbolAddress, with that device current, the first time a
// call on the device succeeds in doing so, and cached from then on; a failed
// lookup (for example one attempted during a stream capture) is not cached,
// so the next call tries again. Host code must never pass the symbol itself
// to a kernel: on the host it names a stand-in, not device memory.
cudaError_t noalloc_compact_scratch(uint32_t** counts, uint32_t** offsets) {
    static std::mutex mu;
    static uint32_t* base[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!base[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_compact_scratch);
        if (e != cudaSuccess) {
            cudaGetLastError();  // leave no sticky launch error behind a failed lookup
            return e;
        }
        base[dev] = static_cast<uint32_t*>(p);
    }
    *counts = base[dev];
    *offsets = base[dev] + kNoAllocMaxTiles;
    return cudaSuccess;
}

// ---- hash check --------------------------------------------------------------

namespace {
__global__ void __launch_bounds__(kThreads) hash_kernel(const uint32_t* __restrict__ idx, uint64_t m, uint32_t d,
                                                        uint32_t w, RowKeys keys, uint32_t* __restrict__ bucket_out,
                                                        int8_t* __restrict__ sign_out) {
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t t = tid; t < m; t += stride) {
        const uint32_t i = idx[t];
        for (uint32_t j = 0; j < d; ++j) {
            bucket_out[(uint64_t)j * m + t] = bucket_of(i, keys.kh[j], w);
            sign_out[(uint64_t)j * m + t] = signbit_of(i, keys.ks[j]) ? (int8_t)-1 : (int8_t)1;
        }
    }
}
}  // namespace

cudaError_t launch_hash(const uint32_t* idx, uint64_t m, uint32_t d, uint32_t w, RowKeys keys,
                        uint32_t* bucket_out, int8_t* sign_out, cudaStream_t s) {
    if (m == 0) return cudaSuccess;
    const uint64_t blocks = (m + kThreads - 1) / kThreads;
    hash_kernel<<<grid_for(hash_kernel, blocks), kThreads, 0, s>>>(idx, m, d, w, keys, bucket_out, sign_out);
    return cudaGetLastError();
}

}  // namespace s2
