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
#include <atomic>

#include "s2_tasks.cuh"

namespace s2 {
namespace {

// Insert value `val` of position `i` into every row of the sketch. The
// reductions carry no L2 policy of their own: the zero fill before the
// encode stored the sketch's lines evict-last and the gradient streams past
// with evict-first loads. Measured on GB300 (ms per step, large LM /
// embedding / top-k): reductions with an evict-last policy on every line
// 1.613 / 0.514 / 0.242, on a quarter of the lines 1.585 / 0.512 / 0.236,
// without a policy 1.571 / 0.509 / 0.235; plain zero-fill stores instead
// cost 18 % on the large LM (1.852). SL: only buckets whose flattened
// index j*w + b lies in the launch's slice [a.x_lo, a.x_lo + a.x_span) are
// updated (a sketch larger than L2 is built one slice per pass).
template <int D, bool SL>
__device__ __forceinline__ void insert(float* __restrict__ sk, uint32_t i, float val, const EncodeArgs& a,
                                       const uint32_t* s_kh, const uint32_t* s_ks) {
    const int rows = D > 0 ? D : a.d;
#pragma unroll
    for (int j = 0; j < (D > 0 ? D : kMaxRows); ++j) {
        if (D > 0 || j < rows) {
            const uint64_t x = (uint64_t)j * a.w + bucket_of(i, s_kh[j], a.w);
            if (!SL || x - a.x_lo < a.x_span) {
                const uint32_t sb = signbit_of(i, s_ks[j]);
                red_add_f32(sk + x, apply_sign(val, sb));
            }
        }
    }
}


// Store word wi of worker k's bitmap (lanes with valid = true hold one). With
// BLK, the bitmap is a block bitmap (one bit per a.block_words words, zeroed
// beforehand): every block that holds a nonzero word is marked once per task
// with an atomicOr; lanes marking the same block are merged first. Called by
// all 32 lanes.
template <bool BLK>
__device__ __forceinline__ void store_bitmap_word(const EncodeArgs& a, uint32_t k, uint64_t wi, uint32_t word,
                                                  bool valid, int lane) {
    if (!BLK) {
        if (valid) a.bitmaps[(uint64_t)k * a.nw + wi] = word;
    } else {
        const bool mark = valid && word != 0;
        const unsigned long long blk = mark ? wi / a.block_words : ~0ull;
        const unsigned grp = __match_any_sync(kFull, blk);
        if (mark && __ffs(grp) - 1 == lane)
            atomicOr(a.bitmaps + (uint64_t)k * a.nbw + (blk >> 5), 1u << (blk & 31));
    }
}

// Nonzeros of sparse tasks wait in a per-warp list until 32 of them can be
// inserted at once, one per lane (see encode_f32_vec).
constexpr uint32_t kListCap = 64;
constexpr uint32_t kDenseTask = 32;  // a task with at least this many nonzeros is walked per lane

template <int D, bool SL>
__device__ __forceinline__ void insert_listed(const uint32_t* lpos, const float* lval, uint32_t cnt, int lane,
                                              float* sk, const EncodeArgs& a, const uint32_t* s_kh,
                                              const uint32_t* s_ks) {
    if ((uint32_t)lane < cnt) insert<D, SL>(sk, lpos[lane], lval[lane], a, s_kh, s_ks);
}

// fp32 rows, 16-byte aligned. Dense tasks (>= kDenseTask nonzeros, e.g. the
// whole embedding rows) are inserted by each lane walking its own slots;
// the nonzeros of sparse tasks (a few scattered values per 512 positions)
// are appended to a per-warp list in shared memory instead, and inserted 32
// at a time with every lane busy, so their d reductions do not run on lone
// lanes. The list only holds one worker's entries; it is drained when the
// warp moves on to another worker and at the end.
template <int D, bool BLK, bool SL>
__global__ void __launch_bounds__(kThreads) encode_f32_vec(EncodeArgs a) {
    __shared__ uint32_t s_kh[kMaxRows], s_ks[kMaxRows];
    __shared__ uint32_t s_lpos[kThreads / 32][kListCap];
    __shared__ float s_lval[kThreads / 32][kListCap];
    load_keys(a.keys, s_kh, s_ks);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t* lpos = s_lpos[warp];
    float* lval = s_lval[warp];
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    uint32_t k = 0;
    uint32_t local = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    while (local >= a.tasks_per_worker && k < a.workers) {
        local -= a.tasks_per_worker;
        ++k;
    }
    const float* grad = reinterpret_cast<const float*>(a.grad);
    uint32_t lcount = 0, lk = k;  // listed entries and their worker (warp-uniform)
    uint4 v[4];
    if (k < a.workers) load_f32_task(v, grad + (uint64_t)k * a.n, (uint64_t)local * kTaskElems, a.n, lane);
    for (; k < a.workers;) {
        const uint64_t e0 = (uint64_t)local * kTaskElems;
        // the warp's next task, whose loads go out before this task is processed
        uint32_t nk = k, nlocal = local + nwarps;
        while (nlocal >= a.tasks_per_worker && nk < a.workers) {
            nlocal -= a.tasks_per_worker;
            ++nk;
        }
        uint4 nv[4];
        if (nk < a.workers)
            load_f32_task(nv, grad + (uint64_t)nk * a.n, (uint64_t)nlocal * kTaskElems, a.n, lane);
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
        {
            const uint64_t wi = (uint64_t)local * kTaskWords + lane;
            store_bitmap_word<BLK>(a, k, wi, my_word, lane < kTaskWords && wi < a.nw, lane);
        }
        uint32_t total;
        const uint32_t excl = warp_exclusive_scan(__popc(mask), lane, &total);
        if (total >= kDenseTask) {
            float* sk = a.sketches + (uint64_t)k * a.dw;
            while (mask) {
                const int slot = __ffs(mask) - 1;
                mask &= mask - 1;
                const uint32_t i = (uint32_t)(e0 + (slot >> 2) * 128 + lane * 4 + (slot & 3));
                insert<D, SL>(sk, i, __uint_as_float(pick16(v, slot)), a, s_kh, s_ks);
            }
        } else if (total > 0) {
            if (k != lk && lcount > 0) {  // the list belongs to another worker: drain it first
                insert_listed<D, SL>(lpos, lval, lcount, lane, a.sketches + (uint64_t)lk * a.dw, a, s_kh, s_ks);
                __syncwarp();
                lcount = 0;
            }
            lk = k;
            uint32_t at = lcount + excl;
            for (uint32_t m = mask; m; m &= m - 1, ++at) {
                const int slot = __ffs(m) - 1;
                lpos[at] = (uint32_t)(e0 + (slot >> 2) * 128 + lane * 4 + (slot & 3));
                lval[at] = __uint_as_float(pick16(v, slot));
            }
            lcount += total;  // at most 31 + 31 < kListCap
            __syncwarp();
            if (lcount >= 32) {
                insert_listed<D, SL>(lpos, lval, 32, lane, a.sketches + (uint64_t)lk * a.dw, a, s_kh, s_ks);
                const uint32_t rest = lcount - 32;
                uint32_t p = 0;
                float q = 0.f;
                if ((uint32_t)lane < rest) {
                    p = lpos[32 + lane];
                    q = lval[32 + lane];
                }
                __syncwarp();
                if ((uint32_t)lane < rest) {
                    lpos[lane] = p;
                    lval[lane] = q;
                }
                __syncwarp();
                lcount = rest;
            }
        }
        k = nk;
        local = nlocal;
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = nv[u];
    }
    if (lcount > 0)
        insert_listed<D, SL>(lpos, lval, lcount, lane, a.sketches + (uint64_t)lk * a.dw, a, s_kh, s_ks);
}

// ---- bf16, 16-byte vector loads --------------------------------------------
// Lane l loads positions u*256 + 8l .. +7 for u = 0..1; slot 8u + c is
// position u*256 + 8l + c. Word q of chunk u is made of the bytes of lanes
// 4q .. 4q+3.
template <int D, bool BLK, bool SL>
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
        {
            const uint64_t wi = (uint64_t)local * kTaskWords + lane;
            store_bitmap_word<BLK>(a, k, wi, my_word, lane < kTaskWords && wi < a.nw, lane);
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
            insert<D, SL>(sk, i, __uint_as_float(bits), a, s_kh, s_ks);
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
template <int D, bool BF16, bool BLK, bool SL>
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
        {
            const uint64_t wi = (uint64_t)local * kTaskWords + lane;
            store_bitmap_word<BLK>(a, k, wi, my_word, lane < kTaskWords && wi < a.nw, lane);
        }
        float* sk = a.sketches + (uint64_t)k * a.dw;
        while (mask) {
            const int slot = __ffs(mask) - 1;
            mask &= mask - 1;
            uint32_t bits = x[0];
#pragma unroll
            for (int s = 1; s < 16; ++s) bits = (slot == s) ? x[s] : bits;
            const uint32_t i = (uint32_t)(e0 + slot * 32 + lane);
            insert<D, SL>(sk, i, __uint_as_float(bits), a, s_kh, s_ks);
        }
        local += nwarps;
        while (local >= a.tasks_per_worker && k < a.workers) {
            local -= a.tasks_per_worker;
            ++k;
        }
    }
}

// ---- shared-memory privatised sketch ----------------------------------------
// For a sketch small enough to live in shared memory (4*d*w at most
// kPrivMaxBytes), each block owns a contiguous range of one worker's tasks
// and accumulates that range's inserts in a private d x w copy in shared
// memory; lanes of a warp that hit the same bucket in the same step are
// merged first (AGG), so each shared-memory atomic carries one bucket's sum.
// At the end the copy is added into the worker's sketch in global memory
// with d*w/4 vector reductions (or stored, when one block covers the whole
// worker): the L2 sees d*w/4 operations per block instead of d per nonzero.
//
// The four load layouts L of a task are those of s2_tasks.cuh.
constexpr int kPrivThreads = 1024;

// Add v into tile[x] for every lane with act set; lanes with the same x are
// merged first: the lowest of them adds the group's sum, taken in ascending
// lane order. Called by all 32 lanes.
__device__ __forceinline__ void smem_add_merged(float* tile, uint32_t x, float v, bool act, int lane) {
    const uint32_t key = act ? x : 0xffffffffu;
    const unsigned grp = __match_any_sync(kFull, key);
    const int leader = __ffs(grp) - 1;
    unsigned others = grp & (grp - 1);  // the group without its lowest lane
    const int extra = (act && lane == leader) ? __popc(others) : 0;
    const int rounds = __reduce_max_sync(kFull, (unsigned)extra);
    float s = v;
    for (int r = 0; r < rounds; ++r) {
        const int src = others ? __ffs(others) - 1 : lane;
        const float o = __shfl_sync(kFull, v, src);
        if (others) {
            s += o;
            others &= others - 1;
        }
    }
    if (act && lane == leader) atomicAdd(tile + x, s);
}

template <int D, int L, bool BLK, bool AGG>
__global__ void __launch_bounds__(kPrivThreads) encode_priv(EncodeArgs a, uint32_t per_worker, int store) {
    extern __shared__ __align__(16) float s_tile[];  // [d][w]
    __shared__ uint32_t s_kh[kMaxRows], s_ks[kMaxRows];
    const uint32_t dw = (uint32_t)a.dw;
    for (uint32_t x = threadIdx.x; x < dw; x += blockDim.x) s_tile[x] = 0.f;
    load_keys(a.keys, s_kh, s_ks);  // ends with __syncthreads
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t k = blockIdx.x / per_worker, part = blockIdx.x - k * per_worker;
    const uint64_t T = a.tasks_per_worker;
    const uint64_t t1 = T * (part + 1) / per_worker;
    constexpr uint64_t esz = (L == 1 || L == 3) ? 2 : 4;
    const void* row = static_cast<const char*>(a.grad) + (uint64_t)k * a.n * esz;
    const int rows = D > 0 ? D : a.d;
    uint64_t t = T * part / per_worker + warp;
    uint4 v[4];
    if (t < t1) load_task<L>(v, row, t * kTaskElems, a.n, lane);
    for (; t < t1; t += nwarps) {
        const uint64_t e0 = t * kTaskElems;
        const bool more = t + nwarps < t1;
        uint4 nv[4];
        if (more) load_task<L>(nv, row, (t + nwarps) * kTaskElems, a.n, lane);
        uint32_t my_word;
        uint32_t mask = task_bits<L>(v, lane, &my_word);
        const uint64_t wi = t * kTaskWords + lane;
        store_bitmap_word<BLK>(a, k, wi, my_word, lane < kTaskWords && wi < a.nw, lane);
        while (__any_sync(kFull, mask != 0)) {
            const bool act = mask != 0;
            const int slot = act ? __ffs(mask) - 1 : 0;
            mask &= mask - 1;
            const uint32_t i = slot_position<L>(e0, slot, lane);
            const float val = __uint_as_float(slot_bits<L>(v, slot));
#pragma unroll
            for (int j = 0; j < (D > 0 ? D : kMaxRows); ++j) {
                if (D > 0 || j < rows) {
                    const uint32_t x = (uint32_t)j * a.w + bucket_of(i, s_kh[j], a.w);
                    const float sv = apply_sign(val, signbit_of(i, s_ks[j]));
                    if (AGG)
                        smem_add_merged(s_tile, x, sv, act, lane);
                    else if (act)
                        atomicAdd(s_tile + x, sv);
                }
            }
        }
        if (more) {
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = nv[u];
        }
    }
    __syncthreads();
    float* sk = a.sketches + (uint64_t)k * a.dw;
    if ((dw & 3u) == 0) {  // every worker's sketch starts on a 16-byte boundary
        const float4* t4 = reinterpret_cast<const float4*>(s_tile);
        for (uint32_t x = threadIdx.x; x < dw / 4; x += blockDim.x) {
            const float4 q = t4[x];
            if (store)
                reinterpret_cast<float4*>(sk)[x] = q;
            else if (q.x != 0.f || q.y != 0.f || q.z != 0.f || q.w != 0.f)
                red_add_f32x4(sk + 4 * x, q);
        }
    } else {
        for (uint32_t x = threadIdx.x; x < dw; x += blockDim.x) {
            const float q = s_tile[x];
            if (store)
                sk[x] = q;
            else if (q != 0.f)
                red_add_f32(sk + x, q);
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
    const uint64_t keep = policy_evict_last();  // the encode that follows updates these lines
    for (uint64_t x = tid; x < n4; x += stride) st_f4_hint(p4 + x, make_float4(0.f, 0.f, 0.f, 0.f), keep);
    for (uint64_t x = head + n4 * 4 + tid; x < count; x += stride) p[x] = 0.f;
}

template <int D, bool BLK, bool SL>
cudaError_t launch_encode_dbs(const EncodeArgs& a, int dtype, bool vec, cudaStream_t s) {
    const uint64_t tasks = (uint64_t)a.workers * a.tasks_per_worker;
    const uint64_t blocks = (tasks + (kThreads / 32) - 1) / (kThreads / 32);
    if (vec && dtype == 0) {
        encode_f32_vec<D, BLK, SL><<<grid_for(encode_f32_vec<D, BLK, SL>, blocks), kThreads, 0, s>>>(a);
    } else if (vec && dtype == 1) {
        encode_bf16_vec<D, BLK, SL><<<grid_for(encode_bf16_vec<D, BLK, SL>, blocks), kThreads, 0, s>>>(a);
    } else if (dtype == 0) {
        encode_scalar<D, false, BLK, SL><<<grid_for(encode_scalar<D, false, BLK, SL>, blocks), kThreads, 0, s>>>(a);
    } else {
        encode_scalar<D, true, BLK, SL><<<grid_for(encode_scalar<D, true, BLK, SL>, blocks), kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

// Slices (x_span < d*w) are only used with the element bitmap.
template <int D, bool BLK>
cudaError_t launch_encode_db(const EncodeArgs& a, int dtype, bool vec, cudaStream_t s) {
    if (!BLK && a.x_span < a.dw) return launch_encode_dbs<D, false, true>(a, dtype, vec, s);
    return launch_encode_dbs<D, BLK, false>(a, dtype, vec, s);
}

// ---- shared-memory path: planning and launch ------------------------------
// Buckets per row up to which lanes hitting the same bucket are merged
// before the shared-memory atomic. Measured on GB300 (8 workers of 2^22
// positions, d = 3): merging pays only in rows of about 16 buckets with half
// of the positions nonzero; from 64 buckets up, the match/shuffle work costs
// more than the serialised same-address atomics it saves (up to 2.3x slower).
constexpr uint32_t kAggMaxW = 16;

template <int D, int L, bool BLK, bool AGG>
cudaError_t launch_priv_t(const EncodeArgs& a, bool only_if_preferred, bool* launched, cudaStream_t s) {
    auto kern = encode_priv<D, L, BLK, AGG>;
    const size_t smem = (size_t)a.dw * 4;
    static std::atomic<bool> configured[64];  // cudaFuncSetAttribute is idempotent
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !configured[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrivMaxBytes);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    DeviceInfo di{};
    e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int per_sm = blocks_per_sm(reinterpret_cast<const void*>(kern), kPrivThreads, smem);
    // blocks per worker: enough to fill every SM, at most one per warp's task
    const uint64_t slots = (uint64_t)di.sms * (uint64_t)(per_sm > 0 ? per_sm : 1);
    uint64_t per_worker = (slots + a.workers - 1) / a.workers;
    const uint64_t most = ((uint64_t)a.tasks_per_worker + kPrivThreads / 32 - 1) / (kPrivThreads / 32);
    if (per_worker > most) per_worker = most;
    if (per_worker < 1) per_worker = 1;
    if (only_if_preferred) {
        // Taken when a row has few buckets for the positions (at least 4096
        // positions per bucket: from about 1% density on, every bucket takes
        // tens of adds, which serialise in L2 but not in shared memory) and
        // the blocks' final additions (d*w/4 operations each) cost at most
        // half the sectors of the worker's gradient row (n*esz/32). Measured
        // on GB300: 1.1x slower than the L2 path at 1% density, 2.5-20x
        // faster at 10-50%; with the paper's sketch sizing (w about half the
        // nonzeros, so fewer than 2000 positions per bucket) the L2 path,
        // 5-15% faster there, is kept.
        const uint64_t esz = (L == 1 || L == 3) ? 2 : 4;
        if (a.n < (uint64_t)a.w * 4096 || per_worker * a.dw * 16 > a.n * esz) {
            *launched = false;
            return cudaSuccess;
        }
    }
    if (per_worker > 1) {
        e = launch_zero(a.sketches, (uint64_t)a.workers * a.dw, s);
        if (e != cudaSuccess) return e;
    }
    const uint64_t esz = (L == 1 || L == 3) ? 2 : 4;
    const uint64_t chunk = 0x7fffffffull / per_worker;  // workers per launch: grid below 2^31 blocks
    for (uint64_t k0 = 0; k0 < a.workers; k0 += chunk) {
        EncodeArgs b = a;
        b.workers = (uint32_t)((a.workers - k0) < chunk ? (a.workers - k0) : chunk);
        b.grad = static_cast<const char*>(a.grad) + k0 * a.n * esz;
        b.bitmaps = a.bitmaps + k0 * (BLK ? a.nbw : a.nw);
        b.sketches = a.sketches + k0 * a.dw;
        kern<<<(unsigned)(b.workers * per_worker), kPrivThreads, smem, s>>>(b, (uint32_t)per_worker,
                                                                          per_worker == 1 ? 1 : 0);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    *launched = true;
    return cudaSuccess;
}

template <int D, int L, bool BLK>
cudaError_t launch_priv_l(const EncodeArgs& a, bool only_if_preferred, bool* launched, cudaStream_t s) {
    return a.w <= kAggMaxW ? launch_priv_t<D, L, BLK, true>(a, only_if_preferred, launched, s)
                           : launch_priv_t<D, L, BLK, false>(a, only_if_preferred, launched, s);
}

template <int D, bool BLK>
cudaError_t launch_priv_db(const EncodeArgs& a, int dtype, bool vec, bool only_if_preferred, bool* launched,
                           cudaStream_t s) {
    if (vec) {
        return dtype == 0 ? launch_priv_l<D, 0, BLK>(a, only_if_preferred, launched, s)
                          : launch_priv_l<D, 1, BLK>(a, only_if_preferred, launched, s);
    }
    return dtype == 0 ? launch_priv_l<D, 2, BLK>(a, only_if_preferred, launched, s)
                      : launch_priv_l<D, 3, BLK>(a, only_if_preferred, launched, s);
}

template <int D>
cudaError_t launch_priv_d(const EncodeArgs& a, int dtype, bool vec, bool only_if_preferred, bool* launched,
                          cudaStream_t s) {
    return a.block_words ? launch_priv_db<D, true>(a, dtype, vec, only_if_preferred, launched, s)
                         : launch_priv_db<D, false>(a, dtype, vec, only_if_preferred, launched, s);
}

template <int D>
cudaError_t launch_encode_d(const EncodeArgs& a, int dtype, bool vec, cudaStream_t s) {
    return a.block_words ? launch_encode_db<D, true>(a, dtype, vec, s) : launch_encode_db<D, false>(a, dtype, vec, s);
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

cudaError_t launch_encode_smem(const EncodeArgs& a, int dtype, bool vec, bool only_if_preferred, bool* launched,
                               cudaStream_t s) {
    *launched = false;
    if ((uint64_t)a.dw * 4 > kPrivMaxBytes) return cudaSuccess;
    if (a.workers == 0 || a.tasks_per_worker == 0) {  // nothing to read: the sketches are zero
        *launched = true;
        return launch_zero(a.sketches, (uint64_t)a.workers * a.dw, s);
    }
    switch (a.d) {
        case 3: return launch_priv_d<3>(a, dtype, vec, only_if_preferred, launched, s);
        case 5: return launch_priv_d<5>(a, dtype, vec, only_if_preferred, launched, s);
        default: return launch_priv_d<0>(a, dtype, vec, only_if_preferred, launched, s);
    }
}

cudaError_t launch_zero(float* p, uint64_t count, cudaStream_t s) {
    if (count == 0) return cudaSuccess;
    const uint64_t blocks = (count / 4 + kThreads - 1) / kThreads + 1;
    zero_f32<<<grid_for(zero_f32, blocks), kThreads, 0, s>>>(p, count);
    return cudaGetLastError();
}

}  // namespace s2
