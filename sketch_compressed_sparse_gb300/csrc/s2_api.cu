// C ABI of libs2: argument validation and dispatch to the kernels. Every
// entry point checks its arguments completely before anything is launched,
// then queues its kernels on the caller's stream and returns.
#include <cstring>
#include <mutex>

#include "s2.h"  // include/ is on the include path
#include "s2_internal.h"

namespace s2 {

cudaError_t device_info(DeviceInfo* out) {
    static DeviceInfo cache[64];
    static std::once_flag once[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaError_t err = cudaSuccess;
    std::call_once(once[dev], [&] {
        DeviceInfo di{};
        err = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&di.l2_bytes, cudaDevAttrL2CacheSize, dev);
        cache[dev] = di;
    });
    if (err != cudaSuccess) return err;
    if (cache[dev].sms <= 0) return cudaErrorInvalidDevice;
    *out = cache[dev];
    return cudaSuccess;
}

int blocks_per_sm(const void* fn, int threads, size_t smem) {
    struct Entry {
        int dev;
        const void* fn;
        int threads;
        size_t smem;
        int per_sm;
    };
    static std::mutex mu;
    static Entry table[512];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int x = 0; x < used; ++x)
            if (table[x].dev == dev && table[x].fn == fn && table[x].threads == threads && table[x].smem == smem)
                return table[x].per_sm;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();  // a failed query is not a launch error
        return 1;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (used < 512) table[used++] = Entry{dev, fn, threads, smem, per_sm};
    return per_sm;
}

static uint32_t host_fmix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x85ebca6bu;
    x ^= x >> 13;
    x *= 0xc2b2ae35u;
    x ^= x >> 16;
    return x;
}

RowKeys make_keys(uint32_t seed, uint32_t d) {
    RowKeys k;
    std::memset(&k, 0, sizeof(k));
    const uint32_t golden = 0x9E3779B9u;
    for (uint32_t j = 0; j < d && j < (uint32_t)kMaxRows; ++j) {
        k.kh[j] = host_fmix32(seed ^ (uint32_t)(golden * (2u * j + 1u)));
        k.ks[j] = host_fmix32(seed ^ (uint32_t)(golden * (2u * j + 2u)));
    }
    return k;
}

}  // namespace s2

using namespace s2;

namespace {

constexpr uint64_t kMaxN = 0xffffffffull;  // positions are 32-bit
static_assert(kPrivMaxBytes == S2_SMEM_SKETCH_MAX_BYTES, "shared-memory sketch limit differs from the header");

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Byte ranges [a, a+na) and [b, b+nb) intersect (empty ranges never do).
inline bool overlap(const void* a, uint64_t na, const void* b, uint64_t nb) {
    if (na == 0 || nb == 0 || a == nullptr || b == nullptr) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

inline s2_status check_params(const s2_params& p) {
    if (p.d < 1 || p.d > S2_MAX_ROWS) return S2_ERR_INVALID_ARG;
    if (p.w < 1 || p.w > (1u << 31)) return S2_ERR_INVALID_ARG;
    return S2_OK;
}

inline uint64_t words_of(uint64_t n) { return (n + 31) / 32; }

inline s2_status cuda_status(cudaError_t e) { return e == cudaSuccess ? S2_OK : S2_ERR_CUDA; }

inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Encode W workers: zero the sketches and fill them, in groups of workers
// whose sketches fit in half of L2 together, so that each group's
// sketches are zeroed, updated and written back once.
s2_status encode_impl(const void* grad, s2_dtype dt, uint32_t W, uint64_t n, s2_params p, uint32_t* bitmaps,
                      float* sketches, cudaStream_t stream, uint32_t block = 0,
                      s2_encode_path path = S2_PATH_AUTO) {
    const uint64_t esz = dt == S2_F32 ? 4 : 2;
    const uint64_t nw = words_of(n);
    const uint64_t dw = (uint64_t)p.d * p.w;
    DeviceInfo di{};
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return S2_ERR_CUDA;
    const uint64_t sk_bytes = dw * 4;
    uint64_t group = sk_bytes ? ((uint64_t)di.l2_bytes / 2) / sk_bytes : W;
    if (group < 1) group = 1;
    if (group > W) group = W;
    // A sketch too large to stay in L2 while it is built (above 3/4 of L2:
    // its reductions would go to DRAM) is built one worker at a time in
    // `passes` slices of its flattened buckets, each pass re-reading the
    // worker's gradient and updating only its slice. Element bitmaps only.
    // Measured on GB300 (8 workers of 2^27 positions at 10 % density): a
    // 160 MB sketch in two passes 5.6 ms instead of 10.7 ms; a 96 MB sketch
    // 3.7 ms in one pass, 4.1 ms in two.
    const uint64_t slice_cap = (uint64_t)di.l2_bytes / 4 * 3;
    uint64_t passes = 1;
    if (sk_bytes > slice_cap && path != S2_PATH_SMEM && block == 0) {
        passes = (sk_bytes + slice_cap - 1) / slice_cap;
        group = 1;
    }
    // vector loads need every worker row 16-byte aligned
    const bool vec = ((n * esz) % 16 == 0) || W == 1;
    EncodeArgs a;
    std::memset(&a, 0, sizeof(a));
    a.n = n;
    a.nw = nw;
    a.dw = dw;
    a.tasks_per_worker = (uint32_t)((n + kTaskElems - 1) / kTaskElems);
    a.d = p.d;
    a.w = p.w;
    a.keys = make_keys(p.seed, p.d);
    const uint64_t nbw = block ? words_of((n + block - 1) / block) : 0;
    a.block_words = block / 32;
    a.nbw = nbw;
    a.x_lo = 0;
    a.x_span = dw;
    if (block && W * nbw) {  // block bits are set with atomicOr: start from zero
        e = launch_zero(reinterpret_cast<float*>(bitmaps), W * nbw, stream);
        if (e != cudaSuccess) return S2_ERR_CUDA;
    }
    if (path != S2_PATH_L2 && sk_bytes <= kPrivMaxBytes) {
        a.grad = grad;
        a.bitmaps = bitmaps;
        a.sketches = sketches;
        a.workers = W;
        bool launched = false;
        e = launch_encode_smem(a, dt == S2_F32 ? 0 : 1, vec, path == S2_PATH_AUTO, &launched, stream);
        if (e != cudaSuccess) return S2_ERR_CUDA;
        if (launched) return S2_OK;
    }
    for (uint64_t k0 = 0; k0 < W; k0 += group) {
        const uint64_t g = (W - k0) < group ? (W - k0) : group;
        a.grad = static_cast<const char*>(grad) + k0 * n * esz;
        a.bitmaps = bitmaps + k0 * (block ? nbw : nw);
        a.sketches = sketches + k0 * dw;
        a.workers = (uint32_t)g;
        if (passes == 1) {
            e = launch_zero(sketches + k0 * dw, g * dw, stream);
            if (e != cudaSuccess) return S2_ERR_CUDA;
            e = launch_encode(a, dt == S2_F32 ? 0 : 1, vec, stream);
            if (e != cudaSuccess) return S2_ERR_CUDA;
            continue;
        }
        // one worker, slice by slice (the bitmap is rewritten with the same
        // words on every pass; block bits are ORed again)
        const uint64_t span = (dw + passes - 1) / passes;
        for (uint64_t x0 = 0; x0 < dw; x0 += span) {
            a.x_lo = x0;
            a.x_span = (dw - x0) < span ? (dw - x0) : span;
            e = launch_zero(sketches + k0 * dw + x0, a.x_span, stream);
            if (e != cudaSuccess) return S2_ERR_CUDA;
            e = launch_encode(a, dt == S2_F32 ? 0 : 1, vec, stream);
            if (e != cudaSuccess) return S2_ERR_CUDA;
        }
        a.x_lo = 0;
        a.x_span = dw;
    }
    return S2_OK;
}

s2_status check_encode(const void* grad, s2_dtype dt, uint32_t W, uint64_t n, s2_params p, const uint32_t* bitmaps,
                       const float* sketches) {
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (dt != S2_F32 && dt != S2_BF16) return S2_ERR_INVALID_ARG;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    if (W == 0) return S2_OK;
    const uint64_t esz = dt == S2_F32 ? 4 : 2;
    const uint64_t gbytes = (uint64_t)W * n * esz, bbytes = (uint64_t)W * words_of(n) * 4,
                   sbytes = (uint64_t)W * p.d * p.w * 4;
    if (!sketches || (n > 0 && (!grad || !bitmaps))) return S2_ERR_INVALID_ARG;
    if (!aligned(grad, 16) || !aligned(bitmaps, 16) || !aligned(sketches, 16)) return S2_ERR_ALIGNMENT;
    if (overlap(grad, gbytes, bitmaps, bbytes) || overlap(grad, gbytes, sketches, sbytes) ||
        overlap(bitmaps, bbytes, sketches, sbytes))
        return S2_ERR_INVALID_ARG;
    return S2_OK;
}

s2_status check_reduce(const uint32_t* bitmaps, const float* sketches, uint32_t W, uint64_t n, s2_params p,
                       const uint32_t* bitmap_out, const float* sketch_out) {
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    const uint64_t nw = words_of(n), dw = (uint64_t)p.d * p.w;
    if (!sketch_out || (nw > 0 && !bitmap_out)) return S2_ERR_INVALID_ARG;
    if (W > 0 && (!sketches || (nw > 0 && !bitmaps))) return S2_ERR_INVALID_ARG;
    if (!aligned(bitmaps, 16) || !aligned(sketches, 16) || !aligned(bitmap_out, 16) || !aligned(sketch_out, 16))
        return S2_ERR_ALIGNMENT;
    const uint64_t ib = (uint64_t)W * nw * 4, is = (uint64_t)W * dw * 4;
    if (overlap(bitmaps, ib, bitmap_out, nw * 4) || overlap(bitmaps, ib, sketch_out, dw * 4) ||
        overlap(sketches, is, bitmap_out, nw * 4) || overlap(sketches, is, sketch_out, dw * 4) ||
        overlap(bitmap_out, nw * 4, sketch_out, dw * 4))
        return S2_ERR_INVALID_ARG;
    return S2_OK;
}

s2_status check_decode_dense(const uint32_t* bitmap, const float* sketch, uint64_t n, s2_params p, const float* out) {
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    if (n == 0) return S2_OK;
    if (!bitmap || !sketch || !out) return S2_ERR_INVALID_ARG;
    if (!aligned(bitmap, 16) || !aligned(sketch, 16) || !aligned(out, 16)) return S2_ERR_ALIGNMENT;
    const uint64_t dw = (uint64_t)p.d * p.w;
    if (overlap(out, n * 4, bitmap, words_of(n) * 4) || overlap(out, n * 4, sketch, dw * 4))
        return S2_ERR_INVALID_ARG;
    return S2_OK;
}

DecodeArgs make_decode_args(const uint32_t* bitmap, const float* sketch, uint64_t n, s2_params p, float scale) {
    DecodeArgs a;
    std::memset(&a, 0, sizeof(a));
    a.bitmap = bitmap;
    a.sketch = sketch;
    a.n = n;
    a.nw = words_of(n);
    a.d = p.d;
    a.w = p.w;
    a.scale = scale;
    a.keys = make_keys(p.seed, p.d);
    return a;
}

// Device address of page-locked host memory at `p` that the current device
// can access in place (16-byte aligned), or nullptr for any other memory.
const void* mapped_host(const void* p) {
    if (!p) return nullptr;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer is not an error here
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || !at.devicePointer || !aligned(at.devicePointer, 16)) return nullptr;
    return at.devicePointer;
}

struct PipelineLayout {
    size_t grad, bitmaps, sketches, bitmap, sketch, out, dec_ws, total;
};

PipelineLayout pipeline_layout(s2_dtype dt, uint32_t W, uint64_t n, s2_params p) {
    const uint64_t esz = dt == S2_F32 ? 4 : 2, nw = words_of(n), dw = (uint64_t)p.d * p.w;
    PipelineLayout L{};
    size_t off = 0;
    L.grad = off;
    off += round256((size_t)W * n * esz);
    L.bitmaps = off;
    off += round256((size_t)W * nw * 4);
    L.sketches = off;
    off += round256((size_t)W * dw * 4);
    L.bitmap = off;
    off += round256((size_t)nw * 4);
    L.sketch = off;
    off += round256((size_t)dw * 4);
    L.out = off;
    off += round256((size_t)n * 4);
    L.dec_ws = off;
    off += round256(dense_workspace_bytes(n, p.d));
    L.total = off;
    return L;
}

}  // namespace

extern "C" {

s2_status s2_encode(const void* grad, s2_dtype dt, uint64_t n, s2_params p, uint32_t* bitmap, float* sketch,
                    s2_stream_t stream) {
    s2_status st = check_encode(grad, dt, 1, n, p, bitmap, sketch);
    if (st != S2_OK) return st;
    return encode_impl(grad, dt, 1, n, p, bitmap, sketch, reinterpret_cast<cudaStream_t>(stream));
}

s2_status s2_encode_batched(const void* grad, s2_dtype dt, uint32_t W, uint64_t n, s2_params p, uint32_t* bitmaps,
                            float* sketches, s2_stream_t stream) {
    s2_status st = check_encode(grad, dt, W, n, p, bitmaps, sketches);
    if (st != S2_OK || W == 0) return st;
    return encode_impl(grad, dt, W, n, p, bitmaps, sketches, reinterpret_cast<cudaStream_t>(stream));
}

s2_status s2_encode_batched_path(const void* grad, s2_dtype dt, uint32_t W, uint64_t n, s2_params p,
                                 s2_encode_path path, uint32_t* bitmaps, float* sketches, s2_stream_t stream) {
    if (path != S2_PATH_AUTO && path != S2_PATH_L2 && path != S2_PATH_SMEM) return S2_ERR_INVALID_ARG;
    s2_status st = check_encode(grad, dt, W, n, p, bitmaps, sketches);
    if (st != S2_OK) return st;
    if (path == S2_PATH_SMEM && (uint64_t)p.d * p.w * 4 > S2_SMEM_SKETCH_MAX_BYTES) return S2_ERR_UNSUPPORTED;
    if (W == 0) return S2_OK;
    return encode_impl(grad, dt, W, n, p, bitmaps, sketches, reinterpret_cast<cudaStream_t>(stream), 0, path);
}

s2_status s2_encode_batched_blocks(const void* grad, s2_dtype dt, uint32_t W, uint64_t n, uint32_t block,
                                   s2_params p, uint32_t* block_bitmaps, float* sketches, s2_stream_t stream) {
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (dt != S2_F32 && dt != S2_BF16) return S2_ERR_INVALID_ARG;
    if (block == 0 || block % 32 != 0) return S2_ERR_UNSUPPORTED;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    if (W == 0) return S2_OK;
    const uint64_t esz = dt == S2_F32 ? 4 : 2;
    const uint64_t nbw = words_of((n + block - 1) / block);
    const uint64_t gbytes = (uint64_t)W * n * esz, bbytes = (uint64_t)W * nbw * 4,
                   sbytes = (uint64_t)W * p.d * p.w * 4;
    if (!sketches || (n > 0 && (!grad || !block_bitmaps))) return S2_ERR_INVALID_ARG;
    if (!aligned(grad, 16) || !aligned(block_bitmaps, 16) || !aligned(sketches, 16)) return S2_ERR_ALIGNMENT;
    if (overlap(grad, gbytes, block_bitmaps, bbytes) || overlap(grad, gbytes, sketches, sbytes) ||
        overlap(block_bitmaps, bbytes, sketches, sbytes))
        return S2_ERR_INVALID_ARG;
    return encode_impl(grad, dt, W, n, p, block_bitmaps, sketches, reinterpret_cast<cudaStream_t>(stream), block);
}

s2_status s2_decode_dense_blocks(const uint32_t* block_bitmap, const float* sketch, uint64_t n, uint32_t block,
                                 s2_params p, float scale, float* out, s2_stream_t stream) {
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (block == 0 || block % 32 != 0 || n > kMaxN) return S2_ERR_UNSUPPORTED;
    if (n == 0) return S2_OK;
    if (!block_bitmap || !sketch || !out) return S2_ERR_INVALID_ARG;
    if (!aligned(block_bitmap, 16) || !aligned(sketch, 16) || !aligned(out, 16)) return S2_ERR_ALIGNMENT;
    const uint64_t dw = (uint64_t)p.d * p.w, nbw = words_of((n + block - 1) / block);
    if (overlap(out, n * 4, block_bitmap, nbw * 4) || overlap(out, n * 4, sketch, dw * 4)) return S2_ERR_INVALID_ARG;
    DecodeArgs a = make_decode_args(block_bitmap, sketch, n, p, scale);
    a.nw = nbw;
    a.block = block;
    return cuda_status(launch_decode_dense(a, out, reinterpret_cast<cudaStream_t>(stream)));
}

s2_status s2_block_topk_workspace_size(uint32_t W, uint64_t n, uint32_t block, size_t* bytes) {
    if (!bytes) return S2_ERR_INVALID_ARG;
    if (block == 0 || block % 32 != 0 || n > kMaxN) return S2_ERR_UNSUPPORTED;
    *bytes = topk_workspace_bytes(W, n, block);
    return S2_OK;
}

s2_status s2_block_topk(const float* grad, float* residual, uint32_t W, uint64_t n, uint32_t block, uint64_t K,
                        float* sparse_out, void* workspace, size_t workspace_bytes, s2_stream_t stream) {
    if (block == 0 || block % 32 != 0 || n > kMaxN) return S2_ERR_UNSUPPORTED;
    const uint64_t nb = (n + block - 1) / block, bytes = (uint64_t)W * n * 4;
    if (K > nb) return S2_ERR_INVALID_ARG;
    if (bytes == 0) return S2_OK;
    const size_t need = topk_workspace_bytes(W, n, block);
    if (!grad || !residual || !sparse_out || !workspace || workspace_bytes < need) return S2_ERR_INVALID_ARG;
    if (!aligned(grad, 16) || !aligned(residual, 16) || !aligned(sparse_out, 16) || !aligned(workspace, 16))
        return S2_ERR_ALIGNMENT;
    if (overlap(grad, bytes, residual, bytes) || overlap(grad, bytes, sparse_out, bytes) ||
        overlap(residual, bytes, sparse_out, bytes) || overlap(workspace, need, grad, bytes) ||
        overlap(workspace, need, residual, bytes) || overlap(workspace, need, sparse_out, bytes))
        return S2_ERR_INVALID_ARG;
    return cuda_status(
        launch_block_topk(grad, residual, W, n, block, K, sparse_out, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

s2_status s2_sparse_pack_workspace_size(uint32_t W, uint64_t n, size_t* bytes) {
    if (!bytes) return S2_ERR_INVALID_ARG;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    *bytes = pack_workspace_bytes(W, n);
    return S2_OK;
}

s2_status s2_sparse_pack(const float* grad, uint32_t W, uint64_t n, uint32_t* idx_out, float* val_out,
                         uint64_t capacity, uint64_t* counts_out, void* workspace, size_t workspace_bytes,
                         s2_stream_t stream) {
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    if (W == 0) return S2_OK;
    const size_t need = pack_workspace_bytes(W, n);
    const uint64_t gbytes = (uint64_t)W * n * 4, lbytes = (uint64_t)W * capacity * 4;
    if (!counts_out || (n > 0 && (!grad || !workspace || workspace_bytes < need)) ||
        (capacity > 0 && (!idx_out || !val_out)))
        return S2_ERR_INVALID_ARG;
    if (!aligned(grad, 16) || !aligned(idx_out, 4) || !aligned(val_out, 4) || !aligned(counts_out, 8) ||
        !aligned(workspace, 16))
        return S2_ERR_ALIGNMENT;
    const void* outs[4] = {idx_out, val_out, counts_out, workspace};
    const uint64_t osz[4] = {lbytes, lbytes, (uint64_t)W * 8, need};
    for (int o = 0; o < 4; ++o) {
        if (overlap(grad, gbytes, outs[o], osz[o])) return S2_ERR_INVALID_ARG;
        for (int q = o + 1; q < 4; ++q)
            if (overlap(outs[o], osz[o], outs[q], osz[q])) return S2_ERR_INVALID_ARG;
    }
    return cuda_status(launch_sparse_pack(grad, W, n, idx_out, val_out, capacity,
                                          reinterpret_cast<unsigned long long*>(counts_out), workspace,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

s2_status s2_sparse_sum(const uint32_t* idx, const float* val, const uint64_t* counts, uint32_t W, uint64_t capacity,
                        uint64_t n, float* out, s2_stream_t stream) {
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    if (n == 0) return S2_OK;
    const uint64_t lbytes = (uint64_t)W * capacity * 4;
    if (!out || (W > 0 && (!counts || (capacity > 0 && (!idx || !val))))) return S2_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(idx, 4) || !aligned(val, 4) || !aligned(counts, 8)) return S2_ERR_ALIGNMENT;
    if (overlap(out, n * 4, idx, lbytes) || overlap(out, n * 4, val, lbytes) || overlap(out, n * 4, counts, W * 8ull))
        return S2_ERR_INVALID_ARG;
    return cuda_status(launch_sparse_sum(idx, val, reinterpret_cast<const unsigned long long*>(counts), W, capacity, n,
                                         out, reinterpret_cast<cudaStream_t>(stream)));
}

s2_status s2_reduce(const uint32_t* bitmaps, const float* sketches, uint32_t W, uint64_t n, s2_params p,
                    uint32_t* bitmap_out, float* sketch_out, s2_stream_t stream) {
    s2_status st = check_reduce(bitmaps, sketches, W, n, p, bitmap_out, sketch_out);
    if (st != S2_OK) return st;
    const uint64_t nw = words_of(n), dw = (uint64_t)p.d * p.w;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (W == 0) {
        cudaError_t e = launch_zero(sketch_out, dw, s);
        if (e == cudaSuccess && nw) e = launch_zero(reinterpret_cast<float*>(bitmap_out), nw, s);
        return cuda_status(e);
    }
    return cuda_status(launch_reduce(bitmaps, sketches, W, nw, dw, bitmap_out, sketch_out, s));
}

s2_status s2_encode_reduce_fused(const void* grad, s2_dtype dt, uint32_t W, uint64_t n, s2_params p,
                                 uint32_t* bitmap_out, float* sketch_out, s2_stream_t stream) {
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (dt != S2_F32 && dt != S2_BF16) return S2_ERR_INVALID_ARG;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    const uint64_t esz = dt == S2_F32 ? 4 : 2, nw = words_of(n), dw = (uint64_t)p.d * p.w;
    const uint64_t gbytes = (uint64_t)W * n * esz;
    if (!sketch_out || (nw > 0 && !bitmap_out) || (gbytes > 0 && !grad)) return S2_ERR_INVALID_ARG;
    if (!aligned(grad, 16) || !aligned(bitmap_out, 16) || !aligned(sketch_out, 16)) return S2_ERR_ALIGNMENT;
    if (overlap(grad, gbytes, bitmap_out, nw * 4) || overlap(grad, gbytes, sketch_out, dw * 4) ||
        overlap(bitmap_out, nw * 4, sketch_out, dw * 4))
        return S2_ERR_INVALID_ARG;
    FusedArgs a;
    std::memset(&a, 0, sizeof(a));
    a.grad = grad;
    a.bitmap = bitmap_out;
    a.sketch = sketch_out;
    a.n = n;
    a.nw = nw;
    a.workers = W;
    a.d = p.d;
    a.w = p.w;
    a.keys = make_keys(p.seed, p.d);
    return cuda_status(launch_fused(a, dt == S2_F32 ? 0 : 1, reinterpret_cast<cudaStream_t>(stream)));
}

s2_status s2_decode_dense(const uint32_t* bitmap, const float* sketch, uint64_t n, s2_params p, float scale,
                          float* out, s2_stream_t stream) {
    s2_status st = check_decode_dense(bitmap, sketch, n, p, out);
    if (st != S2_OK || n == 0) return st;
    return cuda_status(
        launch_decode_dense(make_decode_args(bitmap, sketch, n, p, scale), out, reinterpret_cast<cudaStream_t>(stream)));
}

s2_status s2_decode_dense_workspace_size(uint64_t n, s2_params p, size_t* bytes) {
    if (!bytes) return S2_ERR_INVALID_ARG;
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    *bytes = dense_workspace_bytes(n, p.d);
    return S2_OK;
}

s2_status s2_decode_dense_ws(const uint32_t* bitmap, const float* sketch, uint64_t n, s2_params p, float scale,
                             float* out, void* workspace, size_t workspace_bytes, s2_stream_t stream) {
    s2_status st = check_decode_dense(bitmap, sketch, n, p, out);
    if (st != S2_OK || n == 0) return st;
    const size_t need = dense_workspace_bytes(n, p.d);
    if (workspace_bytes < need || (need > 0 && !workspace)) return S2_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return S2_ERR_ALIGNMENT;
    const uint64_t dw = (uint64_t)p.d * p.w;
    if (overlap(workspace, need, out, n * 4) || overlap(workspace, need, bitmap, words_of(n) * 4) ||
        overlap(workspace, need, sketch, dw * 4))
        return S2_ERR_INVALID_ARG;
    return cuda_status(launch_decode_dense_ws(make_decode_args(bitmap, sketch, n, p, scale), out,
                                              static_cast<float*>(workspace), reinterpret_cast<cudaStream_t>(stream)));
}

s2_status s2_decode_workspace_size(uint64_t n, size_t* bytes) {
    if (!bytes) return S2_ERR_INVALID_ARG;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    *bytes = compact_workspace_bytes(n);
    return S2_OK;
}

}  // extern "C"

namespace {
// Argument checks shared by both compacted decodes (everything but the workspace).
s2_status check_decode_compact(const uint32_t* bitmap, const float* sketch, uint64_t n, s2_params p,
                               const uint32_t* idx_out, const float* val_out, uint64_t capacity,
                               const uint64_t* count_out, const void* workspace, size_t ws_bytes) {
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    if (!count_out) return S2_ERR_INVALID_ARG;
    if (n > 0 && (!bitmap || !sketch)) return S2_ERR_INVALID_ARG;
    if (capacity > 0 && (!idx_out || !val_out)) return S2_ERR_INVALID_ARG;
    if (!aligned(bitmap, 16) || !aligned(sketch, 16) || !aligned(workspace, 16) || !aligned(idx_out, 4) ||
        !aligned(val_out, 4) || !aligned(count_out, 8))
        return S2_ERR_ALIGNMENT;
    const uint64_t nw = words_of(n), dw = (uint64_t)p.d * p.w, cap = capacity < n ? capacity : n;
    const void* ins[2] = {bitmap, sketch};
    const uint64_t insz[2] = {nw * 4, dw * 4};
    const void* outs[4] = {idx_out, val_out, count_out, workspace};
    const uint64_t outsz[4] = {cap * 4, cap * 4, 8, ws_bytes};
    for (int i = 0; i < 2; ++i)
        for (int o = 0; o < 4; ++o)
            if (overlap(ins[i], insz[i], outs[o], outsz[o])) return S2_ERR_INVALID_ARG;
    for (int o = 0; o < 4; ++o)
        for (int q = o + 1; q < 4; ++q)
            if (overlap(outs[o], outsz[o], outs[q], outsz[q])) return S2_ERR_INVALID_ARG;
    return S2_OK;
}
}  // namespace

extern "C" {

s2_status s2_decode_compact(const uint32_t* bitmap, const float* sketch, uint64_t n, s2_params p, float scale,
                            uint32_t* idx_out, float* val_out, uint64_t capacity, uint64_t* count_out,
                            void* workspace, size_t workspace_bytes, s2_stream_t stream) {
    if (n <= kMaxN) {
        const size_t need = compact_workspace_bytes(n);
        if (workspace_bytes < need || (need > 0 && !workspace)) {
            s2_status st = check_params(p);
            return st != S2_OK ? st : S2_ERR_INVALID_ARG;
        }
    }
    s2_status st = check_decode_compact(bitmap, sketch, n, p, idx_out, val_out, capacity, count_out, workspace,
                                        n <= kMaxN ? compact_workspace_bytes(n) : 0);
    if (st != S2_OK) return st;
    const uint64_t tiles = compact_tiles(words_of(n));
    uint32_t* counts = static_cast<uint32_t*>(workspace);
    uint32_t* offsets = counts + (round256(tiles * 4) / 4);
    return cuda_status(launch_decode_compact(make_decode_args(bitmap, sketch, n, p, scale), idx_out, val_out, capacity,
                                             reinterpret_cast<unsigned long long*>(count_out), counts, offsets,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

s2_status s2_decode_compact_noalloc(const uint32_t* bitmap, const float* sketch, uint64_t n, s2_params p, float scale,
                                    uint32_t* idx_out, float* val_out, uint64_t capacity, uint64_t* count_out,
                                    s2_stream_t stream) {
    s2_status st = check_decode_compact(bitmap, sketch, n, p, idx_out, val_out, capacity, count_out, nullptr, 0);
    if (st != S2_OK) return st;
    if (n > noalloc_compact_max_n()) return S2_ERR_UNSUPPORTED;
    uint32_t* counts = nullptr;
    uint32_t* offsets = nullptr;
    if (noalloc_compact_scratch(&counts, &offsets) != cudaSuccess) return S2_ERR_CUDA;
    return cuda_status(launch_decode_compact(make_decode_args(bitmap, sketch, n, p, scale), idx_out, val_out, capacity,
                                             reinterpret_cast<unsigned long long*>(count_out), counts, offsets,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

s2_status s2_hash(const uint32_t* idx, uint64_t m, s2_params p, uint32_t* bucket_out, int8_t* sign_out,
                  s2_stream_t stream) {
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (m == 0) return S2_OK;
    if (!idx || !bucket_out || !sign_out) return S2_ERR_INVALID_ARG;
    if (!aligned(idx, 4) || !aligned(bucket_out, 4)) return S2_ERR_ALIGNMENT;
    if (overlap(idx, m * 4, bucket_out, m * p.d * 4) || overlap(idx, m * 4, sign_out, m * p.d) ||
        overlap(bucket_out, m * p.d * 4, sign_out, m * p.d))
        return S2_ERR_INVALID_ARG;
    return cuda_status(
        launch_hash(idx, m, p.d, p.w, make_keys(p.seed, p.d), bucket_out, sign_out, reinterpret_cast<cudaStream_t>(stream)));
}

s2_status s2_pipeline_workspace_size(s2_dtype dt, uint32_t W, uint64_t n, s2_params p, size_t* bytes) {
    if (!bytes) return S2_ERR_INVALID_ARG;
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (dt != S2_F32 && dt != S2_BF16) return S2_ERR_INVALID_ARG;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    *bytes = pipeline_layout(dt, W, n, p).total;
    return S2_OK;
}

s2_status s2_pipeline_dense_host(const void* host_grad, s2_dtype dt, uint32_t W, uint64_t n, s2_params p,
                                 float scale, float* host_out, void* workspace, size_t workspace_bytes,
                                 s2_stream_t stream) {
    s2_status st = check_params(p);
    if (st != S2_OK) return st;
    if (dt != S2_F32 && dt != S2_BF16) return S2_ERR_INVALID_ARG;
    if (n > kMaxN) return S2_ERR_UNSUPPORTED;
    const PipelineLayout L = pipeline_layout(dt, W, n, p);
    if (!workspace || workspace_bytes < L.total) return S2_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return S2_ERR_ALIGNMENT;
    if (n > 0 && (!host_out || (W > 0 && !host_grad))) return S2_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    const uint64_t esz = dt == S2_F32 ? 4 : 2;
    void* d_grad = ws + L.grad;
    uint32_t* d_bitmaps = reinterpret_cast<uint32_t*>(ws + L.bitmaps);
    float* d_sketches = reinterpret_cast<float*>(ws + L.sketches);
    uint32_t* d_bitmap = reinterpret_cast<uint32_t*>(ws + L.bitmap);
    float* d_sketch = reinterpret_cast<float*>(ws + L.sketch);
    float* d_out = reinterpret_cast<float*>(ws + L.out);
    // Page-locked host buffers mapped into the device's address space are
    // read and written in place by the kernels (over NVLink-C2C on a
    // Grace-Blackwell node): the encode streams the gradient from host
    // memory once and the decode stores the output there, so no staging
    // copy precedes or follows them. Other host memory is staged through
    // the workspace with copies. A sketch built in several passes (larger
    // than 3/4 of L2) would re-read the gradient per pass: staged too.
    const void* enc_src = d_grad;
    if ((uint64_t)W * n > 0) {
        DeviceInfo di{};
        if (device_info(&di) != cudaSuccess) return S2_ERR_CUDA;
        const bool one_pass = (uint64_t)p.d * p.w * 4 <= (uint64_t)di.l2_bytes / 4 * 3;
        const void* mapped = one_pass ? mapped_host(host_grad) : nullptr;
        if (mapped) {
            enc_src = mapped;
        } else if (cudaMemcpyAsync(d_grad, host_grad, (size_t)W * n * esz, cudaMemcpyHostToDevice, s) !=
                   cudaSuccess) {
            return S2_ERR_CUDA;
        }
        st = encode_impl(enc_src, dt, W, n, p, d_bitmaps, d_sketches, s);
        if (st != S2_OK) return st;
    }
    st = s2_reduce(d_bitmaps, d_sketches, W, n, p, d_bitmap, d_sketch, stream);
    if (st != S2_OK) return st;
    if (n == 0) return S2_OK;
    float* out_mapped = static_cast<float*>(const_cast<void*>(mapped_host(host_out)));
    st = s2_decode_dense_ws(d_bitmap, d_sketch, n, p, scale, out_mapped ? out_mapped : d_out, ws + L.dec_ws,
                            dense_workspace_bytes(n, p.d), stream);
    if (st != S2_OK) return st;
    if (!out_mapped &&
        cudaMemcpyAsync(host_out, d_out, (size_t)n * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return S2_ERR_CUDA;
    return S2_OK;
}

const char* s2_status_string(s2_status st) {
    switch (st) {
        case S2_OK: return "S2_OK";
        case S2_ERR_INVALID_ARG: return "S2_ERR_INVALID_ARG";
        case S2_ERR_ALIGNMENT: return "S2_ERR_ALIGNMENT";
        case S2_ERR_UNSUPPORTED: return "S2_ERR_UNSUPPORTED";
        case S2_ERR_CUDA: return "S2_ERR_CUDA";
    }
    return "S2_UNKNOWN_STATUS";
}

const char* s2_version(void) { return "libs2 0.1 (sm_103a)"; }

}  // extern "C"
