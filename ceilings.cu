// Device ceilings that bound the S2 Reducer kernels on this GPU, measured
// with CUDA events (built and run by `python bench.py --ceilings`).
//
//   stream_read   16-byte streaming loads over 1 GiB            (HBM read rate)
//   red_f32       random red.global.add.f32 into 32 MiB         (scattered L2 reductions)
//   gather_f32    random 4-byte loads from 32 MiB               (scattered L2 reads)
//   read_and_red  both of the above in one kernel, interleaved  (do they share a ceiling?)
//   red_v4_f32    random red.global.add.v4.f32 (4 adds per op)  (cost per op or per float?)
//   smem_atomic   random shared-memory atomicAdd over 192 KiB   (on-chip alternative)
//   concurrent    the stream and the reductions (and a zero write and the
//                 gathers) as two kernels on two streams at once, half the
//                 grid each                                      (do they overlap?)
//   host_*        page-locked host memory mapped into the device: SM reads
//                 and writes of 1 GiB in place, and copy-engine copies of
//                 1 GiB each way                                 (the host link)
//
// Every index is masked to its buffer; no kernel waits on another.
// Prints one JSON object on stdout.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint32_t mix(uint32_t x) {
    x ^= x >> 16; x *= 0x85ebca6bu; x ^= x >> 13; x *= 0xc2b2ae35u; x ^= x >> 16;
    return x;
}

__device__ __forceinline__ uint4 ld_cs(const uint4* p) {
    uint4 v;
    asm("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// do_read: stream n4 16-byte vectors; do_red: nred random reductions into sk[mask+1]
__global__ void read_red(const uint4* src, uint64_t n4, float* sk, uint32_t mask, uint64_t nred, int do_read,
                         int do_red, uint32_t* sink) {
    const uint64_t nth = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t tid = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    const uint64_t rp = do_read ? (n4 + nth - 1) / nth : 0, ap = do_red ? (nred + nth - 1) / nth : 0;
    const uint64_t it = rp > ap ? rp : ap;
    uint32_t acc = 0;
    for (uint64_t k = 0; k < it; ++k) {
        const uint64_t x = tid + k * nth;
        if (k < rp && x < n4) {
            const uint4 v = ld_cs(src + x);
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
        if (k < ap && x < nred)
            asm volatile("red.global.add.f32 [%0], %1;" ::"l"(sk + (mix((uint32_t)x * 2654435761u) & mask)), "f"(1.0f)
                         : "memory");
    }
    if (acc == 0x9abcdef1u) sink[0] = acc;
}

__global__ void gather(const float* sk, uint32_t mask, uint64_t ngat, float* sink) {
    const uint64_t nth = (uint64_t)gridDim.x * blockDim.x;
    float acc = 0.f;
    for (uint64_t x = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; x < ngat; x += 4 * nth) {
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = __ldg(sk + (mix((uint32_t)(x + q * nth) * 2654435761u) & mask));
        acc += v[0] + v[1] + v[2] + v[3];
    }
    if (acc == 1234.5f) sink[0] = acc;
}

__global__ void red_v4(float* sk, uint32_t mask4, uint64_t nops) {
    const uint64_t nth = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t x = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; x < nops; x += nth) {
        float* p = sk + 4 * (mix((uint32_t)x * 2654435761u) & mask4);
        asm volatile("red.global.add.v4.f32 [%0], {%1,%1,%1,%1};" ::"l"(p), "f"(1.0f) : "memory");
    }
}

// Zero 16-byte vectors with evict-first stores.
__global__ void write_zero(uint4* dst, uint64_t n4) {
    const uint64_t nth = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t x = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; x < n4; x += nth)
        asm volatile("st.global.cs.v4.u32 [%0], {%1,%1,%1,%1};" ::"l"(dst + x), "r"(0u) : "memory");
}

constexpr uint32_t kSmemFloats = 48 * 1024;

__global__ void smem_atomic(uint64_t per_thread, float* sink) {
    extern __shared__ float s[];
    for (uint32_t x = threadIdx.x; x < kSmemFloats; x += blockDim.x) s[x] = 0.f;
    __syncthreads();
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    for (uint64_t k = 0; k < per_thread; ++k) atomicAdd(&s[mix(tid * 7919u + (uint32_t)k * 104729u) % kSmemFloats], 1.f);
    __syncthreads();
    if (threadIdx.x == 0 && s[7] < 0.f) sink[0] = s[7];
}

struct Timer {
    cudaEvent_t a, b;
    Timer() { cudaEventCreate(&a); cudaEventCreate(&b); }
    void start() { cudaEventRecord(a); }
    float stop() {
        cudaEventRecord(b);
        cudaEventSynchronize(b);
        float ms = 0.f;
        cudaEventElapsedTime(&ms, a, b);
        return ms;
    }
};

}  // namespace

int main() {
    int sms = 0, l2 = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, 0);
    const uint64_t src_bytes = 1ull << 30, sk_bytes = 32ull << 20;
    uint4* src = nullptr;
    float* sk = nullptr;
    float* fsink = nullptr;
    uint32_t* usink = nullptr;
    if (cudaMalloc(&src, src_bytes) != cudaSuccess || cudaMalloc(&sk, sk_bytes) != cudaSuccess ||
        cudaMalloc(&fsink, 4) != cudaSuccess || cudaMalloc(&usink, 4) != cudaSuccess) {
        printf("{\"error\": \"allocation failed\"}\n");
        return 1;
    }
    cudaMemset(src, 0, src_bytes);
    cudaMemset(sk, 0, sk_bytes);
    const uint64_t n4 = src_bytes / 16;
    const uint32_t mask = (uint32_t)(sk_bytes / 4) - 1;
    const uint64_t nred = 40ull << 20;
    const int grid = sms * 8, block = 256;
    Timer t;
    float ms[6] = {0};
    // warm-up of each kernel, then the timed launch
    for (int rep = 0; rep < 2; ++rep) {
        t.start(); read_red<<<grid, block>>>(src, n4, sk, mask, nred, 1, 0, usink); ms[0] = t.stop();
        t.start(); read_red<<<grid, block>>>(src, n4, sk, mask, nred, 0, 1, usink); ms[1] = t.stop();
        t.start(); gather<<<grid, block>>>(sk, mask, nred, fsink); ms[2] = t.stop();
        t.start(); read_red<<<grid, block>>>(src, n4, sk, mask, nred, 1, 1, usink); ms[3] = t.stop();
        t.start(); red_v4<<<grid, block>>>(sk, mask / 4, nred / 4); ms[4] = t.stop();
    }
    cudaFuncSetAttribute(smem_atomic, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemFloats * 4);
    const uint64_t per = 4096;
    for (int rep = 0; rep < 2; ++rep) {
        t.start();
        smem_atomic<<<sms, 1024, kSmemFloats * 4>>>(per, fsink);
        ms[5] = t.stop();
    }
    // the same work split over two streams at once, half the grid each
    cudaStream_t s1, s2;
    cudaStreamCreateWithFlags(&s1, cudaStreamNonBlocking);
    cudaStreamCreateWithFlags(&s2, cudaStreamNonBlocking);
    cudaEvent_t e1, e2;
    cudaEventCreate(&e1);
    cudaEventCreate(&e2);
    uint4* dst = nullptr;
    float cms[4] = {0};
    if (cudaMalloc(&dst, src_bytes) == cudaSuccess) {
        for (int rep = 0; rep < 2; ++rep) {
            t.start();
            cudaEventRecord(e1, 0);
            cudaStreamWaitEvent(s1, e1, 0);
            cudaStreamWaitEvent(s2, e1, 0);
            read_red<<<grid / 2, block, 0, s1>>>(src, n4, sk, mask, nred, 1, 0, usink);
            read_red<<<grid / 2, block, 0, s2>>>(src, n4, sk, mask, nred, 0, 1, usink);
            cudaEventRecord(e1, s1);
            cudaEventRecord(e2, s2);
            cudaStreamWaitEvent(0, e1, 0);
            cudaStreamWaitEvent(0, e2, 0);
            cms[0] = t.stop();
            t.start(); write_zero<<<grid, block>>>(dst, n4); cms[1] = t.stop();
            t.start();
            cudaEventRecord(e1, 0);
            cudaStreamWaitEvent(s1, e1, 0);
            cudaStreamWaitEvent(s2, e1, 0);
            write_zero<<<grid / 2, block, 0, s1>>>(dst, n4);
            gather<<<grid / 2, block, 0, s2>>>(sk, mask, nred, fsink);
            cudaEventRecord(e1, s1);
            cudaEventRecord(e2, s2);
            cudaStreamWaitEvent(0, e1, 0);
            cudaStreamWaitEvent(0, e2, 0);
            cms[2] = t.stop();
        }
        cudaFree(dst);
    }
    // the host link: mapped page-locked memory read and written by kernels in place, and copies
    void* host = nullptr;
    void* hdev = nullptr;
    float hms[4] = {0};
    if (cudaHostAlloc(&host, src_bytes, cudaHostAllocMapped) == cudaSuccess &&
        cudaHostGetDevicePointer(&hdev, host, 0) == cudaSuccess) {
        memset(host, 0, src_bytes);
        for (int rep = 0; rep < 2; ++rep) {
            t.start(); read_red<<<grid, block>>>(static_cast<const uint4*>(hdev), n4, sk, mask, nred, 1, 0, usink); hms[0] = t.stop();
            t.start(); write_zero<<<grid, block>>>(static_cast<uint4*>(hdev), n4); hms[1] = t.stop();
            t.start(); cudaMemcpyAsync(src, host, src_bytes, cudaMemcpyHostToDevice, 0); hms[2] = t.stop();
            t.start(); cudaMemcpyAsync(host, src, src_bytes, cudaMemcpyDeviceToHost, 0); hms[3] = t.stop();
        }
        cudaFreeHost(host);
    }
    const cudaError_t e = cudaDeviceSynchronize();
    const double sector = 32.0;
    printf("{\"sms\": %d, \"l2_bytes\": %d, "
           "\"stream_read\": {\"ms\": %.4f, \"GBps\": %.1f, \"Gsectors_per_s\": %.1f}, "
           "\"red_f32\": {\"ms\": %.4f, \"Gops_per_s\": %.1f}, "
           "\"gather_f32\": {\"ms\": %.4f, \"Gops_per_s\": %.1f}, "
           "\"read_and_red\": {\"ms\": %.4f, \"sum_of_alone_ms\": %.4f}, "
           "\"red_v4_f32\": {\"ms\": %.4f, \"Gops_per_s\": %.1f, \"Gadds_per_s\": %.1f}, "
           "\"smem_atomic\": {\"ms\": %.4f, \"Gops_per_s\": %.1f}, "
           "\"concurrent\": {\"read_and_red_two_streams_ms\": %.4f, \"write_ms\": %.4f, "
           "\"write_and_gather_two_streams_ms\": %.4f, \"sum_of_alone_ms\": %.4f}, "
           "\"host\": {\"sm_read_GBps\": %.1f, \"sm_write_GBps\": %.1f, \"copy_h2d_GBps\": %.1f, "
           "\"copy_d2h_GBps\": %.1f}, \"status\": \"%s\"}\n",
           sms, l2, ms[0], src_bytes / (ms[0] * 1e6), src_bytes / sector / (ms[0] * 1e6), ms[1], nred / (ms[1] * 1e6),
           ms[2], nred / (ms[2] * 1e6), ms[3], ms[0] + ms[1], ms[4], nred / 4 / (ms[4] * 1e6), nred / (ms[4] * 1e6),
           ms[5], (double)sms * 1024 * per / (ms[5] * 1e6), cms[0], cms[1], cms[2], cms[1] + ms[2],
           hms[0] > 0 ? src_bytes / (hms[0] * 1e6) : 0.0, hms[1] > 0 ? src_bytes / (hms[1] * 1e6) : 0.0,
           hms[2] > 0 ? src_bytes / (hms[2] * 1e6) : 0.0, hms[3] > 0 ? src_bytes / (hms[3] * 1e6) : 0.0,
           cudaGetErrorString(e));
    return e == cudaSuccess ? 0 : 2;
}
