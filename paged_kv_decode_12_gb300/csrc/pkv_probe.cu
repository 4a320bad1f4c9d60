// pkv_probe.cu -- HBM read-bandwidth probes (measurement aid; see include/pkv_probe.h).
//
// The decode path only reads the KV pool, so its ceiling is a read-only stream, not
// a copy.  Two probes read a buffer once each: plain 16-byte vector loads, and 1-D
// TMA bulk copies into a shared-memory ring (the copy engine of the decode kernels).
#include "../../include/pkv_probe.h"
#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int kLdgThreads = 512;
constexpr int kBulkChunk = 32768;
constexpr int kBulkStages = 3;  // 96 KiB of ring: two CTAs fit on an SM

__global__ void __launch_bounds__(kLdgThreads) probe_ldg_kernel(const uint4 *__restrict__ buf, size_t n,
                                                                uint32_t *__restrict__ sink)
{
    const size_t stride = (size_t)gridDim.x * kLdgThreads;
    size_t i = (size_t)blockIdx.x * kLdgThreads + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * stride < n; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                         : "l"(buf + i + u * stride));
#pragma unroll
        for (int u = 0; u < 4; ++u)
            acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n; i += stride) {
        const uint4 v = buf[i];
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    acc = __reduce_xor_sync(kFull, acc);
    if ((threadIdx.x & 31) == 0)
        atomicXor(&sink[blockIdx.x], acc);
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// One thread per CTA streams chunks c = blockIdx.x, blockIdx.x + gridDim.x, ... through
// the ring; the other threads fold each landed chunk's first word into the sink.
__global__ void __launch_bounds__(32) probe_bulk_kernel(const uint8_t *__restrict__ buf, size_t nchunks,
                                                        uint32_t *__restrict__ sink)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + kBulkStages * kBulkChunk);
    const int lane = threadIdx.x;
    if (lane == 0) {
        for (int s = 0; s < kBulkStages; ++s)
            mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    const size_t first = blockIdx.x, step = gridDim.x;
    const size_t mine = first < nchunks ? (nchunks - first + step - 1) / step : 0;
    if (lane == 0)
        for (size_t k = 0; k < kBulkStages && k < mine; ++k) {
            mbar_arrive_expect_tx(&bars[k], kBulkChunk);
            bulk_g2s(ring + k * kBulkChunk, buf + (first + k * step) * kBulkChunk, kBulkChunk, &bars[k]);
        }
    uint32_t acc = 0;
    size_t k = 0;
    for (; k < mine; ++k) {
        const int s = (int)(k % kBulkStages);
        if (!mbar_wait_warp(&bars[s], (uint32_t)((k / kBulkStages) & 1)))
            break;
        acc ^= reinterpret_cast<const uint32_t *>(ring + s * kBulkChunk)[lane];
        __syncwarp();
        if (lane == 0 && k + kBulkStages < mine) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars[s], kBulkChunk);
            bulk_g2s(ring + s * kBulkChunk, buf + (first + (k + kBulkStages) * step) * kBulkChunk, kBulkChunk,
                     &bars[s]);
        }
    }
    if (k < mine) {  // gave up: let the copies in flight land (bounded), count it
        for (size_t kk = k; kk < mine && kk < k + kBulkStages; ++kk)
            (void)mbar_wait_warp(&bars[kk % kBulkStages], (uint32_t)((kk / kBulkStages) & 1));
        if (lane == 0)
            atomicAdd(&sink[gridDim.x], 1u);
    }
    acc = __reduce_xor_sync(kFull, acc);
    if (lane == 0)
        atomicXor(&sink[blockIdx.x], acc);
}

int sm_count(int &sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_probe_read_ldg(const void *buf, size_t bytes, uint32_t *sink, int ctas_per_sm, void *cuda_stream)
{
    using namespace pkv;
    if (!buf || !sink || bytes < 16 || (bytes & 15u) || (reinterpret_cast<uintptr_t>(buf) & 15u) ||
        ctas_per_sm < 1 || ctas_per_sm > 4)
        return PKV_ERR_INVALID_ARG;
    int sms = 0;
    if (sm_count(sms) != PKV_OK)
        return PKV_ERR_CUDA;
    probe_ldg_kernel<<<sms * ctas_per_sm, kLdgThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        static_cast<const uint4 *>(buf), bytes / 16, sink);
    return status_from_cuda(cudaGetLastError());
}

extern "C" int pkv_probe_read_bulk(const void *buf, size_t bytes, uint32_t *sink, int ctas_per_sm,
                                   void *cuda_stream)
{
    using namespace pkv;
    if (!buf || !sink || bytes < (size_t)kBulkChunk || (bytes % kBulkChunk) ||
        (reinterpret_cast<uintptr_t>(buf) & 15u) || ctas_per_sm < 1 || ctas_per_sm > 2)
        return PKV_ERR_INVALID_ARG;
    int sms = 0;
    if (sm_count(sms) != PKV_OK)
        return PKV_ERR_CUDA;
    constexpr int smem = 128 + kBulkStages * kBulkChunk + kBulkStages * 8;
    static PerDeviceOnce attr;
    if (const int st = ensure_smem_attr(attr, probe_bulk_kernel, smem); st != PKV_OK)
        return st;
    probe_bulk_kernel<<<sms * ctas_per_sm, 32, smem, static_cast<cudaStream_t>(cuda_stream)>>>(
        static_cast<const uint8_t *>(buf), bytes / kBulkChunk, sink);
    return status_from_cuda(cudaGetLastError());
}
