// pkv_append.cu -- fused RoPE + page-slot append of one decode token per sequence.
//
// samir-vllm README summary ("从零用 C++ 和 CUDA 实现 Llama 3.2 1B 推理引擎"),
// section "目前已完成的功能": decode appends one new token at its absolute RoPE
// position into the sequence's page of the shared BF16 pool.  Rotary embedding
// ("从零构建大模型推理引擎" section 4.1) is read as rotate-half: dimension i turns
// with dimension i + 32 by the angle pos * theta^(-2i/64); the FP32 factors come
// from a table built once on the host in FP64.
//
// One CTA per sequence.  The work is 8 key rows (+ 32 query rows when q is
// given) of 32 rotation pairs, and the 8 value rows copied unchanged.  A thread
// rotates two adjacent pairs (i, i+1) with 4-byte loads/stores of both halves;
// 64 threads copy the 1 KiB of values with 16-byte moves.  The bytes are tiny
// (about 2 KiB written per sequence); the kernel is latency-bound, so it is launched
// with programmatic dependent launch: its CTAs are scheduled while the previous kernel
// finishes, wait for it (griddepcontrol.wait) before reading or writing anything, and
// then let the next launch (the layer's attention) begin its early work.
#include <cuda_bf16.h>

#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
append_rope_kernel(uint16_t *__restrict__ slab, int num_pages, const uint16_t *__restrict__ k_new,
                   const uint16_t *__restrict__ v_new, uint16_t *__restrict__ q, const int32_t *__restrict__ bt,
                   int max_blocks, const int32_t *__restrict__ pos, const float4 *__restrict__ rope, int max_pos,
                   int32_t *__restrict__ err)
{
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    const int b = blockIdx.x;
    const int p = pos[b];
    const int limit = min(max_pos, max_blocks * kPage);
    if (p < 0 || p >= limit) {
        if (threadIdx.x == 0 && err)
            atomicOr(err, PKV_DEVERR_LENGTH);
        return;
    }
    const int page = bt[(size_t)b * max_blocks + p / kPage];
    if (page < 0 || page >= num_pages) {
        if (threadIdx.x == 0 && err)
            atomicOr(err, PKV_DEVERR_PAGE_RANGE);
        return;
    }
    const int slot = p % kPage;
    uint16_t *page_base = slab + (size_t)page * kPageElems;

    // values: 8 heads x 64 dims x 2 B = 64 chunks of 16 B
    if (threadIdx.x < kHkv * kD * 2 / 16) {
        const int h = threadIdx.x / 8, c = threadIdx.x % 8;
        const uint4 v = reinterpret_cast<const uint4 *>(v_new + ((size_t)b * kHkv + h) * kD)[c];
        reinterpret_cast<uint4 *>(page_base + ((size_t)(kHkv + h) * kPage + slot) * kD)[c] = v;
    }

    // rotations: rows 0..7 are keys, rows 8..39 queries (if given); 16 threads per row
    const float4 *rope_row = rope + (size_t)p * (kD / 2);  // [32 pairs] x {cos, sin hi; cos, sin lo}
    const int rows = kHkv + (q ? kHq : 0);
    for (int item = threadIdx.x; item < rows * 16; item += kAppendThreads) {
        const int r = item / 16, j = item % 16;  // pairs 2j and 2j+1
        const float4 cs0 = rope_row[2 * j], cs1 = rope_row[2 * j + 1];
        const uint16_t *src;
        uint16_t *dst;
        if (r < kHkv) {
            src = k_new + ((size_t)b * kHkv + r) * kD;
            dst = page_base + ((size_t)r * kPage + slot) * kD;
        } else {
            src = dst = q + ((size_t)b * kHq + (r - kHkv)) * kD;
        }
        const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(src + 2 * j);
        const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(src + kD / 2 + 2 * j);
        const float2 x1 = __bfloat1622float2(lo);   // dims 2j, 2j+1
        const float2 x2 = __bfloat1622float2(hi);   // dims 2j+32, 2j+33
        float2 y1, y2;
        dev::rope_rotate_pair(x1.x, x2.x, cs0, y1.x, y2.x);
        dev::rope_rotate_pair(x1.y, x2.y, cs1, y1.y, y2.y);
        *reinterpret_cast<__nv_bfloat162 *>(dst + 2 * j) = __float22bfloat162_rn(y1);
        *reinterpret_cast<__nv_bfloat162 *>(dst + kD / 2 + 2 * j) = __float22bfloat162_rn(y2);
    }
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_append_rope(const pkv_pool *pool, const uint16_t *k_new, const uint16_t *v_new, uint16_t *q,
                               const int32_t *bt_dev, int max_blocks, const int32_t *pos_dev, int B,
                               const float *rope_table, int max_pos, int32_t *dev_err_flag, void *cuda_stream)
{
    using namespace pkv;
    if (!pool || !k_new || !v_new || !bt_dev || !pos_dev || !rope_table)
        return PKV_ERR_INVALID_ARG;
    if (B < 1 || B > INT32_MAX / 2 || max_blocks < 1 || max_pos < 1)
        return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
         reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(rope_table)) & 15u)
        return PKV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (pool->kv_format == PKV_KV_FP8)
        return fp8_append_rope(pool, k_new, v_new, q, bt_dev, max_blocks, pos_dev, B, rope_table, max_pos,
                               dev_err_flag, s);
    return launch_kernel(append_rope_kernel, dim3(B), dim3(kAppendThreads), 0, s, true,
                         reinterpret_cast<uint16_t *>(pool->slab), pool->num_pages, k_new, v_new, q, bt_dev,
                         max_blocks, pos_dev, reinterpret_cast<const float4 *>(rope_table), max_pos, dev_err_flag);
}

// ---------------------------------------------------------------------------
// Prefill page fill: T consecutive tokens of one sequence, every layer.  Same
// rotation and placement as the decode append (one CTA per (token, layer)).
namespace pkv {
namespace {

constexpr int kPrefillThreads = 128;

__global__ void __launch_bounds__(kPrefillThreads)
prefill_append_kernel(uint16_t *__restrict__ slab, int num_pages, const uint16_t *__restrict__ k,
                      const uint16_t *__restrict__ v, const int32_t *__restrict__ bt_rows, int max_blocks, int start_pos,
                      int T, const float4 *__restrict__ rope, int max_pos, int32_t *__restrict__ err)
{
    const int t = blockIdx.x, l = blockIdx.y;
    const int p = start_pos + t;
    if (p < 0 || p >= min(max_pos, max_blocks * kPage)) {
        if (threadIdx.x == 0 && err)
            atomicOr(err, PKV_DEVERR_LENGTH);
        return;
    }
    const int page = bt_rows[(size_t)l * max_blocks + p / kPage];
    if (page < 0 || page >= num_pages) {
        if (threadIdx.x == 0 && err)
            atomicOr(err, PKV_DEVERR_PAGE_RANGE);
        return;
    }
    const int slot = p % kPage;
    uint16_t *page_base = slab + (size_t)page * kPageElems;
    const size_t row0 = ((size_t)l * T + t) * kHkv * kD;  // token t of layer l: [8][64]
    if (threadIdx.x < kHkv * kD * 2 / 16) {                // values: 64 chunks of 16 B
        const int h = threadIdx.x / 8, c = threadIdx.x % 8;
        const uint4 val = reinterpret_cast<const uint4 *>(v + row0 + (size_t)h * kD)[c];
        reinterpret_cast<uint4 *>(page_base + ((size_t)(kHkv + h) * kPage + slot) * kD)[c] = val;
    }
    for (int item = threadIdx.x; item < kHkv * (kD / 2); item += kPrefillThreads) {
        const int h = item / (kD / 2), i = item % (kD / 2);
        const float4 cs = rope[(size_t)p * (kD / 2) + i];
        const uint16_t *src = k + row0 + (size_t)h * kD;
        const float x1 = __uint_as_float((uint32_t)src[i] << 16);
        const float x2 = __uint_as_float((uint32_t)src[i + kD / 2] << 16);
        float y1, y2;
        dev::rope_rotate_pair(x1, x2, cs, y1, y2);
        const __nv_bfloat16 b1 = __float2bfloat16_rn(y1), b2 = __float2bfloat16_rn(y2);
        uint16_t *dst = page_base + ((size_t)h * kPage + slot) * kD;
        dst[i] = *reinterpret_cast<const uint16_t *>(&b1);
        dst[i + kD / 2] = *reinterpret_cast<const uint16_t *>(&b2);
    }
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_prefill_append(const pkv_pool *pool, const uint16_t *k, const uint16_t *v, const int32_t *bt_rows,
                                  int max_blocks, int layers, int start_pos, int T, const float *rope_table,
                                  int max_pos, int32_t *dev_err_flag, void *cuda_stream)
{
    using namespace pkv;
    if (!pool || !k || !v || !bt_rows || !rope_table)
        return PKV_ERR_INVALID_ARG;
    if (T < 1 || T > INT32_MAX / 2 || layers < 1 || layers > 65535 || max_blocks < 1 || max_pos < 1 || start_pos < 0)
        return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(rope_table)) &
        15u)
        return PKV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    pool->serialize_next_launch = true;  // the next decode launch may read these pages
    if (pool->kv_format == PKV_KV_FP8)
        return fp8_prefill_append(pool, k, v, bt_rows, max_blocks, layers, start_pos, T, rope_table, max_pos,
                                  dev_err_flag, s);
    prefill_append_kernel<<<dim3(T, layers), kPrefillThreads, 0, s>>>(
        reinterpret_cast<uint16_t *>(pool->slab), pool->num_pages, k, v, bt_rows, max_blocks, start_pos, T,
        reinterpret_cast<const float4 *>(rope_table), max_pos, dev_err_flag);
    return status_from_cuda(cudaGetLastError());
}
