// pkv_host.cpp -- host side of libpkv: page pool allocator, block-table builder,
// RoPE factor table, tensor-map encoding, status helpers.
//
// The page pool follows the samir-vllm README summary ("从零用 C++ 和 CUDA 实现
// Llama 3.2 1B 推理引擎"), section "目前已完成的功能": one shared BF16 page pool,
// 16 tokens of K and V per physical page, block tables per sequence and layer,
// and section "当前范围": physical pages are allocated lazily and returned on
// finish.  "从零构建大模型推理引擎" section 5.1 recommends one preallocated buffer
// managed by offsets; the caller allocates that slab, the library manages ids.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <new>

#include "pkv_internal.h"

namespace {

// splitmix64: a small, well-known 64-bit mixer used to seed the shuffle.
uint64_t splitmix64(uint64_t &state)
{
    uint64_t z = (state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// uniform integer in [0, n) by the multiply-shift method
uint32_t bounded(uint64_t &state, uint32_t n)
{
    return (uint32_t)(((unsigned __int128)splitmix64(state) * n) >> 64);
}

}  // namespace

extern "C" {

const char *pkv_version(void) { return "pkv 0.1 sm_103a"; }

const char *pkv_status_string(int status)
{
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_OUT_OF_PAGES: return "out of pages";
    case PKV_ERR_DOUBLE_FREE: return "page not allocated (double free)";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE_BOUNDS: return "device bounds check failed";
    case PKV_ERR_BUDGET_EXCEEDS_POOL: return "request budget exceeds the whole pool";
    case PKV_ERR_UNSUPPORTED: return "unsupported geometry";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    default: return "unknown status";
    }
}

}  // extern "C"

namespace {

int create_pool(void *dev_slab, size_t slab_bytes, int kv_format, size_t page_bytes, uint64_t seed, pkv_pool **out)
{
    if (!out)
        return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    if (!dev_slab || (reinterpret_cast<uintptr_t>(dev_slab) & 15u) != 0)
        return PKV_ERR_INVALID_ARG;
    size_t pages = slab_bytes / page_bytes;
    if (pages < 1 || pages > (size_t)INT32_MAX)
        return PKV_ERR_INVALID_ARG;
    pkv_pool *p = new (std::nothrow) pkv_pool();
    if (!p)
        return PKV_ERR_INVALID_ARG;
    p->slab = static_cast<char *>(dev_slab);
    p->slab_bytes = slab_bytes;
    p->num_pages = (int32_t)pages;
    p->kv_format = kv_format;
    p->page_bytes = page_bytes;
    try {
        p->free_list.resize(pages);
        p->allocated.assign(pages, 0);
    } catch (...) {
        delete p;
        return PKV_ERR_INVALID_ARG;
    }
    // Fisher-Yates shuffle of the ids, seeded: pages handed out are scattered
    // through the slab, reproducibly for a given seed.
    for (size_t i = 0; i < pages; ++i)
        p->free_list[i] = (int32_t)i;
    uint64_t state = seed;
    for (size_t i = pages - 1; i > 0; --i) {
        size_t j = bounded(state, (uint32_t)(i + 1));
        std::swap(p->free_list[i], p->free_list[j]);
    }
    *out = p;
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_pool_create(void *dev_slab, size_t slab_bytes, int page_size, int num_kv_heads, int head_dim,
                    uint64_t seed, pkv_pool **out)
{
    if (!out)
        return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    if (!dev_slab || (reinterpret_cast<uintptr_t>(dev_slab) & 15u) != 0)
        return PKV_ERR_INVALID_ARG;
    if (page_size != PKV_PAGE_SIZE || num_kv_heads != PKV_NUM_KV_HEADS || head_dim != PKV_HEAD_DIM)
        return PKV_ERR_UNSUPPORTED;
    return create_pool(dev_slab, slab_bytes, PKV_KV_BF16, PKV_PAGE_BYTES, seed, out);
}

int pkv_pool_create_fp8(void *dev_slab, size_t slab_bytes, uint64_t seed, pkv_pool **out)
{
    return create_pool(dev_slab, slab_bytes, PKV_KV_FP8, PKV_PAGE_BYTES_FP8, seed, out);
}

int pkv_pool_kv_format(const pkv_pool *pool)
{
    return pool ? pool->kv_format : PKV_ERR_INVALID_ARG;
}

int pkv_pool_destroy(pkv_pool *pool)
{
    delete pool;
    return PKV_OK;
}

int pkv_pool_alloc(pkv_pool *pool, int n, int32_t *ids_out)
{
    if (!pool || n < 0 || (n > 0 && !ids_out))
        return PKV_ERR_INVALID_ARG;
    if ((size_t)n > pool->free_list.size())
        return PKV_ERR_OUT_OF_PAGES;
    for (int i = 0; i < n; ++i) {
        int32_t id = pool->free_list.back();
        pool->free_list.pop_back();
        pool->allocated[id] = 1;
        ids_out[i] = id;
    }
    return PKV_OK;
}

int pkv_pool_free(pkv_pool *pool, int n, const int32_t *ids)
{
    if (!pool || n < 0 || (n > 0 && !ids))
        return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= pool->num_pages)
            return PKV_ERR_INVALID_ARG;
    // check every id before freeing any: each must be allocated and appear once
    int status = PKV_OK;
    int i = 0;
    for (; i < n; ++i) {
        if (pool->allocated[ids[i]] != 1) {
            status = PKV_ERR_DOUBLE_FREE;
            break;
        }
        pool->allocated[ids[i]] = 2;  // mark "seen in this call"
    }
    for (int k = 0; k < i; ++k)
        pool->allocated[ids[k]] = 1;  // undo the marks
    if (status != PKV_OK)
        return status;
    for (int k = 0; k < n; ++k) {
        pool->allocated[ids[k]] = 0;
        pool->free_list.push_back(ids[k]);
    }
    return PKV_OK;
}

int pkv_pool_info(const pkv_pool *pool, void **k_base, void **v_base, int64_t *page_stride_bytes,
                  int *num_pages, int *num_free)
{
    if (!pool)
        return PKV_ERR_INVALID_ARG;
    if (k_base)
        *k_base = pool->slab;
    if (v_base)
        *v_base = pool->slab + (pool->kv_format == PKV_KV_FP8 ? pkv::kPage * pkv::kD : PKV_PAGE_BYTES / 2);
    if (page_stride_bytes)
        *page_stride_bytes = (int64_t)pool->page_bytes;
    if (num_pages)
        *num_pages = pool->num_pages;
    if (num_free)
        *num_free = (int)pool->free_list.size();
    return PKV_OK;
}

int pkv_block_tables_build(pkv_pool *pool, int layers, int B, const int32_t *seq_lens, int max_blocks,
                           int32_t *bt_host)
{
    if (!pool || layers < 1 || B < 1 || max_blocks < 1 || !seq_lens || !bt_host)
        return PKV_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < 0)
            return PKV_ERR_INVALID_ARG;
        int64_t need = ((int64_t)seq_lens[b] + PKV_PAGE_SIZE - 1) / PKV_PAGE_SIZE;
        if (need > max_blocks)
            return PKV_ERR_INVALID_ARG;
        total += need;
    }
    total *= layers;
    if (total > (int64_t)pool->free_list.size())
        return PKV_ERR_OUT_OF_PAGES;
    for (int l = 0; l < layers; ++l) {
        for (int b = 0; b < B; ++b) {
            int32_t *row = bt_host + ((size_t)l * B + b) * max_blocks;
            int need = (seq_lens[b] + PKV_PAGE_SIZE - 1) / PKV_PAGE_SIZE;
            (void)pkv_pool_alloc(pool, need, row);
            for (int j = need; j < max_blocks; ++j)
                row[j] = -1;
        }
    }
    return PKV_OK;
}

size_t pkv_rope_table_bytes(int max_pos, int half_dim)
{
    if (max_pos < 1 || half_dim != PKV_HEAD_DIM / 2)
        return 0;
    return (size_t)max_pos * half_dim * 4 * sizeof(float);
}

int pkv_rope_table_init(double theta, int max_pos, int half_dim, float *dev_cos_sin, void *cuda_stream)
{
    if (!dev_cos_sin || max_pos < 1 || half_dim != PKV_HEAD_DIM / 2 || !(theta > 1.0))
        return PKV_ERR_INVALID_ARG;
    std::vector<float> table;
    try {
        table.resize((size_t)max_pos * half_dim * 4);
    } catch (...) {
        return PKV_ERR_INVALID_ARG;
    }
    const double dim = 2.0 * half_dim;
    for (int p = 0; p < max_pos; ++p) {
        for (int i = 0; i < half_dim; ++i) {
            const double angle = (double)p * std::pow(theta, -2.0 * i / dim);
            const double c = std::cos(angle), s = std::sin(angle);
            float *e = &table[((size_t)p * half_dim + i) * 4];
            e[0] = (float)c;                      // nearest FP32
            e[1] = (float)s;
            e[2] = (float)(c - (double)e[0]);     // the rest (exact in FP64), rounded to FP32
            e[3] = (float)(s - (double)e[1]);
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t e = cudaMemcpyAsync(dev_cos_sin, table.data(), table.size() * sizeof(float),
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    return pkv::status_from_cuda(e);
}

int pkv_check_device_error(const int32_t *dev_err_flag, int32_t *host_flag, void *cuda_stream)
{
    if (!dev_err_flag)
        return PKV_ERR_INVALID_ARG;
    int32_t h = 0;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t e = cudaMemcpyAsync(&h, dev_err_flag, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return PKV_ERR_CUDA;
    if (host_flag)
        *host_flag = h;
    return h ? PKV_ERR_DEVICE_BOUNDS : PKV_OK;
}

}  // extern "C"

namespace pkv {

const CUtensorMap *pool_tensor_map(const pkv_pool *cpool)
{
    pkv_pool *pool = const_cast<pkv_pool *>(cpool);
    if (pool->tmap_ready)
        return &pool->tmap;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return nullptr;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    CUresult r;
    cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    if (pool->kv_format == PKV_KV_FP8) {
        // dims innermost first: byte of a 128-byte line, line (17 per unit: 16 of
        // codes, 1 of scales), KV head, page; one box is one head's 2176-byte unit,
        // landing in shared memory exactly as it lies in the page
        constexpr int kLine = 128;
        cuuint64_t dims[4] = {(cuuint64_t)kLine, (cuuint64_t)(kFp8Unit / kLine), (cuuint64_t)kHkv,
                              (cuuint64_t)pool->num_pages};
        cuuint64_t strides[3] = {(cuuint64_t)kLine, (cuuint64_t)kFp8Unit, (cuuint64_t)pool->page_bytes};
        cuuint32_t box[4] = {(cuuint32_t)kLine, (cuuint32_t)(kFp8Unit / kLine), 1, 1};
        r = encode(&pool->tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, pool->slab, dims, strides, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        // dims innermost first: dim, slot, KV head, K/V, page
        cuuint64_t dims[5] = {(cuuint64_t)kD, (cuuint64_t)kPage, (cuuint64_t)kHkv, 2, (cuuint64_t)pool->num_pages};
        cuuint64_t strides[4] = {kD * 2, (cuuint64_t)kPage * kD * 2, (cuuint64_t)kHkv * kPage * kD * 2,
                                 (cuuint64_t)PKV_PAGE_BYTES};
        cuuint32_t box[5] = {(cuuint32_t)kD, (cuuint32_t)kPage, 1, 2, 1};
        r = encode(&pool->tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, pool->slab, dims, strides, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS)
        return nullptr;
    pool->tmap_ready = true;
    return &pool->tmap;
}

}  // namespace pkv
