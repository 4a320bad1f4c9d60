// pkv_internal.h -- definitions shared by libpkv's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "../../include/pkv.h"

struct pkv_pool {
    char *slab = nullptr;          // caller-owned device slab
    size_t slab_bytes = 0;
    int32_t num_pages = 0;
    std::vector<int32_t> free_list;  // stack of free page ids; pop from the back
    std::vector<uint8_t> allocated;  // 1 while a page is handed out
    int kv_format = PKV_KV_BF16;     // PKV_KV_BF16 or PKV_KV_FP8
    size_t page_bytes = PKV_PAGE_BYTES;
    // TMA descriptor of the slab.  BF16 pools: [num_pages][2][8][16][64] BF16,
    // 128-byte swizzle, box = one (page, KV head): its K rows then its V rows
    // (4 KiB).  FP8 pools: the slab as [num_pages][8 heads][17 lines][128 B] (a
    // head's unit: 16 lines of codes, 1 of scales), no swizzle, box = one
    // (page, KV head) unit (2176 B).  Encoded on first use, because encoding
    // needs the CUDA driver.
    CUtensorMap tmap;  // 64-byte aligned by its own declaration
    bool tmap_ready = false;
};

namespace pkv {

constexpr int kPage = PKV_PAGE_SIZE;      // tokens per page
constexpr int kHq = PKV_NUM_Q_HEADS;      // query heads
constexpr int kHkv = PKV_NUM_KV_HEADS;    // KV heads
constexpr int kGroup = kHq / kHkv;        // query heads per KV head
constexpr int kD = PKV_HEAD_DIM;          // head dimension
constexpr int kPageElems = PKV_PAGE_BYTES / 2;
constexpr int kMaxPagesPerChunk = 128;
constexpr int kFp8PageBytes = PKV_PAGE_BYTES_FP8;
constexpr int kFp8Unit = 2 * kPage * (kD + 4);     // one KV head's codes [2][16][64] + scales [2][16]
constexpr int kFp8UnitCodes = 2 * kPage * kD;      // code bytes at the start of a unit

// Encodes the pool's tensor map if needed; returns nullptr on a driver error.
const CUtensorMap *pool_tensor_map(const pkv_pool *pool);

// Log-sum-exp merge of the split kernels' chunk partials (any KV format).
int launch_decode_merge(const int32_t *seq_lens, int max_blocks, int pages_per_chunk, const float2 *part_ml,
                        const float *part_o, int max_chunks, uint16_t *out, int B, cudaStream_t s);

// FP8 pools: quantizing append / prefill and the dequantizing split kernel.  The
// public entry points validate their arguments and dispatch here.
int fp8_append_rope(const pkv_pool *pool, const uint16_t *k_new, const uint16_t *v_new, uint16_t *q,
                    const int32_t *bt, int max_blocks, const int32_t *pos, int B,
                    const float *rope, int max_pos, int32_t *err, cudaStream_t s);
int fp8_prefill_append(const pkv_pool *pool, const uint16_t *k, const uint16_t *v, const int32_t *bt_rows,
                       int max_blocks, int layers, int start_pos, int T, const float *rope, int max_pos,
                       int32_t *err, cudaStream_t s);
int fp8_decode_split(const pkv_pool *pool, const uint16_t *q, const int32_t *bt, int max_blocks,
                     const int32_t *seq_lens, int B, float scale_log2, int pages_per_chunk, float2 *part_ml,
                     float *part_o, int max_chunks, uint16_t *out, int32_t *err, cudaStream_t s);

inline int status_from_cuda(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

}  // namespace pkv
