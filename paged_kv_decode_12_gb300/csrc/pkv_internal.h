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
    // TMA descriptor of the slab seen as [num_pages][2][8][16][64] BF16, 128-byte
    // swizzle, box = one (page, KV head): its K rows then its V rows (4 KiB).
    // Encoded on first use, because encoding needs the CUDA driver.
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

// Encodes the pool's tensor map if needed; returns nullptr on a driver error.
const CUtensorMap *pool_tensor_map(const pkv_pool *pool);

inline int status_from_cuda(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

}  // namespace pkv
