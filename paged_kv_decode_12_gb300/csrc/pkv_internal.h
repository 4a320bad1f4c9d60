// pkv_internal.h -- definitions shared by libpkv's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <utility>
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
    // Set by a prefill on this pool: the prefill wrote cached positions that the next
    // decode launch would otherwise start copying before its dependency wait, so that
    // launch goes without programmatic dependent launch (and clears the flag).
    mutable bool serialize_next_launch = false;
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

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of pkv_decode_attention and pkv_decode_step: the per-(sequence, KV head)
// merge counters [B][8] int32, then the chunk partials (m, l) [B][32][max_chunks]
// float2 and o [B][32][max_chunks][64] float; each region starts 256-byte aligned.
struct WorkspaceLayout {
    size_t counters, ml, o;
    size_t ml_offset() const { return counters; }
    size_t o_offset() const { return counters + ml; }
    size_t total() const { return counters + ml + o; }
};

inline WorkspaceLayout workspace_layout(int B, int max_chunks)
{
    WorkspaceLayout w;
    w.counters = align256((size_t)B * kHkv * sizeof(int));
    w.ml = align256((size_t)B * kHq * max_chunks * sizeof(float) * 2);
    w.o = (size_t)B * kHq * max_chunks * kD * sizeof(float);
    return w;
}

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
// pkv_decode_attention's default form: the fused grid kernel without the append
// (in-kernel LSE merge).  Arguments validated by the caller; `workspace` has
// workspace_layout(B, max_chunks) (may be null when max_chunks == 1); `options` are
// the pkv_decode_attention_variant option bits (policy, NO_PDL, RING, SORTED,
// TEST_EXPIRE_WAIT).
int launch_attention_fused(const pkv_pool *pool, const uint16_t *q, const int32_t *bt, int max_blocks,
                           const int32_t *seq_lens, int B, float scale, int pages_per_chunk, void *workspace,
                           uint16_t *out, int32_t *err, cudaStream_t s, int options);

int fp8_decode_split(const pkv_pool *pool, const uint16_t *q, const int32_t *bt, int max_blocks,
                     const int32_t *seq_lens, int B, float scale_log2, int pages_per_chunk, float2 *part_ml,
                     float *part_o, int max_chunks, uint16_t *out, int32_t *err, cudaStream_t s);

inline int status_from_cuda(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

// A set-up step done once per device, with that device current (a kernel's
// shared-memory attribute, a symbol's device address).  Thread-safe; a step that
// fails is not recorded, so a later call tries again.
constexpr int kMaxDevices = 64;

class PerDeviceOnce {
  public:
    template <class F>
    int run(F step)
    {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
            return PKV_ERR_CUDA;
        std::lock_guard<std::mutex> lock(mu_);
        if (done_[dev])
            return PKV_OK;
        if (step(dev) != cudaSuccess)
            return PKV_ERR_CUDA;
        done_[dev] = true;
        return PKV_OK;
    }

  private:
    std::mutex mu_;
    bool done_[kMaxDevices] = {};
};

// The dynamic shared-memory limit of `kernel` raised to `bytes`, once per device.
template <class Kernel>
int ensure_smem_attr(PerDeviceOnce &once, Kernel kernel, int bytes)
{
    return once.run([&](int) { return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes); });
}

// Programmatic dependent launch: the launch may begin before the previous kernel on
// the stream has finished; the kernel's griddepcontrol.wait orders what follows it.
inline cudaLaunchAttribute pdl_attribute()
{
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    return attr;
}

// Launch `kernel` on `s`, with programmatic dependent launch if `pdl`.
template <class... Params, class... Args>
int launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                  Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[1] = {pdl_attribute()};
    cfg.attrs = attrs;
    cfg.numAttrs = pdl ? 1 : 0;
    return status_from_cuda(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

// Whether a decode launch on `pool` may use programmatic dependent launch: not the
// first one after a prefill on the pool (see pkv_pool::serialize_next_launch).
inline bool take_pdl_permission(const pkv_pool *pool, bool pdl_requested)
{
    const bool fence = pool->serialize_next_launch;
    pool->serialize_next_launch = false;
    return pdl_requested && !fence;
}

}  // namespace pkv
