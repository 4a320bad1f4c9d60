// pkv_decode.cu -- paged decode attention: the entry points, and the two-kernel form
// (split-sequence kernel + log-sum-exp merge kernel).
//
// pkv_decode_attention runs, by default, the grid kernel of pkv_step.cu without the
// append: the same unit of work as below, with the chunk partials merged inside the
// same launch.  The two-kernel form here (PKV_DECODE_SPLIT_MERGE) keeps the merge in a
// second small kernel; it needs no zeroed workspace, which is why the allocation-free
// entry point uses it.  Both merge in chunk order with the same arithmetic, so their
// results are identical bit for bit.
//
// What is computed (samir-vllm README summary, "从零用 C++ 和 CUDA 实现 Llama 3.2 1B
// 推理引擎", section "目前已完成的功能": each query head streams its sequence's
// cached pages with an FP32 online softmax and accumulates weighted values,
// without a contiguous gather or stored scores; "从零构建大模型推理引擎" section
// 3.2: scores q.k / sqrt(d), maximum subtracted, weighted sum of V):
//     out[b][h] = sum_t softmax_t(scale * q[b][h] . K_t) V_t,  t < seq_lens[b].
//
// GB300 design:
//  * One CTA per (sequence b, KV head g, chunk c of pages_per_chunk pages).  The
//    four query heads of group g are served from ONE read of each page, so every
//    KV byte crosses HBM once.  The chunking depends only on the sequence's own
//    length, never on the batch, so results are batch invariant.
//  * 4 warps per CTA; warp w takes pages w, w+4, ... of the chunk and owns a
//    private ring of STAGES 4 KiB shared-memory stages.  Lane 0 of the warp
//    issues one TMA tensor copy per (page, KV head) -- its 16 K rows and 16 V
//    rows, 128-byte swizzled -- completing on the stage's mbarrier.  No
//    CTA-wide barrier is taken inside the page loop.
//  * The online softmax runs in the log2 domain (scale * log2(e) folded in) with
//    running max m, running sum l and an unnormalised FP32 accumulator o per
//    head; the four warps' states are combined in shared memory at the end.
//  * A sequence with one chunk writes BF16 output directly; otherwise chunk
//    partials (m, l, o) go to the workspace and a small merge kernel combines
//    them by log-sum-exp, in chunk order (deterministic).
//  * Two per-page compute policies:
//      SimtWarp  FP32 FMA dot products on CUDA cores; a lane holds 8 dims of 4
//                tokens, partial dot products are reduce-scattered across the 8
//                lanes sharing a token with warp shuffles; P.V with a lane
//                owning 2 output dims of the 4 heads.
//      MmaWarp   the 16-token page tile as warp-level BF16 MMA (m16n8k16, FP32
//                accumulate): S^T = K Q^T with the tokens in M and the 4 heads
//                (padded to 8) in N, then O^T += V^T P^T with P^T moved into the
//                B-operand layout by movmatrix.  P is rounded to BF16 for the
//                second product; l is summed from the unrounded FP32 weights.
//  * Every wait is bounded; a wait that gives up sets PKV_DEVERR_TIMEOUT.
//    Page ids outside the pool and bad lengths are checked before any copy is
//    issued; the unit is skipped and the device error flag set.
#include <cuda_bf16.h>

#include <cmath>

#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

// ------------------------------------------------------------------ kernels

struct SplitArgs {
    int num_pages;
    const uint16_t *q;
    const int32_t *bt;
    int max_blocks;
    const int32_t *seq_lens;
    float scale_log2;
    int pages_per_chunk;
    float2 *part_ml;  // [B][32][max_chunks] (m, l), log2 domain
    float *part_o;    // [B][32][max_chunks][64]
    int max_chunks;
    uint16_t *out;    // [B][32][64]
    int32_t *err;
};

template <int STAGES>
constexpr int split_smem_bytes()
{
    return SmemLayout<STAGES>::kBaseBytes;
}

// Write this CTA's 4 heads as "no contribution": zeros if the sequence has one
// chunk, else an empty partial (m = -inf, l = 0, o = 0).
__device__ void write_empty(const SplitArgs &a, int b, int g, int c, int nchunks)
{
    const int h = g * kGroup + (threadIdx.x >> 5), dp = threadIdx.x & 31;
    if (nchunks <= 1) {
        reinterpret_cast<uint32_t *>(a.out + ((size_t)b * kHq + h) * kD)[dp] = 0u;
    } else {
        const size_t idx = ((size_t)b * kHq + h) * a.max_chunks + c;
        reinterpret_cast<float2 *>(a.part_o + idx * kD)[dp] = make_float2(0.f, 0.f);
        if (dp == 0)
            a.part_ml[idx] = make_float2(-INFINITY, 0.f);
    }
}

template <class Warp, int STAGES>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const __grid_constant__ CUtensorMap tmap, SplitArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    SmemLayout<STAGES> sm(smem_raw);

    const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = a.seq_lens[b];
    if (L < 1 || L > a.max_blocks * kPage) {
        if (c == 0) {
            write_empty(a, b, g, 0, 1);
            if (threadIdx.x == 0 && a.err)
                atomicOr(a.err, PKV_DEVERR_LENGTH);
        }
        return;
    }
    const int npages = (L + kPage - 1) / kPage;
    const int nchunks = (npages + a.pages_per_chunk - 1) / a.pages_per_chunk;
    if (c >= nchunks)
        return;
    const int j0 = c * a.pages_per_chunk;
    const int jn = min(npages - j0, a.pages_per_chunk);
    const int nmine = warp < jn ? (jn - warp + kWarps - 1) / kWarps : 0;  // <= 32

    int my_page = 0;
    bool bad = false;
    if (lane < nmine) {
        my_page = a.bt[(size_t)b * a.max_blocks + j0 + warp + lane * kWarps];
        bad = my_page < 0 || my_page >= a.num_pages;
    }
    if (__syncthreads_or(bad)) {
        write_empty(a, b, g, c, nchunks);
        if (threadIdx.x == 0 && a.err)
            atomicOr(a.err, PKV_DEVERR_PAGE_RANGE);
        return;
    }

    uint64_t *my_bars = sm.bars + warp * STAGES;
    uint8_t *my_stages = sm.stages + warp * STAGES * kStageBytes;
    init_warp_barriers<STAGES>(my_bars, lane);
    const uint64_t policy = l2_evict_first_policy();
    issue_prologue<STAGES>(&tmap, my_stages, my_bars, my_page, nmine, g, lane, policy);

    Warp w;
    w.init(a.q + ((size_t)b * kHq + g * kGroup) * kD, a.scale_log2, lane, sm.scratch + warp * kScratchFloats);
    if (!consume_pages<STAGES>(&tmap, my_stages, my_bars, w, my_page, nmine, j0, warp, lane, L, g, policy,
                               NoPatch{}) &&
        lane == 0 && a.err)
        atomicOr(a.err, PKV_DEVERR_TIMEOUT);

    // ---- combine the 4 warps' (m, l, o) in shared memory (stages are free now)
    __syncthreads();
    float *state = reinterpret_cast<float *>(sm.stages);
    w.store_state(state + warp * kStateFloats);
    __syncthreads();
    const int hl = threadIdx.x >> 5, dp = threadIdx.x & 31;
    float M, lsum, o0, o1;
    combine_warps(state, hl, dp, M, lsum, o0, o1);
    const int h = g * kGroup + hl;
    if (nchunks == 1) {
        reinterpret_cast<uint32_t *>(a.out + ((size_t)b * kHq + h) * kD)[dp] = finish_pair(o0, o1, lsum);
    } else {
        const size_t idx = ((size_t)b * kHq + h) * a.max_chunks + c;
        reinterpret_cast<float2 *>(a.part_o + idx * kD)[dp] = make_float2(o0, o1);
        if (dp == 0)
            a.part_ml[idx] = make_float2(M, lsum);
    }
}

// One CTA per (sequence, group of 4 query heads); thread = (head, dim pair).
// Partials are merged in chunk order, so the result does not depend on timing.
__global__ void __launch_bounds__(kThreads)
decode_merge_kernel(const int32_t *__restrict__ seq_lens, int max_blocks, int pages_per_chunk,
                    const float2 *__restrict__ part_ml, const float *__restrict__ part_o, int max_chunks,
                    uint16_t *__restrict__ out)
{
    const int b = blockIdx.x;
    const int h = blockIdx.y * kGroup + (threadIdx.x >> 5), dp = threadIdx.x & 31;
    const int L = seq_lens[b];
    if (L < 1 || L > max_blocks * kPage)
        return;  // the split kernel wrote zeros and set the flag
    const int nchunks = ((L + kPage - 1) / kPage + pages_per_chunk - 1) / pages_per_chunk;
    if (nchunks <= 1)
        return;  // written directly by the split kernel
    const size_t base = ((size_t)b * kHq + h) * max_chunks;
    float M = -INFINITY;
    for (int c = 0; c < nchunks; ++c)
        M = fmaxf(M, part_ml[base + c].x);
    float lsum = 0.f, o0 = 0.f, o1 = 0.f;
    if (M != -INFINITY) {
        for (int c = 0; c < nchunks; ++c) {
            const float2 ml = part_ml[base + c];
            const float f = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
            const float2 oc = reinterpret_cast<const float2 *>(part_o + (base + c) * kD)[dp];
            lsum = fmaf(f, ml.y, lsum);
            o0 = fmaf(f, oc.x, o0);
            o1 = fmaf(f, oc.y, o1);
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    reinterpret_cast<uint32_t *>(out + ((size_t)b * kHq + h) * kD)[dp] = pack_bf16x2(o0 * inv, o1 * inv);
}

constexpr int kStages = 4;

template <class Warp>
int launch_split(const CUtensorMap *tmap, const SplitArgs &a, int B, cudaStream_t s)
{
    auto kernel = decode_split_kernel<Warp, kStages>;
    constexpr int smem = split_smem_bytes<kStages>();
    static PerDeviceOnce attr;  // set on the first launch per device (before any graph capture)
    if (const int st = ensure_smem_attr(attr, kernel, smem); st != PKV_OK)
        return st;
    dim3 grid(a.max_chunks, kHkv, B);
    kernel<<<grid, kThreads, smem, s>>>(*tmap, a);
    return status_from_cuda(cudaGetLastError());
}

}  // namespace

int launch_decode_merge(const int32_t *seq_lens, int max_blocks, int pages_per_chunk, const float2 *part_ml,
                        const float *part_o, int max_chunks, uint16_t *out, int B, cudaStream_t s)
{
    decode_merge_kernel<<<dim3(B, kHkv), kThreads, 0, s>>>(seq_lens, max_blocks, pages_per_chunk, part_ml, part_o,
                                                            max_chunks, out);
    return status_from_cuda(cudaGetLastError());
}

}  // namespace pkv

extern "C" size_t pkv_decode_workspace_bytes(int B, int max_blocks, int pages_per_chunk)
{
    using namespace pkv;
    if (B < 1 || max_blocks < 1 || pages_per_chunk < 1)
        return 0;
    const size_t chunks = (size_t)(max_blocks + pages_per_chunk - 1) / pages_per_chunk;
    if (chunks > (size_t)INT32_MAX)
        return 0;
    return workspace_layout(B, (int)chunks).total();
}

extern "C" int pkv_decode_attention_variant(const pkv_pool *pool, const uint16_t *q, const int32_t *bt_dev,
                                            int max_blocks, const int32_t *seq_lens_dev, int B, float scale,
                                            int pages_per_chunk, void *workspace, size_t workspace_bytes,
                                            uint16_t *out, int32_t *dev_err_flag, void *cuda_stream, int variant)
{
    using namespace pkv;
    if (!pool || !q || !bt_dev || !seq_lens_dev || !out)
        return PKV_ERR_INVALID_ARG;
    if (B < 1 || B > 65535 || max_blocks < 1 || max_blocks > (1 << 20))
        return PKV_ERR_INVALID_ARG;
    if (pages_per_chunk < 1 || pages_per_chunk > kMaxPagesPerChunk || !(scale > 0.f) || !std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    const int policy = variant & 0xff;
    if (policy < PKV_DECODE_DEFAULT || policy > PKV_DECODE_MMA)
        return PKV_ERR_INVALID_ARG;
    if (pool->kv_format == PKV_KV_FP8 && policy == PKV_DECODE_SIMT)
        return PKV_ERR_UNSUPPORTED;  // FP8 pages have the MMA policy only
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u)
        return PKV_ERR_INVALID_ARG;
    const int max_chunks = (max_blocks + pages_per_chunk - 1) / pages_per_chunk;
    const size_t need = pkv_decode_workspace_bytes(B, max_blocks, pages_per_chunk);
    if (max_chunks > 1) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u))
            return PKV_ERR_INVALID_ARG;
        if (workspace_bytes < need)
            return PKV_ERR_WORKSPACE_TOO_SMALL;
    }
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (!(variant & PKV_DECODE_SPLIT_MERGE))
        return launch_attention_fused(pool, q, bt_dev, max_blocks, seq_lens_dev, B, scale, pages_per_chunk,
                                      workspace, out, dev_err_flag, s, variant);
    // the two-kernel form: split kernel, then the separate LSE merge kernel
    if (variant & ~(0xff | PKV_DECODE_SPLIT_MERGE))
        return PKV_ERR_INVALID_ARG;
    const CUtensorMap *tmap = pool_tensor_map(pool);
    if (!tmap)
        return PKV_ERR_CUDA;
    (void)take_pdl_permission(pool, false);  // this form launches without programmatic dependent launch
    const WorkspaceLayout ws = workspace_layout(B, max_chunks);
    char *wsp = static_cast<char *>(workspace);
    SplitArgs a;
    a.num_pages = pool->num_pages;
    a.q = q;
    a.bt = bt_dev;
    a.max_blocks = max_blocks;
    a.seq_lens = seq_lens_dev;
    a.scale_log2 = scale * kLog2e;
    a.pages_per_chunk = pages_per_chunk;
    a.part_ml = wsp ? reinterpret_cast<float2 *>(wsp + ws.ml_offset()) : nullptr;
    a.part_o = wsp ? reinterpret_cast<float *>(wsp + ws.o_offset()) : nullptr;
    a.max_chunks = max_chunks;
    a.out = out;
    a.err = dev_err_flag;
    const int v = policy == PKV_DECODE_DEFAULT ? PKV_DECODE_MMA : policy;
    int st;
    if (pool->kv_format == PKV_KV_FP8) {
        st = fp8_decode_split(pool, q, bt_dev, max_blocks, seq_lens_dev, B, a.scale_log2, pages_per_chunk,
                              a.part_ml, a.part_o, max_chunks, out, dev_err_flag, s);
    } else {
        st = v == PKV_DECODE_SIMT ? launch_split<SimtWarp>(tmap, a, B, s) : launch_split<MmaWarp>(tmap, a, B, s);
    }
    if (st != PKV_OK || max_chunks == 1)
        return st;
    return launch_decode_merge(seq_lens_dev, max_blocks, pages_per_chunk, a.part_ml, a.part_o, max_chunks, out, B, s);
}

extern "C" int pkv_decode_attention(const pkv_pool *pool, const uint16_t *q, const int32_t *bt_dev, int max_blocks,
                                    const int32_t *seq_lens_dev, int B, float scale, int pages_per_chunk,
                                    void *workspace, size_t workspace_bytes, uint16_t *out, int32_t *dev_err_flag,
                                    void *cuda_stream)
{
    return pkv_decode_attention_variant(pool, q, bt_dev, max_blocks, seq_lens_dev, B, scale, pages_per_chunk,
                                        workspace, workspace_bytes, out, dev_err_flag, cuda_stream,
                                        PKV_DECODE_DEFAULT);
}

// ---------------------------------------------------------------------------
// Decode attention without any allocation by the caller or the library.
//
// For callers that cannot call cudaMalloc: a plugin hosted by an engine that
// owns the whole device-memory budget through its own allocator and hands its
// plugins no workspace; a latency-critical loop that must not call cudaMalloc or
// cudaFree mid-run because they can synchronise the device; a C caller with no
// device allocator of its own.  The chunk partials live in the file-scope array
// below instead of a caller-supplied workspace.  That array is part of this
// library's device image: every GPU that loads the library holds its
// PKV_NOALLOC_SCRATCH_BYTES until the process exits.
//
// In host code `pkv_noalloc_scratch` names a host-side stand-in, not a device
// address; handing it to a kernel would fault (or, where the GPU can reach host
// memory, silently use the wrong memory).  The device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call made on that device; make that first call before any stream
// capture begins.
static __device__ __align__(256) unsigned char pkv_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the static scratch on the current device, looked up on the first
// call per device.  A failed lookup is not remembered: a later call (for example one
// made outside a stream capture) tries again.
void *g_noalloc_address[pkv::kMaxDevices];
pkv::PerDeviceOnce g_noalloc_lookup;

int noalloc_scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= pkv::kMaxDevices)
        return PKV_ERR_CUDA;
    const int st = g_noalloc_lookup.run([](int d) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, pkv_noalloc_scratch);
        if (e == cudaSuccess && p == nullptr)
            return cudaErrorInvalidSymbol;
        if (e == cudaSuccess)
            g_noalloc_address[d] = p;
        return e;
    });
    if (st != PKV_OK)
        return st;
    *out = g_noalloc_address[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_decode_attention_noalloc(const pkv_pool *pool, const uint16_t *q, const int32_t *bt_dev,
                                            int max_blocks, const int32_t *seq_lens_dev, int B, float scale,
                                            int pages_per_chunk, uint16_t *out, int32_t *dev_err_flag,
                                            void *cuda_stream)
{
    if (!pool || !q || !bt_dev || !seq_lens_dev || !out)
        return PKV_ERR_INVALID_ARG;
    const size_t need = pkv_decode_workspace_bytes(B, max_blocks, pages_per_chunk);
    if (need == 0)
        return PKV_ERR_INVALID_ARG;
    if (need > PKV_NOALLOC_SCRATCH_BYTES)
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    const int st = noalloc_scratch_address(&scratch);
    if (st != PKV_OK)
        return st;
    // The two-kernel form: the partials of every chunk are written by the split kernel
    // before the merge kernel reads them, so nothing left in the array by an earlier
    // call is ever read and nothing needs to start at zero.
    return pkv_decode_attention_variant(pool, q, bt_dev, max_blocks, seq_lens_dev, B, scale, pages_per_chunk,
                                        scratch, PKV_NOALLOC_SCRATCH_BYTES, out, dev_err_flag, cuda_stream,
                                        PKV_DECODE_DEFAULT | PKV_DECODE_SPLIT_MERGE);
}
