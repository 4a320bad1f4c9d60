// pkv_fp8.cu -- FP8 E4M3 KV pages: quantizing append and prefill, and the decode
// split kernel that dequantizes in registers.
//
// "从零构建大模型推理引擎：KV缓存、算子融合与量化优化实战", section 5.1, suggests
// keeping the KV cache in low precision and dequantizing before attention; it
// gives no scheme.  The one read here (the same in the oracle):
//   * codes E4M3 without infinities (largest 448), round to nearest even,
//     saturating; one FP32 scale per (token, KV head) row of 64 values,
//     scale = amax / 448 (1 for an all-zero row), code = E4M3(x / scale) with an
//     IEEE FP32 division; x is the BF16 value the BF16 path would store (the
//     rotated key rounded to BF16, or the value);
//   * a page is 8 units of 2176 bytes, one per KV head: the codes [2 (K,V)]
//     [16 slots][64 dims] then the row scales [2][16] FP32 (17408 bytes a page),
//     so one (page, KV head) is one contiguous copy.
//
// Decode (same work split, chunking, online softmax and merge as the BF16 split
// kernel): per (page, KV head) one TMA tensor copy brings the unit -- 16 K and
// 16 V code rows of 64 bytes and the two scale rows -- into a shared-memory
// stage.  The page tile is two warp-level MMAs with FP32 accumulation:
//   S^T = K_codes . (T1 + T2)^T   on E4M3 tensor cores (m16n8k32): the K codes as
//                           stored, Q' = q times a power of two per head split
//                           into two E4M3 terms whose sum is Q' exactly (a BF16
//                           value has 8 significant bits, E4M3 4) except for
//                           entries below 2^-10 of the head's largest
//   x   = S^T * scale_k[token] * 2^e_head * scale * log2(e)
//   O^T += V_codes^T . P''^T   in FP16 (m16n8k16; E4M3 codes are exact in FP16),
//          P'' = p * scale_v[token] / sref (<= 1)
// with sref the largest V scale met so far (O^T kept in units of sref and
// rescaled when it grows), so P'' never overflows FP16 and its rounding is
// relative to the unit's own magnitude; l sums the unscaled FP32 p.
// The MMA operands are built from the codes without a staging pass: the dot
// product's k index and the output-dimension index are permuted so that a lane
// reads 16 contiguous code bytes of a K row and 8 contiguous code bytes of four
// V rows, and byte permutes pair two tokens' codes of one dimension for the
// conversion to FP16x2.

#include <cmath>

#include "pkv_fp8.cuh"

namespace pkv {
namespace {

using namespace dev;
using namespace fp8;

// One warp stores the K row of head h: lane i rotates the pair (i, i + 32) with
// the table's factors, rounds both to BF16 and quantizes them with the row scale.
__device__ __forceinline__ void store_key_row_fp8(uint8_t *page, int h, int slot, const uint16_t *k, float4 cs,
                                                  int lane)
{
    const float x1 = __uint_as_float((uint32_t)k[lane] << 16);
    const float x2 = __uint_as_float((uint32_t)k[lane + kD / 2] << 16);
    float y1, y2;
    rope_rotate_pair(x1, x2, cs, y1, y2);
    uint32_t c1, c2;
    float scale;
    quantize_pair(bf16_round(y1), bf16_round(y2), c1, c2, scale);
    uint8_t *unit = page + (size_t)h * kFp8Unit;
    uint8_t *row = unit + slot * kD;
    row[lane] = (uint8_t)c1;
    row[lane + kD / 2] = (uint8_t)c2;
    if (lane == 0)
        reinterpret_cast<float *>(unit + kFp8UnitCodes)[slot] = scale;
}

// One warp stores the V row of head h: lane i quantizes dims 2i, 2i+1.
__device__ __forceinline__ void store_value_row_fp8(uint8_t *page, int h, int slot, const uint16_t *v, int lane)
{
    const uint32_t w = reinterpret_cast<const uint32_t *>(v)[lane];
    uint32_t c0, c1;
    float scale;
    quantize_pair(bf16lo(w), bf16hi(w), c0, c1, scale);
    const uint32_t c = c0 | (c1 << 8);
    uint8_t *unit = page + (size_t)h * kFp8Unit;
    uint8_t *vt = unit + kFp8Tile;  // token-pair interleaved V codes
    vt[v_code_offset(slot, 2 * lane)] = (uint8_t)c;
    vt[v_code_offset(slot, 2 * lane + 1)] = (uint8_t)(c >> 8);
    if (lane == 0)
        reinterpret_cast<float *>(unit + kFp8UnitCodes)[kPage + slot] = scale;
}

constexpr int kAppendThreads = kHkv * 32;  // one warp per KV head

// Decode append for FP8 pages: one CTA per sequence, warp h stores head h's K and
// V rows; then the 32 query rows are rotated in place (BF16, as the BF16 path).
__global__ void __launch_bounds__(kAppendThreads)
append_rope_fp8_kernel(uint8_t *__restrict__ slab, int num_pages, const uint16_t *__restrict__ k_new,
                       const uint16_t *__restrict__ v_new, uint16_t *__restrict__ q, const int32_t *__restrict__ bt,
                       int max_blocks, const int32_t *__restrict__ pos,
                       const float4 *__restrict__ rope, int max_pos, int32_t *__restrict__ err)
{
    grid_dependency_wait();  // launched with programmatic dependent launch: see append_rope_kernel
    allow_dependent_launch();
    const int b = blockIdx.x;
    const int p = pos[b];
    if (p < 0 || p >= min(max_pos, max_blocks * kPage)) {
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
    const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *page_base = slab + (size_t)page * kFp8PageBytes;
    const float4 *rope_row = rope + (size_t)p * (kD / 2);
    store_key_row_fp8(page_base, h, slot, k_new + ((size_t)b * kHkv + h) * kD, rope_row[lane], lane);
    store_value_row_fp8(page_base, h, slot, v_new + ((size_t)b * kHkv + h) * kD, lane);
    if (!q)
        return;
    // query rows: 32 rows x 32 pairs, one pair per thread and pass
    for (int item = threadIdx.x; item < kHq * (kD / 2); item += kAppendThreads) {
        const int r = item / (kD / 2), i = item % (kD / 2);
        uint16_t *row = q + ((size_t)b * kHq + r) * kD;
        const float4 cs = rope_row[i];
        const float x1 = __uint_as_float((uint32_t)row[i] << 16);
        const float x2 = __uint_as_float((uint32_t)row[i + kD / 2] << 16);
        float y1, y2;
        rope_rotate_pair(x1, x2, cs, y1, y2);
        const __nv_bfloat16 b1 = __float2bfloat16_rn(y1), b2 = __float2bfloat16_rn(y2);
        row[i] = *reinterpret_cast<const uint16_t *>(&b1);
        row[i + kD / 2] = *reinterpret_cast<const uint16_t *>(&b2);
    }
}

constexpr int kPrefillThreads = 128;

// Prefill for FP8 pages: one CTA per (token, layer); warp w stores K and V rows of
// heads w and w + 4.
__global__ void __launch_bounds__(kPrefillThreads)
prefill_append_fp8_kernel(uint8_t *__restrict__ slab, int num_pages, const uint16_t *__restrict__ k,
                          const uint16_t *__restrict__ v, const int32_t *__restrict__ bt_rows, int max_blocks,
                          int start_pos, int T, const float4 *__restrict__ rope, int max_pos,
                          int32_t *__restrict__ err)
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
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *page_base = slab + (size_t)page * kFp8PageBytes;
    const size_t row0 = ((size_t)l * T + t) * kHkv * kD;  // token t of layer l: [8][64]
    const float4 cs = rope[(size_t)p * (kD / 2) + lane];
#pragma unroll
    for (int hh = 0; hh < kHkv / 4; ++hh) {
        const int h = w + 4 * hh;
        store_key_row_fp8(page_base, h, slot, k + row0 + (size_t)h * kD, cs, lane);
        store_value_row_fp8(page_base, h, slot, v + row0 + (size_t)h * kD, lane);
    }
}

}  // namespace
}  // namespace pkv

// ---------------------------------------------------------------------------
// Decode split kernel over FP8 pages.
namespace pkv {
namespace {

using namespace dev;
using namespace fp8;

struct Fp8SplitArgs {
    int num_pages;
    const uint16_t *q;
    const int32_t *bt;
    int max_blocks;
    const int32_t *seq_lens;
    float scale_log2;
    int pages_per_chunk;
    float2 *part_ml;
    float *part_o;
    int max_chunks;
    uint16_t *out;
    int32_t *err;
};

__device__ void fp8_write_empty(const Fp8SplitArgs &a, int b, int g, int c, int nchunks)
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

// One CTA per (chunk c, KV head g, sequence b), as the BF16 split kernel.
template <int STAGES>
__global__ void __launch_bounds__(kThreads, 6)  // six CTAs per SM: at most 85 registers
decode_split_fp8_kernel(const __grid_constant__ CUtensorMap tmap, Fp8SplitArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    Fp8Smem<STAGES> sm(smem_raw);

    const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = a.seq_lens[b];
    if (L < 1 || L > a.max_blocks * kPage) {
        if (c == 0) {
            fp8_write_empty(a, b, g, 0, 1);
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
        fp8_write_empty(a, b, g, c, nchunks);
        if (threadIdx.x == 0 && a.err)
            atomicOr(a.err, PKV_DEVERR_PAGE_RANGE);
        return;
    }

    uint64_t *my_bars = sm.bars + warp * STAGES;
    uint8_t *my_stages = sm.stages + warp * STAGES * kFp8Unit;
    init_warp_barriers<STAGES>(my_bars, lane);
    const uint64_t policy = l2_evict_first_policy();
    const int prologue = min(STAGES, nmine);
    for (int k = 0; k < prologue; ++k) {
        const int pk = __shfl_sync(kFull, my_page, k);
        if (lane == 0)
            fp8_issue(&tmap, my_stages + k * kFp8Unit, &my_bars[k], g, pk, policy);
    }

    Fp8MmaWarp w;
    w.init(a.q + ((size_t)b * kHq + g * kGroup) * kD, a.scale_log2, lane);
    // pages k = k0 + s, the ring unrolled so that every stage address is a constant
    int k = 0;
    bool timed_out = false;
    for (int k0 = 0; k0 < nmine && !timed_out; k0 += STAGES) {
        const uint32_t parity = (uint32_t)((k0 / STAGES) & 1);
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            k = k0 + s;
            if (k >= nmine)
                break;
            if (!mbar_wait_warp(&my_bars[s], parity)) {
                timed_out = true;
                break;
            }
            const int j = j0 + warp + k * kWarps;
            uint8_t *stage = my_stages + s * kFp8Unit;
            w.page(stage, min(kPage, L - j * kPage));
            __syncwarp();
            if (k + STAGES < nmine) {
                const int pk = __shfl_sync(kFull, my_page, k + STAGES);
                if (lane == 0) {
                    fence_proxy_async_smem();
                    fp8_issue(&tmap, stage, &my_bars[s], g, pk, policy);
                }
            }
        }
    }
    if (timed_out) {  // a wait gave up: let the copies in flight land (bounded), flag it
        for (int kk = k; kk < min(nmine, k + STAGES); ++kk)
            (void)mbar_wait_warp(&my_bars[kk % STAGES], (uint32_t)((kk / STAGES) & 1));
        if (lane == 0 && a.err)
            atomicOr(a.err, PKV_DEVERR_TIMEOUT);
    }

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

constexpr int kFp8Stages = 4;  // 35 KiB of shared memory: six CTAs per SM

}  // namespace

// ------------------------------------------------------------------ launchers

int fp8_append_rope(const pkv_pool *pool, const uint16_t *k_new, const uint16_t *v_new, uint16_t *q,
                    const int32_t *bt, int max_blocks, const int32_t *pos, int B, const float *rope,
                    int max_pos, int32_t *err, cudaStream_t s)
{
    return launch_kernel(append_rope_fp8_kernel, dim3(B), dim3(kAppendThreads), 0, s, true,
                         reinterpret_cast<uint8_t *>(pool->slab), pool->num_pages, k_new, v_new, q, bt, max_blocks,
                         pos, reinterpret_cast<const float4 *>(rope), max_pos, err);
}

int fp8_prefill_append(const pkv_pool *pool, const uint16_t *k, const uint16_t *v, const int32_t *bt_rows,
                       int max_blocks, int layers, int start_pos, int T, const float *rope, int max_pos,
                       int32_t *err, cudaStream_t s)
{
    prefill_append_fp8_kernel<<<dim3(T, layers), kPrefillThreads, 0, s>>>(
        reinterpret_cast<uint8_t *>(pool->slab), pool->num_pages, k, v, bt_rows, max_blocks, start_pos, T,
        reinterpret_cast<const float4 *>(rope), max_pos, err);
    return status_from_cuda(cudaGetLastError());
}

int fp8_decode_split(const pkv_pool *pool, const uint16_t *q, const int32_t *bt, int max_blocks,
                     const int32_t *seq_lens, int B, float scale_log2, int pages_per_chunk, float2 *part_ml,
                     float *part_o, int max_chunks, uint16_t *out, int32_t *err, cudaStream_t s)
{
    const CUtensorMap *tmap = pool_tensor_map(pool);
    if (!tmap)
        return PKV_ERR_CUDA;
    auto kernel = decode_split_fp8_kernel<kFp8Stages>;
    constexpr int smem = Fp8Smem<kFp8Stages>::kBytes;
    static PerDeviceOnce attr;  // set on the first launch per device (before any graph capture)
    if (const int st = ensure_smem_attr(attr, kernel, smem); st != PKV_OK)
        return st;
    Fp8SplitArgs a;
    a.num_pages = pool->num_pages;
    a.q = q;
    a.bt = bt;
    a.max_blocks = max_blocks;
    a.seq_lens = seq_lens;
    a.scale_log2 = scale_log2;
    a.pages_per_chunk = pages_per_chunk;
    a.part_ml = part_ml;
    a.part_o = part_o;
    a.max_chunks = max_chunks;
    a.out = out;
    a.err = err;
    kernel<<<dim3(max_chunks, kHkv, B), kThreads, smem, s>>>(*tmap, a);
    return status_from_cuda(cudaGetLastError());
}

}  // namespace pkv
