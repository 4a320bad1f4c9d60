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
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>

#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int kFp8Tile = kPage * kD;  // 1 KiB: one (page, KV head) K or V code tile
static_assert(kFp8Unit == 2176 && kFp8Unit % 128 == 0, "stage = one unit, 128-byte aligned");

// ------------------------------------------------------------------ quantization

__device__ __forceinline__ uint32_t e4m3_code(float x)
{
    return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// Largest |value| over the warp's lanes (each passes its own maximum).
__device__ __forceinline__ float warp_amax(float a)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        a = fmaxf(a, __shfl_xor_sync(kFull, a, off));
    return a;
}

__device__ __forceinline__ float row_scale(float amax)
{
    return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
}

__device__ __forceinline__ float bf16_round(float x)
{
    return __bfloat162float(__float2bfloat16_rn(x));
}

// One warp stores the K row of head h: lane i rotates the pair (i, i + 32) with
// the table's factors, rounds both to BF16 and quantizes them with the row scale.
__device__ __forceinline__ void store_key_row_fp8(uint8_t *page, int h, int slot, const uint16_t *k, float2 cs,
                                                  int lane)
{
    const float x1 = __uint_as_float((uint32_t)k[lane] << 16);
    const float x2 = __uint_as_float((uint32_t)k[lane + kD / 2] << 16);
    float y1, y2;
    rope_rotate_pair(x1, x2, cs.x, cs.y, y1, y2);
    y1 = bf16_round(y1);
    y2 = bf16_round(y2);
    const float scale = row_scale(warp_amax(fmaxf(fabsf(y1), fabsf(y2))));
    uint8_t *unit = page + (size_t)h * kFp8Unit;
    uint8_t *row = unit + slot * kD;
    row[lane] = (uint8_t)e4m3_code(__fdiv_rn(y1, scale));
    row[lane + kD / 2] = (uint8_t)e4m3_code(__fdiv_rn(y2, scale));
    if (lane == 0)
        reinterpret_cast<float *>(unit + kFp8UnitCodes)[slot] = scale;
}

// One warp stores the V row of head h: lane i quantizes dims 2i, 2i+1.
__device__ __forceinline__ void store_value_row_fp8(uint8_t *page, int h, int slot, const uint16_t *v, int lane)
{
    const uint32_t w = reinterpret_cast<const uint32_t *>(v)[lane];
    const float v0 = bf16lo(w), v1 = bf16hi(w);
    const float scale = row_scale(warp_amax(fmaxf(fabsf(v0), fabsf(v1))));
    const uint32_t c = e4m3_code(__fdiv_rn(v0, scale)) | (e4m3_code(__fdiv_rn(v1, scale)) << 8);
    uint8_t *unit = page + (size_t)h * kFp8Unit;
    uint8_t *row = unit + (kPage + slot) * kD;
    reinterpret_cast<uint16_t *>(row)[lane] = (uint16_t)c;
    if (lane == 0)
        reinterpret_cast<float *>(unit + kFp8UnitCodes)[kPage + slot] = scale;
}

constexpr int kAppendThreads = kHkv * 32;  // one warp per KV head

// Decode append for FP8 pages: one CTA per sequence, warp h stores head h's K and
// V rows; then the 32 query rows are rotated in place (BF16, as the BF16 path).
__global__ void __launch_bounds__(kAppendThreads)
append_rope_fp8_kernel(uint8_t *__restrict__ slab, int num_pages, const uint16_t *__restrict__ k_new,
                       const uint16_t *__restrict__ v_new, uint16_t *__restrict__ q, const int32_t *__restrict__ bt,
                       int max_blocks, const int32_t *__restrict__ pos, int pos_offset,
                       const float2 *__restrict__ rope, int max_pos, int32_t *__restrict__ err)
{
    const int b = blockIdx.x;
    const int p = pos[b] + pos_offset;  // pos_offset -1: `pos` holds the lengths
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
    const float2 *rope_row = rope + (size_t)p * (kD / 2);
    store_key_row_fp8(page_base, h, slot, k_new + ((size_t)b * kHkv + h) * kD, rope_row[lane], lane);
    store_value_row_fp8(page_base, h, slot, v_new + ((size_t)b * kHkv + h) * kD, lane);
    if (!q)
        return;
    // query rows: 32 rows x 32 pairs, one pair per thread and pass
    for (int item = threadIdx.x; item < kHq * (kD / 2); item += kAppendThreads) {
        const int r = item / (kD / 2), i = item % (kD / 2);
        uint16_t *row = q + ((size_t)b * kHq + r) * kD;
        const float2 cs = rope_row[i];
        const float x1 = __uint_as_float((uint32_t)row[i] << 16);
        const float x2 = __uint_as_float((uint32_t)row[i + kD / 2] << 16);
        float y1, y2;
        rope_rotate_pair(x1, x2, cs.x, cs.y, y1, y2);
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
                          int start_pos, int T, const float2 *__restrict__ rope, int max_pos,
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
    const float2 cs = rope[(size_t)p * (kD / 2) + lane];
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

// Four E4M3 codes (one byte each of w) as two FP16x2 words (exact): bytes 0, 1 go
// to `lo` (byte 0 in its low half), bytes 2, 3 to `hi`.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Hardware approximations (PTX ex2.approx.ftz / rcp.approx.ftz): the softmax weights
// and the V-scale ratios tolerate their ~2 ulp error; ex2(-inf) = 0.
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// D = A(16x16, row) * B(16x8, col) + D, FP16 inputs, FP32 accumulate
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A(16x32, row) * B(32x8, col) + D, E4M3 inputs (products exact), FP32 accumulate
__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// E4M3 codes of (lo, hi), RNE, saturating; lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi)
{
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_value(uint32_t code)
{
    return __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3)));
}

// One (page, KV head) unit of an FP8 pool (2176 bytes) into a shared-memory stage.
__device__ __forceinline__ void tma_load_unit(void *dst, const CUtensorMap *map, uint64_t *bar, int head, int page,
                                              uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(head), "r"(page), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Per-page policy for FP8 pages.  Lane (gid = lane / 4, tig = lane % 4).
//  * QK^T on E4M3 tensor cores (m16n8k32): Q' = q * 2^(134-e) (|Q'| < 256) is
//    split once per unit into two E4M3 terms T1 = E4M3(Q'), T2 = E4M3(Q' - T1);
//    a BF16 value has 8 significant bits and E4M3 4, so T1 + T2 = Q' exactly
//    whenever |Q'| >= 2^-2 (smaller entries, below 2^-10 of the head's largest,
//    keep an absolute error under 2^-10).  The K codes are the A operand as
//    stored.  MMA h takes k positions 4tig+i / 16+4tig+i as dims 16tig+8h+i /
//    16tig+8h+4+i, so a lane's A fragments of a K row are its 16 code bytes
//    16tig..16tig+15 and its B fragments the same dims of head gid's terms.
//  * PV in FP16 (m16n8k16): in m-tile i the rows gid / gid+8 stand for dims
//    8gid+2i / 8gid+2i+1, so a lane needs dims 8gid..8gid+7 (8 bytes) of tokens
//    2tig, 2tig+1, 2tig+8, 2tig+9; the loads alternate token parity with tig (a
//    half-warp's 8-byte loads then hit 8 distinct bank pairs, two lanes each, the
//    least rows of 64 bytes allow), and byte permutes with lane-dependent
//    selectors pair two tokens' codes of one dim.
//  * V scales: O^T is kept in units of sref, the largest V row scale seen so far
//    by this warp, so P'' = p * scale_v / sref <= 1 fits FP16 with its rounding
//    relative to the unit's own magnitude, and the MMA accumulates straight into
//    O^T; when a page raises sref, O^T is rescaled with the softmax correction.
struct Fp8MmaWarp {
    uint32_t qt[2][4];  // E4M3 terms of Q' for head gid, dims 16tig..16tig+15 (4 bytes per word)
    float hf[2];        // 2^(e-134) * scale * log2(e) for heads 2tig, 2tig+1 (0 for padding heads)
    float o[4][4];      // O^T accumulators, in units of sref
    float m[2], l[2];
    float sref, sinv;   // largest V scale so far (warp-uniform) and its reciprocal
    uint32_t sel_lo, sel_hi;  // byte-permute selectors pairing tokens (2tig, 2tig+1) per dim
    int lane;

    __device__ __forceinline__ void init(const uint16_t *qg, float scale_log2, int lane_)
    {
        lane = lane_;
        const int gid = lane >> 2, tig = lane & 3;
        float qv[16];
        float amax = 0.f;
        if (gid < kGroup) {
            const uint4 *src = reinterpret_cast<const uint4 *>(qg + gid * kD + 16 * tig);
            const uint4 u0 = src[0], u1 = src[1];
            const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                qv[2 * i] = bf16lo(w[i]);
                qv[2 * i + 1] = bf16hi(w[i]);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
                amax = fmaxf(amax, fabsf(qv[i]));
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                qv[i] = 0.f;
        }
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
        // head exponent e: amax < 2^(e-126), so |Q'| = |q| * 2^(134-e) < 256
        const int e = min(max((int)((__float_as_uint(amax) >> 23) & 0xffu), 8), 254);
        const float norm = __uint_as_float((uint32_t)(261 - e) << 23);  // 2^(134-e)
        const float undo = __uint_as_float((uint32_t)(e - 7) << 23);    // 2^(e-134)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t t1 = 0, t2 = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float x0 = qv[4 * j + 2 * h] * norm, x1 = qv[4 * j + 2 * h + 1] * norm;
                const uint32_t c = e4m3x2_of(x0, x1);
                const uint32_t r = e4m3x2_of(x0 - e4m3_value(c & 0xffu), x1 - e4m3_value(c >> 8));
                t1 |= c << (16 * h);
                t2 |= r << (16 * h);
            }
            qt[0][j] = t1;
            qt[1][j] = t2;
        }
        const float hfac = gid < kGroup ? scale_log2 * undo : 0.f;
        hf[0] = __shfl_sync(kFull, hfac, 8 * tig);      // lanes 4h.. hold head h
        hf[1] = __shfl_sync(kFull, hfac, 8 * tig + 4);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int r = 0; r < 4; ++r)
                o[i][r] = 0.f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
        sref = 0.f;
        sinv = 0.f;
        // tokens are loaded in the order (2tig + par, 2tig + 1 - par), par = bit 0 of tig;
        // the selectors put token 2tig's code in the low byte of each pair either way
        const bool par = tig & 1;
        sel_lo = par ? 0x1504u : 0x5140u;  // codes of dims +0, +1 (or +4, +5)
        sel_hi = par ? 0x3726u : 0x7362u;  // codes of dims +2, +3 (or +6, +7)
    }

    // unit: the stage -- K code rows, V code rows (64 bytes each), K scales[16], V scales[16]
    __device__ __forceinline__ void page(const uint8_t *unit, int nvalid)
    {
        const uint8_t *codes = unit;
        const float *scales = reinterpret_cast<const float *>(unit + kFp8UnitCodes);
        const int gid = lane >> 2, tig = lane & 3;
        // ---- S^T[16 tokens][8 heads] = K_codes . (T1 + T2)^T
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const uint4 ka = *reinterpret_cast<const uint4 *>(codes + gid * kD + 16 * tig);
            const uint4 kb = *reinterpret_cast<const uint4 *>(codes + (gid + 8) * kD + 16 * tig);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                mma_e4m3(s, ka.x, kb.x, ka.y, kb.y, qt[t][0], qt[t][1]);
                mma_e4m3(s, ka.z, kb.z, ka.w, kb.w, qt[t][2], qt[t][3]);
            }
        }
        const float sk0 = scales[gid], sk1 = scales[gid + 8];
        float sv0 = scales[kPage + gid], sv1 = scales[kPage + gid + 8];
        float x[4] = {s[0] * (sk0 * hf[0]), s[1] * (sk0 * hf[1]), s[2] * (sk1 * hf[0]), s[3] * (sk1 * hf[1])};
        if (gid >= nvalid) {
            x[0] = x[1] = -INFINITY;
            sv0 = 0.f;
        }
        if (gid + 8 >= nvalid) {
            x[2] = x[3] = -INFINITY;
            sv1 = 0.f;
        }
        float pm0 = fmaxf(x[0], x[2]), pm1 = fmaxf(x[1], x[3]);
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
            pm0 = fmaxf(pm0, __shfl_xor_sync(kFull, pm0, off));
            pm1 = fmaxf(pm1, __shfl_xor_sync(kFull, pm1, off));
        }
        // raise sref when a V scale of this page exceeds it (rare after the first pages)
        float grow = 1.f;
        if (__any_sync(kFull, fmaxf(sv0, sv1) > sref)) {
            float smax = fmaxf(sv0, sv1);
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1)
                smax = fmaxf(smax, __shfl_xor_sync(kFull, smax, off));
            const float inv = rcp_approx(smax);
            grow = sref * inv;  // 0 on the first page
            sref = smax;
            sinv = inv;
        }
        const float mn0 = fmaxf(m[0], pm0), mn1 = fmaxf(m[1], pm1);
        const float al0 = ex2_approx(m[0] - mn0), al1 = ex2_approx(m[1] - mn1);
        const float p0 = ex2_approx(x[0] - mn0), p1 = ex2_approx(x[1] - mn1);
        const float p2 = ex2_approx(x[2] - mn0), p3 = ex2_approx(x[3] - mn1);
        l[0] = fmaf(l[0], al0, p0 + p2);
        l[1] = fmaf(l[1], al1, p1 + p3);
        m[0] = mn0;
        m[1] = mn1;
        // ---- P''^T as the B operand (FP16): p * scale_v / sref, transposed
        const float r0 = sv0 * sinv, r1 = sv1 * sinv;
        const uint32_t b0 = movmatrix_trans(pack_f16x2(p0 * r0, p1 * r0));  // tokens 2tig, 2tig+1 ; head gid
        const uint32_t b1 = movmatrix_trans(pack_f16x2(p2 * r1, p3 * r1));  // tokens 2tig+8, 2tig+9
        const float c0 = al0 * grow, c1 = al1 * grow;
        if (__any_sync(kFull, c0 != 1.f || c1 != 1.f)) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o[i][0] *= c0;
                o[i][1] *= c1;
                o[i][2] *= c0;
                o[i][3] *= c1;
            }
        }
        // ---- V code rows: dims 8gid..8gid+7 of tokens 2tig(+1), 2tig+8(+1)
        const uint8_t *vt = codes + kFp8Tile;
        const int par = tig & 1;
        const uint32_t col = (uint32_t)(8 * gid);
        const uint2 u0 = *reinterpret_cast<const uint2 *>(vt + (2 * tig + par) * kD + col);
        const uint2 u1 = *reinterpret_cast<const uint2 *>(vt + (2 * tig + 1 - par) * kD + col);
        const uint2 u2 = *reinterpret_cast<const uint2 *>(vt + (2 * tig + 8 + par) * kD + col);
        const uint2 u3 = *reinterpret_cast<const uint2 *>(vt + (2 * tig + 9 - par) * kD + col);
        uint32_t a[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t sel = (i & 1) ? sel_hi : sel_lo;
            const uint32_t lo = __byte_perm(i < 2 ? u0.x : u0.y, i < 2 ? u1.x : u1.y, sel);
            const uint32_t hi = __byte_perm(i < 2 ? u2.x : u2.y, i < 2 ? u3.x : u3.y, sel);
            e4m3x4_to_f16x2(lo, a[i][0], a[i][1]);  // dim 8gid+2i | 8gid+2i+1, tokens 2tig, 2tig+1
            e4m3x4_to_f16x2(hi, a[i][2], a[i][3]);  // same dims, tokens 2tig+8, 2tig+9
        }
        if (nvalid < kPage) {  // zero V of slots past the sequence end (their bytes are arbitrary)
            const uint32_t mlo =
                (2 * tig < nvalid ? 0x0000ffffu : 0u) | (2 * tig + 1 < nvalid ? 0xffff0000u : 0u);
            const uint32_t mhi =
                (2 * tig + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * tig + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i][0] &= mlo;
                a[i][1] &= mlo;
                a[i][2] &= mhi;
                a[i][3] &= mhi;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            mma_f16(o[i], a[i], b0, b1);
    }

    // m[4], l[4] (log2 domain) and o[4][64] (true units), the layout of the BF16 policies
    __device__ __forceinline__ void store_state(float *dst)
    {
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
            l[0] += __shfl_xor_sync(kFull, l[0], off);
            l[1] += __shfl_xor_sync(kFull, l[1], off);
        }
        const int gid = lane >> 2, tig = lane & 3;
        if (tig < 2) {
            if (gid == 0) {
                dst[2 * tig] = m[0];
                dst[2 * tig + 1] = m[1];
                dst[4 + 2 * tig] = l[0];
                dst[4 + 2 * tig + 1] = l[1];
            }
            float *h0 = dst + 8 + (2 * tig) * kD + 8 * gid;  // head 2tig, dims 8gid..8gid+7
            float *h1 = h0 + kD;                             // head 2tig+1
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                *reinterpret_cast<float2 *>(h0 + 2 * i) = make_float2(o[i][0] * sref, o[i][2] * sref);
                *reinterpret_cast<float2 *>(h1 + 2 * i) = make_float2(o[i][1] * sref, o[i][3] * sref);
            }
        }
    }
};

template <int STAGES>
struct Fp8Smem {
    static constexpr int kStagesBytes = kWarps * STAGES * kFp8Unit;
    static constexpr int kBarsBytes = kWarps * STAGES * 8;
    static constexpr int kBytes = 128 + kStagesBytes + kBarsBytes;  // incl. alignment slack
    static_assert(kStagesBytes >= kWarps * kStateFloats * 4, "the combine reuses the stages");
    uint8_t *stages;
    uint64_t *bars;

    __device__ __forceinline__ explicit Fp8Smem(uint8_t *raw)
    {
        uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 127) & ~uintptr_t(127));
        stages = base;
        bars = reinterpret_cast<uint64_t *>(base + kStagesBytes);
    }
};

// One stage: the (page, KV head) unit by one TMA copy, completing on `bar`.
__device__ __forceinline__ void fp8_issue(const CUtensorMap *map, uint8_t *stage, uint64_t *bar, int g, int page,
                                          uint64_t policy)
{
    mbar_arrive_expect_tx(bar, kFp8Unit);
    tma_load_unit(stage, map, bar, g, page, policy);
}

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
                    const int32_t *bt, int max_blocks, const int32_t *pos, int pos_offset, int B, const float *rope,
                    int max_pos, int32_t *err, cudaStream_t s)
{
    append_rope_fp8_kernel<<<B, kAppendThreads, 0, s>>>(reinterpret_cast<uint8_t *>(pool->slab), pool->num_pages,
                                                        k_new, v_new, q, bt, max_blocks, pos, pos_offset,
                                                        reinterpret_cast<const float2 *>(rope), max_pos, err);
    return status_from_cuda(cudaGetLastError());
}

int fp8_prefill_append(const pkv_pool *pool, const uint16_t *k, const uint16_t *v, const int32_t *bt_rows,
                       int max_blocks, int layers, int start_pos, int T, const float *rope, int max_pos,
                       int32_t *err, cudaStream_t s)
{
    prefill_append_fp8_kernel<<<dim3(T, layers), kPrefillThreads, 0, s>>>(
        reinterpret_cast<uint8_t *>(pool->slab), pool->num_pages, k, v, bt_rows, max_blocks, start_pos, T,
        reinterpret_cast<const float2 *>(rope), max_pos, err);
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
    static bool attr_set = false;  // set once per process (before any graph capture)
    if (!attr_set) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return PKV_ERR_CUDA;
        attr_set = true;
    }
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
