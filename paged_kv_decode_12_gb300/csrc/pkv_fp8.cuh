// pkv_fp8.cuh -- device building blocks for FP8 E4M3 KV pages, shared by the split
// decode kernel (pkv_fp8.cu) and the fused step kernel (pkv_step.cu): quantization of
// a row, E4M3 -> FP16 conversion, the E4M3 / FP16 warp MMAs, the unit copy, and the
// per-page compute policy Fp8MmaWarp.  Not part of the ABI.
//
// Page format (a reading of "从零构建大模型推理引擎：KV缓存、算子融合与量化优化实战",
// section 5.1, which asks only for a low-precision cache dequantized before attention):
// 8 units of 2176 bytes per page, one per KV head: K code rows [16][64], V code rows
// [16][64] (E4M3, one byte each), K row scales [16], V row scales [16] (FP32); a row x
// is stored as scale = amax|x| / 448 (1 for an all-zero row), codes E4M3_rne_sat(x / scale).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pkv_device.cuh"

namespace pkv {
namespace fp8 {

using namespace dev;

constexpr int kFp8Tile = kPage * kD;  // 1 KiB: one (page, KV head) K or V code tile
constexpr float kDeferLog2 = 8.f;      // softmax reference moves when a score exceeds it by 2^8
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

// Byte offset, inside a unit's V code tile, of the code of (slot, dim): slots 2p and 2p+1
// share a 128-byte line; dims 8c..8c+7 of both form 16-byte chunk c (byte 2 (dim % 8) +
// slot % 2), stored at chunk position c ^ (2p % 8), so that the decode's 16-byte reads of
// one chunk by the lanes of a quarter warp fall in distinct bank groups.
__device__ __forceinline__ int v_code_offset(int slot, int dim)
{
    const int pair = slot >> 1;
    return pair * 2 * kD + (((dim >> 3) ^ ((2 * pair) & 7)) << 4) + ((dim & 7) << 1) + (slot & 1);
}

// The row codes of one warp's BF16-valued pair (y1, y2) per lane (a row of 64 values
// held as lane i: values i and i + 32, or 2i and 2i + 1): the row scale and the two
// lanes' codes, with the arithmetic every FP8 writer uses.
__device__ __forceinline__ void quantize_pair(float y1, float y2, uint32_t &c1, uint32_t &c2, float &scale)
{
    scale = row_scale(warp_amax(fmaxf(fabsf(y1), fabsf(y2))));
    c1 = e4m3_code(__fdiv_rn(y1, scale));
    c2 = e4m3_code(__fdiv_rn(y2, scale));
}

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
        // Exponents relative to the reference maxima m (log2 domain).  m moves only when a
        // score exceeds it by more than kDeferLog2 -- then the page's maxima are reduced
        // across the warp and O^T, l are rescaled -- so most pages need no reduction and
        // the weights stay below 2^kDeferLog2 (m, l, o remain a valid log-sum-exp triple).
        const float skh00 = sk0 * hf[0], skh01 = sk0 * hf[1], skh10 = sk1 * hf[0], skh11 = sk1 * hf[1];
        float z[4] = {fmaf(s[0], skh00, -m[0]), fmaf(s[1], skh01, -m[1]), fmaf(s[2], skh10, -m[0]),
                      fmaf(s[3], skh11, -m[1])};
        if (gid >= nvalid) {
            z[0] = z[1] = -INFINITY;
            sv0 = 0.f;
        }
        if (gid + 8 >= nvalid) {
            z[2] = z[3] = -INFINITY;
            sv1 = 0.f;
        }
        float al0 = 1.f, al1 = 1.f;
        if (__any_sync(kFull, fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3])) > kDeferLog2)) {
            float x[4] = {s[0] * skh00, s[1] * skh01, s[2] * skh10, s[3] * skh11};
            if (gid >= nvalid)
                x[0] = x[1] = -INFINITY;
            if (gid + 8 >= nvalid)
                x[2] = x[3] = -INFINITY;
            float pm0 = fmaxf(x[0], x[2]), pm1 = fmaxf(x[1], x[3]);
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                pm0 = fmaxf(pm0, __shfl_xor_sync(kFull, pm0, off));
                pm1 = fmaxf(pm1, __shfl_xor_sync(kFull, pm1, off));
            }
            const float mn0 = fmaxf(m[0], pm0), mn1 = fmaxf(m[1], pm1);
            al0 = ex2_approx(m[0] - mn0);  // 0 on the first page (m = -inf)
            al1 = ex2_approx(m[1] - mn1);
            m[0] = mn0;
            m[1] = mn1;
            z[0] = x[0] - mn0;
            z[1] = x[1] - mn1;
            z[2] = x[2] - mn0;
            z[3] = x[3] - mn1;
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
        const float p0 = ex2_approx(z[0]), p1 = ex2_approx(z[1]);
        const float p2 = ex2_approx(z[2]), p3 = ex2_approx(z[3]);
        l[0] = fmaf(l[0], al0, p0 + p2);
        l[1] = fmaf(l[1], al1, p1 + p3);
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
        // ---- V codes: dims 8gid..8gid+7 of token pairs tig (2tig, 2tig+1) and tig+4
        // (2tig+8, 2tig+9), one 16-byte chunk each in the token-pair interleaved layout:
        // word i holds dims 8gid+2i, 8gid+2i+1 of both tokens, i.e. m-tile i's rows gid, gid+8
        const uint8_t *vt = codes + kFp8Tile;
        const uint32_t chunk = (uint32_t)((gid ^ (2 * tig)) << 4);
        const uint4 u0 = *reinterpret_cast<const uint4 *>(vt + tig * 2 * kD + chunk);
        const uint4 u1 = *reinterpret_cast<const uint4 *>(vt + (tig + 4) * 2 * kD + chunk);
        const uint32_t w0[4] = {u0.x, u0.y, u0.z, u0.w}, w1[4] = {u1.x, u1.y, u1.z, u1.w};
        uint32_t a[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            e4m3x4_to_f16x2(w0[i], a[i][0], a[i][1]);  // dim 8gid+2i | 8gid+2i+1, tokens 2tig, 2tig+1
            e4m3x4_to_f16x2(w1[i], a[i][2], a[i][3]);  // same dims, tokens 2tig+8, 2tig+9
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

}  // namespace fp8
}  // namespace pkv
