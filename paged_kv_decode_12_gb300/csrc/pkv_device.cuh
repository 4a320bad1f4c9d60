// pkv_device.cuh -- device building blocks shared by the decode kernels (not part of the ABI):
// PTX wrappers (mbarrier, TMA, ldmatrix, movmatrix, warp MMA), the 128-byte swizzle
// of TMA-staged (page, KV head) tiles, the two per-page compute policies, the page
// streaming loop and the combine of the warps' online-softmax states.
#pragma once

#include <cuda_bf16.h>

#include "pkv_internal.h"

namespace pkv {
namespace dev {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileBytes = kPage * kD * 2;   // one (page, KV head) K tile: 2 KiB
constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
constexpr int kStateFloats = 8 + kGroup * kD;  // m[4], l[4], o[4][64] per warp
constexpr int kScratchFloats = 72;           // per-warp p[16][4] + alpha[4], padded
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr unsigned kFull = 0xffffffffu;

static_assert(kThreads == kGroup * 32, "combine maps one thread per (head, dim pair)");

// ------------------------------------------------------------------ PTX helpers

// Programmatic dependent launch: wait until every earlier grid this one depends on
// has completed and its memory is visible; let the next grid on the stream launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;" ::); }

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Warp-uniform bounded wait: true once every lane has observed the phase; false
// after `limit` polls.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, uint32_t limit = kWaitLimit)
{
    for (uint32_t i = 0; i < limit; ++i)
        if (__all_sync(kFull, mbar_try_wait(bar, parity)))
            return true;
    return false;
}

// Hardware approximations (PTX ex2.approx.ftz / rcp.approx.ftz): the softmax weights and
// the FP8 V-scale ratios tolerate their ~2 ulp error; ex2(-inf) = 0.
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

__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// One (page, KV head): 16 K rows then 16 V rows of 128 B, 128-byte swizzled.
__device__ __forceinline__ void tma_load_page_head(void *dst, const CUtensorMap *map, uint64_t *bar, int head,
                                                   int page, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(head), "r"(0), "r"(page), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` in a 128-byte
// swizzled tile (the TMA SWIZZLE_128B pattern on a 1024-byte aligned buffer).
__device__ __forceinline__ uint32_t swz(int row, int chunk)
{
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// a c + b s for BF16-valued a, b and factors held as FP32 pairs c = ch + cl, s = sh + sl
// (about 48 bits each).  a ch and b sh have at most 8 + 24 significant bits, so each is
// split exactly into an FP32 product and its FMA remainder; the two leading products
// are added exactly (two-sum) and everything below them goes into one correction term.
// The FP32 result is within one rounding of the exact value plus a few units of
// 2^-48 max(|a|, |b|): even where a c and b s nearly cancel it rounds to the same BF16
// as the exact rotation, except within that distance of a rounding boundary.  The
// intrinsics keep the compiler from contracting the products into other FMAs.
__device__ __forceinline__ float rope_comb(float a, float b, float ch, float cl, float sh, float sl)
{
    const float p = __fmul_rn(a, ch), pe = __fmaf_rn(a, ch, -p);
    const float r = __fmul_rn(b, sh), re = __fmaf_rn(b, sh, -r);
    const float t = __fadd_rn(p, r), bb = __fsub_rn(t, p);
    const float e = __fadd_rn(__fsub_rn(p, __fsub_rn(t, bb)), __fsub_rn(r, bb));
    const float lo = __fadd_rn(__fadd_rn(pe, re), __fmaf_rn(a, cl, __fmul_rn(b, sl)));
    return __fadd_rn(t, __fadd_rn(e, lo));
}

// Rotary embedding of one (i, i + 32) pair by the table entry {cos_hi, sin_hi, cos_lo,
// sin_lo} of its (position, i): y1 = x1 c - x2 s, y2 = x2 c + x1 s.  Every kernel that
// rotates uses this one function, so the append kernels and the fused step kernel round
// identically.
__device__ __forceinline__ void rope_rotate_pair(float x1, float x2, float4 cs, float &y1, float &y2)
{
    y1 = rope_comb(x1, -x2, cs.x, cs.z, cs.y, cs.w);
    y2 = rope_comb(x2, x1, cs.x, cs.z, cs.y, cs.w);
}

// ------------------------------------------------------------------ SIMT policy

struct SimtWarp {
    float qf[kGroup][8];  // q[h][8*dg .. 8*dg+7] * scale * log2(e)
    float acc[kGroup][2]; // o[h][2*lane], o[h][2*lane+1]
    float m[2], l[2];     // heads h0 = 2*(lane&1), h0+1; l is a per-lane partial sum
    float *ps;            // per-warp scratch: p[16 tokens][4 heads], alpha[4]
    int lane;

    __device__ __forceinline__ void init(const uint16_t *qg, float scale_log2, int lane_, float *scratch)
    {
        lane = lane_;
        ps = scratch;
        const int dg = lane & 7;
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
            const uint4 v = *reinterpret_cast<const uint4 *>(qg + h * kD + 8 * dg);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qf[h][2 * i] = bf16lo(w[i]) * scale_log2;
                qf[h][2 * i + 1] = bf16hi(w[i]) * scale_log2;
            }
            acc[h][0] = acc[h][1] = 0.f;
        }
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
    }

    __device__ __forceinline__ void page(const uint8_t *st, int nvalid)
    {
        const int dg = lane & 7, tg = lane >> 3;
        // ---- partial dot products: tokens 4tg..4tg+3, dims 8dg..8dg+7, 4 heads
        float v[16];  // index i*4 + h
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = 4 * tg + i;
            const uint4 kw = *reinterpret_cast<const uint4 *>(st + swz(t, dg));
            const uint32_t w[4] = {kw.x, kw.y, kw.z, kw.w};
            float k[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                k[2 * j] = bf16lo(w[j]);
                k[2 * j + 1] = bf16hi(w[j]);
            }
#pragma unroll
            for (int h = 0; h < kGroup; ++h) {
                float s = qf[h][0] * k[0];
#pragma unroll
                for (int j = 1; j < 8; ++j)
                    s = fmaf(qf[h][j], k[j], s);
                v[i * 4 + h] = s;
            }
        }
        // ---- reduce-scatter over the 8 lanes of a token group (lane bits 0..2)
        const bool b2 = lane & 4, b1 = lane & 2, b0 = lane & 1;
        float u[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float send = b2 ? v[k] : v[k + 8];
            const float keep = b2 ? v[k + 8] : v[k];
            u[k] = keep + __shfl_xor_sync(kFull, send, 4);
        }
        float w4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float send = b1 ? u[k] : u[k + 4];
            const float keep = b1 ? u[k + 4] : u[k];
            w4[k] = keep + __shfl_xor_sync(kFull, send, 2);
        }
        float s[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float send = b0 ? w4[k] : w4[k + 2];
            const float keep = b0 ? w4[k + 2] : w4[k];
            s[k] = keep + __shfl_xor_sync(kFull, send, 1);
        }
        // this lane now holds token t = 4tg + 2*b2 + b1, heads h0 = 2*b0 and h0+1
        const int t = 4 * tg + (b2 ? 2 : 0) + (b1 ? 1 : 0);
        const int h0 = b0 ? 2 : 0;
        if (t >= nvalid)
            s[0] = s[1] = -INFINITY;
        // ---- online softmax update (log2 domain)
        float pm0 = s[0], pm1 = s[1];
#pragma unroll
        for (int off = 2; off <= 16; off <<= 1) {
            pm0 = fmaxf(pm0, __shfl_xor_sync(kFull, pm0, off));
            pm1 = fmaxf(pm1, __shfl_xor_sync(kFull, pm1, off));
        }
        const float mn0 = fmaxf(m[0], pm0), mn1 = fmaxf(m[1], pm1);
        const float al0 = exp2f(m[0] - mn0), al1 = exp2f(m[1] - mn1);
        const float p0 = exp2f(s[0] - mn0), p1 = exp2f(s[1] - mn1);
        l[0] = fmaf(l[0], al0, p0);
        l[1] = fmaf(l[1], al1, p1);
        m[0] = mn0;
        m[1] = mn1;
        *reinterpret_cast<float2 *>(ps + t * 4 + h0) = make_float2(p0, p1);
        if ((lane >> 1) == 0)
            *reinterpret_cast<float2 *>(ps + 64 + h0) = make_float2(al0, al1);
        __syncwarp();
        // ---- o = alpha * o + sum_t p_t v_t, lane owns dims 2*lane, 2*lane+1
        const float4 al = *reinterpret_cast<const float4 *>(ps + 64);
        acc[0][0] *= al.x; acc[0][1] *= al.x;
        acc[1][0] *= al.y; acc[1][1] *= al.y;
        acc[2][0] *= al.z; acc[2][1] *= al.z;
        acc[3][0] *= al.w; acc[3][1] *= al.w;
        const uint8_t *vt = st + kTileBytes;
        const uint32_t col = (uint32_t)((lane & 3) << 2);
        if (nvalid == kPage) {
#pragma unroll
            for (int tt = 0; tt < kPage; ++tt)
                pv_token(vt, tt, col);
        } else {
            for (int tt = 0; tt < nvalid; ++tt)
                pv_token(vt, tt, col);
        }
        __syncwarp();
    }

    __device__ __forceinline__ void pv_token(const uint8_t *vt, int tt, uint32_t col)
    {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(vt + swz(tt, lane >> 2) + col);
        const float v0 = bf16lo(w), v1 = bf16hi(w);
        const float4 p = *reinterpret_cast<const float4 *>(ps + tt * 4);
        acc[0][0] = fmaf(p.x, v0, acc[0][0]); acc[0][1] = fmaf(p.x, v1, acc[0][1]);
        acc[1][0] = fmaf(p.y, v0, acc[1][0]); acc[1][1] = fmaf(p.y, v1, acc[1][1]);
        acc[2][0] = fmaf(p.z, v0, acc[2][0]); acc[2][1] = fmaf(p.z, v1, acc[2][1]);
        acc[3][0] = fmaf(p.w, v0, acc[3][0]); acc[3][1] = fmaf(p.w, v1, acc[3][1]);
    }

    // write m[4], l[4] (log2 domain) and o[4][64] of this warp
    __device__ __forceinline__ void store_state(float *dst)
    {
#pragma unroll
        for (int off = 2; off <= 16; off <<= 1) {
            l[0] += __shfl_xor_sync(kFull, l[0], off);
            l[1] += __shfl_xor_sync(kFull, l[1], off);
        }
        if ((lane >> 1) == 0) {
            const int h0 = (lane & 1) ? 2 : 0;
            dst[h0] = m[0];
            dst[h0 + 1] = m[1];
            dst[4 + h0] = l[0];
            dst[4 + h0 + 1] = l[1];
        }
#pragma unroll
        for (int h = 0; h < kGroup; ++h)
            *reinterpret_cast<float2 *>(dst + 8 + h * kD + 2 * lane) = make_float2(acc[h][0], acc[h][1]);
    }
};

// ------------------------------------------------------------------ MMA policy

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// D = A(16x16, row) * B(16x8, col) + D, BF16 inputs, FP32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct MmaWarp {
    uint32_t qb[4][2];  // B fragments of Q^T for the 4 k-steps (dims 16ks..16ks+15)
    float o[4][4];      // O^T accumulators, m-tile mt = dims 16mt..16mt+15
    float m[2], l[2];   // heads 2*tig + e (meaningful in lanes with tig < 2)
    float c;            // scale * log2(e)
    int lane;

    __device__ __forceinline__ void init(const uint16_t *qg, float scale_log2, int lane_, float *)
    {
        lane = lane_;
        c = scale_log2;
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            if (gid < kGroup) {
                const uint16_t *row = qg + gid * kD + 16 * ks + 2 * tig;
                qb[ks][0] = *reinterpret_cast<const uint32_t *>(row);
                qb[ks][1] = *reinterpret_cast<const uint32_t *>(row + 8);
            } else {
                qb[ks][0] = qb[ks][1] = 0u;
            }
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[mt][i] = 0.f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
    }

    __device__ __forceinline__ void page(const uint8_t *st, int nvalid)
    {
        const int gid = lane >> 2, tig = lane & 3;
        const uint32_t kbase = smem_addr(st);
        const uint32_t vbase = kbase + kTileBytes;
        // ---- S^T[16 tokens][8 heads] = K . Q^T, the even and the odd k-steps in two
        // accumulators (two MMA chains of two instead of one of four), added at the end
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int mi = lane >> 3, r = lane & 7;
            const int tok = r + ((mi & 1) ? 8 : 0);
            float s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 4; ks += 2) {
                uint32_t a0[4], a1[4];
                ldsm_x4(kbase + swz(tok, 2 * ks + (mi >> 1)), a0);
                ldsm_x4(kbase + swz(tok, 2 * (ks + 1) + (mi >> 1)), a1);
                mma_bf16(s, a0, qb[ks][0], qb[ks][1]);
                mma_bf16(s1, a1, qb[ks + 1][0], qb[ks + 1][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                s[i] += s1[i];
        }
        // s[0], s[1]: token gid, heads 2tig, 2tig+1; s[2], s[3]: token gid+8
        float x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            x[i] = s[i] * c;
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
        const float al0 = ex2_approx(m[0] - mn0), al1 = ex2_approx(m[1] - mn1);
        const float p0 = ex2_approx(x[0] - mn0), p1 = ex2_approx(x[1] - mn1);
        const float p2 = ex2_approx(x[2] - mn0), p3 = ex2_approx(x[3] - mn1);
        l[0] = fmaf(l[0], al0, p0 + p2);
        l[1] = fmaf(l[1], al1, p1 + p3);
        m[0] = mn0;
        m[1] = mn1;
        // ---- P^T as the B operand: transpose the two 8x8 BF16 blocks
        const uint32_t b0 = movmatrix_trans(pack_bf16x2(p0, p1));  // tokens 2tig, 2tig+1 ; head gid
        const uint32_t b1 = movmatrix_trans(pack_bf16x2(p2, p3));  // tokens 2tig+8, 2tig+9
        // ---- O^T = alpha * O^T + V^T . P^T
        const int mi = lane >> 3, r = lane & 7;
        const int tok = r + ((mi >> 1) ? 8 : 0);
        const bool partial = nvalid < kPage;
        // token masks of this lane's A-fragment halves: a0/a1 tokens 2tig, 2tig+1; a2/a3 +8
        const uint32_t mlo = (2 * tig < nvalid ? 0x0000ffffu : 0u) | (2 * tig + 1 < nvalid ? 0xffff0000u : 0u);
        const uint32_t mhi =
            (2 * tig + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * tig + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(vbase + swz(tok, 2 * mt + (mi & 1)), a);
            if (partial) {  // zero V of slots past the sequence end (their bytes are arbitrary)
                a[0] &= mlo;
                a[1] &= mlo;
                a[2] &= mhi;
                a[3] &= mhi;
            }
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
            mma_bf16(o[mt], a, b0, b1);
        }
    }

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
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                float *h0 = dst + 8 + (2 * tig) * kD + 16 * mt + gid;
                float *h1 = h0 + kD;
                h0[0] = o[mt][0];
                h1[0] = o[mt][1];
                h0[8] = o[mt][2];
                h1[8] = o[mt][3];
            }
        }
    }
};



// ------------------------------------------------------------------ page streaming

// Shared-memory carve-up of a decode CTA: STAGES 4 KiB stages per warp (1024-byte
// aligned for the 128-byte swizzle), one mbarrier per stage, per-warp scratch.
template <int STAGES>
struct SmemLayout {
    static constexpr int kStagesBytes = kWarps * STAGES * kStageBytes;
    static constexpr int kBarsBytes = kWarps * STAGES * 8;
    static constexpr int kScratchBytes = kWarps * kScratchFloats * 4;
    static constexpr int kBaseBytes = 1024 + kStagesBytes + kBarsBytes + kScratchBytes;  // incl. alignment slack
    uint8_t *stages;
    uint64_t *bars;
    float *scratch;
    uint8_t *extra;  // first byte after the base layout (16-byte aligned)

    __device__ __forceinline__ explicit SmemLayout(uint8_t *raw)
    {
        uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
        stages = base;
        bars = reinterpret_cast<uint64_t *>(base + kStagesBytes);
        scratch = reinterpret_cast<float *>(base + kStagesBytes + kBarsBytes);
        extra = base + kStagesBytes + kBarsBytes + kScratchBytes;
    }
};

// Lane 0 initialises this warp's stage barriers.
template <int STAGES>
__device__ __forceinline__ void init_warp_barriers(uint64_t *my_bars, int lane)
{
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s)
            mbar_init(&my_bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
}

// Issue the (page, KV head) copies k0 .. k1-1 of this warp into ring stages k0 ..
// k1-1 (k1 <= STAGES).  Lane k of the warp holds the physical id of the warp's k-th
// page in `my_page`; k0 and k1 are warp-uniform.
template <int STAGES>
__device__ __forceinline__ void issue_copies(const CUtensorMap *tmap, uint8_t *my_stages, uint64_t *my_bars,
                                             int my_page, int k0, int k1, int g, int lane, uint64_t policy)
{
    for (int k = k0; k < k1; ++k) {
        const int pk = __shfl_sync(kFull, my_page, k);
        if (lane == 0) {
            mbar_arrive_expect_tx(&my_bars[k], kStageBytes);
            tma_load_page_head(my_stages + k * kStageBytes, tmap, &my_bars[k], g, pk, policy);
        }
    }
}

// Issue the first min(STAGES, nmine) copies of this warp.
template <int STAGES>
__device__ __forceinline__ void issue_prologue(const CUtensorMap *tmap, uint8_t *my_stages, uint64_t *my_bars,
                                               int my_page, int nmine, int g, int lane, uint64_t policy)
{
    issue_copies<STAGES>(tmap, my_stages, my_bars, my_page, 0, min(STAGES, nmine), g, lane, policy);
}

// How many of a warp's first min(stages, nmine) pages (pages j0 + warp + 4k of the
// sequence) hold only positions below L - 2.  A decode launch may copy those before
// its dependency wait: the previous decode step of the same layer wrote position
// L - 2 and the append of this step (fused or a separate kernel just before) writes
// L - 1, so the pages holding either are copied only after the wait.
__device__ __forceinline__ int copies_before_wait(int L, int j0, int warp, int nmine, int stages)
{
    const int jsafe = max(L - 2, 0) / kPage;  // first page holding position L - 2 or later
    const int n = jsafe > j0 + warp ? (jsafe - j0 - warp + kWarps - 1) / kWarps : 0;
    return min(n, min(stages, nmine));
}

struct NoPatch {
    __device__ __forceinline__ void operator()(uint8_t *, int) const {}
};

// Consume this warp's pages j0 + warp + k*kWarps (k < nmine): wait for the stage,
// let `patch(stage, j)` edit it, run the policy's page update, refill the stage
// with page k + STAGES.  Returns false if a bounded wait gave up (after giving
// the copies still in flight a bounded chance to land).  The first wait polls at
// most `first_limit` times (a testing aid can make it give up at once); the others,
// and the drain of copies in flight, kWaitLimit times.
template <int STAGES, class Warp, class Patch>
__device__ __forceinline__ bool consume_pages(const CUtensorMap *tmap, uint8_t *my_stages, uint64_t *my_bars, Warp &w,
                                              int my_page, int nmine, int j0, int warp, int lane, int L, int g,
                                              uint64_t policy, const Patch &patch, uint32_t first_limit = kWaitLimit)
{
    int k = 0;
    for (; k < nmine; ++k) {
        const int s = k % STAGES;
        if (!mbar_wait_warp(&my_bars[s], (uint32_t)((k / STAGES) & 1), k == 0 ? first_limit : kWaitLimit))
            break;
        const int j = j0 + warp + k * kWarps;
        uint8_t *stage = my_stages + s * kStageBytes;
        patch(stage, j);
        w.page(stage, min(kPage, L - j * kPage));
        __syncwarp();
        if (k + STAGES < nmine) {
            const int pk = __shfl_sync(kFull, my_page, k + STAGES);
            if (lane == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&my_bars[s], kStageBytes);
                tma_load_page_head(stage, tmap, &my_bars[s], g, pk, policy);
            }
        }
    }
    if (k < nmine) {
        for (int kk = k; kk < min(nmine, k + STAGES); ++kk)
            (void)mbar_wait_warp(&my_bars[kk % STAGES], (uint32_t)((kk / STAGES) & 1));
        return false;
    }
    return true;
}

// Combine the kWarps warps' (m, l, o) states stored at `state` (kStateFloats per
// warp) for query head hl of the group and output dims 2dp, 2dp+1.
__device__ __forceinline__ void combine_warps(const float *state, int hl, int dp, float &M, float &lsum, float &o0,
                                              float &o1)
{
    M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww)
        M = fmaxf(M, state[ww * kStateFloats + hl]);
    lsum = 0.f;
    o0 = 0.f;
    o1 = 0.f;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) {
        const float mw = state[ww * kStateFloats + hl];
        const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        lsum = fmaf(f, state[ww * kStateFloats + 4 + hl], lsum);
        const float2 ow = *reinterpret_cast<const float2 *>(state + ww * kStateFloats + 8 + hl * kD + 2 * dp);
        o0 = fmaf(f, ow.x, o0);
        o1 = fmaf(f, ow.y, o1);
    }
}

// Normalised BF16 pair, zeros when nothing was accumulated.
__device__ __forceinline__ uint32_t finish_pair(float o0, float o1, float lsum)
{
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    return pack_bf16x2(o0 * inv, o1 * inv);
}

}  // namespace dev
}  // namespace pkv
