// pkv_step.cu -- the fused grid kernel of the decode path, one launch per layer.
//
// pkv_decode_step: RoPE + page-slot append of the new token, paged GQA decode
// attention over the sequence's pages, and the log-sum-exp merge of the chunk
// partials, in one launch.  It computes exactly what pkv_append_rope (positions =
// seq_lens - 1, q rotated in place) followed by pkv_decode_attention computes -- the
// samir-vllm README summary ("从零用 C++ 和 CUDA 实现 Llama 3.2 1B 推理引擎", section
// "目前已完成的功能") describes both steps: decode appends one token at its absolute
// RoPE position, then each query head streams its sequence's pages with an FP32
// online softmax -- with the same arithmetic, so the results are bit-identical to
// the two separate calls.  pkv_decode_attention runs the same kernel without the
// append (APPEND = false): the query rows are read as given and no page is written.
//
// Work unit = (sequence b, KV head g, chunk c of pages_per_chunk pages); one CTA per
// unit (grid = KV heads x B x chunks), optionally dispatched largest unit first.
// Per unit:
//  * the 4 query rows of group g are rotated to position L-1 by the unit itself;
//    the rotated rows are written back once, by the unit that finishes (b, g) last;
//  * the sequence's last chunk computes the new token's rotated key and its value,
//    stores them into their page slot in HBM and patches them into the
//    shared-memory copy of the last page, so no unit waits for an append kernel;
//  * chunk partials are merged in-kernel: each unit publishes its partial and
//    takes a ticket from a per-(b, g) counter (one release-acquire atomicAdd, no
//    waiting); the unit drawing the last ticket merges all chunks in chunk order
//    (deterministic) and resets the counter to zero for the next launch.
// Programmatic dependent launch: before griddepcontrol.wait a CTA reads only this
// step's lengths and block tables and starts the TMA copies of those of its pages
// that hold only positions below L - 2 (no kernel of this step or the previous one
// writes them: the previous step's append of this layer wrote position L - 2, this
// step's writes L - 1, and layers never share pages); the pages holding L - 2 or
// L - 1 are copied after the wait, q, k_new, v_new are read after it, and every
// output is written after it.  A CTA lets the next launch begin only after its own
// wait, so at most one earlier kernel can still be running while it copies early.
#include <cuda_bf16.h>

#include <climits>

#include "pkv_device.cuh"
#include "pkv_fp8.cuh"

namespace pkv {
namespace {

using namespace dev;

struct StepArgs {
    int num_pages;
    uint16_t *slab;
    const uint16_t *k_new;   // [B][8][64] (APPEND)
    const uint16_t *v_new;   // [B][8][64] (APPEND)
    uint16_t *q;             // [B][32][64], rotated in place (APPEND) or read as given
    const int32_t *bt;       // [B][max_blocks]
    int max_blocks;
    const int32_t *seq_lens; // [B]
    const float4 *rope;      // [max_pos][32] {cos, sin} high then low FP32 parts (APPEND)
    int max_pos;             // APPEND: rope rows; otherwise INT_MAX
    float scale_log2;
    int pages_per_chunk;
    int *counters;           // [B][8], zero between launches
    float2 *part_ml;         // [B][32][max_chunks]
    float *part_o;           // [B][32][max_chunks][64]
    int max_chunks;
    uint16_t *out;           // [B][32][64]
    int32_t *err;
    int sorted;              // units dispatched largest first (PKV_STEP_SORTED)
    int expire_seq;          // testing aid: this sequence's first page waits give up at once (-1: none)
};

constexpr int kMaxSortedBatch = 1024;
static_assert(kMaxPagesPerChunk + 1 + kWarps + 5 <= kWarps * kScratchFloats, "sorted-order scratch");

// Take a ticket: atomic increment with release and acquire semantics at GPU scope.
__device__ __forceinline__ int ticket_acq_rel(int *counter)
{
    int t;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(t) : "l"(counter) : "memory");
    return t;
}

__device__ __forceinline__ uint16_t bf16_bits(float x)
{
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<const uint16_t *>(&h);
}

__device__ __forceinline__ float bf16_value(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ bool length_ok(const StepArgs &a, int L)
{
    return L >= 1 && L <= a.max_blocks * kPage && L <= a.max_pos;
}

// ------------------------------------------------------------------ sorted unit order

// A sequence's work units per KV head: nfull chunks of pages_per_chunk pages and,
// if rem > 0, a last chunk of rem pages; an invalid length has one empty unit.
struct SeqUnits {
    int nfull, rem;
    bool valid;
};

__device__ __forceinline__ SeqUnits seq_units(const StepArgs &a, int L)
{
    SeqUnits u;
    u.valid = length_ok(a, L);
    if (!u.valid) {
        u.nfull = 0;
        u.rem = 0;
        return u;
    }
    const int ppc = a.pages_per_chunk;
    const int np = (L + kPage - 1) / kPage, nch = (np + ppc - 1) / ppc, rem = np - (nch - 1) * ppc;
    u.nfull = rem == ppc ? nch : nch - 1;
    u.rem = rem == ppc ? 0 : rem;
    return u;
}

// Units of size s of one sequence (s = pages_per_chunk: full chunks; 0 < s < pages_per_chunk:
// a last chunk; s = 0: the empty unit of an invalid length), all KV heads.
__device__ __forceinline__ int units_of_size(const SeqUnits &u, int s, int ppc)
{
    if (!u.valid)
        return s == 0 ? kHkv : 0;
    if (s == ppc)
        return kHkv * u.nfull;
    return (s != 0 && u.rem == s) ? kHkv : 0;
}

// Exclusive prefix sum over the CTA's kThreads threads; `total` receives the sum.
__device__ __forceinline__ int cta_exclusive_scan(int v, int *wsum, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(kFull, x, off);
        if (lane >= off)
            x += y;
    }
    if (lane == 31)
        wsum[warp] = x;
    __syncthreads();
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const int t = wsum[w];
        before += w < warp ? t : 0;
        total += t;
    }
    __syncthreads();
    return before + x - v;
}

// Sorted dispatch (PKV_STEP_SORTED): the CTA with linear index lin takes the lin-th
// unit in decreasing order of page count (ties by sequence, then chunk, then KV
// head).  The block scheduler places CTAs in index order on whichever SM has room,
// so the largest units are placed first and the small ones fill the gaps (greedy
// largest-first list scheduling), instead of the grid order's mix.  The order only
// decides which CTA computes which unit: every unit's arithmetic and the chunk-order
// merge are unchanged, so results are identical to the unsorted grid.  All threads
// call it (it uses barriers); `scratch` holds kMaxPagesPerChunk + 1 + kWarps + 5 ints.
// Returns false (for the whole CTA) if lin is past the last unit.
__device__ bool sorted_unit(const StepArgs &a, int B, int lin, int *scratch, int &b, int &g, int &c)
{
    constexpr int kPer = kMaxSortedBatch / kThreads;  // sequences per thread, at most
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ppc = a.pages_per_chunk;
    int *hist = scratch;                            // [ppc + 1] units per size
    int *wsum = scratch + kMaxPagesPerChunk + 1;    // [kWarps]
    int *res = wsum + kWarps;                       // size, rank, b, g, c
    for (int i = tid; i <= ppc; i += kThreads)
        hist[i] = 0;
    // this thread's contiguous run of sequences, read once (one memory round trip)
    const int per = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * per), nb = min(B, b0 + per) - b0;
    SeqUnits u[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        u[i] = seq_units(a, i < nb ? a.seq_lens[b0 + i] : 0);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        if (i >= nb)
            break;
        if (!u[i].valid) {
            atomicAdd(&hist[0], kHkv);
        } else {
            if (u[i].nfull)
                atomicAdd(&hist[ppc], kHkv * u[i].nfull);
            if (u[i].rem)
                atomicAdd(&hist[u[i].rem], kHkv);
        }
    }
    __syncthreads();
    if (warp == 0) {  // which size bucket holds rank lin, sizes in decreasing order
        constexpr int kBuckets = (kMaxPagesPerChunk + 1 + 31) / 32;
        int cnt[kBuckets];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < kBuckets; ++i) {
            const int k = lane * kBuckets + i;  // k-th largest size, ppc - k
            cnt[i] = k <= ppc ? hist[ppc - k] : 0;
            sum += cnt[i];
        }
        int x = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(kFull, x, off);
            if (lane >= off)
                x += y;
        }
        const int total = __shfl_sync(kFull, x, 31);
        int start = x - sum;
#pragma unroll
        for (int i = 0; i < kBuckets; ++i) {
            if (lin >= start && lin < start + cnt[i]) {
                res[0] = ppc - (lane * kBuckets + i);
                res[1] = lin - start;
            }
            start += cnt[i];
        }
        if (lane == 0 && lin >= total)
            res[0] = -1;
    }
    __syncthreads();
    const int s = res[0], r = res[1];
    if (s < 0)
        return false;
    int mine = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        mine += i < nb ? units_of_size(u[i], s, ppc) : 0;
    int total;
    const int before = cta_exclusive_scan(mine, wsum, total);
    if (r >= before && r < before + mine) {
        int acc = before;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int n = i < nb ? units_of_size(u[i], s, ppc) : 0;
            if (n > 0 && r >= acc && r < acc + n) {
                const int k = r - acc;
                res[2] = b0 + i;
                if (u[i].valid && s == ppc) {  // full chunks 0 .. nfull-1
                    res[3] = k % kHkv;
                    res[4] = k / kHkv;
                } else {                       // the last chunk, or the empty unit of an invalid length
                    res[3] = k;
                    res[4] = u[i].valid ? u[i].nfull : 0;
                }
            }
            acc += n;
        }
    }
    __syncthreads();
    b = res[2];
    g = res[3];
    c = res[4];
    return true;
}

__device__ __forceinline__ int chunks_of(const StepArgs &a, int L)
{
    return ((L + kPage - 1) / kPage + a.pages_per_chunk - 1) / a.pages_per_chunk;
}

// All kThreads threads: the 4 query rows of group g into q_rot[4][64] (one pair per
// thread) -- rotated to position pos (APPEND), else as given -- and, for the
// sequence's last chunk (APPEND), the new token's rotated key row and its value row
// into new_kv[2][64].
template <bool APPEND>
__device__ __forceinline__ void unit_rows(const StepArgs &a, int b, int g, int pos, bool last_chunk, uint16_t *q_rot,
                                          uint16_t *new_kv)
{
    const int hl = threadIdx.x >> 5, i = threadIdx.x & 31;
    const uint16_t *qrow = a.q + ((size_t)b * kHq + g * kGroup + hl) * kD;
    if (!APPEND) {
        reinterpret_cast<uint32_t *>(q_rot + hl * kD)[i] = reinterpret_cast<const uint32_t *>(qrow)[i];
        return;
    }
    const float4 cs = a.rope[(size_t)pos * (kD / 2) + i];
    float y1, y2;
    rope_rotate_pair(bf16_value(qrow[i]), bf16_value(qrow[i + kD / 2]), cs, y1, y2);
    q_rot[hl * kD + i] = bf16_bits(y1);
    q_rot[hl * kD + i + kD / 2] = bf16_bits(y2);
    if (last_chunk && hl == 0) {
        const uint16_t *krow = a.k_new + ((size_t)b * kHkv + g) * kD;
        rope_rotate_pair(bf16_value(krow[i]), bf16_value(krow[i + kD / 2]), cs, y1, y2);
        new_kv[i] = bf16_bits(y1);
        new_kv[i + kD / 2] = bf16_bits(y2);
    } else if (last_chunk && hl == 1) {
        reinterpret_cast<uint32_t *>(new_kv + kD)[i] =
            reinterpret_cast<const uint32_t *>(a.v_new + ((size_t)b * kHkv + g) * kD)[i];
    }
}

// Threads 0..15: the appended token's K row and V row into their page slot.
__device__ __forceinline__ void store_new_token(const StepArgs &a, int page, int g, int slot, const uint16_t *new_kv)
{
    const int part = threadIdx.x >> 3, ch = threadIdx.x & 7;  // part 0: K row, 1: V row
    uint16_t *row = a.slab + (size_t)page * kPageElems + ((size_t)(part * kHkv + g) * kPage + slot) * kD;
    reinterpret_cast<uint4 *>(row)[ch] = reinterpret_cast<const uint4 *>(new_kv + part * kD)[ch];
}

// The shared-memory copy of the last page carries the slot's previous contents:
// lanes 0..15 overwrite it with the appended token (then the warp syncs).
__device__ __forceinline__ void patch_stage(uint8_t *stage, int slot, const uint16_t *new_kv, int lane)
{
    if (lane < 16) {
        const int part = lane >> 3, ch = lane & 7;
        *reinterpret_cast<uint4 *>(stage + part * kTileBytes + swz(slot, ch)) =
            reinterpret_cast<const uint4 *>(new_kv + part * kD)[ch];
    }
    __syncwarp();
}

// Zeros for the 4 heads of an invalid sequence (one (head, dim pair) per thread).
__device__ __forceinline__ void write_zero_unit(const StepArgs &a, int b, int g)
{
    reinterpret_cast<uint32_t *>(a.out + ((size_t)b * kHq + g * kGroup + (threadIdx.x >> 5)) * kD)[threadIdx.x & 31] =
        0u;
    if (threadIdx.x == 0 && a.err)
        atomicOr(a.err, PKV_DEVERR_LENGTH);
}

// Chunk counts up to which the merging unit holds every partial in registers.
constexpr int kMergeRegs = 8;

// Unit epilogue, all threads: combine the warps' states through `state`, then
// write the output (single chunk) or publish the chunk partial and take a ticket;
// the unit drawing the last ticket merges every chunk of (b, g) in chunk order,
// writes the output (and, WRITE_Q, the rotated query rows), and resets the counter.
template <bool WRITE_Q, class Warp>
__device__ __forceinline__ void finish_unit(const StepArgs &a, Warp &w, float *state, int *ticket,
                                            const uint16_t *q_rot, int b, int g, int c, int nchunks)
{
    const int tid = threadIdx.x, warp = tid >> 5;
    __syncthreads();
    w.store_state(state + warp * kStateFloats);
    __syncthreads();
    const int hl = tid >> 5, dp = tid & 31, h = g * kGroup + hl;
    float M, lsum, o0, o1;
    combine_warps(state, hl, dp, M, lsum, o0, o1);
    uint32_t *out_row = reinterpret_cast<uint32_t *>(a.out + ((size_t)b * kHq + h) * kD);
    uint32_t *q_row = reinterpret_cast<uint32_t *>(a.q + ((size_t)b * kHq + h) * kD);
    const uint32_t q_word = reinterpret_cast<const uint32_t *>(q_rot + hl * kD)[dp];
    if (nchunks == 1) {
        out_row[dp] = finish_pair(o0, o1, lsum);
        if (WRITE_Q)
            q_row[dp] = q_word;
        return;
    }
    const size_t base = ((size_t)b * kHq + h) * a.max_chunks;
    reinterpret_cast<float2 *>(a.part_o + (base + c) * kD)[dp] = make_float2(o0, o1);
    if (dp == 0)
        a.part_ml[base + c] = make_float2(M, lsum);
    // publish: the CTA barrier orders every thread's partial stores before thread 0's
    // release-acquire ticket; the acquire side plus the barrier orders the merging
    // unit's loads after every other unit's partial stores
    __syncthreads();
    if (tid == 0)
        *ticket = ticket_acq_rel(&a.counters[b * kHkv + g]);
    __syncthreads();
    if (*ticket != nchunks - 1)
        return;
    float ls = 0.f, r0 = 0.f, r1 = 0.f;
    const float2 *ml_row = a.part_ml + base;
    const float2 *o_col = reinterpret_cast<const float2 *>(a.part_o + base * kD) + dp;
    if (nchunks <= kMergeRegs) {
        // every partial loaded before the first use: one memory round trip at the end of
        // the sequence's critical path; the arithmetic below is the general loop's
        float2 ml[kMergeRegs], oc[kMergeRegs];
#pragma unroll
        for (int cc = 0; cc < kMergeRegs; ++cc)
            if (cc < nchunks) {
                ml[cc] = __ldcg(ml_row + cc);
                oc[cc] = __ldcg(o_col + cc * (kD / 2));
            }
        float Mx = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < kMergeRegs; ++cc)
            if (cc < nchunks)
                Mx = fmaxf(Mx, ml[cc].x);
        if (Mx != -INFINITY) {
#pragma unroll
            for (int cc = 0; cc < kMergeRegs; ++cc)
                if (cc < nchunks) {
                    const float f = (ml[cc].x == -INFINITY) ? 0.f : exp2f(ml[cc].x - Mx);
                    ls = fmaf(f, ml[cc].y, ls);
                    r0 = fmaf(f, oc[cc].x, r0);
                    r1 = fmaf(f, oc[cc].y, r1);
                }
        }
    } else {
        float Mx = -INFINITY;
        for (int cc = 0; cc < nchunks; ++cc)
            Mx = fmaxf(Mx, __ldcg(ml_row + cc).x);
        if (Mx != -INFINITY) {
            for (int cc = 0; cc < nchunks; ++cc) {
                const float2 ml = __ldcg(ml_row + cc);
                const float f = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - Mx);
                const float2 oc = __ldcg(o_col + cc * (kD / 2));
                ls = fmaf(f, ml.y, ls);
                r0 = fmaf(f, oc.x, r0);
                r1 = fmaf(f, oc.y, r1);
            }
        }
    }
    out_row[dp] = finish_pair(r0, r1, ls);
    if (WRITE_Q)
        q_row[dp] = q_word;
    if (tid == 0)
        a.counters[b * kHkv + g] = 0;
}

// ------------------------------------------------------------------ timeline (PKV_TIMELINE builds)

#ifdef PKV_TIMELINE
// Per-CTA timeline of the grid schedule, compiled only into libraries built with
// -DPKV_TIMELINE: globaltimer stamps (ns) at entry, after the unit is known, after
// the dependency wait, after the page loop and at the end, and (SM, sequence, chunk,
// pages) per CTA linear index; CTAs without a unit store SM -1.  Every launch
// overwrites the records of its linear indices.
constexpr int kTimelineMax = 16384;
__device__ unsigned long long g_timeline_stamps[kTimelineMax * 5];
__device__ int g_timeline_meta[kTimelineMax * 4];

__device__ __forceinline__ unsigned long long timeline_now()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

struct Timeline {
    unsigned long long t[4];
    int lin;
    bool rec;
    __device__ __forceinline__ void begin()
    {
        t[0] = timeline_now();
        lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        rec = threadIdx.x == 0 && lin < kTimelineMax;
    }
    __device__ __forceinline__ void stamp(int i) { t[i] = timeline_now(); }
    __device__ __forceinline__ void none() const
    {
        if (rec)
            g_timeline_meta[lin * 4] = -1;
    }
    __device__ __forceinline__ void end(int b, int c, int pages) const
    {
        if (!rec)
            return;
        unsigned sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        for (int i = 0; i < 4; ++i)
            g_timeline_stamps[lin * 5 + i] = t[i];
        g_timeline_stamps[lin * 5 + 4] = timeline_now();
        g_timeline_meta[lin * 4 + 0] = (int)sm;
        g_timeline_meta[lin * 4 + 1] = b;
        g_timeline_meta[lin * 4 + 2] = c;
        g_timeline_meta[lin * 4 + 3] = pages;
    }
};
#else
struct Timeline {  // compiled out
    __device__ __forceinline__ void begin() {}
    __device__ __forceinline__ void stamp(int) {}
    __device__ __forceinline__ void none() const {}
    __device__ __forceinline__ void end(int, int, int) const {}
};
#endif

// ------------------------------------------------------------------ grid schedule

constexpr int kGridExtraBytes = kGroup * kD * 2 + 2 * kD * 2 + 16;  // rotated q rows, new K/V rows, ticket

template <class Warp, int STAGES, bool APPEND>
__global__ void __launch_bounds__(kThreads) decode_step_kernel(const __grid_constant__ CUtensorMap tmap, StepArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    SmemLayout<STAGES> sm(smem_raw);
    uint16_t *q_rot = reinterpret_cast<uint16_t *>(sm.extra);  // [4][64] query rows (rotated when APPEND)
    uint16_t *new_kv = q_rot + kGroup * kD;                     // [2][64] rotated key row, value row
    int *ticket = reinterpret_cast<int *>(new_kv + 2 * kD);
    Timeline tl;
    tl.begin();

    int g = blockIdx.x, b = blockIdx.y, c = blockIdx.z;
    if (a.sorted) {
        const int lin = blockIdx.x + kHkv * (blockIdx.y + gridDim.y * blockIdx.z);
        if (!sorted_unit(a, gridDim.y, lin, reinterpret_cast<int *>(sm.scratch), b, g, c)) {
            tl.none();
            return;
        }
    }
    tl.stamp(1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j0 = c * a.pages_per_chunk;
    // the length and this chunk's table entries are fetched together (one round trip):
    // entries inside the table row are always readable, whatever the length turns out to be
    const int jcap = min(a.max_blocks - j0, a.pages_per_chunk);
    const int ncap = warp < jcap ? (jcap - warp + kWarps - 1) / kWarps : 0;
    int my_page = 0;
    if (lane < ncap)
        my_page = a.bt[(size_t)b * a.max_blocks + j0 + warp + lane * kWarps];
    const int L = a.seq_lens[b];
    if (!length_ok(a, L)) {
        if (c == 0) {
            grid_dependency_wait();
            write_zero_unit(a, b, g);
        }
        tl.none();
        return;
    }
    const int npages = (L + kPage - 1) / kPage;
    const int nchunks = chunks_of(a, L);
    if (c >= nchunks) {
        tl.none();
        return;
    }
    const bool last_chunk = c == nchunks - 1;
    const int jn = min(npages - j0, a.pages_per_chunk);
    const int nmine = warp < jn ? (jn - warp + kWarps - 1) / kWarps : 0;
    const bool bad = lane < nmine && (my_page < 0 || my_page >= a.num_pages);
    const bool any_bad = __syncthreads_or(bad);  // the new token's page is one of the last chunk's pages

    uint64_t *my_bars = sm.bars + warp * STAGES;
    uint8_t *my_stages = sm.stages + warp * STAGES * kStageBytes;
    const uint64_t policy = l2_evict_first_policy();
    const int nfirst = min(STAGES, nmine);
    const int nearly = any_bad ? 0 : copies_before_wait(L, j0, warp, nmine, STAGES);
    if (!any_bad) {
        init_warp_barriers<STAGES>(my_bars, lane);
        issue_copies<STAGES>(&tmap, my_stages, my_bars, my_page, 0, nearly, g, lane, policy);
    }

    grid_dependency_wait();  // q, k_new, v_new, recently written pages and every output follow it
    tl.stamp(2);
    if (!any_bad)  // the pages holding positions L - 2 and L - 1
        issue_copies<STAGES>(&tmap, my_stages, my_bars, my_page, nearly, nfirst, g, lane, policy);

    const int pos = L - 1, slot = pos % kPage;
    unit_rows<APPEND>(a, b, g, pos, last_chunk, q_rot, new_kv);
    __syncthreads();
    if (APPEND && last_chunk && !any_bad && tid < 16)
        store_new_token(a, a.bt[(size_t)b * a.max_blocks + npages - 1], g, slot, new_kv);
    if (any_bad && tid == 0 && a.err)
        atomicOr(a.err, PKV_DEVERR_PAGE_RANGE);

    Warp w;
    w.init(q_rot, a.scale_log2, lane, sm.scratch + warp * kScratchFloats);
    if (!any_bad) {
        const auto patch = [&](uint8_t *stage, int j) {
            if (APPEND && last_chunk && j == npages - 1)
                patch_stage(stage, slot, new_kv, lane);
        };
        const uint32_t first_limit = b == a.expire_seq ? 0u : kWaitLimit;
        if (!consume_pages<STAGES>(&tmap, my_stages, my_bars, w, my_page, nmine, j0, warp, lane, L, g, policy, patch,
                                   first_limit) &&
            lane == 0 && a.err)
            atomicOr(a.err, PKV_DEVERR_TIMEOUT);
    }
    tl.stamp(3);
    allow_dependent_launch();
    // the stages are free now: they hold the combine area
    finish_unit<APPEND>(a, w, reinterpret_cast<float *>(sm.stages), ticket, q_rot, b, g, c, nchunks);
    tl.end(b, c, jn);
}

// ------------------------------------------------------------------ FP8 pages, grid schedule

// The fused step over FP8 pages: the same unit, prologue, dependency wait, query
// rotation, ticket and merge as decode_step_kernel, with the FP8 unit copy and the
// Fp8MmaWarp page policy.  The new token's rotated key row and value row are
// quantized once per (sequence, KV head) by the unit of the last chunk -- warp 0 the
// key, warp 1 the value, with the FP8 append's arithmetic -- stored into their page
// slot, and patched into the staged copy of that page.
template <int STAGES>
struct Fp8StepSmem {
    static constexpr int kStagesBytes = kWarps * STAGES * kFp8Unit;
    static constexpr int kBarsBytes = kWarps * STAGES * 8;
    static constexpr int kSortInts = kMaxPagesPerChunk + 1 + kWarps + 5;
    static constexpr int kExtraBytes = kGroup * kD * 2 + 2 * kD * 2 + 2 * kD + 16 + 16 + kSortInts * 4;
    static constexpr int kBytes = 128 + kStagesBytes + kBarsBytes + kExtraBytes;  // incl. alignment slack
    static_assert(kStagesBytes >= kWarps * kStateFloats * 4, "the combine reuses the stages");
    uint8_t *stages;
    uint64_t *bars;
    uint16_t *q_rot;      // [4][64] rotated query rows (BF16)
    uint16_t *new_kv;     // [2][64] rotated key row, value row (BF16)
    uint8_t *new_codes;   // [2][64] their E4M3 codes
    float *new_scales;    // [2] their row scales
    int *ticket;
    int *sort_scratch;

    __device__ __forceinline__ explicit Fp8StepSmem(uint8_t *raw)
    {
        uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 127) & ~uintptr_t(127));
        stages = base;
        bars = reinterpret_cast<uint64_t *>(base + kStagesBytes);
        uint8_t *e = base + kStagesBytes + kBarsBytes;
        q_rot = reinterpret_cast<uint16_t *>(e);
        new_kv = q_rot + kGroup * kD;
        new_codes = reinterpret_cast<uint8_t *>(new_kv + 2 * kD);
        new_scales = reinterpret_cast<float *>(new_codes + 2 * kD);
        ticket = reinterpret_cast<int *>(new_scales + 4);
        sort_scratch = ticket + 4;
    }
};

// A warp writes the new token's rows into a unit (a stage or the page): lanes 0-3 the
// K codes (16 bytes each), every lane two V codes (dims 2 lane, 2 lane + 1) at their
// interleaved positions, lanes 0 and 1 the two scales.
__device__ __forceinline__ void put_new_token_fp8(uint8_t *unit, int slot, const uint8_t *codes, const float *scales,
                                                  int lane)
{
    if (lane < 4)
        *reinterpret_cast<uint4 *>(unit + slot * kD + 16 * lane) = reinterpret_cast<const uint4 *>(codes)[lane];
    uint8_t *vt = unit + fp8::kFp8Tile;
    vt[fp8::v_code_offset(slot, 2 * lane)] = codes[kD + 2 * lane];
    vt[fp8::v_code_offset(slot, 2 * lane + 1)] = codes[kD + 2 * lane + 1];
    if (lane < 2)
        reinterpret_cast<float *>(unit + kFp8UnitCodes)[lane * kPage + slot] = scales[lane];
}

// CTAs per SM the register budget is set for.  The 3-stage ring takes 27.5 KB of shared
// memory per CTA, so seven CTAs fit (at most 72 registers, a few spilled) and keep 7 x 4 x 3
// units of 2176 B in flight per SM; the other rings keep six (80 registers, none spilled).
constexpr int fp8_ctas_per_sm(int stages) { return stages == 3 ? 7 : 6; }

template <int STAGES, bool APPEND>
__global__ void __launch_bounds__(kThreads, fp8_ctas_per_sm(STAGES))
    decode_step_fp8_kernel(const __grid_constant__ CUtensorMap tmap, StepArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    Fp8StepSmem<STAGES> sm(smem_raw);

    int g = blockIdx.x, b = blockIdx.y, c = blockIdx.z;
    if (a.sorted) {
        const int lin = blockIdx.x + kHkv * (blockIdx.y + gridDim.y * blockIdx.z);
        if (!sorted_unit(a, gridDim.y, lin, sm.sort_scratch, b, g, c))
            return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j0 = c * a.pages_per_chunk;
    const int jcap = min(a.max_blocks - j0, a.pages_per_chunk);
    const int ncap = warp < jcap ? (jcap - warp + kWarps - 1) / kWarps : 0;
    int my_page = 0;
    if (lane < ncap)
        my_page = a.bt[(size_t)b * a.max_blocks + j0 + warp + lane * kWarps];
    const int L = a.seq_lens[b];
    if (!length_ok(a, L)) {
        if (c == 0) {
            grid_dependency_wait();
            write_zero_unit(a, b, g);
        }
        return;
    }
    const int npages = (L + kPage - 1) / kPage;
    const int nchunks = chunks_of(a, L);
    if (c >= nchunks)
        return;
    const bool last_chunk = c == nchunks - 1;
    const int jn = min(npages - j0, a.pages_per_chunk);
    const int nmine = warp < jn ? (jn - warp + kWarps - 1) / kWarps : 0;
    const bool bad = lane < nmine && (my_page < 0 || my_page >= a.num_pages);
    const bool any_bad = __syncthreads_or(bad);

    uint64_t *my_bars = sm.bars + warp * STAGES;
    uint8_t *my_stages = sm.stages + warp * STAGES * kFp8Unit;
    const uint64_t policy = l2_evict_first_policy();
    const int nfirst = min(STAGES, nmine);
    const int nearly = any_bad ? 0 : copies_before_wait(L, j0, warp, nmine, STAGES);
    const auto issue = [&](int k0, int k1) {
        for (int k = k0; k < k1; ++k) {
            const int pk = __shfl_sync(kFull, my_page, k);
            if (lane == 0)
                fp8::fp8_issue(&tmap, my_stages + k * kFp8Unit, &my_bars[k], g, pk, policy);
        }
    };
    if (!any_bad) {
        init_warp_barriers<STAGES>(my_bars, lane);
        issue(0, nearly);
    }

    grid_dependency_wait();  // q, k_new, v_new, recently written pages and every output follow it
    if (!any_bad)  // the pages holding positions L - 2 and L - 1
        issue(nearly, nfirst);

    const int pos = L - 1, slot = pos % kPage;
    unit_rows<APPEND>(a, b, g, pos, last_chunk, sm.q_rot, sm.new_kv);
    __syncthreads();
    if (APPEND && last_chunk) {
        if (warp == 0) {  // key row: lane holds dims lane, lane + 32 (rotated, BF16)
            uint32_t c1, c2;
            float sc;
            fp8::quantize_pair(bf16_value(sm.new_kv[lane]), bf16_value(sm.new_kv[lane + kD / 2]), c1, c2, sc);
            sm.new_codes[lane] = (uint8_t)c1;
            sm.new_codes[lane + kD / 2] = (uint8_t)c2;
            if (lane == 0)
                sm.new_scales[0] = sc;
        } else if (warp == 1) {  // value row: lane holds dims 2 lane, 2 lane + 1
            const uint32_t w2 = reinterpret_cast<const uint32_t *>(sm.new_kv + kD)[lane];
            uint32_t c0, c1;
            float sc;
            fp8::quantize_pair(bf16lo(w2), bf16hi(w2), c0, c1, sc);
            reinterpret_cast<uint16_t *>(sm.new_codes + kD)[lane] = (uint16_t)(c0 | (c1 << 8));
            if (lane == 0)
                sm.new_scales[1] = sc;
        }
        __syncthreads();
        if (!any_bad && warp == 0) {
            const int page = a.bt[(size_t)b * a.max_blocks + npages - 1];
            uint8_t *unit = reinterpret_cast<uint8_t *>(a.slab) + (size_t)page * kFp8PageBytes + (size_t)g * kFp8Unit;
            put_new_token_fp8(unit, slot, sm.new_codes, sm.new_scales, lane);
        }
    }
    if (any_bad && tid == 0 && a.err)
        atomicOr(a.err, PKV_DEVERR_PAGE_RANGE);

    fp8::Fp8MmaWarp w;
    w.init(sm.q_rot, a.scale_log2, lane);
    if (!any_bad) {
        const uint32_t first_limit = b == a.expire_seq ? 0u : kWaitLimit;
        int k = 0;
        for (; k < nmine; ++k) {
            const int s = k % STAGES;
            if (!mbar_wait_warp(&my_bars[s], (uint32_t)((k / STAGES) & 1), k == 0 ? first_limit : kWaitLimit))
                break;
            const int j = j0 + warp + k * kWarps;
            uint8_t *stage = my_stages + s * kFp8Unit;
            if (APPEND && last_chunk && j == npages - 1) {  // the copy may predate the new token's store
                put_new_token_fp8(stage, slot, sm.new_codes, sm.new_scales, lane);
                __syncwarp();
            }
            w.page(stage, min(kPage, L - j * kPage));
            __syncwarp();
            if (k + STAGES < nmine) {
                const int pk = __shfl_sync(kFull, my_page, k + STAGES);
                if (lane == 0) {
                    fence_proxy_async_smem();
                    fp8::fp8_issue(&tmap, stage, &my_bars[s], g, pk, policy);
                }
            }
        }
        if (k < nmine) {  // a wait gave up: let the copies in flight land (bounded), flag it
            for (int kk = k; kk < min(nmine, k + STAGES); ++kk)
                (void)mbar_wait_warp(&my_bars[kk % STAGES], (uint32_t)((kk / STAGES) & 1));
            if (lane == 0 && a.err)
                atomicOr(a.err, PKV_DEVERR_TIMEOUT);
        }
    }
    allow_dependent_launch();
    // the stages are free now: they hold the combine area
    finish_unit<APPEND>(a, w, reinterpret_cast<float *>(sm.stages), sm.ticket, sm.q_rot, b, g, c, nchunks);
}

// ------------------------------------------------------------------ launch

// Ring depth per warp when the options leave it to the library: 3 stages for long
// chunks (4 CTAs per SM for BF16, 7 for FP8), else 2 (6 per SM), the measured best
// for 128-page chunks and for 16- to 32-page chunks of ragged batches respectively.
int default_ring(int pages_per_chunk) { return pages_per_chunk >= 64 ? 3 : 2; }

template <class Warp, int STAGES, bool APPEND>
int launch_grid(const CUtensorMap *tmap, const StepArgs &a, int B, cudaStream_t s, bool pdl)
{
    auto kernel = decode_step_kernel<Warp, STAGES, APPEND>;
    constexpr int smem = SmemLayout<STAGES>::kBaseBytes + kGridExtraBytes;
    static PerDeviceOnce attr;
    if (const int st = ensure_smem_attr(attr, kernel, smem); st != PKV_OK)
        return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kHkv, B, a.max_chunks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[1] = {pdl_attribute()};
    cfg.attrs = attrs;
    cfg.numAttrs = pdl ? 1 : 0;
    return status_from_cuda(cudaLaunchKernelEx(&cfg, kernel, *tmap, a));
}

// FP8 pages: ring depth per warp 2..4 units (2176 B each).
template <int STAGES, bool APPEND>
int launch_fp8_grid(const CUtensorMap *tmap, const StepArgs &a, int B, cudaStream_t s, bool pdl)
{
    auto kernel = decode_step_fp8_kernel<STAGES, APPEND>;
    constexpr int smem = Fp8StepSmem<STAGES>::kBytes;
    static PerDeviceOnce attr;
    if (const int st = ensure_smem_attr(attr, kernel, smem); st != PKV_OK)
        return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kHkv, B, a.max_chunks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[1] = {pdl_attribute()};
    cfg.attrs = attrs;
    cfg.numAttrs = pdl ? 1 : 0;
    return status_from_cuda(cudaLaunchKernelEx(&cfg, kernel, *tmap, a));
}

template <bool APPEND>
int launch_fp8_depth(const CUtensorMap *tmap, const StepArgs &a, int B, cudaStream_t s, bool pdl, int depth)
{
    switch (depth) {
    case 2: return launch_fp8_grid<2, APPEND>(tmap, a, B, s, pdl);
    case 3: return launch_fp8_grid<3, APPEND>(tmap, a, B, s, pdl);
    default: return launch_fp8_grid<4, APPEND>(tmap, a, B, s, pdl);
    }
}

// Ring depth per warp: 2 stages (36 KB per CTA, 6 CTAs per SM), 3 (4 per SM) or 4 (3 per SM).
template <class Warp, bool APPEND>
int launch_grid_depth(const CUtensorMap *tmap, const StepArgs &a, int B, cudaStream_t s, bool pdl, int depth)
{
    switch (depth) {
    case 2: return launch_grid<Warp, 2, APPEND>(tmap, a, B, s, pdl);
    case 3: return launch_grid<Warp, 3, APPEND>(tmap, a, B, s, pdl);
    default: return launch_grid<Warp, 4, APPEND>(tmap, a, B, s, pdl);
    }
}

// Option bits both entry points accept for the fused grid kernel.
constexpr int kGridOptions = 0xff | PKV_STEP_NO_PDL | PKV_STEP_GRID | PKV_STEP_RING_MASK | PKV_STEP_SORTED |
                             PKV_STEP_TEST_EXPIRE_WAIT;

// Validates the options, fills the launch-dependent fields of `a` and launches the
// kernel for the pool's format.
template <bool APPEND>
int launch_fused(const pkv_pool *pool, StepArgs &a, int B, int max_blocks, int pages_per_chunk, void *workspace,
                 cudaStream_t s, int options)
{
    const int variant = options & 0xff;
    if (variant < PKV_DECODE_DEFAULT || variant > PKV_DECODE_MMA || (options & ~kGridOptions))
        return PKV_ERR_INVALID_ARG;
    if ((options & PKV_STEP_SORTED) && B > kMaxSortedBatch)
        return PKV_ERR_INVALID_ARG;  // the sorted order handles up to 1024 sequences
    const int ring = (options & PKV_STEP_RING_MASK) >> 12;
    if (ring != 0 && (ring < 2 || ring > 4))
        return PKV_ERR_INVALID_ARG;
    if (pool->kv_format == PKV_KV_FP8 && variant == PKV_DECODE_SIMT)
        return PKV_ERR_UNSUPPORTED;  // FP8 pages: the MMA policy only
    const int max_chunks = (max_blocks + pages_per_chunk - 1) / pages_per_chunk;
    if (max_chunks > 65535)  // the chunk index is gridDim.z
        return PKV_ERR_INVALID_ARG;
    const CUtensorMap *tmap = pool_tensor_map(pool);
    if (!tmap)
        return PKV_ERR_CUDA;
    const WorkspaceLayout ws = workspace_layout(B, max_chunks);
    char *wsp = static_cast<char *>(workspace);
    a.num_pages = pool->num_pages;
    a.slab = reinterpret_cast<uint16_t *>(pool->slab);
    a.max_blocks = max_blocks;
    a.pages_per_chunk = pages_per_chunk;
    a.counters = wsp ? reinterpret_cast<int *>(wsp) : nullptr;
    a.part_ml = wsp ? reinterpret_cast<float2 *>(wsp + ws.ml_offset()) : nullptr;
    a.part_o = wsp ? reinterpret_cast<float *>(wsp + ws.o_offset()) : nullptr;
    a.max_chunks = max_chunks;
    a.sorted = (options & PKV_STEP_SORTED) ? 1 : 0;
    a.expire_seq = (options & PKV_STEP_TEST_EXPIRE_WAIT) ? 0 : -1;
    const bool pdl = take_pdl_permission(pool, !(options & PKV_STEP_NO_PDL));
    const int depth = ring ? ring : default_ring(pages_per_chunk);
    if (pool->kv_format == PKV_KV_FP8)
        return launch_fp8_depth<APPEND>(tmap, a, B, s, pdl, depth);
    return variant == PKV_DECODE_SIMT ? launch_grid_depth<SimtWarp, APPEND>(tmap, a, B, s, pdl, depth)
                                      : launch_grid_depth<MmaWarp, APPEND>(tmap, a, B, s, pdl, depth);
}

}  // namespace

int launch_attention_fused(const pkv_pool *pool, const uint16_t *q, const int32_t *bt, int max_blocks,
                           const int32_t *seq_lens, int B, float scale, int pages_per_chunk, void *workspace,
                           uint16_t *out, int32_t *err, cudaStream_t s, int options)
{
    StepArgs a = {};
    a.k_new = nullptr;
    a.v_new = nullptr;
    a.q = const_cast<uint16_t *>(q);  // read only: no append writes the rows back
    a.bt = bt;
    a.seq_lens = seq_lens;
    a.rope = nullptr;
    a.max_pos = INT_MAX;
    a.scale_log2 = scale * kLog2e;
    a.out = out;
    a.err = err;
    return launch_fused<false>(pool, a, B, max_blocks, pages_per_chunk, workspace, s, options);
}

}  // namespace pkv

extern "C" size_t pkv_decode_step_workspace_bytes(int B, int max_blocks, int pages_per_chunk)
{
    return pkv_decode_workspace_bytes(B, max_blocks, pages_per_chunk);
}

extern "C" int pkv_decode_step(const pkv_pool *pool, const uint16_t *k_new, const uint16_t *v_new, uint16_t *q,
                               const int32_t *bt_dev, int max_blocks, const int32_t *seq_lens_dev, int B,
                               const float *rope_table, int max_pos, float scale, int pages_per_chunk,
                               void *workspace, size_t workspace_bytes, uint16_t *out, int32_t *dev_err_flag,
                               void *cuda_stream, int options)
{
    using namespace pkv;
    if (!pool || !k_new || !v_new || !q || !bt_dev || !seq_lens_dev || !rope_table || !out || !workspace)
        return PKV_ERR_INVALID_ARG;
    if (B < 1 || B > 65535 || max_blocks < 1 || max_blocks > (1 << 20) || max_pos < 1)
        return PKV_ERR_INVALID_ARG;
    if (pages_per_chunk < 1 || pages_per_chunk > kMaxPagesPerChunk || !(scale > 0.f) || !(scale < INFINITY))
        return PKV_ERR_INVALID_ARG;
    const uintptr_t align = reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
                            reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
                            reinterpret_cast<uintptr_t>(rope_table) | reinterpret_cast<uintptr_t>(workspace);
    if (align & 15u)
        return PKV_ERR_INVALID_ARG;
    if (workspace_bytes < pkv_decode_step_workspace_bytes(B, max_blocks, pages_per_chunk))
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    StepArgs a = {};
    a.k_new = k_new;
    a.v_new = v_new;
    a.q = q;
    a.bt = bt_dev;
    a.seq_lens = seq_lens_dev;
    a.rope = reinterpret_cast<const float4 *>(rope_table);
    a.max_pos = max_pos;
    a.scale_log2 = scale * kLog2e;
    a.out = out;
    a.err = dev_err_flag;
    return launch_fused<true>(pool, a, B, max_blocks, pages_per_chunk, workspace,
                              static_cast<cudaStream_t>(cuda_stream), options);
}

#ifdef PKV_TIMELINE
extern "C" int pkv_timeline_read(uint64_t *stamps, int32_t *meta, int n)
{
    using namespace pkv;
    if (!stamps || !meta || n < 1)
        return PKV_ERR_INVALID_ARG;
    if (n > kTimelineMax)
        n = kTimelineMax;
    if (cudaMemcpyFromSymbol(stamps, g_timeline_stamps, (size_t)n * 5 * sizeof(uint64_t)) != cudaSuccess ||
        cudaMemcpyFromSymbol(meta, g_timeline_meta, (size_t)n * 4 * sizeof(int32_t)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return n;
}
#endif
