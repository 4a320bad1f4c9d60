// pkv_step.cu -- one fused launch per layer: RoPE + page-slot append of the new
// token, paged GQA decode attention over the sequence's pages, and the
// log-sum-exp merge of the chunk partials.
//
// It computes exactly what pkv_append_rope (positions = seq_lens - 1, q rotated
// in place) followed by pkv_decode_attention computes -- the samir-vllm README
// summary ("从零用 C++ 和 CUDA 实现 Llama 3.2 1B 推理引擎", section "目前已完成的功能")
// describes both steps: decode appends one token at its absolute RoPE position,
// then each query head streams its sequence's pages with an FP32 online softmax
// -- with the same arithmetic, so the results are bit-identical to the two
// separate calls.  What changes is the schedule.
//
// Work unit = (sequence b, KV head g, chunk c of pages_per_chunk pages), as in the
// split kernel.  Per unit:
//  * the 4 query rows of group g are rotated to position L-1 by the unit itself;
//    the rotated rows are written back once, by the unit that finishes (b, g) last;
//  * the sequence's last chunk computes the new token's rotated key and its value,
//    stores them into their page slot in HBM and patches them into the
//    shared-memory copy of the last page, so no unit waits for an append kernel;
//  * chunk partials are merged in-kernel: each unit publishes its partial and
//    takes a ticket from a per-(b, g) counter (one release-acquire atomicAdd, no
//    waiting); the unit drawing the last ticket merges all chunks in chunk order
//    (deterministic) and resets the counter to zero for the next launch.
// Two schedules:
//  * grid: one CTA per unit (grid = chunks x 8 x B); best for long sequences
//    with large chunks;
//  * persistent: a few CTAs per SM walk a compact, device-built list of the
//    non-empty units; each warp's TMA ring keeps prefetching pages ACROSS unit
//    boundaries, so a unit's set-up and epilogue (combine, ticket, merge) hide
//    behind copies already in flight.  Best for ragged and small batches.
// Both use programmatic dependent launch: before griddepcontrol.wait a CTA only
// reads this step's lengths and block tables and starts the TMA copies of this
// layer's cached pages (which no earlier kernel of the step writes: every layer
// has its own pages); q, k_new, v_new are read and every output is written after
// the wait.
#include <cuda_bf16.h>

#include "pkv_device.cuh"
#include "pkv_fp8.cuh"

namespace pkv {
namespace {

using namespace dev;

struct StepArgs {
    int num_pages;
    uint16_t *slab;
    const uint16_t *k_new;   // [B][8][64]
    const uint16_t *v_new;   // [B][8][64]
    uint16_t *q;             // [B][32][64], rotated in place
    const int32_t *bt;       // [B][max_blocks]
    int max_blocks;
    const int32_t *seq_lens; // [B]
    const float2 *rope;      // [max_pos][32] (cos, sin)
    int max_pos;
    float scale_log2;
    int pages_per_chunk;
    int *counters;           // [B][8], zero between launches
    float2 *part_ml;         // [B][32][max_chunks]
    float *part_o;           // [B][32][max_chunks][64]
    int max_chunks;
    uint16_t *out;           // [B][32][64]
    int32_t *err;
    int early_trigger;       // grid schedule: allow the next launch as soon as the copies are issued
    int sorted;              // grid schedule: units dispatched largest first (PKV_STEP_SORTED)
};

constexpr int kStepStages = 4;       // persistent schedule ring depth
constexpr int kDefaultGridRing = 4;  // grid schedule ring depth unless the options choose one
constexpr int kMaxPersistentBatch = 512;
constexpr int kMaxSortedBatch = 1024;
static_assert(kMaxPagesPerChunk + 1 + kWarps + 5 <= kWarps * kScratchFloats, "sorted-order scratch");

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;" ::); }

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

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

// All kThreads threads: the 4 query rows of group g rotated to position pos into
// q_rot[4][64] (one pair per thread) and, for the sequence's last chunk, the new
// token's rotated key row and its value row into new_kv[2][64].
__device__ __forceinline__ void unit_rows(const StepArgs &a, int b, int g, int pos, bool last_chunk, uint16_t *q_rot,
                                          uint16_t *new_kv)
{
    const int hl = threadIdx.x >> 5, i = threadIdx.x & 31;
    const float2 cs = a.rope[(size_t)pos * (kD / 2) + i];
    const uint16_t *qrow = a.q + ((size_t)b * kHq + g * kGroup + hl) * kD;
    float y1, y2;
    rope_rotate_pair(bf16_value(qrow[i]), bf16_value(qrow[i + kD / 2]), cs.x, cs.y, y1, y2);
    q_rot[hl * kD + i] = bf16_bits(y1);
    q_rot[hl * kD + i + kD / 2] = bf16_bits(y2);
    if (last_chunk && hl == 0) {
        const uint16_t *krow = a.k_new + ((size_t)b * kHkv + g) * kD;
        rope_rotate_pair(bf16_value(krow[i]), bf16_value(krow[i + kD / 2]), cs.x, cs.y, y1, y2);
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

// Unit epilogue, all threads: combine the warps' states through `state`, then
// write the output (single chunk) or publish the chunk partial and take a ticket;
// the unit drawing the last ticket merges every chunk of (b, g) in chunk order,
// writes the output and the rotated query rows, and resets the counter.
struct CtaSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// The 4 consumer warps only (named barrier 1), for kernels with a producer warp.
struct ConsumerSync {
    __device__ __forceinline__ void operator()() const { asm volatile("bar.sync 1, 128;" ::: "memory"); }
};

// Chunk counts up to which the merging unit holds every partial in registers.
constexpr int kMergeRegs = 8;

template <class Warp, class Sync = CtaSync>
__device__ __forceinline__ void finish_unit(const StepArgs &a, Warp &w, float *state, int *ticket,
                                            const uint16_t *q_rot, int b, int g, int c, int nchunks,
                                            Sync sync = Sync())
{
    const int tid = threadIdx.x, warp = tid >> 5;
    sync();
    w.store_state(state + warp * kStateFloats);
    sync();
    const int hl = tid >> 5, dp = tid & 31, h = g * kGroup + hl;
    float M, lsum, o0, o1;
    combine_warps(state, hl, dp, M, lsum, o0, o1);
    uint32_t *out_row = reinterpret_cast<uint32_t *>(a.out + ((size_t)b * kHq + h) * kD);
    uint32_t *q_row = reinterpret_cast<uint32_t *>(a.q + ((size_t)b * kHq + h) * kD);
    const uint32_t q_word = reinterpret_cast<const uint32_t *>(q_rot + hl * kD)[dp];
    if (nchunks == 1) {
        out_row[dp] = finish_pair(o0, o1, lsum);
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
    sync();
    if (tid == 0)
        *ticket = ticket_acq_rel(&a.counters[b * kHkv + g]);
    sync();
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

template <class Warp, int STAGES>
__global__ void __launch_bounds__(kThreads) decode_step_kernel(const __grid_constant__ CUtensorMap tmap, StepArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    SmemLayout<STAGES> sm(smem_raw);
    uint16_t *q_rot = reinterpret_cast<uint16_t *>(sm.extra);  // [4][64] rotated query rows
    uint16_t *new_kv = q_rot + kGroup * kD;                     // [2][64] rotated key row, value row
    int *ticket = reinterpret_cast<int *>(new_kv + 2 * kD);
    Timeline tl;
    tl.begin();

    // chunk index slowest: every first chunk is dispatched before any later one, so the
    // CTAs left empty by short sequences come last; or the sorted order
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
    if (!any_bad) {
        init_warp_barriers<STAGES>(my_bars, lane);
        issue_prologue<STAGES>(&tmap, my_stages, my_bars, my_page, nmine, g, lane, policy);
    }
    if (a.early_trigger)
        allow_dependent_launch();

    grid_dependency_wait();  // q, k_new, v_new and every output belong to the dependency chain
    tl.stamp(2);

    const int pos = L - 1, slot = pos % kPage;
    unit_rows(a, b, g, pos, last_chunk, q_rot, new_kv);
    __syncthreads();
    if (last_chunk && !any_bad && tid < 16)
        store_new_token(a, a.bt[(size_t)b * a.max_blocks + npages - 1], g, slot, new_kv);
    if (any_bad && tid == 0 && a.err)
        atomicOr(a.err, PKV_DEVERR_PAGE_RANGE);

    Warp w;
    w.init(q_rot, a.scale_log2, lane, sm.scratch + warp * kScratchFloats);
    if (!any_bad) {
        const auto patch = [&](uint8_t *stage, int j) {
            if (last_chunk && j == npages - 1)
                patch_stage(stage, slot, new_kv, lane);
        };
        if (!consume_pages<STAGES>(&tmap, my_stages, my_bars, w, my_page, nmine, j0, warp, lane, L, g, policy,
                                   patch) &&
            lane == 0 && a.err)
            atomicOr(a.err, PKV_DEVERR_TIMEOUT);
    }
    tl.stamp(3);
    if (!a.early_trigger)
        allow_dependent_launch();
    // the stages are free now: they hold the combine area
    finish_unit(a, w, reinterpret_cast<float *>(sm.stages), ticket, q_rot, b, g, c, nchunks);
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

template <int STAGES>
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
    if (!any_bad) {
        init_warp_barriers<STAGES>(my_bars, lane);
        for (int k = 0; k < min(STAGES, nmine); ++k) {
            const int pk = __shfl_sync(kFull, my_page, k);
            if (lane == 0)
                fp8::fp8_issue(&tmap, my_stages + k * kFp8Unit, &my_bars[k], g, pk, policy);
        }
    }
    if (a.early_trigger)
        allow_dependent_launch();

    grid_dependency_wait();  // q, k_new, v_new and every output belong to the dependency chain

    const int pos = L - 1, slot = pos % kPage;
    unit_rows(a, b, g, pos, last_chunk, sm.q_rot, sm.new_kv);
    __syncthreads();
    if (last_chunk) {
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
        int k = 0;
        for (; k < nmine; ++k) {
            const int s = k % STAGES;
            if (!mbar_wait_warp(&my_bars[s], (uint32_t)((k / STAGES) & 1)))
                break;
            const int j = j0 + warp + k * kWarps;
            uint8_t *stage = my_stages + s * kFp8Unit;
            if (last_chunk && j == npages - 1) {  // the copy may predate the new token's store
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
    if (!a.early_trigger)
        allow_dependent_launch();
    // the stages are free now: they hold the combine area
    finish_unit(a, w, reinterpret_cast<float *>(sm.stages), sm.ticket, sm.q_rot, b, g, c, nchunks);
}

// ------------------------------------------------------------------ persistent schedule

struct UnitInfo {
    int b, g, c, L, nchunks, npages, j0, jn;
    bool valid;
};

// Unit r of the compact list.  prefix[b] is the first unit of sequence b, which owns
// 8 * nchunks(b) units ordered (KV head, chunk); an invalid length owns 8 empty units.
__device__ __forceinline__ UnitInfo decode_unit(const StepArgs &a, const int *prefix, int B, int r)
{
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    UnitInfo u;
    u.b = lo;
    u.nchunks = (prefix[lo + 1] - prefix[lo]) / kHkv;
    const int rem = r - prefix[lo];
    u.g = rem / u.nchunks;
    u.c = rem - u.g * u.nchunks;
    u.L = a.seq_lens[lo];
    u.valid = length_ok(a, u.L);
    u.npages = u.valid ? (u.L + kPage - 1) / kPage : 0;
    u.j0 = u.c * a.pages_per_chunk;
    u.jn = u.valid ? min(u.npages - u.j0, a.pages_per_chunk) : 0;
    return u;
}

__device__ __forceinline__ int warp_pages(const UnitInfo &u, int warp)
{
    return warp < u.jn ? (u.jn - warp + kWarps - 1) / kWarps : 0;
}

template <int STAGES>
constexpr int persistent_smem_bytes(int B)
{
    return SmemLayout<STAGES>::kBaseBytes + kWarps * kStateFloats * 4 + kGroup * kD * 2 + 2 * kD * 2 + 16 +
           kWarps * STAGES * 4 + kWarps * 4 + (B + 1) * 4;
}

template <class Warp, int STAGES>
__global__ void __launch_bounds__(kThreads)
decode_step_persistent_kernel(const __grid_constant__ CUtensorMap tmap, StepArgs a, int B)
{
    extern __shared__ uint8_t smem_raw[];
    SmemLayout<STAGES> sm(smem_raw);
    float *state = reinterpret_cast<float *>(sm.extra);                  // [4 warps][kStateFloats]
    uint16_t *q_rot = reinterpret_cast<uint16_t *>(state + kWarps * kStateFloats);  // [4][64]
    uint16_t *new_kv = q_rot + kGroup * kD;                               // [2][64]
    int *ticket = reinterpret_cast<int *>(new_kv + 2 * kD);              // [4]
    int *stage_bad = ticket + 4;                                          // [4 warps][STAGES]
    int *warp_sums = stage_bad + kWarps * STAGES;                         // [4 warps]
    int *prefix = warp_sums + kWarps;                                     // [B + 1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- compact unit list: exclusive prefix sum over sequences (4 per thread)
    int v[4], local = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int b = 4 * tid + i;
        int n = 0;
        if (b < B) {
            const int L = a.seq_lens[b];
            n = kHkv * (length_ok(a, L) ? chunks_of(a, L) : 1);
        }
        v[i] = n;
        local += n;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, off);
        if (lane >= off)
            incl += t;
    }
    if (lane == 31)
        warp_sums[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int ww = 0; ww < warp; ++ww)
        run += warp_sums[ww];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (4 * tid + i < B)
            prefix[4 * tid + i] = run;
        run += v[i];
    }
    if (tid == kThreads - 1)
        prefix[B] = run;
    __syncthreads();
    const int R = prefix[B];
    const int P = gridDim.x;
    const int my_units = (int)blockIdx.x < R ? (R - 1 - (int)blockIdx.x) / P + 1 : 0;
    if (my_units == 0)
        return;

    uint64_t *my_bars = sm.bars + warp * STAGES;
    uint8_t *my_stages = sm.stages + warp * STAGES * kStageBytes;
    int *my_bad = stage_bad + warp * STAGES;
    init_warp_barriers<STAGES>(my_bars, lane);
    const uint64_t policy = l2_evict_first_policy();

    // ---- producer: walks this CTA's units ahead of the consumer, at most STAGES
    //      pages ahead, across unit boundaries.  Lane k holds the page id of the
    //      warp's k-th page of the unit being issued.
    int p_i = 0;
    UnitInfo pu = decode_unit(a, prefix, B, blockIdx.x);
    int p_n = warp_pages(pu, warp), p_k = 0;
    int p_id = lane < p_n ? a.bt[(size_t)pu.b * a.max_blocks + pu.j0 + warp + lane * kWarps] : 0;
    uint32_t issued = 0, consumed = 0;
    bool dead = false;  // a bounded wait gave up: stop streaming, keep the bookkeeping going
    const auto produce = [&]() {
        while (!dead && (int)(issued - consumed) < STAGES && p_i < my_units) {
            if (p_k >= p_n) {
                if (++p_i >= my_units)
                    break;
                pu = decode_unit(a, prefix, B, blockIdx.x + p_i * P);
                p_n = warp_pages(pu, warp);
                p_k = 0;
                p_id = lane < p_n ? a.bt[(size_t)pu.b * a.max_blocks + pu.j0 + warp + lane * kWarps] : 0;
                continue;
            }
            const int id = __shfl_sync(kFull, p_id, p_k);
            const int s = issued % STAGES;
            if (lane == 0) {
                const bool ok = id >= 0 && id < a.num_pages;
                my_bad[s] = ok ? 0 : 1;
                if (ok) {
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(&my_bars[s], kStageBytes);
                    tma_load_page_head(my_stages + s * kStageBytes, &tmap, &my_bars[s], pu.g, id, policy);
                } else {
                    mbar_arrive(&my_bars[s]);  // completes the phase without a copy
                }
            }
            __syncwarp();
            ++issued;
            ++p_k;
        }
    };
    produce();

    grid_dependency_wait();  // q, k_new, v_new and every output belong to the dependency chain

    for (int i = 0; i < my_units; ++i) {
        const UnitInfo u = decode_unit(a, prefix, B, blockIdx.x + i * P);
        __syncthreads();  // the previous unit's epilogue no longer reads q_rot, new_kv, state
        if (i == my_units - 1)
            allow_dependent_launch();
        if (!u.valid) {
            write_zero_unit(a, u.b, u.g);
            continue;
        }
        const int pos = u.L - 1, slot = pos % kPage;
        const bool last_chunk = u.c == u.nchunks - 1;
        unit_rows(a, u.b, u.g, pos, last_chunk, q_rot, new_kv);
        __syncthreads();
        if (last_chunk && tid < 16) {
            const int page = a.bt[(size_t)u.b * a.max_blocks + u.npages - 1];
            if (page >= 0 && page < a.num_pages)
                store_new_token(a, page, u.g, slot, new_kv);
        }
        Warp w;
        w.init(q_rot, a.scale_log2, lane, sm.scratch + warp * kScratchFloats);
        const int n = warp_pages(u, warp);
        for (int k = 0; k < n; ++k) {
            const int s = consumed % STAGES;
            const int j = u.j0 + warp + k * kWarps;
            if (!dead && !mbar_wait_warp(&my_bars[s], (consumed / STAGES) & 1)) {
                // give the other copies in flight a bounded chance to land, then stop
                for (uint32_t kk = consumed + 1; kk < issued; ++kk)
                    (void)mbar_wait_warp(&my_bars[kk % STAGES], (kk / STAGES) & 1);
                dead = true;
                if (lane == 0 && a.err)
                    atomicOr(a.err, PKV_DEVERR_TIMEOUT);
            }
            if (!dead) {
                uint8_t *stage = my_stages + s * kStageBytes;
                if (my_bad[s]) {
                    if (lane == 0 && a.err)
                        atomicOr(a.err, PKV_DEVERR_PAGE_RANGE);
                } else {
                    if (last_chunk && j == u.npages - 1)
                        patch_stage(stage, slot, new_kv, lane);
                    w.page(stage, min(kPage, u.L - j * kPage));
                }
            }
            __syncwarp();
            ++consumed;
            produce();
        }
        finish_unit(a, w, state, ticket, q_rot, u.b, u.g, u.c, u.nchunks);
    }
}

// ------------------------------------------------------------------ warp-specialised schedule
//
// Per CTA, 4 consumer warps (threads 0..127) and one producer warp (128..159); 2 CTAs
// per SM.  The producer walks the compact unit list -- the CTA's first unit is
// blockIdx.x, every further one is drawn from a work counter after the dependency
// wait -- and for each unit posts a descriptor (the unit's raw query rows, new key
// and value rows and RoPE row, fetched by 1-D bulk copies) and streams the unit's
// pages into a CTA-wide ring of kWsRing stages with full/empty mbarriers.  Consumers
// read a unit's inputs from shared memory only; their epilogue (combine, ticket,
// merge) overlaps the producer's copies of the next units.  The last CTA to finish
// resets the work counter, so the workspace counters are zero between launches.
// A unit's descriptor is posted before any of its pages beyond the first ring-full,
// so the consumers can always drain the ring (no circular wait).

constexpr int kWsRing = 24;
constexpr int kWsUnitSlots = 4;
constexpr int kWsThreads = kThreads + 32;

struct WsDesc {
    int b, g, c, L, nchunks, j0, jn, first, new_page, valid, end, pad[5];  // 64 B
    uint16_t q[kGroup * kD];  // raw query rows of the group (512 B)
    uint16_t k[kD];           // new key row, not yet rotated (128 B)
    uint16_t v[kD];           // new value row (128 B)
    float2 rope[kD / 2];      // (cos, sin) at position L-1 (256 B)
};
constexpr uint32_t kWsDescCopyBytes = kGroup * kD * 2 + kD * 2 + kD * 2 + (kD / 2) * 8;
static_assert(sizeof(WsDesc) == 64 + kWsDescCopyBytes && sizeof(WsDesc) % 16 == 0, "descriptor layout");

constexpr int ws_smem_bytes(int B)
{
    return 1024 + kWsRing * kStageBytes + (2 * kWsRing + 2 * kWsUnitSlots) * 8 + kWsRing * 4 +
           kWsUnitSlots * (int)sizeof(WsDesc) + kWarps * kStateFloats * 4 + kWarps * kScratchFloats * 4 +
           kGroup * kD * 2 + 2 * kD * 2 + 16 + (kWarps + 1) * 4 + (B + 1) * 4;
}

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// OR of a predicate over the 128 consumer threads (named barrier 1).
__device__ __forceinline__ bool consumer_any(bool p)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, 128, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p)
        : "memory");
    return r != 0;
}

template <class Warp>
__global__ void __launch_bounds__(kWsThreads)
decode_step_ws_kernel(const __grid_constant__ CUtensorMap tmap, StepArgs a, int B, int *work_counter, int *exit_counter)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + kWsRing * kStageBytes);
    uint64_t *empty = full + kWsRing;
    uint64_t *ufull = empty + kWsRing;
    uint64_t *uempty = ufull + kWsUnitSlots;
    int *bad = reinterpret_cast<int *>(uempty + kWsUnitSlots);
    WsDesc *desc = reinterpret_cast<WsDesc *>(bad + kWsRing);
    float *state = reinterpret_cast<float *>(desc + kWsUnitSlots);
    float *scratch = state + kWarps * kStateFloats;
    uint16_t *q_rot = reinterpret_cast<uint16_t *>(scratch + kWarps * kScratchFloats);
    uint16_t *new_kv = q_rot + kGroup * kD;
    int *ticket = reinterpret_cast<int *>(new_kv + 2 * kD);
    int *warp_sums = ticket + 4;
    int *prefix = warp_sums + kWarps + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- compact unit list (as the persistent schedule), 4 sequences per thread
    {
        int v[4], local = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = 4 * tid + i;
            int n = 0;
            if (b < B) {
                const int L = a.seq_lens[b];
                n = kHkv * (length_ok(a, L) ? chunks_of(a, L) : 1);
            }
            v[i] = n;
            local += n;
        }
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(kFull, incl, off);
            if (lane >= off)
                incl += t;
        }
        if (lane == 31)
            warp_sums[warp] = incl;
        if (tid == 0) {
            for (int s = 0; s < kWsRing; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], 1);
            }
            for (int s = 0; s < kWsUnitSlots; ++s) {
                mbar_init(&ufull[s], 1);
                mbar_init(&uempty[s], 1);
            }
            fence_barrier_init();
        }
        __syncthreads();
        int run = incl - local;
        for (int ww = 0; ww < warp; ++ww)
            run += warp_sums[ww];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (4 * tid + i < B)
                prefix[4 * tid + i] = run;
            run += v[i];
        }
        if (tid == kWsThreads - 1)
            prefix[B] = run;
        __syncthreads();
    }
    const int R = prefix[B];

    if (warp == kWarps) {
        // ================================================================ producer
        const uint64_t policy = l2_evict_first_policy();
        int r = blockIdx.x;
        uint32_t G = 0, ui = 0;
        bool waited = false, dead = false;
        for (;;) {
            const int us = ui % kWsUnitSlots;
            if (ui >= kWsUnitSlots && !dead &&
                !mbar_wait_warp(&uempty[us], ((ui / kWsUnitSlots) - 1) & 1))
                dead = true;
            WsDesc *d = desc + us;
            if (r >= R || dead) {
                if (!waited)
                    grid_dependency_wait();
                if (lane == 0) {
                    d->end = 1;
                    mbar_arrive(&ufull[us]);
                }
                break;
            }
            const UnitInfo u = decode_unit(a, prefix, B, r);
            int id[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int k = lane + 32 * i;
                id[i] = k < u.jn ? a.bt[(size_t)u.b * a.max_blocks + u.j0 + k] : 0;
            }
            const auto page_id = [&](int k) {
                const int i = k >> 5;
                const int mine = i == 0 ? id[0] : i == 1 ? id[1] : i == 2 ? id[2] : id[3];
                return __shfl_sync(kFull, mine, k & 31);
            };
            // Issue pages k .. k+n-1 (n <= 4) from lanes 0..n-1.  A stage is reused only
            // after its consumer released it (empty barrier, acquire after release); the
            // consumers' reads need no proxy fence before the copy overwrites them.
            const auto issue_pages = [&](int k, int n) {
                for (int i = 0; i < n; ++i) {
                    const uint32_t gi = G + i;
                    if (gi >= kWsRing && !dead &&
                        !mbar_wait_warp(&empty[gi % kWsRing], ((gi / kWsRing) - 1) & 1))
                        dead = true;
                }
                // k is a multiple of 4, so pages k..k+3 share one 32-entry register block
                const int reg = k >> 5;
                const int mine = reg == 0 ? id[0] : reg == 1 ? id[1] : reg == 2 ? id[2] : id[3];
                const int pid = __shfl_sync(kFull, mine, (k & 31) + (lane & 3));
                if (lane < n) {
                    const int s = (G + lane) % kWsRing;
                    const bool ok = pid >= 0 && pid < a.num_pages && !dead;
                    bad[s] = ok ? 0 : 1;
                    if (ok) {
                        mbar_arrive_expect_tx(&full[s], kStageBytes);
                        tma_load_page_head(ring + s * kStageBytes, &tmap, &full[s], u.g, pid, policy);
                    } else {
                        mbar_arrive(&full[s]);
                    }
                }
                __syncwarp();
                G += n;
            };
            const uint32_t first = G;
            int k = 0;
            if (!waited) {
                // before the dependency wait: only this layer's cached pages, at most one ring-full
                const int pre = min(u.jn, kWsRing);
                for (; k < pre; k += 4)
                    issue_pages(k, min(4, pre - k));
                grid_dependency_wait();
                waited = true;
            }
            // the unit's descriptor, then its remaining pages
            const int new_page = (u.valid && u.c == u.nchunks - 1 && u.jn > 0) ? page_id(u.jn - 1) : -1;
            if (lane == 0) {
                d->b = u.b;
                d->g = u.g;
                d->c = u.c;
                d->L = u.L;
                d->nchunks = u.nchunks;
                d->j0 = u.j0;
                d->jn = u.jn;
                d->first = (int)first;
                d->new_page = new_page;
                d->valid = u.valid ? 1 : 0;
                d->end = 0;
                if (u.valid) {
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(&ufull[us], kWsDescCopyBytes);
                    bulk_copy_g2s(d->q, a.q + ((size_t)u.b * kHq + u.g * kGroup) * kD, kGroup * kD * 2, &ufull[us]);
                    bulk_copy_g2s(d->k, a.k_new + ((size_t)u.b * kHkv + u.g) * kD, kD * 2, &ufull[us]);
                    bulk_copy_g2s(d->v, a.v_new + ((size_t)u.b * kHkv + u.g) * kD, kD * 2, &ufull[us]);
                    bulk_copy_g2s(d->rope, a.rope + (size_t)(u.L - 1) * (kD / 2), (kD / 2) * 8, &ufull[us]);
                } else {
                    mbar_arrive(&ufull[us]);
                }
            }
            int nxt = 0;
            if (lane == 0)
                nxt = (int)gridDim.x + atomicAdd(work_counter, 1);
            for (; k < u.jn; k += 4)
                issue_pages(k, min(4, u.jn - k));
            r = __shfl_sync(kFull, nxt, 0);
            ++ui;
        }
        allow_dependent_launch();
    } else {
        // ================================================================ consumers
        const ConsumerSync csync;
        uint32_t ui = 0;
        bool dead = false, waited = false;
        for (;;) {
            const int us = ui % kWsUnitSlots;
            csync();  // the previous unit's epilogue no longer reads q_rot, new_kv, state
            const bool timed_out = !mbar_wait_warp(&ufull[us], (ui / kWsUnitSlots) & 1);
            if (consumer_any(timed_out)) {
                if (tid == 0 && a.err)
                    atomicOr(a.err, PKV_DEVERR_TIMEOUT);
                break;
            }
            const WsDesc *d = desc + us;
            if (d->end)
                break;
            if (!waited) {
                grid_dependency_wait();
                waited = true;
            }
            const int b = d->b, g = d->g, c = d->c, L = d->L, nchunks = d->nchunks, j0 = d->j0, jn = d->jn;
            const int first = d->first, new_page = d->new_page;
            if (!d->valid) {
                csync();
                if (tid == 0)
                    mbar_arrive(&uempty[us]);
                write_zero_unit(a, b, g);
                ++ui;
                continue;
            }
            const int pos = L - 1, slot = pos % kPage, npages = (L + kPage - 1) / kPage;
            const bool last_chunk = c == nchunks - 1;
            {
                const int hl = tid >> 5, i = tid & 31;
                const float2 cs = d->rope[i];
                float y1, y2;
                rope_rotate_pair(bf16_value(d->q[hl * kD + i]), bf16_value(d->q[hl * kD + i + kD / 2]), cs.x, cs.y,
                                 y1, y2);
                q_rot[hl * kD + i] = bf16_bits(y1);
                q_rot[hl * kD + i + kD / 2] = bf16_bits(y2);
                if (last_chunk && hl == 0) {
                    rope_rotate_pair(bf16_value(d->k[i]), bf16_value(d->k[i + kD / 2]), cs.x, cs.y, y1, y2);
                    new_kv[i] = bf16_bits(y1);
                    new_kv[i + kD / 2] = bf16_bits(y2);
                } else if (last_chunk && hl == 1) {
                    reinterpret_cast<uint32_t *>(new_kv + kD)[i] = reinterpret_cast<const uint32_t *>(d->v)[i];
                }
            }
            csync();
            if (tid == 0)
                mbar_arrive(&uempty[us]);  // the descriptor is consumed
            if (last_chunk && tid < 16 && new_page >= 0 && new_page < a.num_pages)
                store_new_token(a, new_page, g, slot, new_kv);
            Warp w;
            w.init(q_rot, a.scale_log2, lane, scratch + warp * kScratchFloats);
            for (int k = warp; k < jn; k += kWarps) {
                const uint32_t gi = (uint32_t)first + k;
                const int s = gi % kWsRing;
                if (!dead && !mbar_wait_warp(&full[s], (gi / kWsRing) & 1)) {
                    dead = true;
                    if (lane == 0 && a.err)
                        atomicOr(a.err, PKV_DEVERR_TIMEOUT);
                }
                if (!dead) {
                    uint8_t *stage = ring + s * kStageBytes;
                    if (bad[s]) {
                        if (lane == 0 && a.err)
                            atomicOr(a.err, PKV_DEVERR_PAGE_RANGE);
                    } else {
                        const int j = j0 + k;
                        const bool patched = last_chunk && j == npages - 1;
                        if (patched)
                            patch_stage(stage, slot, new_kv, lane);
                        w.page(stage, min(kPage, L - j * kPage));
                        if (patched)  // generic stores into the stage precede the next copy into it
                            fence_proxy_async_smem();
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[s]);
            }
            finish_unit(a, w, state, ticket, q_rot, b, g, c, nchunks, csync);
            ++ui;
        }
    }

    // ---- the last CTA to finish resets the work counter for the next launch
    __syncthreads();
    if (tid == 0) {
        grid_dependency_wait();
        __threadfence();
        if (atomicAdd(exit_counter, 1) == (int)gridDim.x - 1) {
            atomicExch(work_counter, 0);
            atomicExch(exit_counter, 0);
        }
    }
}

// ------------------------------------------------------------------ launch

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

cudaLaunchAttribute pdl_attribute()
{
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    return attr;
}

template <class Warp, int STAGES>
int launch_grid(const CUtensorMap *tmap, const StepArgs &a, int B, cudaStream_t s, bool pdl)
{
    auto kernel = decode_step_kernel<Warp, STAGES>;
    constexpr int smem = SmemLayout<STAGES>::kBaseBytes + kGridExtraBytes;
    static bool attr_set = false;  // set once per process (before any graph capture)
    if (!attr_set) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return PKV_ERR_CUDA;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kHkv, B, a.max_chunks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return status_from_cuda(cudaLaunchKernelEx(&cfg, kernel, *tmap, a));
}

// FP8 pages: ring depth per warp 2..4 units (2176 B each).
template <int STAGES>
int launch_fp8_grid(const CUtensorMap *tmap, const StepArgs &a, int B, cudaStream_t s, bool pdl)
{
    auto kernel = decode_step_fp8_kernel<STAGES>;
    constexpr int smem = Fp8StepSmem<STAGES>::kBytes;
    static bool attr_set = false;  // set once per process (before any graph capture)
    if (!attr_set) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return PKV_ERR_CUDA;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kHkv, B, a.max_chunks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return status_from_cuda(cudaLaunchKernelEx(&cfg, kernel, *tmap, a));
}

int launch_fp8_depth(const CUtensorMap *tmap, const StepArgs &a, int B, cudaStream_t s, bool pdl, int depth)
{
    switch (depth) {
    case 2: return launch_fp8_grid<2>(tmap, a, B, s, pdl);
    case 3: return launch_fp8_grid<3>(tmap, a, B, s, pdl);
    default: return launch_fp8_grid<4>(tmap, a, B, s, pdl);
    }
}

// Ring depth per warp: 2 stages (36 KB per CTA, 6 CTAs per SM), 3 (4 per SM) or 4 (3 per SM).
template <class Warp>
int launch_grid_depth(const CUtensorMap *tmap, const StepArgs &a, int B, cudaStream_t s, bool pdl, int depth)
{
    switch (depth) {
    case 2: return launch_grid<Warp, 2>(tmap, a, B, s, pdl);
    case 3: return launch_grid<Warp, 3>(tmap, a, B, s, pdl);
    default: return launch_grid<Warp, 4>(tmap, a, B, s, pdl);
    }
}

// CTAs per SM the persistent kernel is sized for, and the SM count, per device.
struct PersistentShape {
    int sms = 0;
    int ctas_per_sm = 0;
};

template <class Warp>
int launch_persistent(const CUtensorMap *tmap, const StepArgs &a, int B, cudaStream_t s, bool pdl)
{
    auto kernel = decode_step_persistent_kernel<Warp, kStepStages>;
    constexpr int max_smem = persistent_smem_bytes<kStepStages>(kMaxPersistentBatch);
    constexpr int kMaxDevices = 64;
    static PersistentShape shape[kMaxDevices];  // filled on the first call per device (before any capture)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PKV_ERR_CUDA;
    PersistentShape &ps = shape[dev];
    if (ps.sms == 0) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) != cudaSuccess ||
            cudaDeviceGetAttribute(&ps.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ps.ctas_per_sm, kernel, kThreads, max_smem) !=
                cudaSuccess ||
            ps.ctas_per_sm < 1) {
            ps.sms = 0;
            return PKV_ERR_CUDA;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ps.sms * ps.ctas_per_sm);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = persistent_smem_bytes<kStepStages>(B);
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return status_from_cuda(cudaLaunchKernelEx(&cfg, kernel, *tmap, a, B));
}

template <class Warp>
int launch_ws(const CUtensorMap *tmap, const StepArgs &a, int B, cudaStream_t s, bool pdl)
{
    auto kernel = decode_step_ws_kernel<Warp>;
    constexpr int max_smem = ws_smem_bytes(kMaxPersistentBatch);
    constexpr int kMaxDevices = 64;
    static PersistentShape shape[kMaxDevices];  // filled on the first call per device (before any capture)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PKV_ERR_CUDA;
    PersistentShape &ps = shape[dev];
    if (ps.sms == 0) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) != cudaSuccess ||
            cudaDeviceGetAttribute(&ps.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ps.ctas_per_sm, kernel, kWsThreads, max_smem) !=
                cudaSuccess ||
            ps.ctas_per_sm < 1) {
            ps.sms = 0;
            return PKV_ERR_CUDA;
        }
    }
    int *work_counter = a.counters + (size_t)B * kHkv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ps.sms * ps.ctas_per_sm);
    cfg.blockDim = dim3(kWsThreads);
    cfg.dynamicSmemBytes = ws_smem_bytes(B);
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return status_from_cuda(cudaLaunchKernelEx(&cfg, kernel, *tmap, a, B, work_counter, work_counter + 1));
}

}  // namespace
}  // namespace pkv

extern "C" size_t pkv_decode_step_workspace_bytes(int B, int max_blocks, int pages_per_chunk)
{
    using namespace pkv;
    if (B < 1 || max_blocks < 1 || pages_per_chunk < 1)
        return 0;
    return align256(((size_t)B * kHkv + 2) * sizeof(int)) + pkv_decode_workspace_bytes(B, max_blocks, pages_per_chunk);
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
    const int variant = options & 0xff;
    if (variant < PKV_DECODE_DEFAULT || variant > PKV_DECODE_MMA ||
        (options & ~(0xff | PKV_STEP_NO_PDL | PKV_STEP_GRID | PKV_STEP_PERSISTENT | PKV_STEP_WS |
                     PKV_STEP_RING_MASK | PKV_STEP_EARLY_TRIGGER | PKV_STEP_SORTED)) ||
        (!!(options & PKV_STEP_GRID) + !!(options & PKV_STEP_PERSISTENT) + !!(options & PKV_STEP_WS) > 1))
        return PKV_ERR_INVALID_ARG;
    if ((options & (PKV_STEP_PERSISTENT | PKV_STEP_WS)) && B > kMaxPersistentBatch)
        return PKV_ERR_INVALID_ARG;
    if ((options & PKV_STEP_SORTED) && ((options & (PKV_STEP_PERSISTENT | PKV_STEP_WS)) || B > kMaxSortedBatch))
        return PKV_ERR_INVALID_ARG;  // the sorted order is a grid-schedule option, up to 1024 sequences
    const uintptr_t align = reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
                            reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
                            reinterpret_cast<uintptr_t>(rope_table) | reinterpret_cast<uintptr_t>(workspace);
    if (align & 15u)
        return PKV_ERR_INVALID_ARG;
    if (workspace_bytes < pkv_decode_step_workspace_bytes(B, max_blocks, pages_per_chunk))
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (pool->kv_format == PKV_KV_FP8 &&
        (variant == PKV_DECODE_SIMT || (options & (PKV_STEP_PERSISTENT | PKV_STEP_WS))))
        return PKV_ERR_UNSUPPORTED;  // FP8 pages: the grid schedule and the MMA policy only
    const CUtensorMap *tmap = pool_tensor_map(pool);
    if (!tmap)
        return PKV_ERR_CUDA;
    const int max_chunks = (max_blocks + pages_per_chunk - 1) / pages_per_chunk;
    if (max_chunks > 65535)  // the grid schedule puts the chunk index in gridDim.z
        return PKV_ERR_INVALID_ARG;
    char *ws = static_cast<char *>(workspace);
    const size_t counters_bytes = align256(((size_t)B * kHkv + 2) * sizeof(int));
    const size_t ml_bytes = align256((size_t)B * kHq * max_chunks * sizeof(float2));
    StepArgs a;
    a.num_pages = pool->num_pages;
    a.slab = reinterpret_cast<uint16_t *>(pool->slab);
    a.k_new = k_new;
    a.v_new = v_new;
    a.q = q;
    a.bt = bt_dev;
    a.max_blocks = max_blocks;
    a.seq_lens = seq_lens_dev;
    a.rope = reinterpret_cast<const float2 *>(rope_table);
    a.max_pos = max_pos;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.pages_per_chunk = pages_per_chunk;
    a.counters = reinterpret_cast<int *>(ws);
    a.part_ml = reinterpret_cast<float2 *>(ws + counters_bytes);
    a.part_o = reinterpret_cast<float *>(ws + counters_bytes + ml_bytes);
    a.max_chunks = max_chunks;
    a.out = out;
    a.err = dev_err_flag;
    a.early_trigger = (options & PKV_STEP_EARLY_TRIGGER) ? 1 : 0;
    a.sorted = (options & PKV_STEP_SORTED) ? 1 : 0;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const bool pdl = !(options & PKV_STEP_NO_PDL);
    // the grid schedule is the measured default; the persistent one is chosen explicitly
    if (options & PKV_STEP_WS)
        return variant == PKV_DECODE_SIMT ? launch_ws<SimtWarp>(tmap, a, B, s, pdl)
                                          : launch_ws<MmaWarp>(tmap, a, B, s, pdl);
    const bool persistent = (options & PKV_STEP_PERSISTENT) != 0;
    if (persistent)
        return variant == PKV_DECODE_SIMT ? launch_persistent<SimtWarp>(tmap, a, B, s, pdl)
                                          : launch_persistent<MmaWarp>(tmap, a, B, s, pdl);
    const int ring = (options & PKV_STEP_RING_MASK) >> 12;
    if (ring != 0 && (ring < 2 || ring > 4))
        return PKV_ERR_INVALID_ARG;
    const int depth = ring ? ring : kDefaultGridRing;
    if (pool->kv_format == PKV_KV_FP8)
        return launch_fp8_depth(tmap, a, B, s, pdl, depth);
    return variant == PKV_DECODE_SIMT ? launch_grid_depth<SimtWarp>(tmap, a, B, s, pdl, depth)
                                      : launch_grid_depth<MmaWarp>(tmap, a, B, s, pdl, depth);
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
