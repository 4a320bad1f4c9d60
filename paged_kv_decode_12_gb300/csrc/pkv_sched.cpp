// pkv_sched.cpp -- host-side request scheduler over the page pool: page-budget
// admission, FIFO waiting, lazy page allocation, continuous or static batching.
//
// Rules restated from the samir-vllm README summary ("从零用 C++ 和 CUDA 实现
// Llama 3.2 1B 推理引擎"), section "当前范围" (current scope):
//  * admission reserves, for each request, its largest processed prefix:
//    prompt_tokens + allowed_new_tokens - 1, rounded up to 16-token pages in every
//    one of the layers; the allowed output budget is capped by the context limit
//    (the last predicted token is returned without being processed);
//  * these admission credits are separate from physical pages, which are taken
//    lazily, when a sequence first needs them; finishing (or stopping early)
//    returns both the pages and the remaining credits;
//  * when a budget cannot coexist with the active requests, requests wait in FIFO
//    order; active requests always have room to finish, so growth across page
//    boundaries never exhausts the pool and nothing deadlocks; a budget larger
//    than the whole pool is rejected with an explicit error; no preemption;
//  * the statistics of --stats: pool size, peak active requests, largest decode
//    batch, peak allocated pages, admission waits, final free pages;
//  * prompts are prefilled one at a time between decode iterations; continuous
//    batching admits waiting requests whenever credits allow, static batching
//    admits the next group only after the current group has finished
//    (same page, "构建": --static / --continuous).
#include <algorithm>
#include <deque>
#include <new>
#include <unordered_set>
#include <vector>

#include "pkv_internal.h"

struct pkv_sched {
    pkv_pool *pool = nullptr;
    int layers = 0, max_blocks = 0, max_context = 0, max_batch = 0, mode = 0;
    int64_t total_credits = 0, free_credits = 0;
    struct Req {
        int64_t id = 0;
        int prompt = 0, allowed = 0;  // allowed output tokens (capped by the context)
        int length = 0;               // tokens whose K/V are (or are being) written
        int remaining = 0;            // decode steps still to run
        int64_t budget_pages = 0;     // credits held
        int npages = 0;               // physical pages per layer so far
        std::vector<int32_t> pages;   // [layers][max_blocks], -1 padded
    };
    std::deque<Req> waiting;
    std::vector<Req> active;       // admission order = decode batch order
    std::unordered_set<int64_t> ids;  // submitted and not yet finished
    pkv_sched_stats st = {};
    int64_t allocated = 0;
};

namespace {

int64_t pages_for(int tokens) { return (tokens + PKV_PAGE_SIZE - 1) / PKV_PAGE_SIZE; }

// Give every layer of r the pages it needs for `tokens` tokens, all or nothing.  The
// credits guarantee success while the scheduler is the pool's only user; if pages were
// taken from the pool outside it, the pages this call took go back and the status of the
// failed allocation is returned, with r unchanged.
int grow(pkv_sched *s, pkv_sched::Req &r, int tokens)
{
    const int need = (int)pages_for(tokens);
    if (need > s->max_blocks)
        return PKV_ERR_INVALID_ARG;
    if (need <= r.npages)
        return PKV_OK;
    const int add = need - r.npages;
    for (int l = 0; l < s->layers; ++l) {
        int32_t *row = &r.pages[(size_t)l * s->max_blocks];
        const int st = pkv_pool_alloc(s->pool, add, row + r.npages);
        if (st != PKV_OK) {
            for (int k = 0; k < l; ++k) {  // undo the layers already grown
                int32_t *done = &r.pages[(size_t)k * s->max_blocks] + r.npages;
                (void)pkv_pool_free(s->pool, add, done);
                std::fill(done, done + add, -1);
            }
            return st;
        }
    }
    s->allocated += (int64_t)add * s->layers;
    r.npages = need;
    if (s->allocated > s->st.peak_allocated_pages)
        s->st.peak_allocated_pages = s->allocated;
    return PKV_OK;
}

void release(pkv_sched *s, pkv_sched::Req &r)
{
    for (int l = 0; l < s->layers; ++l) {
        const int32_t *row = &r.pages[(size_t)l * s->max_blocks];
        if (r.npages > 0)
            (void)pkv_pool_free(s->pool, r.npages, row);
    }
    s->allocated -= (int64_t)r.npages * s->layers;
    s->free_credits += r.budget_pages;
    s->ids.erase(r.id);
    ++s->st.finished;
}

// Requests whose last decode step has run leave; their pages and credits return.
void retire_done(pkv_sched *s)
{
    std::vector<pkv_sched::Req> keep;
    keep.reserve(s->active.size());
    for (auto &r : s->active) {
        if (r.remaining <= 0)
            release(s, r);
        else
            keep.push_back(std::move(r));
    }
    s->active.swap(keep);
}

void refresh_free(pkv_sched *s)
{
    int nf = 0;
    (void)pkv_pool_info(s->pool, nullptr, nullptr, nullptr, nullptr, &nf);
    s->st.final_free_pages = nf;
}

}  // namespace

extern "C" {

int pkv_sched_create(pkv_pool *pool, int layers, int max_blocks, int max_context, int max_batch, int mode,
                     pkv_sched **out)
{
    if (!out)
        return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    if (!pool || layers < 1 || max_blocks < 1 || max_context < 1 || max_batch < 1 ||
        (mode != PKV_SCHED_CONTINUOUS && mode != PKV_SCHED_STATIC) ||
        pages_for(max_context) > max_blocks)
        return PKV_ERR_INVALID_ARG;
    int num_pages = 0, num_free = 0;
    (void)pkv_pool_info(pool, nullptr, nullptr, nullptr, &num_pages, &num_free);
    pkv_sched *s = new (std::nothrow) pkv_sched();
    if (!s)
        return PKV_ERR_INVALID_ARG;
    s->pool = pool;
    s->layers = layers;
    s->max_blocks = max_blocks;
    s->max_context = max_context;
    s->max_batch = max_batch;
    s->mode = mode;
    s->total_credits = s->free_credits = num_free;  // credits are drawn from the pages free now
    s->st.pool_pages = num_pages;
    s->st.final_free_pages = num_free;
    *out = s;
    return PKV_OK;
}

int pkv_sched_destroy(pkv_sched *s)
{
    if (s) {
        for (auto &r : s->active)
            release(s, r);
    }
    delete s;
    return PKV_OK;
}

int pkv_sched_submit(pkv_sched *s, int64_t id, int prompt_tokens, int max_new_tokens)
{
    if (!s || prompt_tokens < 1 || max_new_tokens < 1 || prompt_tokens > s->max_context)
        return PKV_ERR_INVALID_ARG;
    if (s->ids.count(id))
        return PKV_ERR_INVALID_ARG;
    ++s->st.submitted;
    pkv_sched::Req r;
    r.id = id;
    r.prompt = prompt_tokens;
    // the processed prefix prompt + allowed - 1 may not exceed the context
    r.allowed = max_new_tokens;
    if (r.allowed > s->max_context + 1 - prompt_tokens)
        r.allowed = s->max_context + 1 - prompt_tokens;
    r.budget_pages = pages_for(prompt_tokens + r.allowed - 1) * s->layers;
    if (r.budget_pages > s->total_credits) {
        ++s->st.rejected;
        return PKV_ERR_BUDGET_EXCEEDS_POOL;
    }
    s->ids.insert(id);
    s->waiting.push_back(std::move(r));
    return PKV_OK;
}

int pkv_sched_admit(pkv_sched *s, int max_n, int64_t *ids_out, int32_t *prompt_lens_out, int32_t *bt_rows_out,
                    int *n_out)
{
    if (!s || max_n < 0 || !n_out || (max_n > 0 && (!ids_out || !prompt_lens_out || !bt_rows_out)))
        return PKV_ERR_INVALID_ARG;
    *n_out = 0;
    retire_done(s);
    if (s->mode == PKV_SCHED_STATIC && !s->active.empty())
        return PKV_OK;  // static batching: the current group must finish first
    int n = 0;
    while (!s->waiting.empty() && n < max_n && (int)s->active.size() < s->max_batch) {
        pkv_sched::Req &head = s->waiting.front();
        if (head.budget_pages > s->free_credits) {
            ++s->st.admission_waits;  // FIFO: nobody overtakes the head
            break;
        }
        head.pages.assign((size_t)s->layers * s->max_blocks, -1);
        if (grow(s, head, head.prompt) != PKV_OK) {
            // pages were taken from the pool outside the scheduler: the head waits, as for
            // credits, until enough pages are back
            ++s->st.admission_waits;
            break;
        }
        pkv_sched::Req r = std::move(head);
        s->waiting.pop_front();
        s->free_credits -= r.budget_pages;
        r.length = r.prompt;
        r.remaining = r.allowed - 1;
        ids_out[n] = r.id;
        prompt_lens_out[n] = r.prompt;
        std::copy(r.pages.begin(), r.pages.end(), bt_rows_out + (size_t)n * s->layers * s->max_blocks);
        s->active.push_back(std::move(r));
        ++n;
        ++s->st.admitted;
    }
    if ((int64_t)s->active.size() > s->st.peak_active)
        s->st.peak_active = (int64_t)s->active.size();
    *n_out = n;
    refresh_free(s);
    return PKV_OK;
}

int pkv_sched_decode_batch(pkv_sched *s, int max_b, int64_t *ids_out, int32_t *seq_lens_out, int32_t *bt_out,
                           int *B_out)
{
    if (!s || !B_out || max_b < 0 || (max_b > 0 && (!ids_out || !seq_lens_out || !bt_out)))
        return PKV_ERR_INVALID_ARG;
    *B_out = 0;
    // requests whose last decode step has run leave now (their pages are free for the
    // next admission; later GPU work is ordered after that step on the stream)
    retire_done(s);
    const int B = (int)s->active.size();
    if (B > max_b)
        return PKV_ERR_INVALID_ARG;
    // every new token's page first (lazily), then the step: a failed allocation advances
    // no request, and the pages already taken stay with their requests (within budget)
    for (int i = 0; i < B; ++i) {
        const int st = grow(s, s->active[i], s->active[i].length + 1);
        if (st != PKV_OK) {
            refresh_free(s);
            return st;
        }
    }
    for (int i = 0; i < B; ++i) {
        pkv_sched::Req &r = s->active[i];
        r.length += 1;
        r.remaining -= 1;
        ids_out[i] = r.id;
        seq_lens_out[i] = r.length;
    }
    for (int l = 0; l < s->layers; ++l)
        for (int i = 0; i < B; ++i)
            std::copy(&s->active[i].pages[(size_t)l * s->max_blocks],
                      &s->active[i].pages[(size_t)l * s->max_blocks] + s->max_blocks,
                      bt_out + ((size_t)l * B + i) * s->max_blocks);
    if (B > s->st.max_decode_batch)
        s->st.max_decode_batch = B;
    *B_out = B;
    refresh_free(s);
    return PKV_OK;
}

int pkv_sched_finish(pkv_sched *s, int64_t id)
{
    if (!s)
        return PKV_ERR_INVALID_ARG;
    for (size_t i = 0; i < s->active.size(); ++i) {
        if (s->active[i].id == id) {
            release(s, s->active[i]);
            s->active.erase(s->active.begin() + (std::ptrdiff_t)i);
            refresh_free(s);
            return PKV_OK;
        }
    }
    for (auto it = s->waiting.begin(); it != s->waiting.end(); ++it) {
        if (it->id == id) {
            s->ids.erase(id);
            s->waiting.erase(it);
            return PKV_OK;
        }
    }
    return PKV_ERR_INVALID_ARG;
}

int pkv_sched_get_stats(const pkv_sched *s, pkv_sched_stats *out)
{
    if (!s || !out)
        return PKV_ERR_INVALID_ARG;
    *out = s->st;
    out->active = (int64_t)s->active.size();
    out->waiting = (int64_t)s->waiting.size();
    out->allocated_pages = s->allocated;
    out->free_credits = s->free_credits;
    return PKV_OK;
}

}  // extern "C"
