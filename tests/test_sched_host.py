"""CPU tests of the native request scheduler (pkv_sched_*): page-budget admission,
FIFO waiting, rejection, lazy page allocation, finish and early stop, static vs
continuous batching, statistics.

Rules (samir-vllm README summary, section "当前范围"): a request reserves
prompt + allowed_new - 1 tokens rounded up to 16-token pages in every layer, as
credits separate from physical pages; allowed_new is capped by the context;
requests wait in FIFO order; a budget larger than the pool is rejected; pages are
taken lazily and returned, with the credits, on finish.  `RefScheduler` below
restates those rules in plain Python, independently of the C++ code, and random
traces are checked against it step by step.
"""
import math

import numpy as np
import pytest

from paged_kv_decode_12_gb300 import pkv

FAKE_SLAB = 0x7F0000000000
PS = 16


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_decode_12_gb300 import _build

    _build.build()


def make(pages, layers=2, max_blocks=8, ctx=128, max_batch=64, mode=pkv.PKV_SCHED_CONTINUOUS, seed=3):
    pool = pkv.pkv_pool_create(FAKE_SLAB, pages * pkv.PKV_PAGE_BYTES, seed=seed)
    sched = pkv.pkv_sched_create(pool, layers, max_blocks, ctx, max_batch, mode)
    return pool, sched


class RefScheduler:
    """Plain restatement of the admission rules (no page ids, only counts)."""

    def __init__(self, pages, layers, ctx, max_batch, static):
        self.credits, self.layers, self.ctx, self.max_batch, self.static = pages, layers, ctx, max_batch, static
        self.total = pages
        self.waiting, self.active = [], []
        self.waits = 0

    def budget(self, prompt, new):
        allowed = min(new, self.ctx + 1 - prompt)
        return allowed, math.ceil((prompt + allowed - 1) / PS) * self.layers

    def submit(self, rid, prompt, new):
        allowed, b = self.budget(prompt, new)
        if b > self.total:
            return False
        self.waiting.append(dict(id=rid, prompt=prompt, allowed=allowed, budget=b, length=prompt,
                                 remaining=allowed - 1))
        return True

    def retire(self):
        for r in [r for r in self.active if r["remaining"] <= 0]:
            self.active.remove(r)
            self.credits += r["budget"]

    def admit(self):
        self.retire()
        if self.static and self.active:
            return []
        out = []
        while self.waiting and len(self.active) < self.max_batch:
            head = self.waiting[0]
            if head["budget"] > self.credits:
                self.waits += 1
                break
            self.waiting.pop(0)
            self.credits -= head["budget"]
            self.active.append(head)
            out.append(head["id"])
        return out

    def decode(self):
        self.retire()
        for r in self.active:
            r["length"] += 1
            r["remaining"] -= 1
        return [r["id"] for r in self.active], [r["length"] for r in self.active]

    def allocated(self):
        return sum(math.ceil(r["length"] / PS) * self.layers for r in self.active)


def test_budget_rejection_and_validation():
    pool, s = make(pages=10, layers=2)
    # prompt 100 + 29 allowed (capped: 128 + 1 - 100) - 1 = 128 tokens -> 8 pages x 2 layers = 16 > 10
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_sched_submit(s, 1, 100, 500)
    assert e.value.status == pkv.PKV_ERR_BUDGET_EXCEEDS_POOL
    for bad in [(2, 0, 5), (3, 10, 0), (4, 129, 5)]:
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_sched_submit(s, *bad)
        assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    pkv.pkv_sched_submit(s, 5, 16, 1)                       # 16 tokens -> 1 page x 2
    with pytest.raises(pkv.PkvError):
        pkv.pkv_sched_submit(s, 5, 16, 1)                   # duplicate id
    st = pkv.pkv_sched_get_stats(s)
    assert st["rejected"] == 1 and st["submitted"] == 2 and st["pool_pages"] == 10
    pkv.pkv_sched_destroy(s)
    pkv.pkv_pool_destroy(pool)


def test_fifo_head_blocks_later_requests():
    pool, s = make(pages=20, layers=2)
    pkv.pkv_sched_submit(s, 1, 60, 30)    # 89 tokens -> 6 pages x 2 = 12 credits
    pkv.pkv_sched_submit(s, 2, 60, 30)    # 12 credits: does not fit beside request 1
    pkv.pkv_sched_submit(s, 3, 10, 2)     # 11 tokens -> 2 credits: fits, but must not overtake 2
    ids, lens, bt = pkv.pkv_sched_admit(s, 8, 2, 8)
    assert ids.tolist() == [1] and lens.tolist() == [60]
    assert np.all(bt[0, :, :4] >= 0) and np.all(bt[0, :, 4:] == -1)   # 60 tokens: 4 pages now (lazy)
    st = pkv.pkv_sched_get_stats(s)
    assert st["admission_waits"] == 1 and st["waiting"] == 2 and st["allocated_pages"] == 8
    pkv.pkv_sched_finish(s, 1)            # early stop returns pages and credits
    ids, _, _ = pkv.pkv_sched_admit(s, 8, 2, 8)
    assert ids.tolist() == [2, 3]
    pkv.pkv_sched_destroy(s)
    pkv.pkv_pool_destroy(pool)


def test_lazy_growth_and_retirement():
    pool, s = make(pages=64, layers=3)
    pkv.pkv_sched_submit(s, 7, 15, 4)     # decode positions 15, 16, 17: page 1 is taken at length 17
    ids, lens, bt0 = pkv.pkv_sched_admit(s, 4, 3, 8)
    assert pkv.pkv_sched_get_stats(s)["allocated_pages"] == 3
    seen = []
    for step in range(3):
        ids, lens, bt = pkv.pkv_sched_decode_batch(s, 4, 3, 8)
        seen.append((ids.tolist(), lens.tolist()))
        npages = math.ceil(lens[0] / PS)
        assert np.all(bt[:, 0, :npages] >= 0) and np.all(bt[:, 0, npages:] == -1)
        assert np.array_equal(bt[:, 0, 0], bt0[0, :, 0])          # earlier pages never move
    assert seen == [([7], [16]), ([7], [17]), ([7], [18])]  # 4 allowed tokens -> 3 decode steps
    ids, _, _ = pkv.pkv_sched_decode_batch(s, 4, 3, 8)          # retired before the next step
    assert ids.size == 0
    st = pkv.pkv_sched_get_stats(s)
    assert st["finished"] == 1 and st["allocated_pages"] == 0 and st["final_free_pages"] == 64
    assert st["peak_allocated_pages"] == 6 and st["free_credits"] == 64
    pkv.pkv_sched_destroy(s)
    pkv.pkv_pool_destroy(pool)


def test_static_batching_waits_for_the_group():
    pool, s = make(pages=64, layers=1, mode=pkv.PKV_SCHED_STATIC)
    pkv.pkv_sched_submit(s, 1, 10, 4)                            # 3 decode steps
    pkv.pkv_sched_submit(s, 2, 10, 2)                            # 1 decode step
    ids, _, _ = pkv.pkv_sched_admit(s, 8, 1, 8)
    assert ids.tolist() == [1, 2]
    pkv.pkv_sched_submit(s, 3, 10, 2)
    assert pkv.pkv_sched_decode_batch(s, 8, 1, 8)[0].tolist() == [1, 2]
    assert pkv.pkv_sched_admit(s, 8, 1, 8)[0].size == 0          # group still running
    assert pkv.pkv_sched_decode_batch(s, 8, 1, 8)[0].tolist() == [1]   # request 2 retired
    assert pkv.pkv_sched_admit(s, 8, 1, 8)[0].size == 0
    assert pkv.pkv_sched_decode_batch(s, 8, 1, 8)[0].tolist() == [1]   # request 1's last step
    ids, _, _ = pkv.pkv_sched_admit(s, 8, 1, 8)                  # group done: next group
    assert ids.tolist() == [3]
    pkv.pkv_sched_destroy(s)
    pkv.pkv_pool_destroy(pool)


def test_batch_cap():
    pool, s = make(pages=256, layers=1, max_batch=3)
    for i in range(5):
        pkv.pkv_sched_submit(s, i, 20, 10)
    assert pkv.pkv_sched_admit(s, 8, 1, 8)[0].tolist() == [0, 1, 2]
    ids, lens, bt = pkv.pkv_sched_decode_batch(s, 8, 1, 8)
    assert ids.tolist() == [0, 1, 2] and pkv.pkv_sched_get_stats(s)["max_decode_batch"] == 3
    pkv.pkv_sched_destroy(s)
    pkv.pkv_pool_destroy(pool)


@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_trace_matches_reference(seed, static):
    rng = np.random.default_rng(seed)
    layers, max_blocks, ctx, pages, max_batch = 4, 16, 256, 160, 12
    mode = pkv.PKV_SCHED_STATIC if static else pkv.PKV_SCHED_CONTINUOUS
    pool, s = make(pages, layers, max_blocks, ctx, max_batch, mode, seed=seed)
    ref = RefScheduler(pages, layers, ctx, max_batch, static)
    rid = 0
    for step in range(300):
        for _ in range(int(rng.poisson(0.5))):
            prompt, new = int(rng.integers(1, 200)), int(rng.integers(1, 120))
            ok = ref.submit(rid, prompt, new)
            if ok:
                pkv.pkv_sched_submit(s, rid, prompt, new)
            else:
                with pytest.raises(pkv.PkvError):
                    pkv.pkv_sched_submit(s, rid, prompt, new)
            rid += 1
        got, _, bt_rows = pkv.pkv_sched_admit(s, 64, layers, max_blocks)
        assert got.tolist() == ref.admit()
        ids, lens, bt = pkv.pkv_sched_decode_batch(s, 64, layers, max_blocks)
        rids, rlens = ref.decode()
        assert ids.tolist() == rids and lens.tolist() == rlens
        # every (request, layer) row holds exactly its pages, and no page is held twice
        held = []
        for b, L in enumerate(lens):
            n = math.ceil(L / PS)
            assert np.all(bt[:, b, :n] >= 0) and np.all(bt[:, b, n:] == -1)
            held.extend(bt[:, b, :n].ravel().tolist())
        assert len(held) == len(set(held))
        st = pkv.pkv_sched_get_stats(s)
        assert st["allocated_pages"] == ref.allocated() <= pages - st["free_credits"]
        assert st["final_free_pages"] == pages - st["allocated_pages"]
        assert st["admission_waits"] == ref.waits
    pkv.pkv_sched_destroy(s)
    pkv.pkv_pool_destroy(pool)


def test_outputs_written_into_given_arrays():
    # the trace runner hands the scheduler views of pinned host buffers; the results must be
    # exactly those of the wrapper-allocated call, written in place (the block tables of a
    # decode batch compact: layer l's rows start at l * B * max_blocks)
    results = []
    for given in (False, True):
        pool, sched = make(64, layers=2, max_blocks=8, max_batch=4)
        for rid, (p, n) in enumerate([(20, 5), (40, 3), (3, 9)]):
            pkv.pkv_sched_submit(sched, rid, p, n)
        bufs = dict(ids_out=np.full(4, -7, np.int64), lens_out=np.full(4, -7, np.int32),
                    bt_out=np.full(4 * 2 * 8, -7, np.int32)) if given else {}
        a = pkv.pkv_sched_admit(sched, 4, 2, 8, **bufs)
        if given:
            assert np.shares_memory(a[2], bufs["bt_out"]) and np.shares_memory(a[0], bufs["ids_out"])
        dbufs = dict(ids_out=np.full(4, -7, np.int64), lens_out=np.full(4, -7, np.int32),
                     bt_out=np.full(2 * 4 * 8, -7, np.int32)) if given else {}
        d = pkv.pkv_sched_decode_batch(sched, 4, 2, 8, **dbufs)
        if given:
            B = d[0].size
            assert np.array_equal(dbufs["bt_out"][: 2 * B * 8], d[2].reshape(-1))
        results.append([np.array(x) for x in a + d])
        pkv.pkv_sched_destroy(sched)
        pkv.pkv_pool_destroy(pool)
    for x, y in zip(*results):
        assert np.array_equal(x, y)
    pool, sched = make(8)
    with pytest.raises(ValueError):     # too small / wrong dtype output arrays are refused
        pkv.pkv_sched_decode_batch(sched, 4, 2, 8, bt_out=np.empty(10, np.int32))
    with pytest.raises(ValueError):
        pkv.pkv_sched_admit(sched, 4, 2, 8, ids_out=np.empty(4, np.int32))
    pkv.pkv_sched_destroy(sched)
    pkv.pkv_pool_destroy(pool)


def test_pages_taken_outside_the_scheduler():
    # credits are the pool's free pages when the scheduler was created; pages a caller takes
    # from the pool directly afterwards make allocations fail: admission then waits (nothing
    # of the head is allocated) and a decode step advances no request until pages are back
    pool, s = make(pages=12, layers=2)
    outside = pkv.pkv_pool_alloc(pool, 9)                       # 3 pages left
    pkv.pkv_sched_submit(s, 1, 48, 2)                           # 49 tokens: 4 pages x 2 layers of credit
    ids, _, _ = pkv.pkv_sched_admit(s, 4, 2, 8)                 # its prompt needs 3 x 2 = 6 pages now
    st = pkv.pkv_sched_get_stats(s)
    assert ids.size == 0 and st["waiting"] == 1 and st["admission_waits"] == 1
    assert st["allocated_pages"] == 0 and st["free_credits"] == 12 and st["final_free_pages"] == 3
    pkv.pkv_pool_free(pool, outside[:6])                        # 9 free
    ids, lens, bt = pkv.pkv_sched_admit(s, 4, 2, 8)
    assert ids.tolist() == [1] and lens.tolist() == [48] and np.all(bt[0, :, :3] >= 0)
    assert pkv.pkv_sched_get_stats(s)["allocated_pages"] == 6
    again = pkv.pkv_pool_alloc(pool, 3)                         # the pool is empty now
    with pytest.raises(pkv.PkvError) as e:                      # length 49 needs page 3 in both layers
        pkv.pkv_sched_decode_batch(s, 4, 2, 8)
    assert e.value.status == pkv.PKV_ERR_OUT_OF_PAGES
    st = pkv.pkv_sched_get_stats(s)
    assert st["allocated_pages"] == 6 and st["final_free_pages"] == 0
    pkv.pkv_pool_free(pool, again)
    ids, lens, bt = pkv.pkv_sched_decode_batch(s, 4, 2, 8)      # repeated: the request advances once
    assert ids.tolist() == [1] and lens.tolist() == [49] and np.all(bt[:, 0, :4] >= 0)
    assert pkv.pkv_sched_get_stats(s)["allocated_pages"] == 8
    pkv.pkv_sched_destroy(s)
    pkv.pkv_pool_free(pool, outside[6:])
    pkv.pkv_pool_destroy(pool)
