"""The host half of LORA_DEBUG_CHECKS (CPU only).

lora_plan_check plans a table and checks every index the kernels derive from the plan against the buffer it
addresses.  These tests run it on the workloads' full-size tables and on many seeded random tables (decode,
prefill and fine-tuning segments, ranks 1..128, ragged K and N, sliced layers), forward and backward; and they
plant a mistake in a copy of the planner, built on its own with the host compiler, and check that the checker
reports it.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import lora_co_serving_gb300 as lm
import workloads
from gpu_util import RESPLIT_SMALL, grad_split_table

CSRC = os.path.join(os.path.dirname(lm.__file__), "csrc")
INCLUDE = os.path.join(os.path.dirname(os.path.dirname(lm.__file__)), "include")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lm.build()
    lm.library()


def _pool(wl):
    return lm.Pool(None, None, wl.a_off, wl.b_off, wl.rank, wl.scale)


def _check(wl, bounds=None):
    for bwd in (False, True):
        lm.plan_check(wl.T, wl.K, wl.N, _pool(wl), wl.segs, backward=bwd, bounds=bounds)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_full_size_tables(cfg):
    kw = {"K": 512, "N": 1024} if cfg in (3, 4, 5) else {}
    _check(workloads.config(cfg, **kw))


def _random_table(rng):
    n_ad = int(rng.integers(1, 40))
    rank = [int(rng.integers(1, 129)) for _ in range(n_ad)]
    segs, t, n_train = [], 0, 0
    for _ in range(int(rng.integers(1, 60))):
        kind = rng.integers(0, 3)
        if kind == 0:
            ln, tr = 1, 0
        elif kind == 1:
            ln, tr = int(rng.integers(2, 700)), 0
        else:
            ln, tr = int(rng.integers(1, 600)), 1
        if tr and n_train >= 40:
            tr = 0
        a = int(rng.integers(0 if tr else -1, n_ad))
        segs.append((t, ln, a, tr))
        n_train += tr
        t += ln
    order = rng.permutation(len(segs))
    return [segs[i] for i in order], t, rank


@pytest.mark.parametrize("seed", range(12))
def test_random_tables(seed):
    rng = np.random.default_rng(seed)
    segs, T, rank = _random_table(rng)
    K = int(rng.choice([8, 64, 136, 520, 1024]))
    N = int(rng.choice([8, 72, 256, 776, 2048]))
    _check(workloads.custom(seed, T, K, N, segs, rank, want_dy=False))


@pytest.mark.parametrize("seed", range(4))
def test_random_sliced_tables(seed):
    rng = np.random.default_rng(100 + seed)
    segs, T, rank = _random_table(rng)
    S = int(rng.integers(2, 5))
    widths = [256 * int(rng.integers(1, 4)) for _ in range(S - 1)] + [int(rng.choice([8, 136, 256]))]
    bounds = np.concatenate([[0], np.cumsum(widths)]).astype(np.int32)
    wl = workloads.sliced(seed, T, int(rng.choice([64, 520])), bounds, segs, rank, want_dy=False)
    _check(wl, bounds=bounds)


# A driver for a planner built on its own with g++: validate, plan, check (the same calls lora_plan_check makes).
DRIVER = r'''
#include <string>
#include "plan.h"
namespace lora { void set_last_error(const char*) {} }
extern "C" int check_table(int T, int K, int N, const lora_pool_t* pool, const lora_segment_t* segs, int n,
                           int backward) {
    lora::Problem p;
    std::string err;
    int rc = lora::validate(T, K, N, LORA_BF16, pool, segs, n, &p, &err);
    if (rc) return rc;
    lora::Plan pl;
    if (backward) lora::plan_backward(p, true, true, true, true, &pl);
    else lora::plan_forward(p, &pl);
    return lora::check_plan(p, pl, backward != 0, &err);
}
// number of items of the backward's gradient launch (-1: the table does not validate); slices may be NULL
extern "C" int grad_items(int T, int K, int N, const lora_pool_t* pool, const lora_slices_t* slices,
                          const lora_segment_t* segs, int n) {
    lora::Problem p;
    std::string err;
    if (lora::validate(T, K, N, LORA_BF16, pool, segs, n, &p, &err, slices)) return -1;
    lora::Plan pl;
    lora::plan_backward(p, true, true, true, true, &pl);
    return int(pl.items[2].size());
}
// assign_items on n random items over G CTAs against a plain greedy (each item, in order, to the CTA with the least
// summed estimated cost, the lowest index on a tie): 0 when the two agree
extern "C" int assign_matches_greedy(int n, int G, unsigned seed) {
    std::vector<lora::WorkItem> items(n);
    unsigned x = seed * 2654435761u + 1u;
    auto rnd = [&](unsigned m) { x ^= x << 13; x ^= x >> 17; x ^= x << 5; return int(x % m); };
    for (auto& w : items) {
        w = lora::WorkItem{};
        w.kind = rnd(7);
        w.nk = 1 + rnd(200);
        w.n_ext = rnd(40);
        w.mma_n = 16 * (1 + rnd(16));
    }
    lora::Plan pl;
    std::vector<int32_t> off, lst;
    lora::assign_items(items, pl, G, &off, &lst);
    std::vector<int64_t> load(G, 0);
    std::vector<std::vector<int32_t>> mine(G);
    for (int i = 0; i < n; ++i) {
        int best = 0;
        for (int c = 1; c < G; ++c)
            if (load[c] < load[best]) best = c;
        load[best] += lora::item_cost_estimate(items[i]);
        mine[best].push_back(i);
    }
    if ((int)off.size() != G + 1 || (int)lst.size() != n) return 1;
    for (int c = 0; c < G; ++c) {
        if (off[c + 1] - off[c] != (int)mine[c].size()) return 2;
        for (size_t j = 0; j < mine[c].size(); ++j)
            if (lst[off[c] + j] != mine[c][j]) return 3;
    }
    return 0;
}
// backward shrink items: out[0] of the dY B^T passes, out[1] of the x A recompute (-1: the table does not validate)
extern "C" int bwd_shrink_items(int T, int K, int N, const lora_pool_t* pool, const lora_segment_t* segs, int n,
                                int* out) {
    lora::Problem p;
    std::string err;
    if (lora::validate(T, K, N, LORA_BF16, pool, segs, n, &p, &err)) return -1;
    lora::Plan pl;
    lora::plan_backward(p, true, true, true, true, &pl);
    out[0] = out[1] = 0;
    for (const lora::WorkItem& w : pl.items[0]) out[w.kind == lora::kShrinkDyb ? 0 : 1]++;
    return 0;
}
'''

def _build_driver(tmp_path, src):
    (tmp_path / "plan.cpp").write_text(src)
    (tmp_path / "driver.cpp").write_text(DRIVER)
    so = str(tmp_path / "libplan.so")
    cxx = os.environ.get("CXX", "g++")
    res = subprocess.run([cxx, "-O1", "-std=c++17", "-shared", "-fPIC", "-I", CSRC, "-I", INCLUDE,
                          str(tmp_path / "plan.cpp"), str(tmp_path / "driver.cpp"), "-o", so],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    lib = ctypes.CDLL(so)
    lib.check_table.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    lib.grad_items.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p] * 3 + [ctypes.c_int]
    lib.bwd_shrink_items.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2 + [ctypes.c_int, ctypes.c_void_p]
    lib.assign_matches_greedy.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint]
    return lib


def _decode_table():
    """Decode rows (atoms of several adapters) and a small split main pass."""
    return workloads.config2(T=256, K=256, N=512, n_adapters=20)


# (name, original text in plan.cpp, planted mistake, table, backward)
PLANTED = [
    ("atom_row_past_block", "pl->atoms_a.push_back(ch.prow_a + sl * ch.r + std::min(o, last));",
     "pl->atoms_a.push_back(ch.prow_a + sl * ch.r + o + 8);", _decode_table, 0),
    ("split_slot_reused", "pl->main_slots += nsplit;", "pl->main_slots += nsplit - 1;", _decode_table, 0),
    ("grad_split_partial_overlap", "v.part = u.part0 + sp * w.mma_n;", "v.part = u.part0;", grad_split_table, 1),
]


@pytest.mark.parametrize("name,orig,bad,table,backward", PLANTED, ids=[p[0] for p in PLANTED])
def test_planted_planner_mistake_is_reported(tmp_path, name, orig, bad, table, backward):
    src = open(os.path.join(CSRC, "plan.cpp")).read()
    assert src.count(orig) == 1, "anchor not unique: " + orig
    lib = _build_driver(tmp_path, src.replace(orig, bad))
    wl = table()
    pool = _pool(wl)
    segs = lm.segments(wl.segs)
    rc = lib.check_table(wl.T, wl.K, wl.N, pool.cptr(), segs.ctypes.data, segs.shape[0], backward)
    assert rc == -12, "planted mistake %s not reported (rc %d)" % (name, rc)


@pytest.mark.parametrize("sliced", [False, True], ids=["plain", "sliced"])
def test_gradient_items_split_three_ways(tmp_path, sliced):
    """The tables of the GPU tests of split gradients do split: 12 gradient items (16 on the sliced layer), each
    into 3 token ranges (the shortest group has 25 token blocks; 4 ways would leave splits under 8 blocks)."""
    lib = _build_driver(tmp_path, open(os.path.join(CSRC, "plan.cpp")).read())
    wl = grad_split_table(sliced=sliced)
    pool = _pool(wl)
    segs = lm.segments(wl.segs)
    sl = lm.Slices(wl.bounds) if sliced else None
    n = lib.grad_items(wl.T, wl.K, wl.N, pool.cptr(), sl.cptr() if sl else None, segs.ctypes.data, segs.shape[0])
    assert n == (48 if sliced else 36)
    if not sliced:
        assert lib.check_table(wl.T, wl.K, wl.N, pool.cptr(), segs.ctypes.data, segs.shape[0], 1) == 0
    else:
        lm.plan_check(wl.T, wl.K, wl.N, pool, wl.segs, backward=True, bounds=wl.bounds)


def _table_pool(K, N, rank):
    rank = np.asarray(rank, np.int32)
    a_off, b_off = workloads._pool_offsets(rank, K, N)
    return lm.Pool(None, None, a_off, b_off, rank, np.full(rank.shape, 2.0, np.float32))


@pytest.mark.parametrize("case", ["ftbwd_5120", "ftbwd_5120_reordered", "cosrv_8192x28672", "small_4096x256x4096"])
def test_backward_shrink_split_fills_waves(tmp_path, case):
    """The dY B^T passes of the backward shrink take the split count whose schedule ends first: on the 5120^2
    fine-tuning batch (32 tiles, 80 k-blocks a pass) 4 pieces of 20 k-blocks instead of 5 of 16 (288 items on 152
    CTAs: two waves, against 320, whose third wave holds 16 items), the same whatever the segment order; the x A
    recompute keeps the forward's 5 splits.  On the co-serving batch's fine-tuning rows (16 tiles, 448 k-blocks
    a pass) the default 14 splits already fill two waves and stay.  The small table of the GPU test of this split
    (32 tiles, 64 k-blocks a pass: 160 items at the default leave 8 in a last wave) takes 8 pieces instead of 4."""
    lib = _build_driver(tmp_path, open(os.path.join(CSRC, "plan.cpp")).read())
    if case.startswith("ftbwd"):
        K = N = 5120
        segs = [(i * 1024, 1024, 0, 1) for i in range(4)]
        if case.endswith("reordered"):
            segs = segs[::-1]
        T, rank, want = 4096, [16], (32 * 4, 32 * 5)
    elif case.startswith("small"):
        T, K, N, segs, rank = (RESPLIT_SMALL[k] for k in ("T", "K", "N", "segs", "rank"))
        want = (32 * 8, 32)
    else:
        K, N = 8192, 28672
        segs = [(t, 1, t % 7, 0) for t in range(2048)] + [(2048, 4096, 3, 0), (6144, 1024, 5, 1), (7168, 1024, 5, 1)]
        T, rank, want = 8192, [8, 16, 32, 64, 128, 64, 16], (16 * 14, 16 * 4)
    pool = _table_pool(K, N, rank)
    s = lm.segments(np.asarray(segs, np.int32))
    out = (ctypes.c_int * 2)()
    assert lib.bwd_shrink_items(T, K, N, pool.cptr(), s.ctypes.data, s.shape[0], out) == 0
    assert (out[0], out[1]) == want
    assert lib.check_table(T, K, N, pool.cptr(), s.ctypes.data, s.shape[0], 1) == 0


def test_item_assignment_is_the_plain_greedy(tmp_path):
    """The persistent launches' item lists: every item, in plan order, to the CTA with the least summed estimated
    cost so far (the lowest index on a tie), for random costs and CTA counts that are and are not powers of two,
    fewer CTAs than items and more."""
    lib = _build_driver(tmp_path, open(os.path.join(CSRC, "plan.cpp")).read())
    for n, G in [(1, 1), (5, 1), (3, 8), (100, 76), (3584, 76), (452, 152), (1000, 7), (64, 64), (129, 128)]:
        for seed in range(3):
            assert lib.assign_matches_greedy(n, G, seed) == 0, (n, G, seed)
