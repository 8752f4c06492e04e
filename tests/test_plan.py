"""Host-side schedule of the persistent kernel (CPU only, no CUDA calls).

The kernel's three roles walk the work list that gemm_relu_plan_work_item
reports, so checking it here checks what the GPU will do: every
(tile, k-block) unit is covered exactly once, split tiles are shared by
consecutive slots in K order, rasterisation is a bijection, and resource
use stays inside GB300 limits.
"""
import random
from collections import defaultdict

import pytest

from tiled_dense_gemm_gb300.workloads import WORKLOADS

SMEM_LIMIT = 227 * 1024
SHAPES = [(w.M, w.N, w.K) for w in WORKLOADS.values()] + [
    (1, 8, 8), (8, 8, 8), (127, 8, 64), (129, 136, 72), (257, 264, 2056), (128, 128, 128),
    (256, 512, 64), (4096, 8192, 64), (64, 4096, 16384), (1000, 1000, 8), (2048, 2048, 2048),
    (8192, 8192, 8192), (130, 24, 4104), (16, 65536, 512), (100000, 8, 8), (48, 6144, 2048),
    (8, 4864, 1024),
]


def _check(gemm_lib, M, N, K, sms, forced=False):
    p = gemm_lib.plan(M, N, K, sms)
    d = p.as_dict()
    if forced:
        assert d["path"] in (2, 3, 4)
    elif M <= 32:
        assert d["path"] == 3  # swapped operands for very small M
    elif M <= 64:
        # swapped operands only with a cluster or plain split of K
        assert d["path"] == 2 or (d["path"] == 3 and (d["cluster"] == 2 or d["splits"] > 1))
    elif M <= 128:
        assert d["path"] == 2
    else:
        assert d["path"] in (2, 4)
    csk = d["path"] in (2, 3) and d["cluster"] > 1  # cluster split-K
    if csk:
        assert d["cluster"] == 2 and d["dp_tiles"] == d["num_tiles"] == d["grid"]
        assert d["sk_tiles"] == 0 and d["workspace_bytes"] == 0
    if d["path"] == 3:
        assert d["mma_n"] == ((M + 15) // 16) * 16
        assert d["tile_n"] == 128
        assert d["mma_m"] == 128 and (d["cluster"] == 1 or csk)
    elif d["path"] == 2:
        assert d["mma_n"] in (64, 128, 256) and d["tile_m"] == 128
        assert d["mma_m"] == 128 and (d["cluster"] == 1 or csk)
    else:
        assert d["mma_n"] == 256
        assert (d["mma_m"], d["tile_m"], d["tile_n"], d["cluster"]) == (256, 256, d["mma_n"], 2)
        assert d["stage_bytes"] == (128 + d["mma_n"] // 2) * d["block_k"] * 2
    assert d["mma_n"] % 16 == 0 and 16 <= d["mma_n"] <= 256
    assert d["tiles_m"] * d["tile_m"] >= M and d["tiles_n"] * d["tile_n"] >= N
    want_bk = 64 if (d["path"] in (2, 4) and d["mma_n"] == 256) else 128
    assert d["block_k"] == want_bk
    assert d["num_kb"] == (K + d["block_k"] - 1) // d["block_k"]
    assert 2 <= d["num_stages"] <= 16
    assert d["smem_bytes"] <= SMEM_LIMIT
    # A is copied to a 128-byte pitch only when neither pitch is aligned
    assert d["pack_a"] in (0, 1)
    if d["pack_a"]:
        assert d["path"] in (2, 4) and K % 64 != 0
        assert forced or (d["path"] == 4 and N % 64 != 0 and d["tiles_n"] >= 4)
    assert d["tmem_cols"] in (32, 64, 128, 256, 512) and d["tmem_cols"] >= 2 * d["mma_n"]
    assert 1 <= d["grid"] * d["cluster"] <= sms
    assert d["dp_tiles"] + d["sk_tiles"] == d["num_tiles"]
    assert d["workspace_bytes"] == d["sk_tiles"] * d["cluster"] * d["max_slots"] * 128 * d["mma_n"] * 4
    assert d["counter_count"] == d["sk_tiles"] * d["cluster"]

    # split tiles: the last sk_tiles in raster order, or the first ones when
    # their slots share the reduction (their items then run first)
    chunk = 16 if d["path"] == 3 else 64
    concurrent = (d["splits"] > 1 and d["sk_tiles"] * d["splits"] <= d["grid"]
                  and d["mma_n"] % (d["splits"] * chunk) == 0)
    split_lo = 0 if concurrent else d["dp_tiles"]
    split_hi = split_lo + d["sk_tiles"]
    cover = defaultdict(int)
    slots = defaultdict(dict)
    coords = {}
    sk_units = []
    n_cta = d["grid"] * d["cluster"] if csk else d["grid"]
    for cta in range(n_cta):
        items = gemm_lib.plan_work_items(p, cta)
        units = 0
        for it in items:
            assert 0 <= it["kb0"] < it["kb1"] <= d["num_kb"]
            assert 0 <= it["tm"] < d["tiles_m"] and 0 <= it["tn"] < d["tiles_n"]
            if it["tile"] in coords:
                assert coords[it["tile"]] == (it["tm"], it["tn"])
            coords[it["tile"]] = (it["tm"], it["tn"])
            for kb in range(it["kb0"], it["kb1"]):
                cover[(it["tile"], kb)] += 1
            if csk:
                r = cta % d["cluster"]
                assert it["slot"] == r and it["nslots"] == d["cluster"]
                assert it["kb0"] == r * d["num_kb"] // d["cluster"]
                assert it["kb1"] == (r + 1) * d["num_kb"] // d["cluster"]
            elif not split_lo <= it["tile"] < split_hi:
                assert (it["kb0"], it["kb1"], it["nslots"]) == (0, d["num_kb"], 1)
            else:
                units += it["kb1"] - it["kb0"]
                assert 0 <= it["slot"] < it["nslots"] <= d["max_slots"]
                assert it["slot"] not in slots[it["tile"]]
                slots[it["tile"]][it["slot"]] = (it["kb0"], it["kb1"], it["nslots"])
        if d["sk_tiles"]:
            sk_units.append(units)
    # every unit exactly once
    assert len(cover) == d["num_tiles"] * d["num_kb"]
    assert set(cover.values()) == {1}
    # rasterisation is a bijection
    assert len(coords) == d["num_tiles"]
    assert len(set(coords.values())) == d["num_tiles"]
    # split tiles: slots 0..n-1, contiguous K ranges in slot order
    for t, s in slots.items():
        n = next(iter(s.values()))[2]
        assert sorted(s) == list(range(n))
        kb = 0
        for i in range(n):
            assert s[i][0] == kb and s[i][2] == n
            kb = s[i][1]
        assert kb == d["num_kb"]
    # stream-K runs differ by at most one k-block
    if sk_units and d["splits"] == 1:
        assert max(sk_units) - min(sk_units) <= 1
        assert sum(sk_units) == d["sk_tiles"] * d["num_kb"]
    return d


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("sms", [152, 148, 7])
def test_schedule_covers_every_unit_once(gemm_lib, shape, sms):
    _check(gemm_lib, *shape, sms)


@pytest.mark.parametrize("force", ["tiled256", "tiled128", "pair", "tiled256:dp", "pair:dp",
                                   "swap", "swap:dp", "swap:s19", "tiled128:s8", "pair:s3",
                                   "tiled128:c2", "tiled256:c2", "swap:c2", "swap:sk",
                                   "tiled128:sk", "tiled64", "tiled64:s3", "tiled64:c2", "pair:t2"])
def test_forced_paths(gemm_lib, monkeypatch, force):
    monkeypatch.setenv("GEMM_RELU_FORCE_PATH", force)
    want = {"tiled256": (2, 256), "tiled128": (2, 128), "pair": (4, 256), "tiled64": (2, 64)}
    for shape in SHAPES:
        d = _check(gemm_lib, *shape, 152, forced=True)
        if force.startswith("swap"):
            assert d["path"] == (3 if shape[0] <= 128 else d["path"])
        else:
            assert (d["path"], d["mma_n"]) == want[force.split(":")[0]]
        if force.endswith(":dp"):
            assert d["sk_tiles"] == 0
        if ":c2" in force and d["num_tiles"] <= 76 and d["num_kb"] >= 2:
            assert d["cluster"] == 2 and d["grid"] == d["num_tiles"]
        if force.endswith(":sk"):
            assert d["dp_tiles"] == 0 and d["sk_tiles"] == d["num_tiles"] and d["splits"] == 1
            workers = 76 if d["path"] == 4 else 152  # CTA pairs on 152 SMs
            assert d["grid"] == min(workers, d["num_tiles"] * d["num_kb"])
        elif ":s" in force and force.split(":s")[1][:1].isdigit():
            want_s = min(int(force.split(":s")[1]), d["num_kb"])
            assert d["dp_tiles"] == 0 and d["max_slots"] == want_s
            assert d["splits"] == (want_s if want_s > 1 else 1)


@pytest.mark.parametrize("force,sp", [("pair:t2", 2), ("pair:t3", 3), ("tiled256:t4", 4)])
def test_tail_wave_split(gemm_lib, monkeypatch, force, sp):
    monkeypatch.setenv("GEMM_RELU_FORCE_PATH", force)
    for shape in [(4096, 4096, 4096), (3000, 5000, 2056), (8192, 8192, 2048)]:
        d = _check(gemm_lib, *shape, 152, forced=True)
        workers = d["grid"]
        T = d["num_tiles"]
        if T % workers:
            assert d["dp_tiles"] == (T // workers) * workers
            assert d["sk_tiles"] == T % workers and d["splits"] == sp and d["max_slots"] == sp


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (3000, 5000, 2056), (8192, 8192, 2048)])
def test_split_items_come_first_when_the_reduction_is_shared(gemm_lib, monkeypatch, shape):
    """With a split tail whose slots share the reduction (every worker has
    at most one split item, and the columns divide into whole epilogue
    chunks per slot), each worker runs its split item first, so that all
    slots of a split tile run together and the reduction overlaps the
    worker's next tile."""
    monkeypatch.delenv("GEMM_RELU_FORCE_PATH", raising=False)
    p = gemm_lib.plan(*shape, 152)
    d = p.as_dict()
    assert d["splits"] > 1 and d["sk_tiles"] * d["splits"] <= d["grid"]
    assert d["mma_n"] % (d["splits"] * 64) == 0
    for w in range(d["grid"]):
        items = gemm_lib.plan_work_items(p, w)
        split = [i for i, it in enumerate(items) if it["nslots"] > 1]
        if w < d["sk_tiles"] * d["splits"]:
            assert split == [0], (w, items[:2])
        else:
            assert split == []


def test_copy_of_a_decision(gemm_lib, monkeypatch):
    monkeypatch.delenv("GEMM_RELU_FORCE_PATH", raising=False)
    assert gemm_lib.plan(3000, 5000, 2056, 152).pack_a == 1      # both pitches misaligned
    assert gemm_lib.plan(3000, 5120, 2056, 152).pack_a == 0      # B's pitch aligned
    assert gemm_lib.plan(3000, 5000, 2048, 152).pack_a == 0      # A's pitch aligned
    assert gemm_lib.plan(4096, 4096, 4096, 152).pack_a == 0
    assert gemm_lib.plan(16, 8192, 8200, 152).pack_a == 0        # swapped operands
    assert gemm_lib.plan(300, 264, 2056, 152).pack_a == 0        # A read by too few tiles
    monkeypatch.setenv("GEMM_RELU_FORCE_PATH", "tiled128:pk")
    assert gemm_lib.plan(300, 264, 2056, 152).pack_a == 1
    monkeypatch.setenv("GEMM_RELU_FORCE_PATH", "pair:npk")
    assert gemm_lib.plan(3000, 5000, 2056, 152).pack_a == 0


def test_random_shapes(gemm_lib):
    rng = random.Random(0)
    for _ in range(60):
        M = rng.randint(1, 3000)
        N = 8 * rng.randint(1, 700)
        K = 8 * rng.randint(1, 600)
        _check(gemm_lib, M, N, K, rng.choice([152, 148, 100, 33]))


def test_degenerate_plans(gemm_lib):
    assert gemm_lib.plan(0, 8, 8, 152).path == 0
    assert gemm_lib.plan(8, 0, 8, 152).path == 0
    assert gemm_lib.plan(8, 8, 0, 152).path == 1
    with pytest.raises(gemm_lib.GemmReluError):
        gemm_lib.plan(-1, 8, 8, 152)
    with pytest.raises(gemm_lib.GemmReluError):
        gemm_lib.plan(8, 8, 8, 0)


def test_headline_shapes_use_the_intended_kernels(gemm_lib):
    sq = gemm_lib.plan(4096, 4096, 4096, 152)
    assert sq.path == 4 and sq.grid == 76 and sq.cluster == 2
    sk = gemm_lib.plan(16, 8192, 8192, 152)
    # 64 tiles of 128 columns, each by a 2-CTA cluster (one K half each)
    assert sk.path == 3 and sk.mma_n == 16 and sk.tile_n == 128
    assert sk.cluster == 2 and sk.grid == 64 and sk.dp_tiles == 64


def _check_boxes(gemm_lib, M, N, K, layout, no3d=False):
    """The TMA boxes of one ring stage agree with the stage the kernel
    reserves: the copies of a stage deliver exactly stage_bytes per CTA, a
    3-D copy fills the shared-memory region of its operand, and no 3-D view
    reaches past the end of a matrix row."""
    p = gemm_lib.plan(M, N, K, 152)
    d = p.as_dict()
    if d["path"] < 2:
        return
    bx = gemm_lib.plan_boxes(p, M, N, K, layout).as_dict()
    swap, pair = d["path"] == 3, d["path"] == 4
    bk = d["block_k"]
    sub = bk // 64
    for box in (bx["a_box"], bx["b_box"]):
        assert all(1 <= v <= 256 for v in box)
    # A
    rows_a = d["tile_m"] if swap else 128
    assert bx["a_box"][:2] == [64, rows_a]
    if bx["a_3d"]:
        assert not no3d and K % 64 == 0 and sub == 2 and bx["a_box"][2] == sub
    else:
        assert bx["a_box"][2] == 1
        assert no3d or K % 64 != 0 or sub == 1
    a_bytes = 64 * rows_a * sub * 2  # one stage of A, 3-D or one 2-D box per 64-k block
    # B
    if layout == "kn":
        cols = 128 if swap else (d["mma_n"] // 2 if pair else d["mma_n"])
        if bx["b_3d"]:
            assert not no3d and N >= 64 and cols % 64 == 0 and cols >= 128
            assert bx["b_box"] == [64, bk, cols // 64]
            assert bx["b_view_inner"] == (N // 64) * 64 <= N
            assert bx["b2_box"] == [64, bk]  # the partial chunk's 2-D boxes
        else:
            assert bx["b_box"][1] == bk and bx["b_box"][2] == 1
            assert bx["b_box"][0] == 64 and bx["b2_box"] == [64, bk]
            assert no3d or N < 64 or cols % 64 != 0 or cols < 128
        b_bytes = cols * bk * 2
    else:
        rows_b = 128 if swap else (d["mma_n"] // 2 if pair else d["mma_n"])
        assert bx["b_box"][:2] == [64, rows_b] and bx["b2_box"] == [64, rows_b]
        if bx["b_3d"]:
            assert not no3d and K % 64 == 0 and sub == 2
            assert bx["b_box"][2] == sub
        else:
            assert bx["b_box"][2] == 1
        b_bytes = rows_b * 64 * sub * 2
    assert a_bytes + b_bytes == d["stage_bytes"], (M, N, K, layout, d, bx)


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("force", ["", "tiled256", "tiled128", "tiled64", "pair", "swap", "tiled128:c2", "swap:c2",
                                   "tiled128:no3d", "pair:no3d", "swap:no3d"])
def test_copy_boxes_match_the_stage(gemm_lib, monkeypatch, layout, force):
    if force:
        monkeypatch.setenv("GEMM_RELU_FORCE_PATH", force)
    else:
        monkeypatch.delenv("GEMM_RELU_FORCE_PATH", raising=False)
    rng = random.Random(3)
    shapes = list(SHAPES) + [(rng.randint(1, 3000), 8 * rng.randint(1, 700), 8 * rng.randint(1, 600))
                             for _ in range(25)]
    for M, N, K in shapes:
        _check_boxes(gemm_lib, M, N, K, layout, no3d=":no3d" in force)
