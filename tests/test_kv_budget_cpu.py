"""gk_kv_budget (host only): the KV-pool sizing of "determine_available_memory
design" (sections "Heuristic formula", "Minimum KV guard") and the block count
for the group-buffer layout, pinned by the page's printed 120B figures and by
cases worked by hand from the formula."""
import os

import pytest

import paged_fp8_kv_gk_gb300 as gk

GiB = 1 << 30
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_budget_gk.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def _shape(groups, kv, block, d):
    return gk.Shape.make(num_layers=2 * groups, batch=1, num_q_heads=8 * kv, num_kv_heads=kv,
                         head_dim=d, block_size=block, num_blocks=1, window=128,
                         max_blocks_full=1, max_blocks_swa=1)


def test_page_120b_pool_gives_its_block_count():
    """GPT-OSS-120B giga-kernel decode, section "KV budget": 18 groups, kv 1,
    block 128, head 64 -> ~36,175 blocks, ~9.94 GiB."""
    g = _golden()
    sh = _shape(int(g["group_size"]), int(g["kv_heads"]), int(g["block"]), int(g["head_size"]))
    per_block = int(g["group_size"]) * 2 * int(g["kv_heads"]) * int(g["block"]) * int(g["head_size"])
    nb = int(g["num_blocks"])
    for extra in (0, per_block - 1):   # any budget inside the last block gives the same count
        total = 10 ** 12
        used = 0
        # choose gmu so that total_budget = nb * per_block + extra exactly; no cap binding
        budget = nb * per_block + extra
        st, avail, blocks = gk.gk_kv_budget(budget, used, 1.0, 1.0, 1.0, sh)
        assert st == gk.GK_OK and avail == budget and blocks == nb
        assert round(avail / GiB, 2) == g["kv_gib"]


@pytest.mark.parametrize("total,used,gmu,cap,expect", [
    # user budget binds: int(1000e9*0.9)=900e9; 900e9-100e9=800e9 < cap int(900e9*0.95)
    (1000 * 10 ** 9, 100 * 10 ** 9, 0.9, 0.95, 800 * 10 ** 9),
    # cap binds: 0.30 of the 900e9 budget = 270e9 < 800e9
    (1000 * 10 ** 9, 100 * 10 ** 9, 0.9, 0.30, 270 * 10 ** 9),
    # used above the budget: kv budget clamps at 0
    (100 * GiB, 95 * GiB, 0.9, 0.30, 0),
    # truncation of the products: int(7 * 0.5) = 3, int(3 * 0.5) = 1
    (7, 0, 0.5, 0.5, 1),
])
def test_formula_cases_worked_by_hand(total, used, gmu, cap, expect):
    st, avail, nb = gk.gk_kv_budget(total, used, gmu, cap, 0.0)
    assert avail == expect and nb is None
    assert st == gk.GK_OK


def test_minimum_guard_and_too_few_blocks():
    st, avail, _ = gk.gk_kv_budget(10 * GiB, 9 * GiB, 1.0, 1.0, 1.0)
    assert st == gk.GK_OK and avail == GiB
    st, avail, _ = gk.gk_kv_budget(10 * GiB, 9 * GiB + 1, 1.0, 1.0, 1.0)
    assert st == gk.GK_ERR_BUDGET and avail == GiB - 1          # reported, not hidden
    sh = _shape(18, 8, 32, 64)                                   # 589,824 B per block
    st, avail, nb = gk.gk_kv_budget(589824 * 2 - 1, 0, 1.0, 1.0, 0.0, sh)
    assert st == gk.GK_ERR_BUDGET and nb == 1
    st, avail, nb = gk.gk_kv_budget(589824 * 2, 0, 1.0, 1.0, 0.0, sh)
    assert st == gk.GK_OK and nb == 2


def test_invalid_arguments():
    L = gk.lib()
    import ctypes
    a = ctypes.c_uint64()
    for gmu, cap, mn in ((0.0, 0.3, 1.0), (1.5, 0.3, 1.0), (0.9, 0.0, 1.0), (0.9, 1.2, 1.0),
                         (0.9, 0.3, -1.0)):
        assert L.gk_kv_budget(10, 0, gmu, cap, mn, None, ctypes.byref(a), None) == gk.GK_ERR_INVALID_ARG
    assert L.gk_kv_budget(10, 0, 0.9, 0.3, 0.0, None, None, None) == gk.GK_ERR_INVALID_ARG
