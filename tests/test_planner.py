"""Host split planner (mla_plan_splits): the plan image covers every page exactly once, in
order, balanced over CTA pairs, with consistent partial slots and merge entries."""
import numpy as np
import pytest
import torch

from mla_latent_kv_absorb_gb300 import binding, synth

HDR = dict(magic=0, version=1, batch=2, clusters=3, items=4, partials=5, combine=6, cl_off=7, it_off=8, cb_off=9,
           total=10, max_splits=11)


def decode_plan(plan):
    h = {k: int(plan[v]) for k, v in HDR.items()}
    cl = plan[h["cl_off"]: h["cl_off"] + h["clusters"] + 1]
    items = plan[h["it_off"]: h["it_off"] + 8 * h["items"]].reshape(-1, 8)[:, :5]
    comb = plan[h["cb_off"]: h["cb_off"] + 4 * h["combine"]].reshape(-1, 4)[:, :3]
    return h, cl, items, comb


def check_plan(lens, num_sms=152, **kw):
    lens = np.asarray(lens, dtype=np.int32)
    plan, info = binding.mla_plan_splits(lens, num_sms, **kw)
    h, cl, items, comb = decode_plan(plan)
    B = lens.size
    pages = (lens.astype(np.int64) + 63) // 64
    assert h["magic"] == 0x504C4D41 and h["version"] == 2 and h["batch"] == B
    assert h["total"] == pages.sum() == info.total_pages
    assert 1 <= h["clusters"] <= num_sms // 2 and h["clusters"] == info.num_clusters
    assert cl[0] == 0 and cl[-1] == h["items"] and np.all(np.diff(cl) >= 0)
    # coverage: items in order tile every sequence's pages exactly once
    covered = {b: [] for b in range(B)}
    for seq, pb, pe, slen, slot in items:
        assert 0 <= seq < B and 0 <= pb < pe <= pages[seq] and slen == lens[seq]
        covered[seq].append((pb, pe))
    for b in range(B):
        rng = covered[b]
        assert rng[0][0] == 0 and rng[-1][1] == pages[b]
        assert all(rng[i][1] == rng[i + 1][0] for i in range(len(rng) - 1))
    # partial slots: -1 for single-item sequences, consecutive per sequence otherwise
    n_items = np.bincount(items[:, 0], minlength=B)
    assert info.max_splits == n_items.max()
    slots = items[:, 4]
    assert np.all(slots[n_items[items[:, 0]] == 1] == -1)
    multi = slots[n_items[items[:, 0]] > 1]
    assert sorted(multi.tolist()) == list(range(info.num_partials))
    assert info.num_combine == (n_items > 1).sum() == h["combine"]
    for seq, first, n in comb:
        assert n == n_items[seq] > 1
        own = items[items[:, 0] == seq]
        assert own[:, 4].tolist() == list(range(first, first + n))
    assert info.workspace_bytes == info.num_partials * (128 * 512 * 4 + 128 * 4)
    # balance: no CTA pair has more than its share plus one sequence edge's slack
    per = np.zeros(h["clusters"], dtype=np.int64)
    for k in range(h["clusters"]):
        for seq, pb, pe, _, _ in items[cl[k]:cl[k + 1]]:
            per[k] += pe - pb
    assert per.sum() == pages.sum()
    return info, per, items


def test_single_long_sequence_is_split_evenly():
    info, per, _ = check_plan([65536], item_cost_pages=-1)
    assert info.num_clusters == 76 and info.num_combine == 1 and info.max_splits == 76
    assert per.max() - per.min() <= 1


def test_64k_workload_balance():
    info, per, _ = check_plan([65536] * 16, item_cost_pages=-1)
    assert info.num_clusters == 76
    share = 16384 / 76
    assert per.max() <= share + 8 + 1  # min-split snapping moves an edge by < 8 pages


def test_short_sequences_stay_whole():
    info, per, items = check_plan([2048], item_cost_pages=-1)
    # 32 pages with the default minimum of 8 pages per item: 4 pairs
    assert info.num_clusters == 4 and info.num_items == 4 and info.num_combine == 1


def test_ragged_workload():
    g = torch.Generator().manual_seed(42)
    lens = synth.ragged_lengths(64, 128, 32768, g)
    info, per, _ = check_plan(lens, item_cost_pages=-1)
    assert info.total_pages == 17480
    assert per.max() <= 17480 / 76 + 8 + 1


@pytest.mark.parametrize("lens", [[1], [1, 1, 1], [64], [65], [63, 64, 65, 129], [1] * 300, [5000, 1, 70000, 3]])
def test_edge_lengths(lens):
    check_plan(lens)


@pytest.mark.parametrize("min_pages,max_clusters", [(1, 0), (2, 3), (64, 0), (8, 1)])
def test_options(min_pages, max_clusters):
    info, per, items = check_plan([100, 3000, 9000, 64 * 7], min_pages_per_split=min_pages, max_clusters=max_clusters)
    if max_clusters:
        assert info.num_clusters <= max_clusters


def test_randomised_plans():
    rng = np.random.default_rng(0)
    for _ in range(200):
        B = int(rng.integers(1, 200))
        lens = rng.integers(1, 70000, size=B)
        sms = int(rng.choice([2, 16, 148, 152]))
        check_plan(lens, num_sms=sms, min_pages_per_split=int(rng.integers(0, 20)))


def test_timeout_option_recorded():
    plan, info = binding.mla_plan_splits([100], 152, wait_timeout_ns=123456789)
    assert info.wait_timeout_ns == 123456789
    assert int(plan[12]) + (int(plan[13]) << 32) == 123456789


def _pair_costs(lens, c, **kw):
    plan, info = binding.mla_plan_splits(np.asarray(lens, np.int32), 152, item_cost_pages=c, **kw)
    h, cl, items, _ = decode_plan(plan)
    return np.array([int((items[cl[k]:cl[k + 1], 2] - items[cl[k]:cl[k + 1], 1]).sum())
                     + c * max(0, int(cl[k + 1] - cl[k]) - 1) for k in range(h["clusters"])]), info


@pytest.mark.parametrize("cost", [1, 7, 50])
def test_item_cost_plans_are_valid(cost):
    g = torch.Generator().manual_seed(42)
    for lens in ([65536] * 16, synth.ragged_lengths(64, 128, 32768, g), [1] * 300, [5000, 1, 70000, 3], [65536],
                 [4096] * 16, [2048]):
        check_plan(lens, item_cost_pages=cost)
    rng = np.random.default_rng(cost)
    for _ in range(100):
        lens = rng.integers(1, 70000, size=int(rng.integers(1, 200)))
        check_plan(lens, num_sms=int(rng.choice([2, 16, 152])), min_pages_per_split=int(rng.integers(0, 20)),
                   item_cost_pages=cost)


def test_item_cost_balances_pairs():
    """With a per-item charge the pairs that hold two items get fewer pages: the largest pair
    cost (pages + charge per extra item) drops below that of equal page runs and comes within
    one charge and one sequence-edge snap of the mean."""
    c = 7
    for lens in ([65536] * 16, [4096] * 16):
        base_plan, base_info = binding.mla_plan_splits(np.asarray(lens, np.int32), 152, item_cost_pages=-1)
        h, cl, items, _ = decode_plan(base_plan)
        base = np.array([int((items[cl[k]:cl[k + 1], 2] - items[cl[k]:cl[k + 1], 1]).sum())
                         + c * max(0, int(cl[k + 1] - cl[k]) - 1) for k in range(h["clusters"])])
        costs, info = _pair_costs(lens, c)
        assert costs.max() < base.max(), (lens[0], costs.max(), base.max())
        assert costs.max() <= costs.sum() / costs.size + c + 8


def test_item_cost_default_and_off():
    """0 asks for the library's default charge (7 pages), a negative value for equal page runs."""
    lens = np.asarray([65536] * 16, np.int32)
    p0, _ = binding.mla_plan_splits(lens, 152)
    p7, _ = binding.mla_plan_splits(lens, 152, item_cost_pages=7)
    pe, _ = binding.mla_plan_splits(lens, 152, item_cost_pages=-1)
    assert np.array_equal(p0, p7) and not np.array_equal(p0, pe)


def test_plan_rejects_bad_queries_per_seq():
    """queries_per_seq must lie in [0, MLA_MAX_QUERIES_PER_SEQ] and no sequence may be shorter
    than its query tokens."""
    import ctypes
    buf = np.zeros(1 << 16, np.int32)
    info = binding.PlanInfo()
    lens = np.array([100, 3], np.int32)
    for q, want in ((-1, binding.MLA_ERR_INVALID_ARG), (4097, binding.MLA_ERR_INVALID_ARG),
                    (4, binding.MLA_ERR_INVALID_ARG), (3, binding.MLA_OK)):
        opts = binding.PlanOptions(0, 0, 0, 0, q)
        st = binding.lib().mla_plan_splits(lens.ctypes.data_as(ctypes.c_void_p), 2, 152, ctypes.byref(opts),
                                           buf.ctypes.data_as(ctypes.c_void_p), buf.nbytes, ctypes.byref(info))
        assert st == want, q


def _items(plan):
    off, n = int(plan[8]), int(plan[4])
    return plan[off: off + 8 * n].reshape(n, 8)


@pytest.mark.parametrize("q", [2, 5])
def test_multi_query_rows(q):
    """With q query tokens per sequence the plan covers B * q rows: row b * q + t has visible
    length S_b - q + 1 + t, every page of it once, and reads block-table row b."""
    lens = np.array([700, 64 * 9 + q - 1, 5000, q], np.int32)
    plan, info = binding.mla_plan_splits(lens, 152, min_pages_per_split=2, queries_per_seq=q)
    assert info.batch == lens.size * q and info.queries_per_seq == q and int(plan[14]) == q
    items = _items(plan)
    for b in range(lens.size):
        for t in range(q):
            row = b * q + t
            mine = items[items[:, 0] == row]
            L = int(lens[b]) - q + 1 + t
            assert (mine[:, 3] == L).all() and (mine[:, 5] == b).all()
            covered = sorted(p for it in mine for p in range(it[1], it[2]))
            assert covered == list(range((L + 63) // 64))
    assert info.total_pages == sum((int(lens[b]) - q + 1 + t + 63) // 64 for b in range(lens.size) for t in range(q))


def test_single_query_rows_read_their_own_table_row():
    lens = np.array([3000, 700, 64 * 9 + 1], np.int32)
    for q in (0, 1):
        plan, info = binding.mla_plan_splits(lens, 152, min_pages_per_split=2, queries_per_seq=q)
        items = _items(plan)
        assert (items[:, 0] == items[:, 5]).all() and info.queries_per_seq == 1 and info.batch == 3
