"""The launch model's reading of a CSR matrix's data (host only, no GPU): a strided
sample of row lengths and of column indices sets the fp64 lane groups, the split of
shared memory between the scatter window and the copy of y, and where both sit.
Synthetic structures with known answers pin each decision."""
import numpy as np
import pytest

import dense_linear_algebra_gb300 as fx
import inputgen

SAMPLES = 8192


def _window(desc, key):
    """(start, length) of 'window=[c0,+len)' or 'y_window=[c0,+len)' in a plan description."""
    for tok in desc.split():
        if tok.startswith(key + "=["):
            a, b = tok[len(key) + 2:-1].split(",+")
            return int(a), int(b)
    raise KeyError(key)


def _csr_from_lengths(lens, cols_fn):
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    ci = cols_fn(int(rp[-1])).astype(np.int32)
    return rp, ci


def test_unsampled_plan_leaves_placement_to_the_device():
    p = inputgen.csr_powerlaw(m=20_000, n=1_000_000)
    d = fx.plan_describe("csr", "f32", p.m, p.n, p.nnz)
    assert "placement=device" in d and _window(d, "window")[0] == 0
    # every column inside both windows: nothing to place
    d = fx.plan_describe("csr", "f64", 1000, 5000, 20_000)
    assert "placement=whole" in d


@pytest.mark.parametrize("offset", [0, 400_000, 777_777])
def test_window_follows_the_hot_columns(offset):
    """Zipf columns rotated by `offset`: both windows start at the head of the hot range, and
    catch the same share of sampled columns as on the unrotated matrix."""
    n = 1_000_000
    p = inputgen.csr_powerlaw(m=50_000, n=n, col_offset=offset)
    base = inputgen.csr_powerlaw(m=50_000, n=n)
    d, st = fx.csr_plan_describe_host(p.row_ptr, p.col_idx, n, "f32")
    _, st0 = fx.csr_plan_describe_host(base.row_ptr, base.col_idx, n, "f32")
    assert "placement=sampled" in d
    bw = -(-n // 1024)  # columns per histogram bin
    for c0, ln in (_window(d, "window"), _window(d, "y_window")):
        assert 0 <= c0 and c0 + ln <= n
        # column `offset` (the Zipf head, 12 % of all entries) lies inside each window
        assert c0 <= offset < c0 + ln or (offset == 0 and c0 == 0)
        assert abs(c0 - offset) <= ln  # the window starts at most one window-width away from the head
    assert abs(st["window_hit_share"] - st0["window_hit_share"]) < 0.02
    assert abs(st["y_hit_share"] - st0["y_hit_share"]) < 0.02
    assert st["window_hit_share"] > 0.4  # Zipf(1.1): the hottest ~3 % of columns hold over 40 % of entries


def test_uniform_columns_hit_in_proportion_to_the_window():
    rng = np.random.default_rng(5)
    n = 400_000
    rp, ci = _csr_from_lengths(np.full(30_000, 40), lambda nnz: rng.integers(0, n, nnz))
    d, st = fx.csr_plan_describe_host(rp, ci, n, "f32")
    c0, ln = _window(d, "window")
    assert st["col_samples"] == SAMPLES
    assert abs(st["window_hit_share"] - ln / n) < 0.03


def test_row_length_statistics():
    rng = np.random.default_rng(9)
    n = 10_000
    # constant rows of 40 entries
    rp, ci = _csr_from_lengths(np.full(20_000, 40), lambda nnz: rng.integers(0, n, nnz))
    _, st = fx.csr_plan_describe_host(rp, ci, n, "f64")
    assert st["mean_row_len"] == 40 and st["cv_row_len"] == 0 and st["p50_row_len"] == st["p90_row_len"] == 40
    assert st["long_row_share"] == 0 and st["row_samples"] == SAMPLES
    assert (st["group_lanes"], st["group_entries"]) == (4, 16)  # 40 entries: 4 lanes x 16
    # rows of 20 entries with one row in 64 of 20,000: the mean is 332, the 75th percentile 20,
    # and the groups follow the typical row, not the mean
    lens = np.full(16_384, 20)
    lens[::64] = 20_000
    rp, ci = _csr_from_lengths(lens, lambda nnz: rng.integers(0, n, nnz))
    _, st = fx.csr_plan_describe_host(rp, ci, n, "f64")
    assert st["p75_row_len"] == 20 and st["mean_row_len"] > 300
    assert (st["group_lanes"], st["group_entries"]) == (2, 16)
    # the long rows (over 2,048 entries) hold 20,000 / (20,000 + 63 * 20) of the entries; the
    # sample (every other row, at hashed offsets) estimates that share
    assert abs(st["long_row_share"] - 20_000 / (20_000 + 63 * 20)) < 0.02
    # fp32 rows are packed whatever their lengths
    _, st32 = fx.csr_plan_describe_host(rp, ci, n, "f32")
    assert st32["group_lanes"] == 0


def test_small_matrices_are_sampled_whole():
    rp = np.array([0, 3, 3, 7], np.int64)
    ci = np.array([1, 2, 5, 0, 1, 2, 3], np.int32)
    _, st = fx.csr_plan_describe_host(rp, ci, 6, "f32")
    assert st["row_samples"] == 3 and st["col_samples"] == 7
    assert st["max_sampled_row_len"] == 4 and st["p50_row_len"] == 3
    _, st = fx.csr_plan_describe_host(np.zeros(1, np.int64), np.zeros(0, np.int32), 6, "f32")
    assert st["row_samples"] == 0 and st["col_samples"] == 0


def test_split_follows_the_column_skew():
    """Skewed columns: the model compares the ½, ¾ and ⅞ window/y splits on the sample and
    keeps a split whose two windows both hold the head; uniform columns over many more
    columns than fit keep the default ¾ split (no split catches more than its share)."""
    p = inputgen.csr_powerlaw(m=50_000, n=1_000_000, col_offset=123_457)
    d, st = fx.csr_plan_describe_host(p.row_ptr, p.col_idx, p.n, "f32")
    room = _window(d, "window")[1] + _window(d, "y_window")[1]
    assert _window(d, "window")[1] in (room // 2, room * 3 // 4, room * 7 // 8, room * 3 // 4 + 1, room // 2 + 1)
    rng = np.random.default_rng(2)
    n = 5_000_000
    rp, ci = _csr_from_lengths(np.full(20_000, 30), lambda nnz: rng.integers(0, n, nnz))
    d, _ = fx.csr_plan_describe_host(rp, ci, n, "f32")
    w, y = _window(d, "window")[1], _window(d, "y_window")[1]
    assert abs(w / (w + y) - 0.75) < 0.01


def test_analyze_refuses_bad_arguments_without_a_device():
    st = fx.CsrStats()
    assert fx.fxtx_csr_analyze(0, -1, 4, 0, None, None, None, None) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_csr_analyze(0, 3, 4, 2, None, None, None, None) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_csr_plan_describe_host(0, 3, 4, 2, None, None, None, None, 0) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_csr_analysis_clear() == fx.FXTX_OK
    del st
