"""Invariants of the launch model over a sweep of shapes (host only, no GPU): every
plan fits the GB300's per-CTA shared-memory limit, uses at most one CTA per SM for
the persistent kernels, sizes its workspace for its grid, and picks kernel shapes
the library instantiates."""
import itertools

import pytest

import dense_linear_algebra_gb300 as fx

SMS = 152
SMEM_LIMIT = 227 * 1024


def fields(desc):
    out = {}
    for kv in desc.split()[1:]:
        if "=" in kv:
            k, v = kv.split("=", 1)
            out[k] = v
    return out


DENSE_SHAPES = list(itertools.product(
    (0, 1, 7, 100, 4097, 1_000_000, 16_000_000),
    (1, 3, 4, 8, 16, 31, 32, 33, 64, 100, 128, 512, 513, 2048, 20_000),
))


@pytest.mark.parametrize("dtype,elem", [("f32", 4), ("f64", 8)])
def test_dense_plans(dtype, elem):
    for m, n in DENSE_SHAPES:
        for ld in (n, n + 1, n + 8):
            f = fields(fx.plan_describe("dense", dtype, m, n, 0, ld))
            kind = f["kind"]
            where = (dtype, m, n, ld, f)
            if m == 0:
                assert kind == "empty_rows", where
                continue
            assert kind in ("tile_tma", "narrow_tma", "narrow_direct", "wide"), where
            ctas, warps, smem, ws = int(f["ctas"]), int(f["warps"]), int(f["smem"]), int(f["ws"])
            assert smem <= SMEM_LIMIT, where
            assert 1 <= ctas, where
            assert float(f["est_us"]) >= 4.0, where
            if kind == "tile_tma":
                # tensor copies need a 16-byte row pitch; a tile kernel is persistent (one CTA per SM)
                assert (ld * elem) % 16 == 0 and ctas <= SMS and int(f["stages"]) >= 2, where
                # the row's column boxes cover it: blocks of `box` bytes, at most 2 KB a row
                blocks, box = int(f["blocks"]), int(f["box"])
                assert box in (64, 128) and 1 <= blocks <= 16 and blocks * box >= n * elem > (blocks - 1) * box, where
                # one fp64 partial per column per CTA, plus the ticket
                assert ws >= ctas * n * 8, where
            if kind == "narrow_tma":
                assert (ld * elem) % 16 == 0 and (n * elem) % 16 == 0, where
            if kind == "wide":
                assert n * elem > 2048 and ws >= ctas * n * 8, where
            if kind in ("tile_tma", "narrow_tma", "narrow_direct"):
                rows = int(f["rows_per_tile"])
                assert rows >= 1 and warps >= 1 and warps * 32 <= 1024, where


@pytest.mark.parametrize("dtype,elem", [("f32", 4), ("f64", 8)])
def test_csr_plans(dtype, elem):
    for m, n, avg in itertools.product((1, 1000, 4_000_000), (1, 100, 10_000, 1_000_000), (0, 1, 16, 17, 50, 100, 5000)):
        nnz = m * avg
        f = fields(fx.plan_describe("csr", dtype, m, n, nnz))
        where = (dtype, m, n, nnz, f)
        c0, wlen = f["window"].strip("[)").split(",+")
        y0, ylen = f["y_window"].strip("[)").split(",+")
        wlen, ylen = int(wlen), int(ylen)
        assert int(c0) == 0 and int(y0) == 0 and 0 <= wlen <= n and 0 <= ylen <= n, where
        # without a sample the windows are placed per call on the device, unless they cover every column
        assert f["placement"] == ("whole" if wlen >= n and ylen >= n else "device"), where
        # window and copy of y share the dynamic shared memory
        assert int(f["smem"]) <= SMEM_LIMIT and (wlen + ylen) * elem <= int(f["smem"]), where
        assert 1 <= int(f["ctas"]) <= SMS and int(f["long_ctas"]) == SMS, where
        lpr, kg = int(f["group_lanes"]), int(f["group_entries"])
        if elem == 8:
            # fp64 short rows go to lane groups of an instantiated shape, 768 threads a CTA
            assert lpr in (2, 4, 8, 16) and kg in (8, 16) and f["threads"] == "768", where
            assert lpr * kg >= min(avg, 256) or lpr == 16, where
        else:
            assert lpr == 0 and f["threads"] == "1024", where
        # every row longer than the one-warp limit fits its bucket of the long-row queue
        longest_count = nnz // (int(f["warp_cap"]) + 1)
        assert int(f["queue_cap"]) >= min(m, longest_count), where


def test_autotune_candidates_are_valid_plans():
    """Every candidate the tuner would time is a plan of the same kind that fits the limits."""
    for kind, dtype, m, n, nnz in (("dense", "f32", 16_000_000, 32, 0), ("dense", "f64", 20_000, 20_000, 0),
                                   ("dense", "f64", 1000, 64, 0), ("csr", "f64", 4_000_000, 10_000, 200_000_000),
                                   ("csr", "f32", 2_000_000, 1_000_000, 200_000_000)):
        cands = fx.autotune_candidates(kind, dtype, m, n, nnz)
        assert cands[0] == fx.plan_describe(kind, dtype, m, n, nnz), cands[0]
        for c in cands:
            f = fields(c)
            assert int(f["smem"]) <= SMEM_LIMIT, c
            if kind == "csr":
                assert f["threads"] == fields(cands[0])["threads"], c
