"""The binning's two-stage order, on the CPU: sorting the visible rows by depth
(stable), emitting each row's tiles in that order and then sorting stably by
tile gives exactly the order of one stable sort of (tile << 32 | depth) keys
emitted with rows in order and tiles row-major -- the definition the oracle
implements.  Equal depths (within and across views) and empty rows included."""
import numpy as np


def _rows(rng, n_views, n, tiles_x, tiles_y):
    rows = []
    depths = rng.choice(np.array([0.5, 2.0, 2.0000002, 7.0, 7.0], np.float32), n_views * n)
    for r in range(n_views * n):
        w, h = rng.integers(0, min(4, tiles_x + 1)), rng.integers(0, min(4, tiles_y + 1))
        x0, y0 = rng.integers(0, tiles_x - w + 1), rng.integers(0, tiles_y - h + 1)
        rows.append((r // n, r % n, x0, x0 + w, y0, y0 + h, depths[r]))
    return rows


def _one_sort(rows, T, tiles_x):
    keys, ids = [], []
    for view, g, x0, x1, y0, y1, d in rows:  # rows in order, tiles row-major
        for ty in range(y0, y1):
            for tx in range(x0, x1):
                flat = view * T + ty * tiles_x + tx
                keys.append((flat << 32) | int(np.float32(d).view(np.uint32)))
                ids.append(g)
    keys = np.array(keys, np.uint64)
    o = np.argsort(keys, kind="stable")
    return keys[o], np.array(ids)[o]


def _two_stage(rows, T, tiles_x):
    visible = [r for r in rows if (r[3] - r[2]) * (r[5] - r[4]) > 0]  # compaction, row order
    dbits = np.array([int(np.float32(r[6]).view(np.uint32)) for r in visible], np.uint64)
    by_depth = np.argsort(dbits, kind="stable")                       # depth passes
    flat, comp = [], []
    for c in by_depth:                                                # emission in depth order
        view, g, x0, x1, y0, y1, d = visible[c]
        for ty in range(y0, y1):
            for tx in range(x0, x1):
                flat.append(view * T + ty * tiles_x + tx)
                comp.append(c)
    flat, comp = np.array(flat, np.uint64), np.array(comp)
    o = np.argsort(flat, kind="stable")                               # tile passes
    keys = (flat[o] << np.uint64(32)) | dbits[comp[o]]
    ids = np.array([visible[c][1] for c in comp[o]])
    return keys, ids


def test_depth_then_tile_equals_one_sort_of_tile_depth_keys():
    rng = np.random.default_rng(3)
    for n_views, n, tiles_x, tiles_y in ((1, 300, 5, 4), (3, 200, 7, 3), (2, 1, 2, 2), (4, 50, 1, 1)):
        T = tiles_x * tiles_y
        rows = _rows(rng, n_views, n, tiles_x, tiles_y)
        k1, v1 = _one_sort(rows, T, tiles_x)
        k2, v2 = _two_stage(rows, T, tiles_x)
        assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
