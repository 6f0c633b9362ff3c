"""The numpy reference planner against brute-force loops and invariants (CPU)."""
import numpy as np
import pytest

import graphgen
from oracle import planner


def _graphs():
    yield "random", graphgen.random_csr(70, 30, seed=1, zero_frac=0.2)
    yield "unsorted", graphgen.random_csr(53, 40, seed=2, zero_frac=0.1, sorted_rows=False)
    yield "multigraph", graphgen.random_csr(45, 25, seed=3, zero_frac=0.2, multigraph=True)
    yield "tiny", graphgen.tiny_poisson(num_nodes=37, seed=4)
    yield "dense", graphgen.batched_dense(num_graphs=5, seed=5)
    yield "one_row", graphgen.random_csr(1, 1, seed=6, zero_frac=0.0)


def brute_bsb(row_ptr, col, n):
    """Window-by-window restatement with Python loops (tiny graphs only)."""
    W = (n + 15) // 16
    tile_ptr, cols, bits, nnz, dup = [0], [], [], [], []
    for w in range(W):
        rows = range(16 * w, min(16 * w + 16, n))
        srcs = sorted({int(col[e]) for r in rows for e in range(row_ptr[r], row_ptr[r + 1])})
        nt = (len(srcs) + 7) // 8
        tile_ptr.append(tile_ptr[-1] + nt)
        padded = srcs + [-1] * (8 * nt - len(srcs))
        cols += padded
        for t in range(nt):
            word = [0, 0, 0, 0]
            for r in rows:
                present = {int(col[e]) for e in range(row_ptr[r], row_ptr[r + 1])}
                for c in range(8):
                    s = padded[8 * t + c]
                    if s >= 0 and s in present:
                        b = (r - 16 * w) * 8 + c
                        word[b // 32] |= 1 << (b % 32)
            bits.append(word)
        nnz.append(sum(int(row_ptr[r + 1] - row_ptr[r]) for r in rows))
        d = False
        for r in rows:
            s = [int(col[e]) for e in range(row_ptr[r], row_ptr[r + 1])]
            d |= len(s) != len(set(s))
        dup.append(d)
    return (np.array(tile_ptr), np.array(cols, dtype=np.int64), np.array(bits, dtype=np.uint64).reshape(-1, 4),
            np.array(nnz), np.array(dup, bool))


@pytest.mark.parametrize("name,g", list(_graphs()), ids=[n for n, _ in _graphs()])
def test_bsb_matches_brute_force(name, g):
    b = planner.bsb(g.row_ptr, g.col_idx, g.num_nodes)
    tp, cols, bits, nnz, dup = brute_bsb(g.row_ptr, g.col_idx, g.num_nodes)
    assert np.array_equal(b["win_tile_ptr"], tp)
    assert np.array_equal(b["tile_cols"], cols)
    assert np.array_equal(b["tile_bits"].astype(np.uint64), bits.reshape(-1, 4))
    assert np.array_equal(b["win_nnz"], nnz)
    assert np.array_equal(b["win_dup"], dup)


@pytest.mark.parametrize("name,g", list(_graphs()), ids=[n for n, _ in _graphs()])
def test_bsb_decodes_to_csr(name, g):
    b = planner.bsb(g.row_ptr, g.col_idx, g.num_nodes)
    n = g.num_nodes
    got = set()
    bits = b["tile_bits"]
    popc = 0
    for w in range(b["win_tile_ptr"].size - 1):
        t0, t1 = b["win_tile_ptr"][w], b["win_tile_ptr"][w + 1]
        cw = b["tile_cols"][8 * t0:8 * t1]
        real = cw[cw >= 0]
        assert np.all(np.diff(real) > 0)  # strictly increasing
        assert np.all(cw[real.size:] == -1)  # padding only at the end
        assert t1 - t0 == (real.size + 7) // 8  # minimal tile count
        for t in range(t0, t1):
            for bit in range(128):
                if (int(bits[t, bit // 32]) >> (bit % 32)) & 1:
                    r, c = divmod(bit, 8)
                    assert b["tile_cols"][8 * t + c] >= 0
                    got.add((16 * w + r, int(b["tile_cols"][8 * t + c])))
                    popc += 1
    want = {(i, int(s)) for i in range(n) for s in g.col_idx[g.row_ptr[i]:g.row_ptr[i + 1]]}
    assert got == want
    if name != "multigraph":
        assert popc == g.num_edges


def test_degree_buckets_brute_force():
    g = graphgen.powerlaw(num_nodes=3000, max_degree=2500, seed=9)
    bounds = (3, 10, 100)
    b = planner.degree_buckets(g.row_ptr, bounds)
    deg = g.degrees()
    lists = [[], [], [], [], []]
    for i, d in enumerate(deg):
        if d == 0:
            k = 0
        elif d <= 3:
            k = 1
        elif d <= 10:
            k = 2
        elif d <= 100:
            k = 3
        else:
            k = 4
        lists[k].append(i)
    flat = [i for lst in lists for i in lst]
    assert np.array_equal(b["bucket_rows"], flat)
    assert np.array_equal(b["bucket_ptr"], np.cumsum([0] + [len(x) for x in lists]))


def test_heavy_chunks_cover_rows():
    g = graphgen.powerlaw(num_nodes=3000, max_degree=2500, seed=10)
    T, C = 40, 16
    h = planner.heavy_chunks(g.row_ptr, T, C)
    deg = g.degrees()
    assert np.array_equal(h["heavy_rows"], np.flatnonzero(deg > T))
    ch = h["chunks"]
    for k, r in enumerate(h["heavy_rows"]):
        mine = ch[h["heavy_chunk_ptr"][k]:h["heavy_chunk_ptr"][k + 1]]
        assert np.all(mine[:, 0] == r)
        assert mine[0, 1] == g.row_ptr[r] and mine[-1, 2] == g.row_ptr[r + 1]
        assert np.all(mine[1:, 1] == mine[:-1, 2])
        assert np.all(mine[:, 2] - mine[:, 1] <= C) and np.all(mine[:, 2] > mine[:, 1])
        assert np.all(mine[:-1, 2] - mine[:-1, 1] == C)


def test_tile_selection_brute_force():
    g = graphgen.batched_dense(num_graphs=12, seed=11)
    b = planner.bsb(g.row_ptr, g.col_idx, g.num_nodes)
    deg = g.degrees()
    W = b["win_nnz"].size
    elig = []
    for w in range(W):
        nt = b["win_tile_ptr"][w + 1] - b["win_tile_ptr"][w]
        md = deg[16 * w:16 * w + 16].max()
        elig.append((not b["win_dup"][w]) and 1 <= nt <= 6 and md <= 40 and b["win_nnz"][w] / (128.0 * nt) >= 0.2)
    nt = np.diff(b["win_tile_ptr"])
    pooled = b["win_nnz"][elig].sum() / (128.0 * nt[elig].sum())
    assert 0 < sum(elig) < W and 0.2 < pooled < 0.9
    for pool_milli, take in ((0, True), (int(1000 * pooled) - 1, True), (int(1000 * pooled) + 1, False)):
        sel = planner.tile_selection(g.row_ptr, b, True, heavy_threshold=40, max_tiles=6, density_milli=200,
                                     pool_milli=pool_milli)
        for w in range(W):
            assert bool(sel["win_flags"][w] & planner.FLAG_TILE) == (elig[w] and take)
        assert np.array_equal(sel["tile_windows"], np.flatnonzero(sel["win_flags"] & planner.FLAG_TILE))
        # every window is on exactly one of the two lists, each ascending
        tile, core = list(sel["tile_windows"]), list(sel["core_windows"])
        assert sorted(tile + core) == list(range(W)) and tile == sorted(tile) and core == sorted(core)
        assert (0 < len(tile) < W) == take


def test_tile_items_pairing():
    """Every tile-path window sits in exactly one item; two windows share an
    item only when their 16-column units (ceil(T/2)) fit the 8 of an item,
    the narrower first; no two single windows could have shared one; and on
    small random unit mixes the number of items equals the fewest any pairing
    reaches (brute force over all pairings)."""
    from functools import lru_cache
    g = graphgen.batched_dense(num_graphs=60, seed=12)
    b = planner.bsb(g.row_ptr, g.col_idx, g.num_nodes)
    sel = planner.tile_selection(g.row_ptr, b, True, heavy_threshold=100, max_tiles=16, density_milli=0)
    tw = sel["tile_windows"]
    items = planner.tile_items(g.row_ptr, b, tw)
    ptr = b["win_tile_ptr"]
    units = lambda w: (ptr[w + 1] - ptr[w] + 1) // 2  # noqa: E731
    seen, singles = [], []
    for it in items:
        nwin, u0 = it[3] & 0xFF, it[3] >> 8
        assert nwin in (1, 2)
        wins = [it[0]] + ([it[4]] if nwin == 2 else [])
        for w, first, t in zip(wins, (it[1], it[5]), (it[2], it[6])):
            assert first == ptr[w] and t == ptr[w + 1] - ptr[w]
        assert u0 == units(it[0])
        if nwin == 2:
            assert units(it[0]) <= units(it[4]) and units(it[0]) + units(it[4]) <= 8
        else:
            assert not np.any(it[4:])
            singles.append(units(it[0]))
        seen += wins
    assert sorted(seen) == sorted(tw)
    singles.sort()
    assert len(singles) < 2 or singles[0] + singles[1] > 8
    assert len(items) < 0.6 * len(tw)

    rng = np.random.default_rng(13)
    for _ in range(60):
        n = int(rng.integers(1, 10))
        T = rng.integers(1, 17, n)
        fake = {"win_tile_ptr": np.concatenate([[0], np.cumsum(T)]).astype(np.int64)}
        got = planner.tile_items(None, fake, np.arange(n))
        u = [(int(t) + 1) // 2 for t in T]

        @lru_cache(maxsize=None)
        def fewest(mask):
            if mask == (1 << n) - 1:
                return 0
            i = next(k for k in range(n) if not mask >> k & 1)
            best = 1 + fewest(mask | 1 << i)
            for j in range(i + 1, n):
                if not mask >> j & 1 and u[i] + u[j] <= 8:
                    best = min(best, 1 + fewest(mask | 1 << i | 1 << j))
            return best
        assert got.shape[0] == fewest(0), (u, got)


def _split_graph():
    """Windows of every kind: clustered heavy-row windows (split), a sparse
    wide window (too sparse to split), batched windows (pairs) and a ragged
    tail of random rows, with empty rows among them."""
    parts = [graphgen.clustered_heavy(num_windows=12, pool=300, degree=150, light_frac=0.2, empty_frac=0.1, seed=21),
             graphgen.clustered_heavy(num_windows=12, pool=1000, degree=30, light_frac=0.0, seed=22),
             graphgen.batched_dense(num_graphs=6, seed=23),
             graphgen.random_csr(37, 9, seed=24, zero_frac=0.3)]
    n, rp, cols = 0, [np.zeros(1, np.int64)], []
    for g in parts:
        rp.append(rp[-1][-1] + g.row_ptr[1:])
        cols.append(g.col_idx.astype(np.int64) + n)
        n += g.num_nodes
    return graphgen.Graph(np.concatenate(rp).astype(np.int32), np.concatenate(cols).astype(np.int32))


@pytest.mark.parametrize("edge_parallel", [True, False])
def test_split_windows_invariants(edge_parallel):
    """Split selection, slice items and the merge list of the reference planner:
    a split window is exactly a window of more than 16 tiles, no repeated pair
    and density >= split_milli / 1000; its slices cover its tiles in order, 16
    at a time; the partial indices of (slice, row) pairs cover [n_chunks,
    n_chunks + 16 x slices) once each; the merge list holds every row of a split
    window with the indices its slices write, and every other heavy row with its
    chunks.  Node-parallel, a slice carries (s, S) instead and the merge list
    holds only the heavy rows outside split windows."""
    g = _split_graph()
    b = planner.bsb(g.row_ptr, g.col_idx, g.num_nodes)
    deg = g.degrees()
    T = 100
    hc = planner.heavy_chunks(g.row_ptr, T, 64)
    n_chunks = hc["chunks"].shape[0]
    ptr = b["win_tile_ptr"].astype(np.int64)
    nt = np.diff(ptr)
    W = nt.size
    for split_milli in (250, 500):
        sel = planner.tile_selection(g.row_ptr, b, True, heavy_threshold=T, max_tiles=16, density_milli=100,
                                     pool_milli=0, split_milli=split_milli)
        fl = sel["win_flags"]
        split = [w for w in range(W) if fl[w] & planner.FLAG_SPLIT]
        for w in range(W):
            dense = b["win_nnz"][w] * 1000 >= split_milli * 128 * nt[w]
            assert (w in split) == (bool(nt[w] > 16) and not b["win_dup"][w] and bool(dense)), w
            if w in split:
                assert fl[w] & planner.FLAG_TILE
        assert 0 < len(split) < W
        assert set(split).isdisjoint(sel["tile_windows"]) and set(split).isdisjoint(sel["core_windows"])
        assert sorted(list(sel["tile_windows"]) + split + list(sel["core_windows"])) == list(range(W))
        items = planner.tile_items(g.row_ptr, b, sel["tile_windows"], sel["split_windows"], n_chunks, edge_parallel)
        n_pair = planner.tile_items(g.row_ptr, b, sel["tile_windows"]).shape[0]
        sitems = items[n_pair:]
        flag = planner.ITEM_PARTIAL if edge_parallel else planner.ITEM_CHAIN
        assert np.all(sitems[:, 3] & flag) and not np.any(items[:n_pair, 3] & (planner.ITEM_PARTIAL | planner.ITEM_CHAIN))
        assert not np.any(sitems[:, 3] & (planner.ITEM_PARTIAL ^ planner.ITEM_CHAIN ^ flag))
        hit = {}
        k = 0
        for w in split:
            S = -(-int(nt[w]) // 16)
            mine = sitems[k:k + S]
            k += S
            assert np.all(mine[:, 0] == w) and np.all(mine[:, 5] == S)
            assert mine[0, 1] == ptr[w] and np.all(mine[1:, 1] == mine[:-1, 1] + 16)
            assert mine[:, 2].sum() == nt[w] and np.all(mine[:-1, 2] == 16)
            assert np.all((mine[:, 3] & 0xFF) == 1) and np.all(((mine[:, 3] >> 8) & 0xFF) == (mine[:, 2] + 1) // 2)
            if not edge_parallel:
                assert list(mine[:, 4]) == list(range(S))
                continue
            for it in mine:
                for r in range(16):
                    hit.setdefault(int(it[4] + r * S), []).append((w, r))
        assert k == len(sitems)
        if edge_parallel:
            total = 16 * sum(-(-int(nt[w]) // 16) for w in split)
            assert sorted(hit) == list(range(n_chunks, n_chunks + total)) and all(len(v) == 1 for v in hit.values())
        ml = planner.merge_list(g.row_ptr, b, fl, T, hc["heavy_chunk_ptr"], n_chunks, edge_parallel)
        rows, ranges = list(ml["merge_rows"]), ml["merge_ranges"]
        heavy = list(hc["heavy_rows"])
        want = sorted(set(r for r in range(g.num_nodes) if (r // 16) in split and edge_parallel) |
                      set(r for r in heavy if (r // 16) not in split))
        assert rows == want
        for r, (lo, hi) in zip(rows, ranges):
            if (r // 16) in split:
                assert sorted(hit_r for hit_r, v in hit.items() if v[0] == (r // 16, r % 16)) == list(range(lo, hi))
            else:
                i = heavy.index(r)
                assert (lo, hi) == (hc["heavy_chunk_ptr"][i], hc["heavy_chunk_ptr"][i + 1])
                assert np.array_equal(hc["chunks"][lo:hi, 0], np.full(hi - lo, r))
        # a heavy row inside a split window is merged from its slices, not its chunks
        assert any(deg[r] > T and (r // 16) in split for r in range(g.num_nodes))
    off = planner.tile_selection(g.row_ptr, b, True, heavy_threshold=T, max_tiles=16, density_milli=100, split_milli=0)
    assert not np.any(off["win_flags"] & planner.FLAG_SPLIT)
