"""Reference planner (numpy) -- the bit-exact target of the device planner.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.

Three outputs, all integer, all unique under the canonical orderings below.

1. Degree buckets.  deg_i = row_ptr[i+1] - row_ptr[i].  With inclusive upper
   bounds b_1 < ... < b_{B-2}: bucket 0 holds deg 0, bucket k (1 <= k <= B-2)
   holds b_{k-1} < deg <= b_k (b_0 = 0), bucket B-1 holds deg > b_{B-2}.
   ``bucket_rows`` lists rows grouped by bucket, ascending id inside a bucket;
   ``bucket_ptr`` (B+1) is the exclusive scan of bucket sizes.

2. Heavy-row chunks.  A row is heavy when deg > heavy_threshold.  Heavy rows in
   ascending id; row r is cut into ceil(deg/C) chunks of C consecutive CSR
   positions (the last one shorter).  ``chunks`` is (n_chunks, 3) int32 of
   (row, e_begin, e_end); ``heavy_chunk_ptr`` (n_heavy+1) the scan of chunk
   counts.

3. Binary Sparse Block (BSB) tiles of 16-row windows, after the Fused3S
   figure 1 caption (sciencestack.ai/paper/2505.08098, Figure 1: a row window
   is "compacted, tiled, and stored in BSB format", TCB 16x8).  Window w holds
   rows [16w, 16w+16).  U_w = sorted unique sources of its edges.  It gets
   T_w = ceil(|U_w| / 8) tiles; tile t covers U_w[8t .. 8t+8), padded with -1.
   ``win_tile_ptr`` (W+1) is the scan of T_w.  Each tile has a 128-bit
   bitmap stored as four little-endian uint32 words: bit r*8 + c (word
   (r*8+c)//32) is set iff the CSR holds an edge (16w + r <- tile_cols[8t+c]).
   ``win_nnz`` counts CSR entries per window; ``win_flags`` bit 0 marks a
   window with a repeated (row, source) pair, bit 1 a window that takes the
   tile path.  With the tile path enabled, a window is eligible when it has
   no repeated pair, 1 <= T_w <= max_tiles, no heavy row, and
   1000 * nnz >= density_milli * 128 * T_w; the eligible windows take the tile
   path together when 1000 * (sum of their nnz) >= pool_milli * 128 * (sum of
   their T_w), and none does otherwise.  ``tile_windows`` lists them in
   ascending order, ``core_windows`` the other windows (whose rows the
   CUDA-core kernel takes), also ascending.

4. Split windows (the edge-parallel form of the Fused3S Figure 2 caption,
   columns split as in its Figure 3 caption).  With split_milli > 0, a window
   with no repeated pair, T_w > 16 and 1000 * nnz >= split_milli * 128 * T_w
   takes the tile path on its own (bits 1 and 3 of ``win_flags``), heavy rows
   included; it is not in ``tile_windows`` (the pairs' list) nor in
   ``core_windows``.  It is cut into S_w = ceil(T_w / 16) slices of 16 tiles,
   one tile item each, after the pairs' items, windows ascending.
   Edge-parallel, window w's partial states occupy indices n_chunks + 16 B_w
   .. n_chunks + 16 (B_w + S_w) - 1, B_w = the slices of the split windows
   before w: row r, slice s at n_chunks + 16 B_w + r S_w + s, and a forward
   merges (``merge_rows``, ascending, with ``merge_ranges`` [begin, end))
   every row of a split window over its S_w partials and every heavy row
   outside split windows over its chunks.  Node-parallel, one CTA takes a
   window's slices in order (a slice carries s and S_w), the split windows'
   rows need no merge, and the merge list holds the heavy rows outside split
   windows only.
"""
from __future__ import annotations

import numpy as np

WIN_ROWS = 16
TILE_COLS = 8
FLAG_DUP = 1
FLAG_TILE = 2
FLAG_SPLIT = 8
SPLIT_TILES = 16   # tiles per slice of a split window (128 columns)
ITEM_PARTIAL = 1 << 16
ITEM_CHAIN = 1 << 17


def degrees(row_ptr: np.ndarray) -> np.ndarray:
    return np.diff(row_ptr.astype(np.int64))


def degree_buckets(row_ptr: np.ndarray, bounds) -> dict:
    deg = degrees(row_ptr)
    bounds = np.asarray(bounds, dtype=np.int64)
    nb = len(bounds) + 2
    bucket = np.where(deg == 0, 0, 1 + np.searchsorted(bounds, deg, side="left"))
    order = np.argsort(bucket, kind="stable")  # stable: ascending id inside a bucket
    counts = np.bincount(bucket, minlength=nb)
    ptr = np.zeros(nb + 1, np.int64)
    np.cumsum(counts, out=ptr[1:])
    return dict(bucket_of=bucket.astype(np.uint8), bucket_ptr=ptr.astype(np.int32),
                bucket_rows=order.astype(np.int32))


def auto_heavy_threshold(num_nodes: int, num_edges: int) -> int:
    """The planner's default heavy-row threshold (a scheduling choice of this
    library, not of the pages): ten times the mean degree, rounded to the
    nearest integer, clamped to [64, 512]; 512 for an empty graph."""
    if num_nodes <= 0:
        return 512
    t = (10 * int(num_edges) + int(num_nodes) // 2) // int(num_nodes)
    return int(min(max(t, 64), 512))


def heavy_chunks(row_ptr: np.ndarray, heavy_threshold: int, chunk_edges: int) -> dict:
    deg = degrees(row_ptr)
    heavy = np.flatnonzero(deg > heavy_threshold)
    nch = (deg[heavy] + chunk_edges - 1) // chunk_edges
    hptr = np.zeros(heavy.size + 1, np.int64)
    np.cumsum(nch, out=hptr[1:])
    rows = np.repeat(heavy, nch)
    local = np.arange(int(hptr[-1])) - np.repeat(hptr[:-1], nch)
    start = row_ptr[rows].astype(np.int64) + local * chunk_edges
    end = np.minimum(start + chunk_edges, row_ptr[rows + 1].astype(np.int64))
    chunks = np.stack([rows, start, end], axis=1).astype(np.int32).reshape(-1, 3)
    return dict(heavy_rows=heavy.astype(np.int32), heavy_chunk_ptr=hptr.astype(np.int32),
                chunks=chunks)


def bsb(row_ptr: np.ndarray, col_idx: np.ndarray, num_nodes: int) -> dict:
    n = int(num_nodes)
    deg = degrees(row_ptr)
    W = (n + WIN_ROWS - 1) // WIN_ROWS
    rows = np.repeat(np.arange(n, dtype=np.int64), deg)
    src = col_idx.astype(np.int64)
    win = rows // WIN_ROWS
    r_in = rows % WIN_ROWS

    # sorted unique (window, source) pairs
    key = win * n + src
    order = np.argsort(key, kind="stable")
    ks = key[order]
    first = np.ones(ks.size, dtype=bool)
    first[1:] = ks[1:] != ks[:-1]
    ukey = ks[first]
    uwin = ukey // n
    usrc = ukey % n
    ucount = np.bincount(uwin, minlength=W).astype(np.int64)
    ntiles = (ucount + TILE_COLS - 1) // TILE_COLS
    win_tile_ptr = np.zeros(W + 1, np.int64)
    np.cumsum(ntiles, out=win_tile_ptr[1:])
    T = int(win_tile_ptr[-1])
    ustart = np.zeros(W + 1, np.int64)
    np.cumsum(ucount, out=ustart[1:])
    upos = np.arange(ukey.size, dtype=np.int64) - ustart[uwin]  # rank inside U_w

    tile_cols = np.full(T * TILE_COLS, -1, np.int64)
    tile_cols[win_tile_ptr[uwin] * TILE_COLS + upos] = usrc

    # every edge -> (tile, column slot) -> bit
    uid_sorted = np.cumsum(first) - 1
    uid = np.empty_like(uid_sorted)
    uid[order] = uid_sorted
    pos = upos[uid]
    tile = win_tile_ptr[win] + pos // TILE_COLS
    bit = r_in * TILE_COLS + pos % TILE_COLS
    words = np.zeros((T, 4), np.uint32)
    np.bitwise_or.at(words, (tile, bit // 32), (np.uint32(1) << (bit % 32).astype(np.uint32)))

    # repeated (row, source) pairs
    rkey = np.sort(rows * n + src)
    dup_at = np.flatnonzero(rkey[1:] == rkey[:-1])
    win_dup = np.zeros(W, bool)
    win_dup[(rkey[dup_at] // n) // WIN_ROWS] = True

    win_nnz = np.bincount(win, minlength=W).astype(np.int64)
    return dict(win_tile_ptr=win_tile_ptr.astype(np.int32),
                tile_cols=tile_cols.astype(np.int32),
                tile_bits=words,
                win_nnz=win_nnz.astype(np.int32),
                win_dup=win_dup)


def tile_selection(row_ptr: np.ndarray, b: dict, enabled: bool, heavy_threshold: int,
                   max_tiles: int, density_milli: int, pool_milli: int = 0, split_milli: int = 0) -> dict:
    W = b["win_nnz"].shape[0]
    flags = np.where(b["win_dup"], FLAG_DUP, 0).astype(np.uint8)
    if enabled and split_milli > 0:
        nt = np.diff(b["win_tile_ptr"].astype(np.int64))
        nnz = b["win_nnz"].astype(np.int64)
        split = (~b["win_dup"]) & (nt > SPLIT_TILES) & (1000 * nnz >= int(split_milli) * 128 * nt)
        flags = flags | np.where(split, FLAG_TILE | FLAG_SPLIT, 0).astype(np.uint8)
    if enabled:
        deg = degrees(row_ptr)
        n = deg.shape[0]
        pad = np.zeros(W * WIN_ROWS, np.int64)
        pad[:n] = deg
        maxdeg = pad.reshape(W, WIN_ROWS).max(axis=1)
        nt = np.diff(b["win_tile_ptr"].astype(np.int64))
        nnz = b["win_nnz"].astype(np.int64)
        elig = (~b["win_dup"]) & (nt >= 1) & (nt <= max_tiles) & (maxdeg <= heavy_threshold) \
            & (1000 * nnz >= int(density_milli) * 128 * nt)
        pool_nnz, pool_tiles = int(nnz[elig].sum()), int(nt[elig].sum())
        take = pool_tiles > 0 and 1000 * pool_nnz >= int(pool_milli) * 128 * pool_tiles
        if take:
            flags = flags | np.where(elig, FLAG_TILE, 0).astype(np.uint8)
    tile_windows = np.flatnonzero((flags & (FLAG_TILE | FLAG_SPLIT)) == FLAG_TILE).astype(np.int32)
    split_windows = np.flatnonzero(flags & FLAG_SPLIT).astype(np.int32)
    core_windows = np.flatnonzero((flags & FLAG_TILE) == 0).astype(np.int32)
    return dict(win_flags=flags, tile_windows=tile_windows, split_windows=split_windows, core_windows=core_windows)


def tile_items(row_ptr: np.ndarray, b: dict, tile_windows: np.ndarray, split_windows=(), n_chunks: int = 0,
               edge_parallel: bool = False) -> np.ndarray:
    """Work items of the tile kernel, (n_items, 8) int32.  A window of T
    tiles takes u = ceil(T/2) units of 16 columns (1..8); two windows share an
    item when their units sum to at most 8.  The tile-path list is sorted by
    (u, position in the list) and matched from both ends: the widest
    remaining window takes the narrowest remaining one when the two fit,
    else it is an item on its own; items come in that order.  Per item:
    (w0, first tile of w0, T0, nwin | u0 << 8, w1, first tile of w1, T1, 0)
    with window 0 the narrower of a pair, the second half zero when nwin = 1.
    Then one item per slice s of each split window w (point 4 above): (w,
    first tile + 16 s, its tiles t_s, 1 | ceil(t_s/2) << 8 | 1 << 16,
    n_chunks + 16 B_w + s, S_w, 0, 0) edge-parallel, (w, first tile + 16 s,
    t_s, 1 | ceil(t_s/2) << 8 | 1 << 17, s, S_w, 0, 0) node-parallel."""
    ptr = b["win_tile_ptr"].astype(np.int64)
    out = []

    def entry(w):
        w = int(w)
        return w, int(ptr[w]), int(ptr[w + 1] - ptr[w])

    units = [(int(ptr[w + 1] - ptr[w]) + 1) // 2 for w in tile_windows]
    order = sorted(range(len(tile_windows)), key=lambda i: (units[i], i))
    lo, hi = 0, len(order) - 1
    while lo <= hi:
        wh, fh, th = entry(tile_windows[order[hi]])
        uh = units[order[hi]]
        if lo < hi and units[order[lo]] + uh <= 8:
            wl, fl, tl = entry(tile_windows[order[lo]])
            out.append([wl, fl, tl, 2 | (units[order[lo]] << 8), wh, fh, th, 0])
            lo += 1
        else:
            out.append([wh, fh, th, 1 | (uh << 8), 0, 0, 0, 0])
        hi -= 1
    slices_before = 0
    for w in split_windows:
        w = int(w)
        first, T = int(ptr[w]), int(ptr[w + 1] - ptr[w])
        S = -(-T // SPLIT_TILES)
        for sl in range(S):
            ts = min(SPLIT_TILES, T - SPLIT_TILES * sl)
            if edge_parallel:
                out.append([w, first + SPLIT_TILES * sl, ts, 1 | (((ts + 1) // 2) << 8) | ITEM_PARTIAL,
                            n_chunks + WIN_ROWS * slices_before + sl, S, 0, 0])
            else:
                out.append([w, first + SPLIT_TILES * sl, ts, 1 | (((ts + 1) // 2) << 8) | ITEM_CHAIN, sl, S, 0, 0])
        slices_before += S
    return np.asarray(out, np.int32).reshape(-1, 8)


def merge_list(row_ptr: np.ndarray, b: dict, win_flags: np.ndarray, heavy_threshold: int,
               heavy_chunk_ptr: np.ndarray, n_chunks: int, edge_parallel: bool = False) -> dict:
    """The rows a forward merges when the plan has split windows (point 4):
    ``merge_rows`` ascending and ``merge_ranges`` (n, 2) [begin, end) partial
    indices -- edge-parallel, a split window's row r: n_chunks + 16 B_w + r S_w
    + [0, S_w); a heavy row outside split windows: its chunks."""
    deg = degrees(row_ptr)
    ptr = b["win_tile_ptr"].astype(np.int64)
    W = len(win_flags)
    S = np.zeros(W, np.int64)
    split = (win_flags & FLAG_SPLIT) != 0
    S[split] = -(-(ptr[1:][split] - ptr[:-1][split]) // SPLIT_TILES)
    base = np.concatenate([[0], np.cumsum(S)[:-1]])  # slices before each window
    rows, ranges = [], []
    heavy_ordinal = 0
    for r in range(len(deg)):
        w = r // WIN_ROWS
        heavy = deg[r] > heavy_threshold
        if split[w]:
            if edge_parallel:
                lo = n_chunks + WIN_ROWS * int(base[w]) + (r % WIN_ROWS) * int(S[w])
                rows.append(r)
                ranges.append([lo, lo + int(S[w])])
        elif heavy:
            rows.append(r)
            ranges.append([int(heavy_chunk_ptr[heavy_ordinal]), int(heavy_chunk_ptr[heavy_ordinal + 1])])
        heavy_ordinal += int(heavy)
    return dict(merge_rows=np.asarray(rows, np.int32),
                merge_ranges=np.asarray(ranges, np.int32).reshape(-1, 2))


def full_plan(row_ptr, col_idx, num_nodes, bounds=(32, 256, 2048), heavy_threshold=512,
              chunk_edges=256, with_bsb=True, tile_enabled=False, max_tiles=16,
              density_milli=150) -> dict:
    out = {}
    out.update(degree_buckets(row_ptr, bounds))
    out.update(heavy_chunks(row_ptr, heavy_threshold, chunk_edges))
    if with_bsb:
        b = bsb(row_ptr, col_idx, num_nodes)
        out.update(b)
        out.update(tile_selection(row_ptr, b, tile_enabled, heavy_threshold, max_tiles, density_milli))
    return out
