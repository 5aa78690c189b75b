"""Layout algebra, written out from its definitions.  TEST INFRASTRUCTURE ONLY.

Sources (restated, not copied):
  * "Advanced CUTLASS Architecture and Kernel Optimization", section "CuTe
    Layout Algebra" (oboe.com): a layout is a pair (Shape, Stride) of integer
    tuples; crd2idx is the dot product of a coordinate with the stride;
    composition A o B is the function c -> A(B(c)); logical_divide(L, S)
    splits L into a within-tile and an across-tile mode.
  * "4.21 What is CuTe?" (gpu-glossary-zh): shapes and strides are
    hierarchical tuples; tiled_divide keeps the tile's own modes first and the
    tile index after them, which fixes the mode order of a divide.

Conventions (the standard CuTe ones, where the pages are silent):
  * an integer index is turned into a coordinate colexicographically (the
    leftmost mode varies fastest);
  * complement(L, M) lists the gaps in the image of L, ordered by stride, and
    ends with the mode that repeats the whole covered range up to M;
  * logical_divide(L, T) = L o (T, complement(T, size(L))).

A layout here is a pair (shape, stride) of equally nested tuples of ints (a
bare int is a rank-0 leaf).  Results of composition/divide are returned as a
*function table* over the right operand's domain, plus that domain's shape:
the oracle needs no closed form for them.
"""
from __future__ import annotations

from math import prod


def is_tuple(x):
    return isinstance(x, tuple)


def flatten(t):
    if is_tuple(t):
        out = []
        for e in t:
            out.extend(flatten(e))
        return out
    return [t]


def size(shape):
    return prod(flatten(shape))


def idx2crd(i, shape):
    """Colexicographic integer -> hierarchical coordinate inside `shape`."""
    if is_tuple(shape):
        out = []
        for s in shape:
            n = size(s)
            out.append(idx2crd(i % n, s))
            i //= n
        return tuple(out)
    return i


def crd2idx(crd, shape, stride):
    """Dot product of a (possibly integer, possibly hierarchical) coordinate with the stride."""
    if is_tuple(shape):
        if not is_tuple(crd):
            crd = idx2crd(crd, shape)
        assert len(crd) == len(shape) == len(stride)
        return sum(crd2idx(c, s, d) for c, s, d in zip(crd, shape, stride))
    if is_tuple(crd):
        raise ValueError("coordinate deeper than shape")
    assert 0 <= crd < shape or shape == 0, (crd, shape)
    return crd * stride


def evaluate(shape, stride, i):
    return crd2idx(idx2crd(i, shape) if is_tuple(shape) else i, shape, stride)


def table(shape, stride):
    """The layout as the list of its values over 0 .. size-1."""
    return [evaluate(shape, stride, i) for i in range(size(shape))]


def cosize(shape, stride):
    """1 + the largest value the layout takes (for non-negative strides)."""
    return max(table(shape, stride)) + 1 if size(shape) else 0


def compose_table(a_shape, a_stride, b_shape, b_stride):
    """(A o B)(i) = A(B(i)) for every i in B's domain."""
    return [evaluate(a_shape, a_stride, evaluate(b_shape, b_stride, i)) for i in range(size(b_shape))]


def complement(shape, stride, m):
    """complement(L, m) as a flat (shape, stride) pair of tuples.

    Modes of L with extent 1 or stride 0 take no part.  The rest are sorted by
    stride; each gap between the running product of (extent x stride) and the
    next stride becomes a mode, and a last mode extends the covered range to m."""
    modes = sorted((d, s) for s, d in zip(flatten(shape), flatten(stride)) if s != 1 and d != 0)
    out_s, out_d = [], []
    cur = 1
    for d, s in modes:
        if d % cur:
            raise ValueError("complement: stride not divisible by the covered range")
        gap = d // cur
        if gap > 1:
            out_s.append(gap)
            out_d.append(cur)
        cur = s * d
    rest = -(-m // cur)
    out_s.append(rest)
    out_d.append(cur)
    # a gap-free complement of a covering layout is the trivial 1:cur mode
    return tuple(out_s), tuple(out_d)


def logical_divide_table(l_shape, l_stride, t_shape, t_stride):
    """logical_divide(L, T) = L o (T, complement(T, size(L))).

    Returns (domain shape, table): domain shape is (T's shape, complement's
    shape), i.e. within-tile mode first, tile index second."""
    c_shape, c_stride = complement(t_shape, t_stride, size(l_shape))
    b_shape = (t_shape, c_shape)
    b_stride = (t_stride, c_stride)
    return b_shape, compose_table(l_shape, l_stride, b_shape, b_stride)


def is_bijective_onto(shape, stride, n):
    """True when the layout's values are exactly {0, .., n-1}, each once."""
    return sorted(table(shape, stride)) == list(range(n))


# ---------------------------------------------------------------- thread maps

def stripmined_coords(rows, cols, threads, vec, tid, it):
    """PitchLinearStripminedThreadMap walkthrough (lpnh.cn/news/2469163), sec. 3.1:
    columns are dealt out first: column_groups = cols / vec, the column group
    is tid mod column_groups, the row anchor is tid div column_groups, and
    iteration `it` moves down by row_stride = rows / iterations rows, where
    iterations = rows * cols / threads / vec (sec. 2.1's invariant).
    Returns the (row, col) of the first element of the vector."""
    assert (rows * cols) % (threads * vec) == 0
    iterations = rows * cols // threads // vec
    column_groups = cols // vec
    row_stride = rows // iterations
    cg = tid % column_groups
    ra = tid // column_groups
    return ra + it * row_stride, cg * vec


def stripmined_predicate(rows, cols, threads, vec, extent_rows, extent_cols, tid, it):
    """Sec. 4.2's guard: the access is live when row < extent_rows and the
    vector's first column < extent_cols (row_stride from the tile, sec. 4.3)."""
    r, c = stripmined_coords(rows, cols, threads, vec, tid, it)
    return r < extent_rows and c < extent_cols


# ---------------------------------------------------------------- per-mode tiling

def zipped_divide_table(shape, stride, tilers):
    """zipped_divide of a rank-r layout by r contiguous tilers (t_i:1), from the
    definition: element (within-tile coordinate w, tile coordinate q) sits at
    per-mode coordinate w_i + t_i * q_i.  Domain: ((t_0, .., t_r-1), (n_0/t_0, ..)),
    colexicographic.  Returns (domain shape, table)."""
    modes = [(s, d) for s, d in zip(shape, stride)]
    rests = [size(m[0]) // t for m, t in zip(modes, tilers)]
    dom = (tuple(tilers), tuple(rests))
    tab = []
    for i in range(size(dom)):
        crd = idx2crd(i, dom)
        w, q = crd
        val = 0
        for k, (s, d) in enumerate(modes):
            val += evaluate(s, d, w[k] + tilers[k] * q[k])
        tab.append(val)
    return dom, tab


def local_partition_offsets(tile_shape, tile_stride, thr_shape, thr_stride, idx):
    """Offsets of the tile elements thread `idx` owns: the thread at position
    (c_0, c_1, ..) of the thread grid (the coordinate whose thread-layout value
    is idx) owns per-mode coordinates c_k + T_k * a_k, walked colexicographically
    over a.  From the definition on "4.21 What is CuTe?" (local_partition)."""
    pos = next(i for i in range(size(thr_shape)) if evaluate(thr_shape, thr_stride, i) == idx)
    c = idx2crd(pos, tuple(size(s) for s in thr_shape))
    T = [size(s) for s in thr_shape]
    reps = tuple(size(s) // t for s, t in zip(tile_shape, T))
    out = []
    for a_i in range(size(reps)):
        a = idx2crd(a_i, reps)
        out.append(sum(evaluate(s, d, c[k] + T[k] * a[k]) for k, (s, d) in enumerate(zip(tile_shape, tile_stride))))
    return out
