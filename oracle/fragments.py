"""Register-fragment maps of the warp-level m16n8k16 product (oracle side).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: "Warp Matrix Instructions", section "From Shared Memory to a Matrix
Product".  That page fixes, for one warp computing Out(16x8) = A(16x16) @
B(8x16).T with fp16 inputs and fp32 accumulation:
  * the per-lane register counts: ``ar`` four 32-bit words (eight fp16), ``br``
    two words (four fp16), ``dr`` four fp32 values;
  * the ldmatrix views: A's words regrouped as (chunk group) x row x word with
    row-of-matrix = group*8 + row and word-of-row = chunk*4 + word; B's words as
    chunk x row x word;
  * five layouts written as ``S[shape : stride]`` where a stride tagged
    ``@laneid`` steps the lane index and an untagged stride steps the register
    index within the lane;
  * the store loop Out[lane//4 + 8*(r//2), 2*(lane%4) + r%2] = dr[r] and the
    lane-0 example Out[0,0], Out[0,1], Out[8,0], Out[8,1].
"copy -> ldstmatrix", section "Algorithm" step 2, adds: lane i holds row i//4
and column pair i%4 of each 8x8 matrix.

This module interprets the printed layouts literally (a tiny evaluator of the
``S[shape : stride]`` notation), and derives every map from them; the tests pin
the result against the page's independent statements (the store loop, the
lane-0 example, the ldstmatrix lane rule) and against the plain product.
"""
import itertools

import numpy as np

LANE = "lane"
REG = "reg"

# The five layouts of the page, transcribed as (extent, stride, axis) triples.
# ``4 @ laneid`` -> (.., 4, LANE); a bare stride -> (.., s, REG).
A_LOAD = [(4, 1, REG), (8, 4, LANE), (4, 1, LANE)]
B_LOAD = [(2, 1, REG), (8, 4, LANE), (4, 1, LANE)]
A_MMA = [(1, 4, REG), (1, 4, REG), (2, 1, REG), (8, 4, LANE), (2, 2, REG), (4, 1, LANE)]
B_MMA = [(1, 2, REG), (1, 2, REG), (8, 4, LANE), (2, 1, REG), (4, 1, LANE)]
D_MMA = [(1, 4, REG), (1, 4, REG), (2, 2, REG), (8, 4, LANE), (4, 1, LANE), (2, 1, REG)]


def place(layout, coord):
    """(lane, reg) of a coordinate given in the layout's own (fine) shape."""
    lane = reg = 0
    for (extent, stride, axis), c in zip(layout, coord):
        if not 0 <= c < extent:
            raise IndexError("coordinate %r outside layout %r" % (coord, layout))
        if axis == LANE:
            lane += c * stride
        else:
            reg += c * stride
    return lane, reg


def split(value, extents):
    """Split an index over a view axis into the layout's finer axes (outer first)."""
    out = []
    for e in reversed(extents):
        out.append(value % e)
        value //= e
    if value:
        raise IndexError("index too large for extents %r" % (extents,))
    return tuple(reversed(out))


def a_word_to_matrix(m, row, word):
    """A's ldmatrix view (matrix, row, word) -> (row of A, word of row).

    The rearrange "(group row) (chunk word) -> (chunk group) row word" with
    group=2, chunk=2, word=4 makes matrix index m = chunk*2 + group.
    """
    chunk, group = divmod(m, 2)
    return group * 8 + row, chunk * 4 + word


def b_word_to_matrix(m, row, word):
    """B's ldmatrix view (chunk, row, word) -> (row of B, word of row)."""
    return row, m * 4 + word


def a_load_map():
    """dict (lane, reg) -> (row of A, word of row) from the A load layout."""
    out = {}
    for m, r, w in itertools.product(range(4), range(8), range(4)):
        out[place(A_LOAD, (m, r, w))] = a_word_to_matrix(m, r, w)
    return out


def b_load_map():
    """dict (lane, reg) -> (row of B, word of row) from the B load layout."""
    out = {}
    for m, r, w in itertools.product(range(2), range(8), range(4)):
        out[place(B_LOAD, (m, r, w))] = b_word_to_matrix(m, r, w)
    return out


def a_mma_map():
    """dict (lane, reg) -> (row, word) of A from the MMA operand view (1,1,16,8)."""
    out = {}
    for row, word in itertools.product(range(16), range(8)):
        out[place(A_MMA, (0, 0) + split(row, (2, 8)) + split(word, (2, 4)))] = (row, word)
    return out


def b_mma_map():
    """dict (lane, reg) -> (row n, word) of B from the MMA operand view (1,1,8,8)."""
    out = {}
    for n, word in itertools.product(range(8), range(8)):
        out[place(B_MMA, (0, 0, n) + split(word, (2, 4)))] = (n, word)
    return out


def d_mma_map():
    """dict (lane, reg) -> (row, col) of Out from the D view (1,1,16,8)."""
    out = {}
    for row, col in itertools.product(range(16), range(8)):
        out[place(D_MMA, (0, 0) + split(row, (2, 8)) + split(col, (4, 2)))] = (row, col)
    return out


def store_loop_coords(lane, r):
    """The page's explicit store loop: where dr[r] of ``lane`` goes in Out."""
    return lane // 4 + 8 * (r // 2), 2 * (lane % 4) + r % 2


def fragments_from_matrices(A, B):
    """Per-lane register contents after the two ldmatrix loads.

    A: (16,16) fp16, B: (8,16) fp16.  Returns (ar, br): uint32 arrays (32,4) and
    (32,2); each word packs two fp16 with the lower-index element in the low half.
    """
    a_words = np.ascontiguousarray(A, dtype=np.float16).view(np.uint32)  # (16, 8)
    b_words = np.ascontiguousarray(B, dtype=np.float16).view(np.uint32)  # (8, 8)
    ar = np.zeros((32, 4), dtype=np.uint32)
    br = np.zeros((32, 2), dtype=np.uint32)
    for (lane, reg), (row, word) in a_load_map().items():
        ar[lane, reg] = a_words[row, word]
    for (lane, reg), (row, word) in b_load_map().items():
        br[lane, reg] = b_words[row, word]
    return ar, br


def warp_mma_via_fragments(A, B):
    """Out = A @ B.T computed the way the warp example moves data.

    1. ldmatrix: matrices -> per-lane words via the load layouts;
    2. the MMA reads the same registers through its operand layouts, so A and B
       are re-assembled from the registers with the *MMA* maps;
    3. D = A @ B.T in double (the instruction's definition, C = 0);
    4. D is handed back to lanes through the D layout, and the page's store loop
       writes dr[r] to Out.
    A mismatch between any load layout and its MMA layout scrambles the result,
    which is what the tests check.
    """
    ar, br = fragments_from_matrices(A, B)
    a_seen = np.zeros((16, 8), dtype=np.uint32)
    b_seen = np.zeros((8, 8), dtype=np.uint32)
    for (lane, reg), (row, word) in a_mma_map().items():
        a_seen[row, word] = ar[lane, reg]
    for (lane, reg), (n, word) in b_mma_map().items():
        b_seen[n, word] = br[lane, reg]
    a_val = a_seen.view(np.float16).astype(np.float64)  # (16,16)
    b_val = b_seen.view(np.float16).astype(np.float64)  # (8,16)
    d = a_val @ b_val.T
    dr = np.zeros((32, 4), dtype=np.float64)
    for (lane, reg), (row, col) in d_mma_map().items():
        dr[lane, reg] = d[row, col]
    out = np.full((16, 8), np.nan)
    for lane in range(32):
        for r in range(4):
            out[store_loop_coords(lane, r)] = dr[lane, r]
    return out, dr


def tmem_row_of_thread(tid):
    """"Blackwell Tensor Cores", "The Accumulator's Lifetime": with the 32x32b
    TMEM load at warpgroup scope, warp w reads TMEM lanes 32w..32w+31 and the
    register fragment gives thread tid one accumulator row (row tid)."""
    return tid
