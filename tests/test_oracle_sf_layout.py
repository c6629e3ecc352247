"""Pins of the tiled scale order (oracle/sf_layout.py) against what fixes it.

The order is the tensor core's: a 512-byte atom is the 32-row x 16-byte block that
tcgen05.cp.32x128b.warpx4 reads, its row l holding the words of rows l, 32 + l, 64 + l,
96 + l of a 128-row tile.  The chunk test reads atoms in exactly that view (reshape to
[atom, l, c, byte]); the others check that the order is a bijection with zero padding, that
it inverts, a few hand-worked positions, and that the library's size function agrees.
The GPU tests then check that the block-scaled GEMM fed tiled scales returns the same
products as with [rows, cols] scales, which only holds if the hardware reads this order.
"""
import numpy as np
import pytest

from oracle import sf_layout as L


@pytest.mark.parametrize("rows,cols", [(1, 1), (32, 4), (128, 16), (130, 9), (300, 10), (513, 64)])
def test_atom_rows_are_the_copy_blocks(rows, cols):
    rng = np.random.default_rng(rows * 1000 + cols)
    sf = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
    tiled = L.tile_scales(sf)
    words = -(-cols // 4)
    tiles = -(-rows // 128)
    padded = np.zeros((tiles * 128, words * 4), dtype=np.uint8)
    padded[:rows, :cols] = sf
    atoms = tiled.reshape(tiles * words, 32, 4, 4)       # [atom, l, c, byte]
    for t in range(tiles):
        block = padded[128 * t:128 * (t + 1)].reshape(4, 32, words, 4)   # [c, l, w, byte]
        for w in range(words):
            assert np.array_equal(atoms[t * words + w], block[:, :, w, :].transpose(1, 0, 2))


@pytest.mark.parametrize("rows,cols", [(50, 5), (1, 255), (255, 1), (17, 15)])
def test_bijection_with_zero_padding(rows, cols):
    sf = (np.arange(rows * cols) % 255 + 1).astype(np.uint8).reshape(rows, cols)
    tiled = L.tile_scales(sf)
    assert tiled.size == L.tiled_bytes(rows, cols)
    assert np.count_nonzero(tiled) == rows * cols
    assert np.array_equal(np.sort(tiled[tiled != 0]), np.sort(sf.ravel()))


@pytest.mark.parametrize("rows,cols", [(1, 3), (129, 7), (256, 128), (1000, 33)])
def test_untile_inverts_tile(rows, cols):
    sf = np.random.default_rng(rows + cols).integers(0, 256, (rows, cols), dtype=np.uint8)
    assert np.array_equal(L.untile_scales(L.tile_scales(sf), rows, cols), sf)


def test_hand_worked_positions():
    rows, cols = 130, 9          # 2 row tiles, 3 words a row: 6 atoms
    sf = np.zeros((rows, cols), dtype=np.uint8)
    marks = {(0, 0): 0, (31, 0): 496, (32, 0): 4, (127, 3): 511, (0, 4): 512, (0, 8): 1024,
             (128, 0): 1536, (129, 6): 2066}
    for k, (r, j) in enumerate(marks):
        sf[r, j] = k + 1
    tiled = L.tile_scales(sf)
    assert tiled.size == 6 * 512
    for k, ((r, j), pos) in enumerate(marks.items()):
        assert tiled[pos] == k + 1, (r, j, pos)


def test_library_size_matches_oracle():
    gtp = pytest.importorskip("param_buffers_gb300")
    try:
        lib = gtp.lib()
    except Exception as e:               # the library is built by __graft_entry__.build()
        pytest.skip(f"libgtp.so not loadable: {e}")
    for rows, cols in [(0, 0), (1, 1), (128, 4), (129, 5), (8192, 128), (2048, 512), (7, 1000)]:
        assert lib.gtp_sf_tiled_bytes(rows, cols) == L.tiled_bytes(rows, cols)
    assert lib.gtp_sf_tiled_bytes(-1, 4) == -1
