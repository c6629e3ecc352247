"""The tiled order of block-scale arrays (oracle; test infrastructure).

Only tests/ may import this module; the product path never calls it.

The pages fix the scale values of the MXFP8 / NVFP4 formats ([GTP] §1.3: one scale byte per
block of 32 / 16 elements along K) but not their order in memory.  The tiled order is the
tensor core's: a block-scaled tcgen05.mma reads the scale of row 32 c + l from tensor-memory
lane l, column c, and tcgen05.cp.32x128b.warpx4 fills those columns from a 32-row x 16-byte
block of shared memory whose row l holds, in 4-byte steps, the words of rows l, 32 + l,
64 + l, 96 + l (PTX ISA, tcgen05 scale-factor layout).  Laid out in global memory so that a
128-row tile's word w is one such 512-byte block ("atom"):

  scale array sf[rows, cols] (bytes); word w of row r = bytes sf[r, 4w .. 4w + 3]
  atom (t, w), t = r // 128, at byte 512 * (t * ceil(cols / 4) + w)
  inside it, the word of row 128 t + 32 c + l at byte 16 l + 4 c
  bytes of rows >= rows or of columns >= cols: zero

Written out element by element, as the definition reads.
"""
from __future__ import annotations

import numpy as np


def tiled_bytes(rows: int, cols: int) -> int:
    """Size of the tiled form of a [rows, cols] scale array."""
    return -(-rows // 128) * -(-cols // 4) * 512


def tile_scales(sf: np.ndarray) -> np.ndarray:
    """[rows, cols] uint8 -> the tiled uint8 array (padding zero)."""
    sf = np.asarray(sf, dtype=np.uint8)
    rows, cols = sf.shape
    words = -(-cols // 4)
    out = np.zeros(tiled_bytes(rows, cols), dtype=np.uint8)
    r = np.arange(rows)[:, None]
    j = np.arange(cols)[None, :]
    t, c, l = r // 128, (r % 128) // 32, r % 32
    w, byte = j // 4, j % 4
    pos = 512 * (t * words + w) + 16 * l + 4 * c + byte
    out[pos] = sf
    return out


def untile_scales(tiled: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """The inverse: the [rows, cols] scale bytes held by a tiled array."""
    tiled = np.asarray(tiled, dtype=np.uint8)
    words = -(-cols // 4)
    r = np.arange(rows)[:, None]
    j = np.arange(cols)[None, :]
    pos = 512 * ((r // 128) * words + j // 4) + 16 * (r % 32) + 4 * ((r % 128) // 32) + j % 4
    return tiled[pos]
