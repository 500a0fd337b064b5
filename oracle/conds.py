"""Host helpers of the conditioning pass: areas to latent slices, and packing cond
entries into model calls (test infrastructure; see ``oracle/__init__``).

Source: [SAMPLING] "calc_cond_batch()：最密集的条件逻辑".  For every conditioning entry
the pass turns its area, given as a percentage or as coordinates, into a latent slice;
it then decides which entries can share one model call and, from the free memory, how
many to merge at once.  The section after it ("为什么要自己拼 batch") adds that cond,
uncond and several regions batch together when their shapes and control options are
compatible, are split when memory runs short, and that the batch is not a fixed size
but a packing problem solved at run time.  "一步采样的数据形状" notes that pixel sizes
are divided by the VAE scale to give latent sizes.

Readings (the pages fix neither rounding nor a packing order):

* Area -> slice: the area in latent units (pixels divided by the VAE scale, fractions
  multiplied by the latent height or width, latent units as given) covers rows
  [y0, y0 + h) and columns [x0, x0 + w) of the continuous latent plane; its slice is
  the smallest whole-pixel rectangle that contains it, floor(y0) .. ceil(y0 + h),
  clipped to the frame, in binary64.  An area that covers no latent pixel (outside
  the frame, or of zero height or width) gives an empty slice (h = w = 0).
* Packing: entries are compatible when their latent shape (h, w) and their control
  options key are equal.  A call of shape (h, w) holds at most
  capacity = max(1, floor(budget / (h * w))) rows, budget being the latent pixels the
  free memory allows per call.  Entries are taken in order; an entry's rows go first
  into the last call opened for its key while it has room, the rest into new calls of
  that key, each filled to capacity.  Calls are numbered in the order they open.
"""

from __future__ import annotations

import math
from typing import List, Sequence, Tuple

LATENT, PIXELS, FRACTION = 0, 1, 2


def area_to_latent(units: int, y0: float, x0: float, h: float, w: float, H: int, W: int,
                   scale: int = 8) -> Tuple[int, int, int, int]:
    """(y0, x0, h, w) of the latent slice covering one area, clipped to H x W."""
    if H < 1 or W < 1:
        raise ValueError("the latent frame must be at least 1 x 1")
    vals = (float(y0), float(x0), float(h), float(w))
    if not all(math.isfinite(v) for v in vals) or vals[2] < 0.0 or vals[3] < 0.0:
        raise ValueError("area corner and size must be finite, the size non-negative")
    if units == LATENT:
        ly0, lx0, lh, lw = vals
    elif units == PIXELS:
        if scale < 1:
            raise ValueError("the VAE scale must be at least 1")
        ly0, lx0, lh, lw = (v / float(scale) for v in vals)
    elif units == FRACTION:
        ly0, lh = vals[0] * float(H), vals[2] * float(H)
        lx0, lw = vals[1] * float(W), vals[3] * float(W)
    else:
        raise ValueError(f"unknown area units {units}")
    if lh == 0.0 or lw == 0.0:
        return 0, 0, 0, 0                 # an empty interval covers no pixel
    top = max(math.floor(ly0), 0)
    bottom = min(math.ceil(ly0 + lh), H)
    left = max(math.floor(lx0), 0)
    right = min(math.ceil(lx0 + lw), W)
    if bottom <= top or right <= left:
        return 0, 0, 0, 0
    return int(top), int(left), int(bottom - top), int(right - left)


def pack_conds(entries: Sequence[Tuple[int, int, int, int]], budget: int
               ) -> Tuple[int, List[Tuple[int, int, int, int]]]:
    """Pack cond entries (h, w, rows, options) into model calls.

    Returns (number of calls, chunks), each chunk (call, entry, row0, rows): rows
    [row0, row0 + rows) of that entry run in that call.  Chunks are listed entry by
    entry in row order.
    """
    if budget < 1:
        raise ValueError("the budget must be at least one latent pixel")
    open_call = {}            # key -> [call index, rows used]
    n_calls = 0
    chunks = []
    for e, (h, w, rows, options) in enumerate(entries):
        if h < 1 or w < 1 or rows < 1:
            raise ValueError(f"entry {e}: shape and rows must be positive")
        key = (h, w, options)
        cap = max(1, budget // (h * w))
        row = 0
        while row < rows:
            cur = open_call.get(key)
            if cur is None or cur[1] >= cap:
                cur = [n_calls, 0]
                open_call[key] = cur
                n_calls += 1
            take = min(rows - row, cap - cur[1])
            chunks.append((cur[0], e, row, take))
            cur[1] += take
            row += take
    return n_calls, chunks
