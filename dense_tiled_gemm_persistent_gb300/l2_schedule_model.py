"""A host-side model of L2 reuse under the pair kernel's persistent schedule.

It estimates the DRAM bytes one launch reads, for choosing the band height
(GROUP_SIZE_M) of the grouped tile order.  It is not part of the GEMM path.

The model:
  * L2 is one fully associative LRU cache of `cap_bytes`.
  * Data moves in 32 KiB units, one TMA block each: 256 rows (or columns)
    by 64 K elements of 2 bytes.
  * The pairs of a wave run in lockstep over the k-blocks; odd waves run K
    backwards, as the kernel's whole tiles do.  Each pair touches its A row
    block and its B column block at every k-block.
  * A wave's C tiles are written into the cache as it ends.

A miss is one unit read from DRAM.  With a 64 MiB cache the model ranks the
band heights as ncu measured them on 8192^3 FP16 and 16384 x 14336 x 4096
BF16; its byte counts are 6-15 % below the measured ones.

    python -m dense_tiled_gemm_persistent_gb300.l2_schedule_model 8192 8192 8192
"""
from __future__ import annotations

import sys
from collections import OrderedDict

UNIT = 32 << 10          # one 256 x 64 block of 2-byte elements
TILE = 256               # pair tile edge
KBLOCK = 64


def grouped_tile(tiles_m: int, tiles_n: int, group_m: int, bid: int):
    """The grouped order: bands of group_m tile rows, down a band's rows first."""
    band_tiles = group_m * tiles_n
    band = bid // band_tiles
    row0 = band * group_m
    rows = min(group_m, tiles_m - row0)
    return row0 + bid % rows, (bid - band * band_tiles) // rows


def dram_read_bytes(M: int, N: int, K: int, group_m: int, resident: int = 76, cap_bytes: int = 64 << 20,
                    alternate_k: bool = True, out_bytes: int = 2) -> int:
    """Bytes the modelled launch reads from DRAM (whole tiles only, no stream-K tail)."""
    tm, tn, kb = -(-M // TILE), -(-N // TILE), -(-K // KBLOCK)
    cap = cap_bytes // UNIT
    c_units = max(1, TILE * TILE * out_bytes // UNIT)
    lru: OrderedDict = OrderedDict()
    misses = 0
    order = [grouped_tile(tm, tn, group_m, t) for t in range(tm * tn)]
    c_id = 0
    for w in range(0, len(order), resident):
        wave = order[w:w + resident]
        ks = range(kb - 1, -1, -1) if (alternate_k and (w // resident) % 2) else range(kb)
        for k in ks:
            for r, c in wave:
                for key in (("A", r, k), ("B", c, k)):
                    if key in lru:
                        lru.move_to_end(key)
                    else:
                        misses += 1
                        lru[key] = None
                        if len(lru) > cap:
                            lru.popitem(last=False)
        for _ in wave:
            for u in range(c_units):
                lru[("C", c_id, u)] = None
                if len(lru) > cap:
                    lru.popitem(last=False)
            c_id += 1
    return misses * UNIT


def main(argv) -> None:
    M, N, K = (int(x) for x in argv[:3])
    heights = [int(x) for x in argv[3:]] or [4, 6, 8, 10, 11, 12, 13, 14, 16, 20, 24, 32]
    for g in heights:
        if g <= -(-M // TILE):
            print("group %2d: %.3f GB" % (g, dram_read_bytes(M, N, K, g) / 1e9), flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])
