"""FNV-1a 64-bit hash over raw bytes in memory order.

The Rocket blog entry "A reduction barrier makes Qwen GDN graph replay bit
exact" hashes output, convolution state and recurrent state with FNV64 to show
replays are bit-identical. The variant is not named there; this is FNV-1a 64
with its published offset basis 14695981039346656037 and prime
1099511628211.
"""
from __future__ import annotations

import numpy as np

OFFSET = 14695981039346656037
PRIME = 1099511628211
MASK = (1 << 64) - 1


def fnv1a64(data) -> int:
    """FNV-1a 64 of the bytes of a contiguous array (or bytes object)."""
    if isinstance(data, (bytes, bytearray)):
        b = bytes(data)
    else:
        b = np.ascontiguousarray(data).tobytes()
    h = OFFSET
    for byte in b:
        h = ((h ^ byte) * PRIME) & MASK
    return h
