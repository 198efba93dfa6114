"""Runs a single-threaded oracle function once per attention head on all host
cores, for comparisons of every output at full workload sizes."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


def by_head(fn, H, *args, **kw):
    """A single-threaded oracle KV-mode function run once per head, on all host
    cores (the C call releases the GIL): every 4-D [B, S, H, D] argument is
    cut to one head. Heads are independent, so every element is computed by
    the function's own arithmetic; the per-head results are joined along the
    head axis."""
    def one(h):
        return fn(*[np.ascontiguousarray(a[:, :, h:h + 1])
                    if isinstance(a, np.ndarray) and a.ndim == 4 else a for a in args], **kw)

    with ThreadPoolExecutor(max(1, os.cpu_count() or 1)) as ex:
        parts = list(ex.map(one, range(H)))
    if isinstance(parts[0], tuple):
        return tuple(np.concatenate([p[i] for p in parts], axis=2) for i in range(len(parts[0])))
    return np.concatenate(parts, axis=2)
