"""Gradient-bucket formation and the flat-bucket gather (oracle; test
infrastructure).

DeepSpeed ZeRO-3 source walkthrough, section 3.1 and 5.1: gradients arrive one
parameter at a time; each is placed at the bucket's running offset
(offset += numel), and the bucket is reduced early once adding the next
gradient would take it past reduce_bucket_size; after backward the partly
filled last bucket is flushed too (section 5.4).  Section 3.2: with
contiguous_gradients the bucket is one preallocated flat buffer and each
parameter's gradient occupies [offset, offset + numel) of it.

In the simulation every rank's gradients already exist as separate buffers, so
the flat bucket is filled by an explicit copy at each gradient's offset.

Readings where the pages leave a step open:
  * a gradient larger than the cap is never split: it forms a bucket of its
    own (the flush rule applied literally: the running bucket is flushed first,
    the next gradient flushes it again);
  * the bucket's element count is rounded up to a multiple of `pad_to`
    (default K) so that the ring can split it into K equal chunks; the padding
    is never written by the gather and must be zero in the caller's buffer.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class Bucket:
    params: list          # parameter indices (arrival order) in this bucket
    offsets: list         # element offset of each parameter in the flat buffer
    used: int             # sum of numels
    numel: int            # used rounded up to a multiple of pad_to


def assign_buckets(numel: list, cap: int, pad_to: int = 1) -> list:
    """Greedy bucket formation over gradients in arrival order."""
    if cap <= 0 or pad_to <= 0:
        raise ValueError("cap and pad_to must be positive")
    buckets = []
    cur_p, cur_off, used = [], [], 0

    def flush():
        nonlocal cur_p, cur_off, used
        if cur_p:
            padded = -(-used // pad_to) * pad_to
            buckets.append(Bucket(cur_p, cur_off, used, padded))
        cur_p, cur_off, used = [], [], 0

    for p, n in enumerate(numel):
        if n <= 0:
            raise ValueError("every gradient must have at least one element")
        if cur_p and used + n > cap:
            flush()
        cur_p.append(p)
        cur_off.append(used)
        used += n
    flush()
    return buckets


def flatten_bucket(src: list, numel: list, offset: list, bucket_numel: int,
                   dst_init: list | None = None) -> list:
    """Copy rank r's gradient p (src[r][p], uint16 bf16 bits) to elements
    [offset[p], offset[p] + numel[p]) of rank r's flat bucket.  Positions no
    gradient covers keep dst_init's value (zeros by default)."""
    K = len(src)
    P = len(numel)
    spans = sorted((offset[p], offset[p] + numel[p]) for p in range(P))
    for (a0, a1), (b0, _) in zip(spans, spans[1:]):
        if b0 < a1:
            raise ValueError("gradients overlap in the bucket")
    if spans and (spans[0][0] < 0 or spans[-1][1] > bucket_numel):
        raise ValueError("gradient outside the bucket")
    out = []
    for r in range(K):
        d = (np.zeros(bucket_numel, dtype=np.uint16) if dst_init is None
             else np.asarray(dst_init[r], dtype=np.uint16).copy())
        for p in range(P):
            s = np.asarray(src[r][p], dtype=np.uint16).reshape(-1)
            if len(s) != numel[p]:
                raise ValueError("numel does not match the gradient")
            d[offset[p]:offset[p] + numel[p]] = s
        out.append(d)
    return out
