"""Splitting one batch across data-parallel ranks.

Tokens of the layer are independent in the forward, so a batch shards by segment.  With
adapter-affine placement (every segment of an adapter on the same rank, as when requests are routed
to the GPU that holds their adapter -- "Data-Driven Optimization of GPU efficiency for Distributed
LLM-Adapter Serving", adapter placement and routing) the LoRA backward needs no exchange: each
fine-tuning adapter's dA/dB is produced on one rank.  When an adapter's segments do span ranks, the
ranks' dA/dB blocks are summed (an all-reduce of the fp32 gradient pools).

Host logic only; each rank then calls the library on its own rows.
"""
import numpy as np

__all__ = ["shard_segments", "gather_rows"]


def shard_segments(segs, world, affine=True):
    """Split a segment table over `world` ranks.

    Returns one dict per rank: ``rows`` (global token rows in local order) and ``segs`` (the local
    segment table, starts re-based to the local row order).  With ``affine``, all segments of an adapter
    go to one rank (adapters placed largest-first onto the least-loaded rank, base-only segments filling
    in); otherwise segments are dealt out round-robin in start order.
    """
    segs = [tuple(int(v) for v in s) for s in np.asarray(segs, dtype=np.int64).reshape(-1, 4) if s[1] > 0]
    segs.sort()
    owner = {}
    if affine:
        load = [0] * world
        per_ad = {}
        for st, ln, a, tr in segs:
            if a >= 0:
                per_ad[a] = per_ad.get(a, 0) + ln
        for a, n in sorted(per_ad.items(), key=lambda kv: (-kv[1], kv[0])):
            r = min(range(world), key=lambda i: (load[i], i))
            owner[("a", a)] = r
            load[r] += n
        for st, ln, a, tr in segs:
            if a < 0:
                r = min(range(world), key=lambda i: (load[i], i))
                owner[("s", st)] = r
                load[r] += ln
    out = [{"rows": [], "segs": []} for _ in range(world)]
    for i, (st, ln, a, tr) in enumerate(segs):
        if affine:
            r = owner[("a", a)] if a >= 0 else owner[("s", st)]
        else:
            r = i % world
        d = out[r]
        local = len(d["rows"])
        d["rows"].extend(range(st, st + ln))
        d["segs"].append((local, ln, a, tr))
    for d in out:
        d["rows"] = np.asarray(d["rows"], dtype=np.int64)
        d["segs"] = np.asarray(d["segs"], dtype=np.int32).reshape(-1, 4)
    return out


def gather_rows(shards, local_outputs, T):
    """Reassemble per-rank row outputs ([T_r, ...] each) into the global [T, ...] order."""
    first = np.asarray(local_outputs[0])
    out = np.zeros((T,) + first.shape[1:], dtype=first.dtype)
    for d, y in zip(shards, local_outputs):
        out[d["rows"]] = np.asarray(y)
    return out
