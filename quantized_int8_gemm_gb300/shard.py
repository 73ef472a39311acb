"""Column-parallel split of the GEMM over ranks (one GPU per rank).

Output rows of W are independent: Y[:, o] needs only row o of W and the whole
activation plane.  Rank r therefore registers its own contiguous slice of W's
rows, [o0, o1), receives the same activations as every other rank, and writes
Y[:, o0:o1] -- no reduction, no exchange inside the GEMM.  The slices are
multiples of the GEMM's 128-row weight tile (the last one takes the ragged
remainder), so no rank pads a tile another rank also computes.  A consumer
that needs the whole Y gathers the column slices once (one all-gather); a
consumer that is itself sharded by columns needs nothing.

Host-side planning and marshalling only: the packed rows of a slice are a
contiguous byte range of W (od rows of id/256 blocks), and the gather is a
torch.distributed all-gather of equal-width padded slices.
"""
from __future__ import annotations

TILE_ROWS = 128  # the GEMM's weight tile; slices are multiples of it
BLOCK_BYTES = {"q4_K": 144, "q6_K": 210}


def od_slices(od: int, world: int, align: int = TILE_ROWS) -> list[tuple[int, int]]:
    """Row ranges [o0, o1) of rank 0 .. world-1: the od rows cut into
    ceil(od/align) units of `align` rows (the last unit ragged) and the units
    shared out as evenly as possible, the first ranks taking one more.  A rank
    left without a unit gets an empty range (o0 == o1)."""
    if od <= 0 or world <= 0 or align <= 0:
        raise ValueError("od, world and align must be positive")
    units = -(-od // align)
    out, u = [], 0
    for r in range(world):
        n = units // world + (1 if r < units % world else 0)
        o0, o1 = min(od, u * align), min(od, (u + n) * align)
        out.append((o0, o1))
        u += n
    return out


def weight_rows(W, qtype: str, id_: int, o0: int, o1: int):
    """The packed bytes of rows [o0, o1) of a k-quant weight (a 1-D byte array
    or tensor holding od rows of id/256 blocks): a contiguous slice, no copy."""
    if id_ % 256:
        raise ValueError("id must be a multiple of 256")
    row = (id_ // 256) * BLOCK_BYTES[qtype]
    return W[o0 * row:o1 * row]


def gather_columns(y_local, slices, group=None):
    """Y (nt x od) on every rank from each rank's Y[:, o0:o1] (y_local, nt x
    (o1 - o0)): one all-gather of slices padded to the widest, then the columns
    put in place.  Works for any torch.distributed backend (gloo on CPU, NCCL
    on GPUs)."""
    import torch
    import torch.distributed as dist
    nt = y_local.shape[0]
    wmax = max(o1 - o0 for o0, o1 in slices)
    od = slices[-1][1]
    pad = torch.zeros((nt, wmax), dtype=y_local.dtype, device=y_local.device)
    pad[:, :y_local.shape[1]] = y_local
    parts = [torch.empty_like(pad) for _ in slices]
    dist.all_gather(parts, pad, group=group)
    y = torch.empty((nt, od), dtype=y_local.dtype, device=y_local.device)
    for (o0, o1), p in zip(slices, parts):
        y[:, o0:o1] = p[:, :o1 - o0]
    return y
