"""Expert-parallel dispatch and combine of the routed rows, in FP8.

With P ranks, rank r owns experts [r E/P, (r + 1) E/P). Every rank routes and
quantises its own tokens with mgq_moe_permute (rows grouped by global expert,
each group padded to a multiple of 128 rows), so the rows it owes rank d for
d's j-th expert are one contiguous, 128-row-aligned slice of its permuted
buffer, and so are their MX (E8M0) or NVFP4 (ue4m3) scale tiles. The exchange
moves those already-quantised rows: one byte per element plus the scales,
about half the bytes of bf16 rows, as the FP8 all-gather discussion of
"FP8BlockQuantizer not work on TE" (TransformerEngine issue #2393, maintainer
replies) points out for quantise-before-communicate.

dispatch: one all_to_all per local expert j. Rank s sends its slice of expert
  (d, j) to every rank d; rank d receives them into consecutive slices of its
  receive buffer, source ranks in order, each source's padded group whole. The
  receive buffer is then expert-major with every group a multiple of 128 rows:
  exactly the layout the grouped GEMMs take, with group offsets
  `recv_offsets` over the E/P local experts.
combine: the reverse exchange of the expert outputs (bf16 rows), back into
  each source rank's own permuted layout, where mgq_moe_unpermute finishes.

Only tensors and torch.distributed collectives are used here (NCCL on GPUs,
gloo on CPU tensors). The slices are views: with NCCL each all_to_all reads
and writes them in place; gloo has only the single-buffer form, so there the
send slices are packed into one buffer and the received bytes copied into
their slots. Per-tensor scaled codes can be exchanged too, when the
ranks share the scale (their amax reduced across ranks first: `allreduce_amax`);
MX and NVFP4 block scales travel with their rows. The blockwise 1x128 scale
layout ([K/128][R_cap], block-major) is not row-contiguous and is not
exchanged here.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

TILE = 128      # rows per scale tile; every group is padded to a multiple of it


class EPExchange:
    """Bookkeeping of one exchange, from the padded group sizes of every rank.

    sizes  [P, E] rows of each (source rank, global expert) group, multiples
           of 128 (the offsets differences of each rank's mgq_moe_permute)
    rank   this rank
    """

    def __init__(self, sizes, rank: int):
        sizes = np.asarray(sizes, dtype=np.int64)
        self.P, self.E = sizes.shape
        if self.E % self.P:
            raise ValueError("the experts must divide evenly over the ranks")
        if np.any(sizes % TILE):
            raise ValueError("group sizes must be multiples of 128 rows")
        self.rank = rank
        self.El = self.E // self.P
        self.sizes = sizes
        # each source's group offsets in its own permuted buffer
        self.src_off = np.concatenate([np.zeros((self.P, 1), np.int64), np.cumsum(sizes, axis=1)], axis=1)
        # receive layout: local expert j, then source rank s
        mine = sizes[:, rank * self.El:(rank + 1) * self.El]            # [P, El]
        self.recv_sizes = mine.T.copy()                                  # [El, P]
        flat = np.concatenate([[0], np.cumsum(self.recv_sizes.reshape(-1))])
        self.recv_slot = flat[:-1].reshape(self.El, self.P)              # start of (j, s)
        self.recv_offsets = np.concatenate([[0], np.cumsum(self.recv_sizes.sum(axis=1))]).astype(np.int32)
        self.R_recv = int(self.recv_offsets[-1])
        self.R_send = int(self.src_off[rank, -1])

    def send_range(self, d: int, j: int):
        """Rows of this rank's buffer that go to rank d for its expert j."""
        e = d * self.El + j
        return int(self.src_off[self.rank, e]), int(self.src_off[self.rank, e + 1])

    def recv_range(self, j: int, s: int):
        """Rows of the receive buffer that come from rank s for local expert j."""
        a = int(self.recv_slot[j, s])
        return a, a + int(self.recv_sizes[j, s])


def exchange_sizes(offsets: torch.Tensor, group=None) -> np.ndarray:
    """All ranks' padded group sizes [P, E] from this rank's offsets [E + 1]
    (device or host int32; one host synchronisation)."""
    off = offsets.to(torch.int64)
    mine = (off[1:] - off[:-1]).contiguous()
    world = dist.get_world_size(group)
    out = torch.empty(world * mine.numel(), dtype=torch.int64, device=mine.device)
    dist.all_gather_into_tensor(out, mine, group=group)
    return out.cpu().numpy().reshape(world, -1)


def _row_view(t: torch.Tensor, a: int, b: int) -> torch.Tensor:
    return t[a:b]


def _tile_view(scales: torch.Tensor, a: int, b: int, tile_bytes: int) -> torch.Tensor:
    """The scale bytes of rows [a, b) of a 128x4-tiled scale buffer (a, b
    multiples of 128): tile_bytes bytes per 128 rows."""
    flat = scales.view(-1)
    return flat[(a // TILE) * tile_bytes:(b // TILE) * tile_bytes]


def _exchange(ex: EPExchange, send_view, recv_view, reverse: bool, group=None):
    """One all_to_all per local expert j. Forward: this rank sends its slice of
    (d, j) to d and receives (j, s) from s. Reverse: it sends (j, s) back to s
    and receives its own (d, j) slice from d."""
    for j in range(ex.El):
        if not reverse:
            ins = [send_view(*ex.send_range(d, j)) for d in range(ex.P)]
            outs = [recv_view(*ex.recv_range(j, s)) for s in range(ex.P)]
        else:
            ins = [send_view(*ex.recv_range(j, s)) for s in range(ex.P)]
            outs = [recv_view(*ex.send_range(d, j)) for d in range(ex.P)]
        _all_to_all(outs, ins, group)


def _all_to_all(outs, ins, group=None):
    """all_to_all over per-rank views (empty views allowed): in place with
    NCCL; gloo packs into one buffer (it has only the single-buffer form)."""
    if dist.get_backend(group) == "nccl":
        dist.all_to_all(outs, [t.contiguous() for t in ins], group=group)
        return
    ins = [t.contiguous() for t in ins]
    send = torch.cat([t.reshape(-1) for t in ins]) if ins else None
    in_splits = [t.numel() for t in ins]
    out_splits = [t.numel() for t in outs]
    recv = torch.empty(sum(out_splits), dtype=ins[0].dtype, device=ins[0].device)
    dist.all_to_all_single(recv, send, output_split_sizes=out_splits, input_split_sizes=in_splits, group=group)
    pos = 0
    for t, n in zip(outs, out_splits):
        if n:
            t.view(-1).copy_(recv[pos:pos + n])
        pos += n


def dispatch(ex: EPExchange, codes: torch.Tensor, scales: torch.Tensor | None, recv_codes: torch.Tensor,
             recv_scales: torch.Tensor | None, tile_bytes: int = 0, group=None):
    """Moves the quantised rows (codes [R, W] bytes, W = H or H/2 for e2m1)
    and, when given, their 128x4-tiled block scales (`tile_bytes` bytes per
    128 rows: MX H/32*128, NVFP4 H/16*128) to the ranks that own their experts.
    recv_codes [>= R_recv, W], recv_scales >= R_recv/128 * tile_bytes bytes."""
    _exchange(ex, lambda a, b: _row_view(codes, a, b), lambda a, b: _row_view(recv_codes, a, b), False, group)
    if scales is not None:
        _exchange(ex, lambda a, b: _tile_view(scales, a, b, tile_bytes),
                  lambda a, b: _tile_view(recv_scales, a, b, tile_bytes), False, group)


def combine(ex: EPExchange, y_recv: torch.Tensor, y_local: torch.Tensor, group=None):
    """Returns the expert outputs (y_recv [R_recv, H], received-row order) to
    the ranks that own the tokens: y_local [>= R_send, H] in this rank's own
    permuted layout, ready for mgq_moe_unpermute."""
    _exchange(ex, lambda a, b: _row_view(y_recv, a, b), lambda a, b: _row_view(y_local, a, b), True, group)


def allreduce_amax(amax: torch.Tensor, group=None) -> torch.Tensor:
    """Per-tensor scaling across ranks: every rank quantises with the scale of
    the largest amax (in place, MAX reduction)."""
    dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    return amax
