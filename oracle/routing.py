"""Token permutation by expert and its inverse (TEST INFRASTRUCTURE ONLY).

The routed-expert layer groups the rows of its input by expert so that one
grouped GEMM covers all experts ("--moe-grouped-gemm" / TEGroupedMLP,
Megatron-LM issue #1152, repro steps and additional context), with each group
padded for FP8 ("padding inputs for FP8", same page; "Padding is the correct
way", TransformerEngine issue #2393, maintainer replies).

The pages fix neither the order of rows inside a group nor the padding rule;
the readings taken here:
* rows of expert e appear in token order (stable): the destination of entry
  (t, j) is offsets[e] + #{(t', j') : expert(t', j') = e, t' < t};
* group e occupies [offsets[e], offsets[e] + counts[e]) and is padded with
  filler rows up to a multiple of ``align``:
  offsets[e+1] = offsets[e] + roundup(counts[e], align);
* the inverse map src_row holds, for each permuted row, the flattened
  (token, slot) entry t*k + j it came from (so that both the token and its
  routing probability can be found from the row); filler rows have -1.
"""
from __future__ import annotations

import numpy as np


def permute_indices(topk_idx, E, align):
    """Returns (row_id_map [T,k] int32, src_row [R_pad] int32,
    offsets [E+1] int32, counts [E] int32)."""
    topk_idx = np.asarray(topk_idx, dtype=np.int64)
    T, k = topk_idx.shape
    flat = topk_idx.reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    padded = -(-counts // align) * align
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    # a stable sort by expert keeps (t, j) order inside each expert; because a
    # token never picks one expert twice this is token order
    order = np.argsort(flat, kind="stable")
    starts = np.zeros(E + 1, dtype=np.int64)
    starts[1:] = np.cumsum(counts)
    dest = np.empty(flat.size, dtype=np.int64)
    for e in range(E):
        ent = order[starts[e]:starts[e + 1]]
        dest[ent] = offsets[e] + np.arange(ent.size)
    row_id_map = dest.reshape(T, k)
    src_row = np.full(int(offsets[-1]), -1, dtype=np.int64)
    src_row[dest] = np.arange(T * k)
    return (row_id_map.astype(np.int32), src_row.astype(np.int32),
            offsets.astype(np.int32), counts.astype(np.int32))


def permute_indices_bruteforce(topk_idx, E, align):
    """The same definition written as plain loops (for tiny inputs)."""
    T, k = len(topk_idx), len(topk_idx[0]) if len(topk_idx) else 0
    counts = [0] * E
    for t in range(T):
        for j in range(k):
            counts[int(topk_idx[t][j])] += 1
    offsets = [0]
    for e in range(E):
        offsets.append(offsets[-1] + ((counts[e] + align - 1) // align) * align)
    row_id_map = [[0] * k for _ in range(T)]
    for t in range(T):
        for j in range(k):
            e = int(topk_idx[t][j])
            before = 0
            for t2 in range(t):
                for j2 in range(k):
                    if int(topk_idx[t2][j2]) == e:
                        before += 1
            row_id_map[t][j] = offsets[e] + before
    src_row = [-1] * offsets[-1]
    for t in range(T):
        for j in range(k):
            src_row[row_id_map[t][j]] = t * k + j
    return row_id_map, src_row, offsets, counts


def permute_rows(x, row_id_map, R_pad, fill=0):
    """Gather: out[row_id_map[t, j]] = x[t]; filler rows = ``fill``."""
    x = np.asarray(x)
    out = np.full((R_pad,) + x.shape[1:], fill, dtype=x.dtype)
    T, k = row_id_map.shape
    for j in range(k):
        out[row_id_map[:, j]] = x
    return out


def unpermute(y, row_id_map, probs):
    """Combine: out[t] = sum_j probs[t, j] * y[row_id_map[t, j]], j ascending,
    in float64."""
    y = np.asarray(y, dtype=np.float64)
    probs = np.asarray(probs, dtype=np.float64)
    T, k = row_id_map.shape
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for j in range(k):
        out += probs[:, j:j + 1] * y[row_id_map[:, j]]
    return out


def unpermute_bwd(dout, y, row_id_map, probs, R_pad):
    """Backward of ``unpermute``: dY[row(t, j)] = probs[t, j] * dout[t] and
    dprobs[t, j] = <dout[t], y[row(t, j)]> (float64). Filler rows of dY are 0.
    The float32 product probs * dout is what the quantiser sees: returned too."""
    dout = np.asarray(dout, dtype=np.float64)
    probs32 = np.asarray(probs, dtype=np.float32)
    T, k = row_id_map.shape
    H = dout.shape[1]
    dy32 = np.zeros((R_pad, H), dtype=np.float32)
    for j in range(k):
        dy32[row_id_map[:, j]] = probs32[:, j:j + 1] * dout.astype(np.float32)
    y = np.asarray(y, dtype=np.float64)
    dprobs = np.stack([np.sum(dout * y[row_id_map[:, j]], axis=1) for j in range(k)], axis=1)
    return dy32, dprobs


def permute_bwd(da, row_id_map):
    """Backward of the permutation: dX[t] = sum_j dA[row(t, j)], j ascending."""
    da = np.asarray(da, dtype=np.float64)
    T, k = row_id_map.shape
    out = np.zeros((T, da.shape[1]), dtype=np.float64)
    for j in range(k):
        out += da[row_id_map[:, j]]
    return out
