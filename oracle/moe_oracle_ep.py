"""Float64 CPU oracle of expert-parallel (EP) staging for the sparse MoE layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
run this module: only the tests use it. It shares no code with the CUDA path.

Source: "MoE 的核心思想", section Expert Parallelism (专家并行): the experts
are spread over devices, each device holding some of them; the router runs
everywhere and every token goes to the device that holds its expert. Its
subsection 前向传播中的 All-to-All 通信 gives the forward in three steps:
  1. dispatch (分发阶段): each device sends the tokens that its routing gave
     to experts held elsewhere to those devices, in one all-to-all;
  2. local compute (本地计算): each device runs its own experts on the tokens
     it received;
  3. combine (合并阶段): the results go back to the source devices in a second
     all-to-all and are summed there with the gate weights.
"MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战" §四 通信瓶颈 says the same
(two all-to-alls per MoE layer: send, then receive).

What this module fixes (the pages leave the layout open; each reading is
listed in the design notes):
  * which device holds which expert is a map owner[e] in [0, R) given by the
    caller (the pages name no placement); block placement
    owner[e] = floor(e * R / N) is the default of the helpers here;
  * capacity and dispatch stay per source device (each device runs the
    single-device dispatch on its own tokens);
  * send order on a source device: destination rank ascending, then the
    destination's experts ascending, then each expert's slots in slot order
    (so an expert's rows stay contiguous, as the single-device dispatch
    leaves them);
  * receive order is the all-to-all's: source rank ascending, each source's
    block in the order it was sent;
  * the receiving device regroups its rows expert-major (its experts
    ascending, then source rank ascending, then the source's order), runs its
    experts, and regroups the outputs back into receive order for the return
    all-to-all; the source device puts each returned row back at its slot;
  * the expert outputs travel back in float64 here (fp32 on the GPU), so the
    combine is the single-device one;
  * shared experts are not part of the exchange (each device runs them on its
    own tokens).
"""
from __future__ import annotations

import numpy as np


def block_owner(N: int, R: int) -> np.ndarray:
    """owner[e] = floor(e * R / N): R devices, consecutive experts on each
    (every device holds N/R experts when R divides N)."""
    return (np.arange(N, dtype=np.int64) * R) // N


def local_experts(owner, r: int) -> np.ndarray:
    """The experts device r holds, ascending."""
    return np.nonzero(np.asarray(owner) == r)[0].astype(np.int64)


def send_counts(kept, owner, R: int) -> np.ndarray:
    """Rows a source device sends to each destination: the kept assignments
    of the destination's experts."""
    kept = np.asarray(kept, dtype=np.int64)
    return np.array([int(kept[local_experts(owner, r)].sum()) for r in range(R)],
                    dtype=np.int64)


def pack(rows, offsets, owner, R: int):
    """Dispatch step on a source device: its expert-contiguous rows (x_perm,
    expert e at [offsets[e], offsets[e+1])) laid out by destination.
    Returns (send rows, send_counts[R]); the send buffer is destination 0's
    block, then destination 1's, ..."""
    rows = np.asarray(rows)
    offsets = np.asarray(offsets, dtype=np.int64)
    blocks = []
    for r in range(R):
        for e in local_experts(owner, r):
            blocks.append(rows[offsets[e]:offsets[e + 1]])
    send = np.concatenate(blocks, axis=0) if blocks else rows[:0]
    return send, send_counts(np.diff(offsets), owner, R)


def unpack(back, offsets, owner, R: int, n_rows=None):
    """Combine step on a source device: the rows returned by the second
    all-to-all (in the order pack sent them) put back at their slots, i.e.
    the inverse of pack. Returns [n_rows (default offsets[N])][...]."""
    back = np.asarray(back)
    offsets = np.asarray(offsets, dtype=np.int64)
    n = int(offsets[-1]) if n_rows is None else n_rows
    out = np.zeros((n,) + back.shape[1:], dtype=back.dtype)
    pos = 0
    for r in range(R):
        for e in local_experts(owner, r):
            cnt = int(offsets[e + 1] - offsets[e])
            out[offsets[e]:offsets[e + 1]] = back[pos:pos + cnt]
            pos += cnt
    assert pos == back.shape[0], "returned rows do not match the sent layout"
    return out


def exchange(blocks_by_source):
    """An all-to-all: blocks_by_source[s][r] is what source s sends to r;
    returns received[r] = the blocks of every source s ascending, stacked."""
    R = len(blocks_by_source)
    return [np.concatenate([blocks_by_source[s][r] for s in range(R)], axis=0)
            for r in range(R)]


def split_by_counts(buf, counts):
    """A send buffer cut into its per-destination blocks."""
    ends = np.cumsum(counts)
    return np.split(np.asarray(buf), ends[:-1].tolist())


def regroup(recv, kept_all, owner, r: int):
    """Local-compute set-up on device r: its received rows (source-major:
    source s's rows of r's experts, experts ascending) rearranged
    expert-major (r's experts ascending, then sources ascending).
    kept_all[s][e]: the kept assignments of expert e on source s.
    Returns (x_local, local_offsets[E_r + 1])."""
    kept_all = np.asarray(kept_all, dtype=np.int64)
    R = kept_all.shape[0]
    mine = local_experts(owner, r)
    # where each (source, expert) block starts in the receive buffer
    start = {}
    pos = 0
    for s in range(R):
        for e in mine:
            start[(s, int(e))] = pos
            pos += int(kept_all[s, e])
    assert pos == np.asarray(recv).shape[0], "received rows do not match the counts"
    parts, loff = [], [0]
    for e in mine:
        for s in range(R):
            b = start[(s, int(e))]
            parts.append(np.asarray(recv)[b:b + int(kept_all[s, e])])
        loff.append(loff[-1] + int(kept_all[:, e].sum()))
    x_local = np.concatenate(parts, axis=0) if parts else np.asarray(recv)[:0]
    return x_local, np.array(loff, dtype=np.int64)


def regroup_back(o_local, kept_all, owner, r: int):
    """The inverse of regroup on device r: outputs in expert-major order put
    back in receive order (source-major), ready for the return all-to-all."""
    kept_all = np.asarray(kept_all, dtype=np.int64)
    R = kept_all.shape[0]
    mine = local_experts(owner, r)
    o_local = np.asarray(o_local)
    # where each (expert, source) block sits in the expert-major order
    at = {}
    pos = 0
    for e in mine:
        for s in range(R):
            at[(int(e), s)] = pos
            pos += int(kept_all[s, e])
    assert pos == o_local.shape[0]
    parts = []
    for s in range(R):
        for e in mine:
            b = at[(int(e), s)]
            parts.append(o_local[b:b + int(kept_all[s, e])])
    return np.concatenate(parts, axis=0) if parts else o_local[:0]
