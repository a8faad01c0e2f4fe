"""A mixture-of-experts MLP with static shapes -- TEST INFRASTRUCTURE.

"33. Removing overhead", §A MoE layer that never asks the host: instead of one
matmul per expert and a host-side count of each expert's tokens, the
assignments (token, slot) are grouped by expert on the device, each group padded
to a multiple of BLOCK_M rows, and one grouped GEMM multiplies every block of
rows by the weights of the expert that owns it.  Every output shape depends only
on the token count N, the experts per token k, the expert count E and BLOCK_M.

This module states it plainly in float64:
  * ``route``: the router (the pages call it from an earlier chapter that is
    not included; the reading taken is Qwen3-MoE's: softmax over the router
    logits, the k most probable experts with ties to the lower id, their
    probabilities renormalised to sum to 1);
  * ``moe_align``: the grouping, from its definition, expert by expert;
  * ``moe_reference``: the layer as a loop over tokens and their k experts;
  * ``moe_grouped``: the same layer computed the grouped way, block by block
    through ``moe_align``'s output, so that the two can be checked against
    each other.
gate_up[e] holds the expert's gate rows first and its up rows second; the
activation is silu(gate) * up, as in the dense MLP.

Parity: ``moe_align`` against brute-force invariants on random routings and a
hand-worked case; ``moe_grouped`` against ``moe_reference``; ``moe_reference``
against scalar loops on tiny sizes and the linearity / permutation properties
of the definition; ``route`` against a brute-force ranking and the two-expert
closed form.
"""
from __future__ import annotations

import numpy as np

from .model import silu


def route(x: np.ndarray, w_router: np.ndarray, top_k: int) -> tuple[np.ndarray, np.ndarray]:
    """Router weights [N, k] (float64, rows sum to 1) and expert ids [N, k] (int64) for token rows x [N, D]."""
    logits = np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    E = p.shape[1]
    ids = np.empty((p.shape[0], top_k), dtype=np.int64)
    for t in range(p.shape[0]):
        order = np.lexsort((np.arange(E), -p[t]))     # most probable first, ties to the lower id
        ids[t] = order[:top_k]
    w = np.take_along_axis(p, ids, axis=1)
    return w / w.sum(axis=1, keepdims=True), ids


def padded_rows(total: int, num_experts: int, block_m: int) -> int:
    """Rows of the grouped layout: room for every assignment plus block_m - 1 padding rows per expert,
    rounded up to whole blocks."""
    m = total + num_experts * (block_m - 1)
    return -(-m // block_m) * block_m


def moe_align(expert_ids: np.ndarray, num_experts: int, block_m: int):
    """Group the flat assignments a = token * k + slot by expert, each group padded to whole blocks.

    Returns (sorted_ids [M], block_expert [M // block_m], num_padded):
      * sorted_ids[i] is the assignment row i of the grouped GEMM handles, or N * k on a padding row;
        expert 0's group comes first, then expert 1's, ...; inside a group the assignments ascend;
      * block_expert[b] is the expert whose group holds block b; blocks from num_padded on belong to no
        group and name the last expert (they hold padding only);
      * num_padded is the number of rows the groups occupy (a multiple of block_m).
    M = padded_rows(N * k, E, block_m) whatever the routing.
    """
    flat = np.asarray(expert_ids, dtype=np.int64).reshape(-1)
    total = flat.size
    M = padded_rows(total, num_experts, block_m)
    sorted_ids = np.full(M, total, dtype=np.int64)
    block_expert = np.full(M // block_m, num_experts - 1, dtype=np.int64)
    row = 0
    for e in range(num_experts):
        mine = np.flatnonzero(flat == e)                  # ascending assignment order
        sorted_ids[row:row + mine.size] = mine
        blocks = -(-mine.size // block_m)
        block_expert[row // block_m: row // block_m + blocks] = e
        row += blocks * block_m
    return sorted_ids, block_expert, row


def _expert_mlp(x_row: np.ndarray, gate_up_e: np.ndarray, down_e: np.ndarray) -> np.ndarray:
    gu = gate_up_e @ x_row
    inter = gu.shape[0] // 2
    return down_e @ (silu(gu[:inter]) * gu[inter:])


def moe_reference(x, gate_up, down, weights, expert_ids) -> np.ndarray:
    """out[t] = sum_j weights[t, j] * down[e] (silu(gate[e] x[t]) * up[e] x[t]), e = expert_ids[t, j]."""
    x = np.asarray(x, dtype=np.float64)
    gate_up = np.asarray(gate_up, dtype=np.float64)
    down = np.asarray(down, dtype=np.float64)
    out = np.zeros((x.shape[0], down.shape[1]))
    for t in range(x.shape[0]):
        for j in range(expert_ids.shape[1]):
            e = int(expert_ids[t, j])
            out[t] += float(weights[t, j]) * _expert_mlp(x[t], gate_up[e], down[e])
    return out


def moe_grouped(x, gate_up, down, weights, expert_ids, block_m: int = 16) -> np.ndarray:
    """The same layer the grouped way: per block of the aligned layout, its rows' inputs times its
    expert's weights (first GEMM from token rows, second from assignment rows scaled by the router
    weight), then each token's k assignment rows summed."""
    x = np.asarray(x, dtype=np.float64)
    gate_up = np.asarray(gate_up, dtype=np.float64)
    down = np.asarray(down, dtype=np.float64)
    N, k = expert_ids.shape
    total = N * k
    sorted_ids, block_expert, num_padded = moe_align(expert_ids, gate_up.shape[0], block_m)
    flat_w = np.asarray(weights, dtype=np.float64).reshape(-1)
    inter = gate_up.shape[1] // 2
    act = np.zeros((total, inter))
    for b in range(num_padded // block_m):                # first GEMM + SiLU * up, rows = assignments
        rows = sorted_ids[b * block_m:(b + 1) * block_m]
        rows = rows[rows < total]
        e = block_expert[b]
        h = x[rows // k] @ gate_up[e].T
        act[rows] = silu(h[:, :inter]) * h[:, inter:]
    y = np.zeros((total, down.shape[1]))
    for b in range(num_padded // block_m):                # second GEMM, scaled by the router weight
        rows = sorted_ids[b * block_m:(b + 1) * block_m]
        rows = rows[rows < total]
        y[rows] = (act[rows] @ down[block_expert[b]].T) * flat_w[rows][:, None]
    return y.reshape(N, k, -1).sum(axis=1)
