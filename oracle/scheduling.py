"""Host-side scheduling rules of the decode loop, restated -- TEST INFRASTRUCTURE.

Two rules from the pages, written as plain functions on integer arrays:

  * "33. Removing overhead", §Async scheduling: the scheduler prepares step
    N+1 before step N's sampled ids reach the host.  A token whose id is not
    known yet carries a placeholder, and the id that step N sampled for the
    same request is put in its place on the device before the embedding runs.
    ``gather_input_ids`` states which id each token of step N+1 reads.
  * "19. Fast decode", §Host synchronizations (the fast decoder's generate):
    stop tokens are looked for only every ``check_every`` steps, one
    synchronisation per check; decoding ends at the first check where every
    request has produced a stop token, and each request's output is cut after
    its first stop token.  ``stop_trim`` states what that loop returns.

Parity: pinned by hand-worked sequences in tests/test_oracle_scheduling.py.
"""
from __future__ import annotations

import numpy as np


def gather_input_ids(token_ids, prev_row, prev_sampled) -> np.ndarray:
    """Input id of every token of an asynchronously scheduled step.

    token_ids[t]: the id the host knows (ignored where the host does not know it);
    prev_row[t]: -1 when the host knows token t's id, else the row, in the previous
    step, of the request whose sampled id token t is; prev_sampled[r]: the id the
    previous step sampled for its row r.  Token t reads token_ids[t] when
    prev_row[t] is -1, else prev_sampled[prev_row[t]].
    """
    token_ids = np.asarray(token_ids, dtype=np.int64)
    prev_row = np.asarray(prev_row, dtype=np.int64)
    prev_sampled = np.asarray(prev_sampled, dtype=np.int64)
    if token_ids.shape != prev_row.shape:
        raise ValueError("token_ids and prev_row must have one entry per token")
    if np.any(prev_row < -1) or np.any(prev_row >= len(prev_sampled)):
        raise ValueError("prev_row entries must be -1 or a row of the previous step")
    out = token_ids.copy()
    for t in range(len(out)):
        if prev_row[t] >= 0:
            out[t] = prev_sampled[prev_row[t]]
    return out


def stop_trim(tokens, stop_ids, check_every: int, max_steps: int | None = None):
    """What a decode loop that checks for stop ids every ``check_every`` steps returns.

    tokens: [R, n] -- the id request r samples at each step if the loop keeps
    running (n >= the steps that can run).  The loop runs groups of check_every
    steps (the last group cut at max_steps, default n) and, after each group,
    looks at the ids so far; it stops after the first group at whose end every
    request has sampled a stop id.  Returns (out [R, max_steps], lengths [R],
    steps_run): request r keeps its ids up to and including its first stop id
    (lengths[r] = that count), or all steps_run ids when it never stopped; every
    later entry of out is -1.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    R, n = tokens.shape
    max_steps = n if max_steps is None else int(max_steps)
    if check_every < 1 or max_steps > n or max_steps < 0:
        raise ValueError("check_every must be >= 1 and max_steps at most the tokens given")
    stops = set(int(s) for s in stop_ids)
    first = [None] * R                    # 1-based step of each request's first stop id
    for r in range(R):
        for k in range(max_steps):
            if int(tokens[r, k]) in stops:
                first[r] = k + 1
                break
    steps_run = 0
    while steps_run < max_steps:
        steps_run = min(steps_run + check_every, max_steps)
        if all(f is not None and f <= steps_run for f in first):
            break
    out = np.full((R, max_steps), -1, dtype=np.int64)
    lengths = np.zeros(R, dtype=np.int64)
    for r in range(R):
        keep = first[r] if first[r] is not None and first[r] <= steps_run else steps_run
        out[r, :keep] = tokens[r, :keep]
        lengths[r] = keep
    return out, lengths, steps_run
