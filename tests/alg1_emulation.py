"""Independent restatement of the token-count and index-generation stages.

"Scalable Pretraining of Large MoE LMs on Aurora Super Computer", §3.1
FastSparseMoE, Algorithm 1, stages 2 and 3, written out as the thread-block
procedure the page describes (token blocks of TBS tokens, one "thread" per
block, per-(expert, thread) partial counts laid out expert-major, their
prefix sums as bases and a per-(expert, thread) counter for offsets), with
an expert-parallel rank that keeps only its local experts.  Pure Python
loops, for small inputs only.  Used to pin the oracle's plain stable-sort
definition of the same indices; it does not share code with the oracle.
"""
from __future__ import annotations

import math


def _running_sum(values):
    out = [0]
    for v in values:
        out.append(out[-1] + v)
    return out


def index_generation(indices, N, ep=1, rank=0, tbs=8):
    """Return (cum_token_counts, expert_counts, cum_expert_counts,
    input_indices, output_indices, selected_expert_indices) for one rank."""
    T = len(indices)
    K = len(indices[0]) if T else 0
    nr = N // ep
    first, last = rank * nr, rank * nr + nr - 1
    threads = math.ceil(T / tbs)

    def tokens_of(thread):
        return range(thread * tbs, min(T, thread * tbs + tbs))

    # stage 2: counts per (local expert, thread) and local selections per token
    partial = [0] * (nr * threads)
    expert_counts = [0] * T
    for th in range(threads):
        for t in tokens_of(th):
            for slot in range(K):
                n = indices[t][slot]
                if first <= n <= last:
                    partial[(n - first) * threads + th] += 1
                    expert_counts[t] += 1
    partial_cum = _running_sum(partial)
    cum_expert_counts = _running_sum(expert_counts)
    cum_token_counts = [partial_cum[n * threads] for n in range(nr + 1)]

    # stage 3: each (expert, thread) writes from its base, counting up
    routed = cum_token_counts[-1]
    input_indices = [None] * routed
    output_indices = [None] * routed
    selected = [None] * routed
    counter = [[0] * threads for _ in range(nr)]
    for th in range(threads):
        for t in tokens_of(th):
            o = cum_expert_counts[t]
            for slot in range(K):
                n = indices[t][slot]
                if not (first <= n <= last):
                    continue
                ln = n - first
                pos = partial_cum[ln * threads + th] + counter[ln][th]
                counter[ln][th] += 1
                input_indices[pos] = t
                output_indices[o] = pos
                selected[o] = slot
                o += 1
    return (cum_token_counts, expert_counts, cum_expert_counts,
            input_indices, output_indices, selected)
