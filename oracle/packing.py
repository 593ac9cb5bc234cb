"""Plain restatement of the host packer (test infrastructure).

TEST INFRASTRUCTURE ONLY: only the tests may import this module; the library
never calls it and shares no code with it. Pure Python loops, written for
reading, not speed (a few thousand sequences at most).

What it follows (mlx-train-perf changelog, "Added"): the packed batch
iterator fills fixed rows with (tokens, offset) sequences after a seeded
per-epoch shuffle, by first-fit placement, and emits per-token segment
buffers; the packed loss masks segment by segment, so the supervised tokens
are exactly those of an unpacked run (0.5.1 README, "Sequence packing").

Readings where the pages leave a step open:
  * the shuffle is Fisher-Yates driven by the counter-based stream of
    ``synth.uint64s`` with the epoch as the stream number;
  * first-fit: each sequence, whole, into the lowest-numbered row that still
    has room; a sequence no row can take is left out;
  * a row's unfilled tail is one extra segment (padding), never supervised;
  * supervision (the unpacked rule applied per sequence): the token at
    position p of a sequence of length L with prompt length `offset` is
    trained to predict token p + 1, and counts iff offset <= p + 1 <= L - 1;
    the target of a supervised position is that next token, -1 elsewhere.

Pins: tests/test_packer_host.py (published splitmix64 outputs, uniformity of
the shuffle over all permutations of three items, a hand-worked first-fit
fixture, the first-fit half-full property, closed-form supervised counts and
the no-contamination property).
"""
from __future__ import annotations

import synth


def shuffled_order(count: int, seed: int, epoch: int) -> list[int]:
    """The epoch's order of sequence indices (Fisher-Yates, last to first)."""
    order = list(range(count))
    draws = synth.uint64s(seed, epoch, max(count, 1))
    for i in range(count - 1, 0, -1):
        j = int(draws[i]) % (i + 1)
        order[i], order[j] = order[j], order[i]
    return order


def first_fit(lengths_in_order: list[int], rows: int, N: int) -> list[tuple[int, int] | None]:
    """(row, start) for each length in the given order, or None when no row has
    room. Rows are scanned from 0 each time."""
    free = [N] * rows
    out: list[tuple[int, int] | None] = []
    for L in lengths_in_order:
        spot = None
        for r in range(rows):
            if L <= free[r]:
                spot = (r, N - free[r])
                free[r] -= L
                break
        out.append(spot)
    return out


def supervised(L: int, offset: int) -> list[bool]:
    """Per position of one sequence: does its next-token prediction count?"""
    return [offset <= p + 1 <= L - 1 for p in range(L)]


def pack(lengths, rows, N, seed, epoch, offsets=None, tokens=None, pad_token=0) -> dict:
    """Same outputs as the library's packer, as nested Python lists."""
    count = len(lengths)
    offsets = [0] * count if offsets is None else list(offsets)
    starts, acc = [], 0
    for L in lengths:
        starts.append(acc)
        acc += L
    order = shuffled_order(count, seed, epoch)
    spots = first_fit([lengths[s] for s in order], rows, N)

    seg = [[None] * N for _ in range(rows)]
    mask = [[0] * N for _ in range(rows)]
    toks = [[pad_token] * N for _ in range(rows)]
    tgts = [[-1] * N for _ in range(rows)]
    placement = [-1] * count
    next_id = [0] * rows
    placed = 0
    for s, spot in zip(order, spots):
        if spot is None:
            continue
        r, start = spot
        sid = next_id[r]
        next_id[r] += 1
        sup = supervised(lengths[s], offsets[s])
        for p in range(lengths[s]):
            seg[r][start + p] = sid
            mask[r][start + p] = 1 if sup[p] else 0
            if tokens is not None:
                toks[r][start + p] = int(tokens[starts[s] + p])
                if sup[p]:
                    tgts[r][start + p] = int(tokens[starts[s] + p + 1])
        placement[s] = r * N + start
        placed += lengths[s]
    for r in range(rows):
        for t in range(N):
            if seg[r][t] is None:
                seg[r][t] = next_id[r]
    used_rows = [r for r in range(rows) if next_id[r] > 0]
    return {"seg": seg, "loss_mask": mask, "row_tokens": toks if tokens is not None else None,
            "row_targets": tgts if tokens is not None else None,
            "placement": placement, "rows_used": (max(used_rows) + 1) if used_rows else 0,
            "placed_tokens": placed}
