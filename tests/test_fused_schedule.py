"""Host-side model of the fused pair kernel's work split (no GPU needed).

The host decides per launch whether the last round of tiles is split into
K-halves (S split tiles, when the round would leave at least half of the
pairs idle and no pair of that round still holds a whole tile of a row block
with split tiles); the kernel maps unit u to a whole tile, or to the owner
(first K-half) or helper (second K-half) of a split tile, and pair p takes
units p, p + pairs, ...  A pair finishes a tile's epilogue, norm included,
before it starts the next one; a norm waits until every N-tile of its row
block has published its row sums; an owner waits for its helper's half.

This model restates that rule and mapping and checks, over a grid of launch
shapes, that every tile's K-blocks are covered exactly once and that the
waits always resolve (no pair waits on a tile whose work sits behind it on a
blocked pair).  It also shows that splitting without the rule's second
condition could stall: that is why the host has it.
"""
import itertools

import pytest


def split_tiles(tiles, nt, cap, may_split=True, guard=True):
    rem = tiles % cap
    x = (tiles - rem) % nt
    ok = may_split and rem > 0 and (2 * rem + x <= cap if guard else 2 * rem <= cap)
    return rem if ok else 0


def unit_at(u, total, S, KB):
    D = total - S
    if u < D:
        return ("whole", u, 0, KB)
    v = u - D
    h, j = v & 1, v >> 1
    return ("helper" if h else "owner", D + j, KB // 2 if h else 0, KB if h else KB // 2)


def plan(row_blocks, nt, cap, guard=True):
    tiles = row_blocks * nt
    S = split_tiles(tiles, nt, cap, guard=guard)
    pairs = max(1, min(cap, tiles + S))
    return tiles, S, pairs


def covers_exactly_once(tiles, S, pairs, KB=128):
    got = {t: [] for t in range(tiles)}
    for u in range(tiles + S):
        _, t, k0, k1 = unit_at(u, tiles, S, KB)
        got[t].append((k0, k1))
    return all(sorted(v) in ([(0, KB)], [(0, KB // 2), (KB // 2, KB)]) for v in got.values())


def runs_to_completion(tiles, nt, S, pairs):
    """Each pair works through its units in order; returns False on a stall."""
    queues = [[unit_at(u, tiles, S, 2) for u in range(p, tiles + S, pairs)] for p in range(pairs)]
    pos = [0] * pairs
    stage = [0] * pairs            # 0: before the tile's row sums are published, 1: waiting for the norm
    published = [False] * tiles    # row sums of the tile are out
    helper_done = [False] * tiles
    while True:
        moved = False
        for p in range(pairs):
            while pos[p] < len(queues[p]):
                role, t, _, _ = queues[p][pos[p]]
                if role == "helper":
                    helper_done[t] = True
                    pos[p] += 1
                    moved = True
                    continue
                if stage[p] == 0:
                    if role == "owner" and not helper_done[t]:
                        break
                    published[t] = True
                    stage[p] = 1
                    moved = True
                rb = t // nt
                if all(published[rb * nt + n] for n in range(nt)):
                    stage[p] = 0
                    pos[p] += 1
                    moved = True
                else:
                    break
        if all(pos[p] == len(queues[p]) for p in range(pairs)):
            return True
        if not moved:
            return False


GRID = [(rb, nt, cap) for rb, nt, cap in itertools.product(range(1, 13), range(1, 21), list(range(1, 25)) + [36, 64, 72, 76])
        if nt <= cap]   # rows wider than the grid take the PIPELINED path


def test_every_tile_is_covered_once_and_every_launch_completes():
    n_split = 0
    for rb, nt, cap in GRID:
        tiles, S, pairs = plan(rb, nt, cap)
        n_split += S > 0
        assert covers_exactly_once(tiles, S, pairs), (rb, nt, cap)
        assert runs_to_completion(tiles, nt, S, pairs), (rb, nt, cap)
    assert n_split > 100   # the grid exercises the split often


@pytest.mark.parametrize("rb,nt,cap", [(32, 16, 76), (32, 16, 72), (32, 16, 64), (16, 16, 76), (8, 19, 76),
                                        (64, 2, 64), (3, 4, 16), (3, 4, 20)])
def test_launch_shapes_of_the_workloads(rb, nt, cap):
    # Llama-3-8B down_proj (one 8192-token launch, 256-wide tiles on 76, 72 or 64 pairs), o_proj (4096
    # tokens), Gemma-2-9B (192-wide tiles), the 16384-token launch of the split test, and others
    tiles, S, pairs = plan(rb, nt, cap)
    assert covers_exactly_once(tiles, S, pairs)
    assert runs_to_completion(tiles, nt, S, pairs)


def test_the_rule_keeps_pairs_from_waiting_on_work_behind_them():
    # Without the guard on the whole tiles that share a row block with split tiles some shapes stall:
    # their norm waits for a split tile whose helper half is queued behind the waiting tile.
    stalls = [(rb, nt, cap) for rb, nt, cap in GRID
              if not runs_to_completion(*(lambda t, s, p: (t, nt, s, p))(*plan(rb, nt, cap, guard=False)))]
    assert stalls, "the unguarded split never stalls on this grid"
    for rb, nt, cap in stalls:
        tiles, S, pairs = plan(rb, nt, cap)
        assert runs_to_completion(tiles, nt, S, pairs)


# ---------------------------------------------------------------- two epilogue groups
# With eight epilogue warps a pair's k-th unit goes to group k % 2 and to TMEM buffer k % 2: its MMAs
# start once the pair's previous unit's MMAs are done and unit k - 2 has released the buffer (its
# epilogue is complete); a group works through its own units in order; a whole or owner unit publishes
# its row sums (an owner only once its helper's half is out), waits for its row block, then takes the
# quarter's output staging from unit k - 1 and hands it on; a helper unit publishes its half as soon as
# its MMAs are done and its group is free, and only then takes and hands on the staging.  So a helper
# never waits for its pair's previous tile, and the split needs no guard on whole tiles.
def split_tiles_two_groups(tiles, nt, cap):
    rem = tiles % cap
    return rem if (rem > 0 and 2 * rem <= cap) else 0


def runs_to_completion_two_groups(tiles, nt, S, pairs, helper_token_first=False):
    queues = [[unit_at(u, tiles, S, 2) for u in range(p, tiles + S, pairs)] for p in range(pairs)]
    mma = [[False] * len(q) for q in queues]
    done = [[False] * len(q) for q in queues]        # epilogue complete: buffer released, staging handed on
    phase1 = [[False] * len(q) for q in queues]
    published = [False] * tiles
    helper_out = [False] * tiles
    while True:
        moved = False
        for p, q in enumerate(queues):
            for k, (role, t, _, _) in enumerate(q):
                if not mma[p][k] and (k == 0 or mma[p][k - 1]) and (k < 2 or done[p][k - 2]):
                    mma[p][k] = moved = True
                group_free = mma[p][k] and (k < 2 or done[p][k - 2])
                if not group_free or done[p][k]:
                    continue
                token = k == 0 or done[p][k - 1]
                if role == "helper":
                    if helper_token_first:
                        if token:
                            helper_out[t] = done[p][k] = moved = True
                        continue
                    if not helper_out[t]:
                        helper_out[t] = moved = True
                    if token:
                        done[p][k] = moved = True
                    continue
                if not phase1[p][k] and (role == "whole" or helper_out[t]):
                    phase1[p][k] = published[t] = moved = True
                rb = t // nt
                if phase1[p][k] and token and all(published[rb * nt + n] for n in range(nt)):
                    done[p][k] = moved = True
        if all(all(d) for d in done):
            return True
        if not moved:
            return False


def test_two_groups_split_every_tile_covered_once_and_every_launch_completes():
    n_split = 0
    for rb, nt, cap in GRID:
        tiles = rb * nt
        S = split_tiles_two_groups(tiles, nt, cap)
        pairs = max(1, min(cap, tiles + S))
        n_split += S > 0
        assert covers_exactly_once(tiles, S, pairs), (rb, nt, cap)
        assert runs_to_completion_two_groups(tiles, nt, S, pairs), (rb, nt, cap)
        assert runs_to_completion_two_groups(tiles, nt, 0, max(1, min(cap, tiles))), (rb, nt, cap)
    assert n_split > 200


@pytest.mark.parametrize("rb,nt,cap,splits", [(16, 16, 76, True), (8, 14, 76, True), (8, 16, 76, False),
                                               (32, 16, 76, False), (16, 16, 72, False)])
def test_two_groups_split_on_the_workloads(rb, nt, cap, splits):
    # o_proj 4096^3 on 76 pairs (28 split tiles), Gemma-2-9B with 256-wide (36 split tiles) and 224-wide
    # tiles, down_proj; a last round with more than half of the pairs busy is not split
    tiles = rb * nt
    S = split_tiles_two_groups(tiles, nt, cap)
    assert (S > 0) == splits
    assert runs_to_completion_two_groups(tiles, nt, S, min(cap, tiles + S))


def test_one_group_split_without_the_guard_stalls_where_two_groups_do_not():
    # the shapes where the one-group kernel needs the guard are safe with two groups
    stalls = [(rb, nt, cap) for rb, nt, cap in GRID
              if not runs_to_completion(*(lambda t, s, p: (t, nt, s, p))(*plan(rb, nt, cap, guard=False)))]
    assert stalls
    for rb, nt, cap in stalls:
        tiles = rb * nt
        S = split_tiles(tiles, nt, cap, guard=False)
        assert runs_to_completion_two_groups(tiles, nt, S, max(1, min(cap, tiles + S)))


def test_a_helper_that_takes_the_staging_first_can_stall():
    # the order matters: a helper that waited for the output staging before publishing its half would
    # wait for its pair's previous tile, whose norm may need that very half
    stalls = [(rb, nt, cap) for rb, nt, cap in GRID
              if split_tiles_two_groups(rb * nt, nt, cap) and not runs_to_completion_two_groups(
                  rb * nt, nt, split_tiles_two_groups(rb * nt, nt, cap),
                  max(1, min(cap, rb * nt + split_tiles_two_groups(rb * nt, nt, cap))), helper_token_first=True)]
    assert len(stalls) > 100
