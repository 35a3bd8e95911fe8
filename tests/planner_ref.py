"""Reference implementations of librc's host planners (rc_plan_extend_stacking,
rc_plan_decode_groups), in plain Python, for the tests only: the C planners must make exactly
the decisions written out here (tests/test_host_parity.py). Nothing in the package imports this
module.

Extend stacking follows the shared-prefix query stacking of the paper digest's related work
(Sec. 7); the cost model is of this repository's extend kernel, calibrated on GB300.
"""
from __future__ import annotations

import numpy as np


# Cost model of one extend CTA, calibrated on GB300 (fork, two-level and few-shot replays):
# per 128-key tile for a pair of query tiles about 2.15 us in a batch without stacking groups,
# 3.3 us in one with them (the kernel's stacking build; half that for a lone tile, whose key
# tiles split across the two softmax groups), 10 us of fixed cost per CTA, 1 us to merge.
_T_TILE_US, _T_STACK_TILE_US, _C_CTA_US, _C_MERGE_US = 2.15, 3.3, 10.0, 1.0


def _extend_cost_us(P, S, key0, ppt, merge, tile=_T_TILE_US):
    """Estimated CTA-time of one request's per-request pass over keys [key0, P) and its S new
    tokens, ppt query positions per tile."""
    if S <= 0:
        return 0.0
    tiles = -(-(P - key0) // 128) + -(-S // 128)
    pairs = -(-S // (2 * ppt))
    per = tiles * (tile if S > ppt else tile / 2)
    return pairs * (per + _C_CTA_US + (_C_MERGE_US if merge else 0.0))


def _fold_tiles(P, qo, r, shared, end):
    """Remainder key tiles member r of a folded group needs in a CTA whose rows end at stacked
    position `end`: its cached keys past the shared prefix, then its new tokens up to its last
    row before `end` (the kernel's walk)."""
    last = min(qo[r + 1], end) - 1 - qo[r]
    return 0 if last < 0 else -(-(P[r] - shared + last + 1) // 128)


FOLD_TILES, FOLD_MEMBERS = 512, 256   # a folded pass's CTA: remainder tiles, members (kernel table)


def _folded_cost_us(P, S, shared, start, ppt, limits=False):
    """Estimated CTA-time of a folded stacked pass: the members' new tokens stacked against keys
    [start, shared), and in each CTA its members' remainders in the kernel's order (query tile A
    reads a prefix of the CTA's remainder tiles, tile B all of them). limits: return instead
    whether every CTA's remainder tiles and members fit the kernel's table."""
    qo = [0]
    for s in S:
        qo.append(qo[-1] + s)
    U, n_pre = qo[-1], -(-(shared - start) // 128)
    total = 0.0
    r0 = 0
    for iA in range(0, U, 2 * ppt):
        endA, endC = min(iA + ppt, U), min(iA + 2 * ppt, U)
        while qo[r0 + 1] <= iA:
            r0 += 1
        n_rem = n_rem_a = 0
        r = r0
        while r < len(S) and qo[r] < endC:
            nt = _fold_tiles(P, qo, r, shared, endC)
            n_rem += nt
            if qo[r + 1] < endA:
                n_rem_a += nt
            elif qo[r] < endA:
                n_rem_a += _fold_tiles(P, qo, r, shared, endA)
            r += 1
        if limits and (n_rem > FOLD_TILES or r - r0 > FOLD_MEMBERS):
            return False
        nA = n_pre + n_rem_a
        if endC > endA:
            per = max(nA, n_pre + n_rem) * _T_STACK_TILE_US
        else:   # one query tile: its key tiles split across the two softmax groups
            per = nA * _T_STACK_TILE_US / 2
        total += per + _C_CTA_US + (_C_MERGE_US if start > 0 else 0.0)
    return True if limits else total


def _stacking_costs(prefix_len, new_len, shared, group, start):
    """(per-request passes alone, stacked pass + per-request remainder passes, folded pass)
    estimated CTA-time over keys from `start` on."""
    ppt = max(128 // group, 1)
    P = [int(x) for x in prefix_len]
    S = [int(x) for x in new_len]
    alone = sum(_extend_cost_us(p, s, start, ppt, start > 0) for p, s in zip(P, S))
    U = sum(S)
    stacked_tiles = -(-(shared - start) // 128)
    first = -(-U // (2 * ppt)) * (stacked_tiles * (_T_STACK_TILE_US if U > ppt
                                                   else _T_STACK_TILE_US / 2)
                                 + _C_CTA_US + (_C_MERGE_US if start > 0 else 0.0))
    second = sum(_extend_cost_us(p, s, shared, ppt, True, _T_STACK_TILE_US) for p, s in zip(P, S))
    return alone, first + second, _folded_cost_us(P, S, shared, start, ppt)


def stacking_pays(prefix_len, new_len, shared: int, group: int, start: int = 0) -> bool:
    """Whether stacking these requests (one group of consecutive requests) over keys
    [start, shared) -- start > 0: a deeper level whose parent covers the keys before it -- is
    estimated to save at least 10% of their extend time over those keys, as a stacked pass
    followed by per-request passes or as one folded pass. It pays when stacking fills query
    tiles that short suffixes leave mostly empty; with long suffixes or many query heads per
    KV head the tiles are full already and an extra pass only adds CTAs."""
    if sum(int(x) for x in new_len) <= 0:
        return False
    alone, unfolded, folded = _stacking_costs(prefix_len, new_len, shared, group, start)
    return min(unfolded, folded) < 0.9 * alone


def prefix_stacking_groups(rows, prefix_len, new_len, min_shared: int):
    """Host-side grouping for extend: runs of consecutive requests whose slot rows hold the same
    slots over at least min_shared of their matched prefixes. A run grows while the next
    request agrees with the run's first over min_shared or more positions; its shared length is
    the smallest such agreement. Returns (ranges [2 G], shared [G], max_group_rows) -- ranges as
    (first, end) request pairs, max_group_rows the largest total of new tokens of a group."""
    rows = np.asarray(rows)
    P = np.asarray(prefix_len, dtype=np.int64)
    S = np.asarray(new_len, dtype=np.int64)
    B = len(P)
    ranges, shared, max_rows = [], [], 0
    b = 0
    while b < B:
        e, sh = b + 1, int(P[b])
        while e < B:
            n = int(min(sh, P[e]))
            diff = np.flatnonzero(rows[b, :n] != rows[e, :n])
            agree = int(diff[0]) if diff.size else n
            if agree < min_shared:
                break
            sh = agree
            e += 1
        if e - b >= 2 and sh >= min_shared and int(S[b:e].sum()) > 0:
            ranges += [b, e]
            shared.append(sh)
            max_rows = max(max_rows, int(S[b:e].sum()))
        b = e
    return np.asarray(ranges, np.int32), np.asarray(shared, np.int32), max_rows


MAX_STACK_LEVELS = 4


def fold_groups(ranges, shared, level_indptr, prefix_len, new_len, group: int = 1, start=None,
                force: bool = False):
    """Groups whose stacked pass also takes their members' remainders (rc_extend_args
    group_fold): no deeper group lies inside, every CTA of its pass fits the kernel's table of
    remainder tiles, and (unless force) the cost model estimates the folded pass at no more than
    the stacked pass plus the members' own passes. Returns (fold int32 [G], every request of the
    batch folded)."""
    P = np.asarray(prefix_len, dtype=np.int64)
    S = np.asarray(new_len, dtype=np.int64)
    G = len(shared)
    st = np.zeros(G, np.int64) if start is None else np.asarray(start, dtype=np.int64)
    fold = np.zeros(G, np.int32)
    level = np.zeros(G, np.int64)
    for l in range(len(level_indptr) - 1):
        level[level_indptr[l]:level_indptr[l + 1]] = l
    covered = np.zeros(len(P), bool)
    for g in range(G):
        b0, b1 = int(ranges[2 * g]), int(ranges[2 * g + 1])
        inner = any(level[h] > level[g] and b0 <= ranges[2 * h] and ranges[2 * h + 1] <= b1
                    for h in range(G))
        if inner or not _folded_cost_us(P[b0:b1], S[b0:b1], int(shared[g]), int(st[g]),
                                        max(128 // group, 1), limits=True):
            continue
        if not force:
            _, unfolded, folded = _stacking_costs(P[b0:b1], S[b0:b1], int(shared[g]), group,
                                                  int(st[g]))
        if force or folded <= unfolded:
            fold[g] = 1
            covered[b0:b1] = True
    return fold, bool(covered.all())


def prefix_stacking_levels(rows, prefix_len, new_len, min_shared: int, pays=None,
                           max_levels: int = MAX_STACK_LEVELS):
    """Stacking groups over the levels of the tree (cascade): level 0 as prefix_stacking_groups;
    inside each kept group of level l (shared length s), runs whose members agree over at least
    s + min_shared positions form level l + 1, with key start s. pays(b0, b1, shared, start)
    decides whether a candidate is kept (None: all); a group not kept is not searched further.
    Returns (ranges [2 G], shared [G], start [G], level_indptr [L + 1], max_group_rows) as int32
    numpy arrays (and an int), groups listed level by level; G = 0 when there is none."""
    rows = np.asarray(rows)
    P = np.asarray(prefix_len, dtype=np.int64)
    S = np.asarray(new_len, dtype=np.int64)
    parents = [(0, len(P), 0)]
    ranges, shared, start, level_indptr, max_rows = [], [], [], [0], 0
    for _ in range(max_levels):
        found = []
        for p0, p1, psh in parents:
            r, sh, _ = prefix_stacking_groups(rows[p0:p1], P[p0:p1], S[p0:p1], psh + min_shared)
            for g in range(len(sh)):
                b0, b1 = p0 + int(r[2 * g]), p0 + int(r[2 * g + 1])
                if pays is None or pays(b0, b1, int(sh[g]), psh):
                    found.append((b0, b1, int(sh[g]), psh))
        if not found:
            break
        for b0, b1, sh, st in found:
            ranges += [b0, b1]
            shared.append(sh)
            start.append(st)
            max_rows = max(max_rows, int(S[b0:b1].sum()))
        level_indptr.append(len(shared))
        parents = [(b0, b1, sh) for b0, b1, sh, _ in found]
    return (np.asarray(ranges, np.int32), np.asarray(shared, np.int32),
            np.asarray(start, np.int32), np.asarray(level_indptr, np.int32), max_rows)


def shared_context_groups(rows, lengths, group_size: int, min_shared: int):
    """Host-side grouping for decode: requests whose slot rows start with the same slots share
    that prefix's KV. rows: int32 [B, >= max(lengths)] slot rows, lengths: context tokens per
    request. Greedy: the first request of each same-first-slot bucket leads; the others with the
    longest common slot prefix join it, up to group_size members, as long as that prefix is at
    least min_shared tokens; a group's shared length is its members' smallest common prefix.
    Returns (indptr, members, shared) int32 numpy arrays (no groups: three empty arrays)."""
    rows = np.asarray(rows)
    lengths = np.asarray(lengths, dtype=np.int64)
    B = len(lengths)
    indptr, members, shared = [0], [], []
    if group_size < 2 or B < 2:
        return (np.zeros(1, np.int32), np.zeros(0, np.int32), np.zeros(0, np.int32))
    eligible = np.flatnonzero(lengths >= max(min_shared, 1))
    buckets = {}
    for b in eligible:
        buckets.setdefault(int(rows[b, 0]), []).append(int(b))

    def lcp(x, y):
        n = int(min(lengths[x], lengths[y]))
        diff = np.flatnonzero(rows[x, :n] != rows[y, :n])
        return int(diff[0]) if diff.size else n

    for rest in buckets.values():
        while len(rest) >= 2:
            lead = rest[0]
            cand = sorted(((lcp(lead, m), m) for m in rest[1:]), reverse=True)
            take = [(l, m) for l, m in cand[:group_size - 1] if l >= min_shared]
            if not take:
                rest = rest[1:]
                continue
            members += [lead] + [m for _, m in take]
            shared.append(min(l for l, _ in take))
            indptr.append(len(members))
            used = {lead} | {m for _, m in take}
            rest = [m for m in rest if m not in used]
    return (np.asarray(indptr, np.int32), np.asarray(members, np.int32),
            np.asarray(shared, np.int32))
