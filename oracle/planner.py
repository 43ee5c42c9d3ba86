"""CPU re-derivation of the tile work lists (test infrastructure).

The device planner classifies tiles with closed forms.  This module derives
the same lists by counting: for every slice it lists each row's visible key
interval, sums the visible entries of every (q-tile, k-tile) pair, and calls
a tile FULL when it holds 128 * 128 visible entries and PARTIAL when it holds
at least one.  The rest (pairing, merging, costs, splitting, ordering) follows
the work-list specification of the planner:

  * forward visits of a q-tile: one per k-tile seen, in kt order; info is
    (slice << 2) | partial when one slice sees the tile pair, else
    (m << 2) | 3 with a slice list [n, s_0, ..] (ascending) at offset m of
    the direction's list array (lists appended in tile, then kt order);
  * grouped heads (Hq/Hkv >= 2): a unit is one q-tile, items are pairs of
    query heads of one kv head; otherwise a unit is q-tiles (2u, 2u+1), items
    one per head, steps merge the two visit lists on kt;
  * cost = 4 per FULL and 5 per PARTIAL visit over the busy halves;
  * split (when 0 < items with work < threshold): min(16, ceil(threshold /
    live)) chunks per item, capped by its step count, step ranges
    b + k*n//c .. b + (k+1)*n//c, cost scaled by the chunk's share;
  * order: cost octave floor(log2(cost + 1)) descending, then kv head, then
    cost descending, then item index;
  * backward: per k-tile one visit per q-tile seen, merged the same way, one
    item per (kt, kv head), cost g * sum of visit costs;
  * gathered forward units: a unit whose q-tiles meet only FULL slices with
    8-aligned key ranges (the end may be Tk), Tk <= 2^19, is instead listed
    as gathered steps when that takes at most 9/10 of its steps (a gathered
    step costs about as much as a masked tile step): the 8-key blocks any of
    its slices covers, ascending, 16 to a step; a step is (0, info0, info1,
    r + 1) with record r = 16 block starts (key index, -8 for an unused
    slot) then, per half, 16 x 4 words of row bits (bit r of word w: row
    32w + r of the half's q-tile sees the slot's keys); info_h = 0 when all
    16 slots hold keys and every row bit of the half is set (the step needs
    no mask), else 1 when the half has a row bit set, else -1; cost 5 per
    busy half.  At most 2048
    blocks per unit;
  * gathered backward units, the transpose: a k-tile whose slices are all
    FULL with 8-aligned query ranges (the end may be Tq), Tq <= 2^19, lists
    the 8-row query blocks its slices cover, 16 to a step, when that takes
    at most 9/10 of its visits; a step is (0, 1, 0, r + 1) with record r =
    16 block start rows (-8: unused) then 16 x 4 words of key bits (bit i of
    word w: key 32w + i of the k-tile is seen by the slot's rows); cost 5
    per step (times g in the item);
  * head-stacked forward units: with g even and >= 4, Tk <= 2^19, when
    every 64-row slab of the queries meets only FULL slices with 8-aligned
    key ranges (at most 2048 blocks per slab), and ceil(g / 4) times the
    slabs' gathered steps is at most 9/10 of g / 2 times the steps chosen
    above, the forward units become the slabs instead: slab s (rows 64s ..
    64s + 63) lists the 8-key blocks its slices cover, 16 to a step, as
    above, with row bits for tile rows r and r + 64 both meaning row
    64s + r (the same bits in both halves); items are (s, s, h, h + 2) for
    the first query head h = hk * g + 4p of each group of four (half 1 idle,
    s and head -1, when 4p + 2 >= g): a half is the slab's 64 rows of heads
    h and h + 1 (h + 2 and h + 3), stacked in one 128-row tile.  With g a
    multiple of 4, 32-row slabs of four heads per half (tile rows r, r + 32,
    r + 64, r + 96 all mean slab row r; items (s, s, h, h + 4) for h =
    hk * g + 8p, half 1 idle when 8p + 4 >= g) replace the choice above when
    g / 4 times their steps is at most 9/10 of its half-steps (g times the
    tile steps, or g / 2 times the 64-row slab steps).  With 32-row slabs and
    g = 4 (`alternate`) an item is (s, s, h, h): both halves hold the same
    rows and heads, take the slab's steps in turn (step j of the slab is
    (0, i, -1, r + 1) for even j, (0, -1, i, r + 1) for odd j) and are merged
    by logsumexp at the end of the item.  `stacked` is the slab height (64
    or 32), 0 for q-tile units.  Such plans are never split.
"""
from __future__ import annotations

import math

import numpy as np

TILE = 128
FULL_COST, PARTIAL_COST = 4, 5
GATHER_KEYS = 8           # keys per gathered slot (one 8-row TMA box)
GATHER_SLOTS = 16         # slots per gathered step (a 128-key tile)
GATHER_MAX_BLOCKS = 2048  # blocks per gathered unit
GATHER_MAX_TK = 1 << 19
GATHER_WORDS = GATHER_SLOTS + 2 * GATHER_SLOTS * 4
SLAB = 64                 # query rows per head-stacked unit
BGATHER_WORDS = GATHER_SLOTS + GATHER_SLOTS * 4


def row_intervals(qs, qe, ks, ke, t):
    """Rows of the slice and each row's visible key interval [lo, hi)."""
    rows = np.arange(qs, qe, dtype=np.int64)
    lo = ks + ((rows - qs) if (t & 2) else 0)
    hi = ke - ((qe - 1 - rows) if (t & 1) else 0)
    lo = np.broadcast_to(np.asarray(lo, np.int64), rows.shape).copy()
    hi = np.broadcast_to(np.asarray(hi, np.int64), rows.shape).copy()
    return rows, lo, hi


def tile_counts(q_ranges, k_ranges, mask_types):
    """{slice: {(qt, kt): visible entries}} by summing clipped row intervals."""
    out = {}
    for s, ((qs, qe), (ks, ke), t) in enumerate(zip(np.asarray(q_ranges).reshape(-1, 2),
                                                    np.asarray(k_ranges).reshape(-1, 2),
                                                    np.asarray(mask_types).reshape(-1))):
        qs, qe, ks, ke, t = int(qs), int(qe), int(ks), int(ke), int(t)
        d = {}
        out[s] = d
        if qe <= qs or ke <= ks:
            continue
        rows, lo, hi = row_intervals(qs, qe, ks, ke, t)
        ok = hi > lo
        if not ok.any():
            continue
        rows, lo, hi = rows[ok], lo[ok], hi[ok]
        kts = np.arange(lo.min() // TILE, -(-hi.max() // TILE))
        qts = rows // TILE
        for qt in np.unique(qts):
            sel = qts == qt
            l, h = lo[sel][:, None], hi[sel][:, None]
            c = np.clip(np.minimum(h, (kts[None] + 1) * TILE) - np.maximum(l, kts[None] * TILE),
                        0, None).sum(axis=0)
            for kt, n in zip(kts, c):
                if n > 0:
                    d[(int(qt), int(kt))] = int(n)
    return out


def visible_area(q_ranges, k_ranges, mask_types) -> int:
    tot = 0
    for (qs, qe), (ks, ke), t in zip(np.asarray(q_ranges).reshape(-1, 2),
                                     np.asarray(k_ranges).reshape(-1, 2),
                                     np.asarray(mask_types).reshape(-1)):
        if qe <= qs or ke <= ks:
            continue
        _, lo, hi = row_intervals(int(qs), int(qe), int(ks), int(ke), int(t))
        tot += int(np.clip(hi - lo, 0, None).sum())
    return tot


def _info(s, count):
    return (s << 2) | (0 if count == TILE * TILE else 1)


def _merge(visits, masks):
    """Sorted (x, slice, info) visits of one tile -> one (x, info) per x;
    x seen by several slices gets a slice list appended to ``masks``."""
    out, i = [], 0
    while i < len(visits):
        j = i
        while j < len(visits) and visits[j][0] == visits[i][0]:
            j += 1
        if j - i == 1:
            out.append((visits[i][0], visits[i][2]))
        else:
            out.append((visits[i][0], (len(masks) << 2) | 3))
            masks.append(j - i)
            masks.extend(v[1] for v in visits[i:j])
        i = j
    return out


def _cost(info):
    return PARTIAL_COST if info & 1 else FULL_COST


def plan(total_q, total_k, num_heads_q, num_heads_kv, q_ranges, k_ranges, mask_types,
         num_sms, split_below=0):
    """Work lists in the export layout of the device planner."""
    n_qt = -(-total_q // TILE)
    n_kt = -(-total_k // TILE)
    g = num_heads_q // num_heads_kv
    counts = tile_counts(q_ranges, k_ranges, mask_types)
    fvis = [[] for _ in range(n_qt)]
    bvis = [[] for _ in range(n_kt)]
    for s, d in counts.items():
        for (qt, kt), c in d.items():
            fvis[qt].append((kt, s, _info(s, c)))
            bvis[kt].append((qt, s, _info(s, c)))
    fmasks, bmasks = [], []
    fvis = [_merge(sorted(v), fmasks) for v in fvis]
    bvis = [_merge(sorted(v), bmasks) for v in bvis]

    # forward units and steps
    pair_mode = 0 if g >= 2 else 1
    n_units = n_qt if pair_mode == 0 else (n_qt + 1) // 2
    gathered = gather_units(total_q, total_k, q_ranges, k_ranges, mask_types, pair_mode, fvis)
    records = []
    steps, soff, scnt, cost_half = [], [], [], []
    for u in range(n_units):
        soff.append(len(steps))
        if u in gathered:
            st, ca, cb = [], 0, 0
            for rec, (i0, i1) in gathered[u]:
                st.append((0, i0, i1, len(records) + 1))
                records.append(rec)
                ca += PARTIAL_COST if i0 >= 0 else 0
                cb += PARTIAL_COST if i1 >= 0 else 0
            cost_half.append((ca, cb))
        elif pair_mode == 0:
            st = [(kt, i, i, 0) for kt, i in fvis[u]]
            c = sum(_cost(i) for _, i in fvis[u])
            cost_half.append((c, c))
        else:
            a = fvis[2 * u]
            b = fvis[2 * u + 1] if 2 * u + 1 < n_qt else []
            st, i, j, ca, cb = [], 0, 0, 0, 0
            while i < len(a) or j < len(b):
                if j >= len(b) or (i < len(a) and a[i][0] < b[j][0]):
                    st.append((a[i][0], a[i][1], -1, 0)); ca += _cost(a[i][1]); i += 1
                elif i >= len(a) or b[j][0] < a[i][0]:
                    st.append((b[j][0], -1, b[j][1], 0)); cb += _cost(b[j][1]); j += 1
                else:
                    st.append((a[i][0], a[i][1], b[j][1], 0))
                    ca += _cost(a[i][1]); cb += _cost(b[j][1]); i += 1; j += 1
            cost_half.append((ca, cb))
        steps.extend(st)
        scnt.append(len(st))

    stacked = 0  # slab rows of head-stacked units, 0: q-tile units
    half_steps = g * len(steps)  # of the units chosen so far
    if pair_mode == 0 and g >= 4 and g % 2 == 0:
        slabs = gather_slabs(total_q, total_k, q_ranges, k_ranges, mask_types)
        if slabs is not None:
            n_slab_steps = sum(len(v) for v in slabs.values())
            if n_slab_steps > 0 and 10 * (-(-g // 4)) * n_slab_steps <= 9 * (g // 2) * len(steps):
                stacked, half_steps = SLAB, (g // 2) * n_slab_steps
    if pair_mode == 0 and g >= 4 and g % 4 == 0:
        slabs4 = gather_slabs(total_q, total_k, q_ranges, k_ranges, mask_types, SLAB // 2)
        if slabs4 is not None:
            n4 = sum(len(v) for v in slabs4.values())
            if n4 > 0 and 10 * (g // 4) * n4 <= 9 * half_steps:
                stacked, slabs = SLAB // 2, slabs4
    # 32-row slabs with 4 query heads per kv head fill one half of an item;
    # its two halves then take the slab's steps in turn (even steps half 0,
    # odd ones half 1) and are merged by logsumexp at the end of the item
    alternate = stacked == SLAB // 2 and g == 4
    if stacked:
        n_units = -(-total_q // stacked)
        records, steps, soff, scnt, cost_half = [], [], [], [], []
        for u in range(n_units):
            soff.append(len(steps))
            ca = cb = 0
            for j, (rec, (i0, i1)) in enumerate(slabs.get(u, [])):
                if alternate:
                    i0, i1 = (i0, -1) if j % 2 == 0 else (-1, i0)
                steps.append((0, i0, i1, len(records) + 1))
                records.append(rec)
                ca += PARTIAL_COST if i0 >= 0 else 0
                cb += PARTIAL_COST if i1 >= 0 else 0
            cost_half.append((ca, cb))
            scnt.append(len(steps) - soff[-1])

    items = []
    if stacked:
        m = TILE // stacked  # query heads per half
        groups = -(-g // (2 * m))
        for u in range(n_units):
            for hk in range(num_heads_kv):
                for p in range(groups):
                    h0 = hk * g + 2 * m * p
                    h1 = h0 + m if 2 * m * p + m < g else -1
                    if alternate:
                        h1 = h0
                    qt1 = u if h1 >= 0 else -1
                    cost = cost_half[u][0] + (cost_half[u][1] if h1 >= 0 else 0)
                    items.append([u, qt1, h0, h1, soff[u], soff[u] + scnt[u], -1, cost])
    elif pair_mode == 0:
        pairs = (g + 1) // 2
        for u in range(n_units):
            for hk in range(num_heads_kv):
                for p in range(pairs):
                    h0 = hk * g + 2 * p
                    h1 = h0 + 1 if 2 * p + 1 < g else -1
                    qt1 = u if h1 >= 0 else -1
                    cost = cost_half[u][0] + (cost_half[u][1] if h1 >= 0 else 0)
                    items.append([u, qt1, h0, h1, soff[u], soff[u] + scnt[u], -1, cost])
    else:
        for u in range(n_units):
            for h in range(num_heads_q):
                qt1 = 2 * u + 1 if 2 * u + 1 < n_qt else -1
                h1 = h if qt1 >= 0 else -1
                cost = cost_half[u][0] + (cost_half[u][1] if h1 >= 0 else 0)
                items.append([2 * u, qt1, h, h1, soff[u], soff[u] + scnt[u], -1, cost])

    live = sum(1 for it in items if it[5] > it[4])
    threshold = 2 * num_sms if split_below == 0 else split_below
    merges, n_slots = [], 0
    if split_below >= 0 and 0 < live < threshold and not stacked:
        nsplit = min(16, -(-threshold // live))
        new = []
        for it in items:
            b, n = it[4], it[5] - it[4]
            c = max(1, min(nsplit, n))
            if c == 1:
                new.append(list(it))
                continue
            for k in range(c):
                kb, ke = b + k * n // c, b + (k + 1) * n // c
                x = list(it)
                x[4], x[5], x[6] = kb, ke, n_slots + k
                x[7] = it[7] * (ke - kb) // max(n, 1)
                new.append(x)
            merges.append([it[0], it[1], it[2], it[3], n_slots, c, 0, 0])
            n_slots += c
        items = new

    def order_of(costs, heads):
        key = lambda i: (-int(costs[i] + 1).bit_length(), heads[i], -costs[i], i)
        return np.array(sorted(range(len(costs)), key=key), dtype=np.int32)

    fwd_items = np.array(items, dtype=np.int32).reshape(-1, 8)
    fwd_order = order_of([it[7] for it in items], [max(it[2], 0) // g for it in items])

    bgathered = gather_units_bwd(total_q, total_k, q_ranges, k_ranges, mask_types, bvis)
    brecords = []
    bsteps, bitems = [], []
    boff, bn, bcost = [], [], []
    for kt in range(n_kt):
        boff.append(len(bsteps))
        if kt in bgathered:
            for rec in bgathered[kt]:
                bsteps.append((0, 1, 0, len(brecords) + 1))
                brecords.append(rec)
            bn.append(len(bgathered[kt]))
            bcost.append(PARTIAL_COST * len(bgathered[kt]))
        else:
            bsteps.extend((qt, i, 0, 0) for qt, i in bvis[kt])
            bn.append(len(bvis[kt]))
            bcost.append(sum(_cost(i) for _, i in bvis[kt]))
    for kt in range(n_kt):
        for hk in range(num_heads_kv):
            bitems.append([kt, hk, boff[kt], boff[kt] + bn[kt], bcost[kt] * g, 0, 0, 0])
    bwd_items = np.array(bitems, dtype=np.int32).reshape(-1, 8)
    return {
        "fwd_steps": np.array(steps, dtype=np.int32).reshape(-1, 4),
        "fwd_items": fwd_items,
        "fwd_order": fwd_order,
        "bwd_steps": np.array(bsteps, dtype=np.int32).reshape(-1, 4),
        "bwd_items": bwd_items,
        "bwd_order": order_of([it[4] for it in bitems], [it[1] for it in bitems]),
        "merges": np.array(merges, dtype=np.int32).reshape(-1, 8),
        "fwd_masks": np.array(fmasks, dtype=np.int32).reshape(-1, 1),
        "gathers": np.array(records, dtype=np.int32).reshape(-1, GATHER_WORDS),
        "bgathers": np.array(brecords, dtype=np.int32).reshape(-1, BGATHER_WORDS),
        "bwd_masks": np.array(bmasks, dtype=np.int32).reshape(-1, 1),
        "n_slots": n_slots,
        "stacked": stacked,
        "alternate": alternate,
        "grid_fwd": max(1, min(num_sms, len(items))),
        "grid_bwd": max(1, min(num_sms, len(bitems))),
        "area": visible_area(q_ranges, k_ranges, mask_types),
    }


def _tile_slices(total_q, q_ranges, k_ranges, mask_types):
    """Per q-tile: the non-empty slices whose q range meets its rows."""
    n_qt = -(-total_q // TILE)
    out = [[] for _ in range(n_qt)]
    for s, ((qs, qe), (ks, ke), t) in enumerate(zip(np.asarray(q_ranges).reshape(-1, 2),
                                                    np.asarray(k_ranges).reshape(-1, 2),
                                                    np.asarray(mask_types).reshape(-1))):
        qs, qe, ks, ke, t = int(qs), int(qe), int(ks), int(ke), int(t)
        if qe <= qs or ke <= ks:
            continue
        for qt in range(qs // TILE, -(-qe // TILE)):
            out[qt].append((qs, qe, ks, ke, t))
    return out


def gather_units(total_q, total_k, q_ranges, k_ranges, mask_types, pair_mode, fvis):
    """{unit: [(record words, (info0, info1)), ...]} for the gathered units."""
    n_qt = -(-total_q // TILE)
    n_units = n_qt if pair_mode == 0 else (n_qt + 1) // 2
    if total_k > GATHER_MAX_TK:
        return {}
    tiles = _tile_slices(total_q, q_ranges, k_ranges, mask_types)
    out = {}
    for u in range(n_units):
        qts = [u] if pair_mode == 0 else [q for q in (2 * u, 2 * u + 1) if q < n_qt]
        sl = [x for q in qts for x in tiles[q]]
        if not sl or any(t != 0 or ks % GATHER_KEYS or (ke % GATHER_KEYS and ke != total_k)
                         for _, _, ks, ke, t in sl):
            continue
        blocks = sorted({b for _, _, ks, ke, _ in sl
                         for b in range(ks // GATHER_KEYS, -(-ke // GATHER_KEYS))})
        if pair_mode == 0:
            regular = len(fvis[u])
        else:  # steps of the two q-tiles' visit lists merged on kt
            regular = len({kt for q in qts for kt, _ in fvis[q]})
        n_steps = -(-len(blocks) // GATHER_SLOTS)
        if len(blocks) > GATHER_MAX_BLOCKS or 10 * n_steps > 9 * regular:
            continue
        half_tiles = [u, u] if pair_mode == 0 else [2 * u, 2 * u + 1 if 2 * u + 1 < n_qt else -1]
        res = []
        for j in range(n_steps):
            bs = blocks[GATHER_SLOTS * j: GATHER_SLOTS * (j + 1)]
            rec = [GATHER_KEYS * b for b in bs] + [-GATHER_KEYS] * (GATHER_SLOTS - len(bs))
            infos = []
            for qt in half_tiles:
                words = np.zeros((GATHER_SLOTS, 4), dtype=np.uint32)
                if qt >= 0:
                    for slot, b in enumerate(bs):
                        k0, k1 = GATHER_KEYS * b, GATHER_KEYS * (b + 1)
                        for qs, qe, ks, ke, _ in tiles[qt]:
                            if ks < k1 and ke > k0:
                                for r in range(max(qs, TILE * qt), min(qe, TILE * (qt + 1))):
                                    rr = r - TILE * qt
                                    words[slot, rr >> 5] |= np.uint32(1 << (rr & 31))
                rec += [int(w) for w in words.view(np.int32).reshape(-1)]
                infos.append(_half_info(words, rec[:GATHER_SLOTS]))
            res.append((rec, (infos[0], infos[1])))
        out[u] = res
    return out


def _half_info(words, starts):
    """Step info of a gathered half: -1 idle, 0 when all 16 slots hold keys
    and every row of the half sees all of them (no mask), else 1."""
    if not words.any():
        return -1
    full = all(y >= 0 for y in starts[:GATHER_SLOTS]) and bool((words == 0xFFFFFFFF).all())
    return 0 if full else 1


def gather_slabs(total_q, total_k, q_ranges, k_ranges, mask_types, rows=SLAB):
    """{slab: [(record words, (info0, info1)), ...]} of the head-stacked
    units of `rows` query rows, or None when some slab is not eligible."""
    if total_k > GATHER_MAX_TK:
        return None
    SLAB = rows
    n_slabs = -(-total_q // SLAB)
    lists = [[] for _ in range(n_slabs)]
    for (qs, qe), (ks, ke), t in zip(np.asarray(q_ranges).reshape(-1, 2),
                                     np.asarray(k_ranges).reshape(-1, 2),
                                     np.asarray(mask_types).reshape(-1)):
        qs, qe, ks, ke, t = int(qs), int(qe), int(ks), int(ke), int(t)
        if qe <= qs or ke <= ks:
            continue
        for u in range(qs // SLAB, -(-qe // SLAB)):
            lists[u].append((qs, qe, ks, ke, t))
    out = {}
    for u, sl in enumerate(lists):
        if any(t != 0 or ks % GATHER_KEYS or (ke % GATHER_KEYS and ke != total_k)
               for _, _, ks, ke, t in sl):
            return None
        blocks = sorted({b for _, _, ks, ke, _ in sl
                         for b in range(ks // GATHER_KEYS, -(-ke // GATHER_KEYS))})
        if len(blocks) > GATHER_MAX_BLOCKS:
            return None
        res = []
        for j in range(-(-len(blocks) // GATHER_SLOTS)):
            bs = blocks[GATHER_SLOTS * j: GATHER_SLOTS * (j + 1)]
            rec = [GATHER_KEYS * b for b in bs] + [-GATHER_KEYS] * (GATHER_SLOTS - len(bs))
            words = np.zeros((GATHER_SLOTS, 4), dtype=np.uint32)
            for slot, b in enumerate(bs):
                k0, k1 = GATHER_KEYS * b, GATHER_KEYS * (b + 1)
                for qs, qe, ks, ke, _ in sl:
                    if ks < k1 and ke > k0:
                        for r in range(max(qs, SLAB * u), min(qe, SLAB * (u + 1))):
                            for rr in range(r - SLAB * u, TILE, SLAB):
                                words[slot, rr >> 5] |= np.uint32(1 << (rr & 31))
            half = [int(w) for w in words.view(np.int32).reshape(-1)]
            info = _half_info(words, rec)
            res.append((rec + half + half, (info, info)))
        if res:
            out[u] = res
    return out


def _ktile_slices(total_k, q_ranges, k_ranges, mask_types):
    """Per k-tile: the non-empty slices whose k range meets its keys."""
    n_kt = -(-total_k // TILE)
    out = [[] for _ in range(n_kt)]
    for s, ((qs, qe), (ks, ke), t) in enumerate(zip(np.asarray(q_ranges).reshape(-1, 2),
                                                    np.asarray(k_ranges).reshape(-1, 2),
                                                    np.asarray(mask_types).reshape(-1))):
        qs, qe, ks, ke, t = int(qs), int(qe), int(ks), int(ke), int(t)
        if qe <= qs or ke <= ks:
            continue
        for kt in range(ks // TILE, -(-ke // TILE)):
            out[kt].append((qs, qe, ks, ke, t))
    return out


def gather_units_bwd(total_q, total_k, q_ranges, k_ranges, mask_types, bvis):
    """{k-tile: [record words, ...]} for the gathered backward units."""
    if total_q > GATHER_MAX_TK:
        return {}
    tiles = _ktile_slices(total_k, q_ranges, k_ranges, mask_types)
    out = {}
    for kt, sl in enumerate(tiles):
        if not sl or any(t != 0 or qs % GATHER_KEYS or (qe % GATHER_KEYS and qe != total_q)
                         for qs, qe, _, _, t in sl):
            continue
        blocks = sorted({b for qs, qe, _, _, _ in sl
                         for b in range(qs // GATHER_KEYS, -(-qe // GATHER_KEYS))})
        n_steps = -(-len(blocks) // GATHER_SLOTS)
        if len(blocks) > GATHER_MAX_BLOCKS or 10 * n_steps > 9 * len(bvis[kt]):
            continue
        res = []
        for j in range(n_steps):
            bs = blocks[GATHER_SLOTS * j: GATHER_SLOTS * (j + 1)]
            rec = [GATHER_KEYS * b for b in bs] + [-GATHER_KEYS] * (GATHER_SLOTS - len(bs))
            words = np.zeros((GATHER_SLOTS, 4), dtype=np.uint32)
            for slot, b in enumerate(bs):
                r0, r1 = GATHER_KEYS * b, GATHER_KEYS * (b + 1)
                for qs, qe, ks, ke, _ in sl:
                    if qs < r1 and qe > r0:
                        for key in range(max(ks, TILE * kt), min(ke, TILE * (kt + 1))):
                            kk = key - TILE * kt
                            words[slot, kk >> 5] |= np.uint32(1 << (kk & 31))
            res.append(rec + [int(w) for w in words.view(np.int32).reshape(-1)])
        out[kt] = res
    return out
