"""Host model of the on-device split-KV partition (csrc/mla_partition.cu).

The same integer arithmetic, step by step, in plain Python: row groups of
128 query rows, each costing an overhead of 3 tile units plus its KV tiles
(64 rows); the groups laid end to end (lane-major when every request has
the same number G >= 2 of groups and the busy workers split into G lanes of
at least two); busy workers n' = min(n, W // 4); worker p's range of units
starts at boundary(p); a group that straddles a boundary is cut at the
corresponding tile; an item belongs to the worker whose range holds its
first tile.  The CPU tests check its invariants, and a GPU test compares the
kernel's work list with it field by field.  Under sparse top-k selection
(``sparse_k`` > 0) a group is one token's H rows and walks the token's list
of ``sparse_k`` entries instead of the request's cache rows.
"""
from __future__ import annotations

OVERHEAD = 3
MIN_UNITS = 4
TILE = 64
ROWS = 128


def ceil_div(a, b):
    return -(-a // b)


def partition(seq_lens, q_lens, q_starts, num_heads, n_workers, mask_bases, sparse_k=0):
    """Return (items, worker_begin).  items: tuples (b, g, kv_begin, kv_end,
    slot, q_len, seq_len, q_start, comb, mask_base) in the kernel's order."""
    B = len(seq_lens)
    rows = num_heads if sparse_k > 0 else ROWS
    kv_rows = [sparse_k if sparse_k > 0 else int(L) for L in seq_lens]
    gcount = [ceil_div(int(q) * num_heads, rows) if int(L) > 0 else 0
              for L, q in zip(seq_lens, q_lens)]
    n_groups = sum(gcount)
    gbase, acc = [], 0
    for c in gcount:
        gbase.append(acc)
        acc += c
    nz = [c for c in gcount if c > 0]
    g_min, g_max = (min(nz), max(nz)) if nz else (1 << 30, 0)
    tiles = [ceil_div(n_kv, TILE) for n_kv in kv_rows]
    W_total = sum(gcount[b] * (OVERHEAD + tiles[b]) for b in range(B))
    n = n_workers
    n_eff = max(1, min(n, W_total // MIN_UNITS))
    G = g_max
    lanes = G if (g_min == g_max and G >= 2 and n_eff // G >= 2) else 1
    n_req_groups = n_groups // G if lanes > 1 else 0
    slot_req = [0] * n_groups
    slot_k = [0] * n_groups
    for b in range(B):
        for k in range(gcount[b]):
            slot = k * n_req_groups + gbase[b] // G if lanes > 1 else gbase[b] + k
            slot_req[slot], slot_k[slot] = b, k
    cost = [OVERHEAD + tiles[slot_req[g]] for g in range(n_groups)]
    start, acc = [], 0
    for c in cost:
        start.append(acc)
        acc += c
    W = acc
    nl = n_eff // lanes
    WL = W // lanes if lanes else 0

    def boundary(p):
        if p >= lanes * nl:
            return W
        k, i = divmod(p, nl)
        return k * WL + (i * WL) // nl

    table = [boundary(p) for p in range(n + 1)]

    def first_above(x):
        lo, hi = 0, n
        while lo < hi:
            mid = (lo + hi) // 2
            if table[mid] > x:
                hi = mid
            else:
                lo = mid + 1
        return lo

    def owner(x):
        return min(first_above(x) - 1, n - 1)

    chunks = []  # per group: list of (t0, t1, owner)
    for g in range(n_groups):
        b = slot_req[g]
        T, S = tiles[b], start[g]
        c = OVERHEAD + T
        cuts, prev = [], 0
        if W > 0:
            p_lo = first_above(S)
            p_hi = first_above(S + c - 1) - 1
            for q in range(max(p_lo, 1), min(p_hi, n - 1) + 1):
                t = min(max(table[q] - S - OVERHEAD, 0), T)
                if prev < t < T:
                    cuts.append(t)
                    prev = t
        edges = [0] + cuts + [T]
        chunks.append([(edges[i], edges[i + 1], owner(S + OVERHEAD + edges[i]))
                       for i in range(len(edges) - 1)])
    items, owners = [], []
    n_slot = n_comb = 0
    for g in range(n_groups):
        b = slot_req[g]
        L = int(seq_lens[b])
        nch = len(chunks[g])
        for k, (t0, t1, o) in enumerate(chunks[g]):
            items.append((b, slot_k[g], t0 * TILE, min(kv_rows[b], t1 * TILE),
                          n_slot + k if nch > 1 else -1, int(q_lens[b]), L, int(q_starts[b]),
                          n_comb if nch > 1 else -1, int(mask_bases[b])))
            owners.append(o)
        if nch > 1:
            n_slot += nch
            n_comb += 1
    worker_begin = []
    for w in range(n + 1):
        lo = next((i for i, o in enumerate(owners) if o >= w), len(owners))
        worker_begin.append(len(items) if w == n else lo)
    return items, worker_begin, dict(W=W, n_eff=n_eff, lanes=lanes, owners=owners)
