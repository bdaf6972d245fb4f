"""Checks that pin the oracle's bookkeeping to what the pages fix.

Each ``check_*`` takes a page-table class (the oracle's, or a deliberately
broken copy in the mutation tests) and returns a list of problems; empty
means the check passes. The expected values come from the golden files under
``tests/golden/`` (numbers the pages print) or from closed forms the pages
state; none is computed by the oracle itself.
"""

from __future__ import annotations

import os
import random

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.rstrip("\n") for ln in f if ln.strip() and not ln.startswith("#")]


def _ints(s):
    s = s.strip()
    return [] if s in ("", "-") else [int(x) for x in s.split()]


def _kv(s):
    out = {}
    for part in s.split(","):
        k, v = part.split(":")
        out[int(k)] = int(v)
    return out


# ---------------------------------------------------------------------------
# Worked example A (chapter 15): every step's gather, table, dropped, free.
# ---------------------------------------------------------------------------
def check_example_a(PT, OutOfPages=Exception):
    P = []
    lines = _lines("ch15_example_a.txt")
    i = lines.index("part1 page=4 window=6 pages=8") + 1
    pt = PT(8, 4)
    pt.new("A")
    W = 6
    while not lines[i].startswith("used_at_end"):
        step, rows, table, dropped, free = [c.strip() for c in lines[i].split("|")]
        L = int(step)
        n = min(L, W)
        lo = L - n
        got_rows = pt.rows("A", lo, L - 1) if n > 1 else []
        pt.append("A", L - 1)
        pt.trim("A", max(0, L + 1 - W))
        if got_rows != _ints(rows):
            P.append(f"example A step {L}: gathered {got_rows}, page prints {rows}")
        if list(pt.table["A"]) != _ints(table):
            P.append(f"example A step {L}: table {pt.table['A']}, page prints {table}")
        if pt.dropped["A"] != int(dropped):
            P.append(f"example A step {L}: dropped {pt.dropped['A']}, page prints {dropped}")
        if sorted(pt.free) != _ints(free):
            P.append(f"example A step {L}: free {sorted(pt.free)}, page prints {free}")
        i += 1
    if pt.used() != int(lines[i].split()[1]):
        P.append(f"example A: {pt.used()} pages in use at the end")

    part2 = {ln.split()[0]: ln.split()[1:] for ln in lines[lines.index("part2") + 1:]}
    pt2 = PT(8, 4)
    pt2.new("A")
    for r in range(10):
        pt2.append("A", r)

    def refs(ids):
        return {p: pt2.ref[p] for p in sorted(set(ids))}

    bf = part2["before_fork"]
    if pt2.table["A"] != [int(x) for x in bf[0][2:].split(",")] or refs(pt2.table["A"]) != _kv(bf[1][4:]):
        P.append("example A part 2: state before the fork")
    pt2.fork("A", "B")
    af = part2["after_fork"]
    if (pt2.table["B"] != [int(x) for x in af[1][2:].split(",")]
            or refs(pt2.table["A"]) != _kv(af[2][4:])):
        P.append("example A part 2: state after the fork")
    pt2.append("B", 100)
    aa = part2["after_append"]
    if (pt2.table["A"] != [int(x) for x in aa[0][2:].split(",")]
            or pt2.table["B"] != [int(x) for x in aa[1][2:].split(",")]
            or refs(pt2.table["A"] + pt2.table["B"]) != _kv(aa[2][4:])):
        P.append(f"example A part 2: after B appends: A {pt2.table['A']} B {pt2.table['B']}")
    rw = part2["rows"]
    if (pt2.rows("A", 0, 10) != [int(x) for x in rw[0][2:].split(",")]
            or pt2.rows("B", 0, 11) != [int(x) for x in rw[1][2:].split(",")]):
        P.append("example A part 2: rows read back")
    pt2.release("B")
    ar = part2["after_release"]
    if refs(pt2.table["A"]) != _kv(ar[0][4:]) or sorted(pt2.free) != [int(x) for x in ar[1][5:].split(",")]:
        P.append("example A part 2: state after releasing B")
    return P


# ---------------------------------------------------------------------------
# Pages in use during the chapter's 32-step run (page 4, pool 64).
# ---------------------------------------------------------------------------
def run_window_decode(PT, W, page, n_pages, steps):
    """The host loop of chapter 15 (record pages, append, trim) without a model."""
    pt = PT(n_pages, page)
    pt.new(0)
    rec, peak = [], 0
    for L in range(1, steps + 1):
        rec.append(pt.used())
        pt.append(0, L - 1)
        if W is not None:
            pt.trim(0, max(0, L + 1 - W))
        peak = max(peak, pt.used())
    return rec, peak, pt


def check_pages_in_use(PT):
    P = []
    for ln in _lines("ch15_pages_in_use.txt"):
        w, *vals = ln.split()
        W = None if w == "None" else int(w)
        rec, peak, _ = run_window_decode(PT, W, 4, 64, 32)
        got = [rec[1], rec[8], rec[16], rec[-1], peak]
        if got != [int(v) for v in vals]:
            P.append(f"W={W}: pages in use {got}, page prints {vals}")
    return P


def check_exact_counts(PT):
    """Chapter 15, section "Tests", item 3: the exact count at every step."""
    P = []
    for W, page in ((None, 4), (8, 4), (6, 2), (4, 4), (3, 1)):
        rec, _, _ = run_window_decode(PT, W, page, 64, 24)
        for L, got in enumerate(rec, start=1):
            n = L - 1
            kf = 0 if W is None else max(0, L - W)
            want = (-(-n // page) - kf // page) if n > 0 else 0
            if got != want:
                P.append(f"W={W} page={page} step {L}: {got} pages, the window rule says {want}")
        if W is not None:
            bound = -(-(W - 1) // page) + 1
            if max(rec) > bound + 1 or rec[-1] > bound:
                P.append(f"W={W} page={page}: footprint above ceil((W-1)/P)+1")
        elif rec[-1] != -(-23 // page):
            P.append("without a window every page must stay")
    return P


# ---------------------------------------------------------------------------
# Shadow model (chapter 15, section "Tests", item 1).
# ---------------------------------------------------------------------------
def invariants(pt, shadow):
    P = []
    cnt = [0] * len(pt.ref)
    for tb in pt.table.values():
        for p in tb:
            cnt[p] += 1
    if cnt != list(pt.ref):
        P.append("reference counts differ from the block-table entries")
    if len(set(pt.free)) != len(pt.free):
        P.append("a page is on the free list twice")
    if any(pt.ref[p] != 0 for p in pt.free):
        P.append("a referenced page is on the free list")
    if len(pt.free) + sum(1 for r in pt.ref if r > 0) != len(pt.ref):
        P.append("a page is neither free nor referenced")
    for rid, rows in shadow.items():
        lo = pt.dropped[rid] * pt.page
        if pt.length[rid] != len(rows):
            P.append(f"length of request {rid}")
        elif pt.rows(rid, lo, len(rows)) != rows[lo:]:
            P.append(f"rows of request {rid} differ from the shadow")
    return P


def check_shadow(PT, OutOfPages, seed, n_ops=400, n_pages=24, page=4, max_live=5):
    R = random.Random(seed)
    pt = PT(n_pages, page)
    shadow = {}
    nxt = ctr = 0
    for step in range(n_ops):
        op = R.choice(["append"] * 6 + ["new", "fork", "trim", "release"])
        ids = list(shadow)
        try:
            if op == "new" and len(ids) < max_live:
                pt.new(nxt); shadow[nxt] = []; nxt += 1
            elif op == "append" and ids:
                rid = R.choice(ids); ctr += 1; row = (ctr, -ctr)
                pt.append(rid, row); shadow[rid].append(row)
            elif op == "fork" and ids and len(ids) < max_live:
                s = R.choice(ids); pt.fork(s, nxt); shadow[nxt] = list(shadow[s]); nxt += 1
            elif op == "trim" and ids:
                rid = R.choice(ids); pt.trim(rid, R.randrange(0, len(shadow[rid]) + 1))
            elif op == "release" and ids:
                rid = R.choice(ids); pt.release(rid); del shadow[rid]
        except OutOfPages:
            pass
        P = invariants(pt, shadow)
        if P:
            return [f"seed {seed} op {step} ({op}): {p}" for p in P[:3]]
    for rid in list(shadow):
        pt.release(rid)
    if len(pt.free) != n_pages or any(pt.ref):
        return [f"seed {seed}: pages leaked after releasing every request"]
    return []


def check_exhaustion(PT, OutOfPages):
    """Chapter 15, section "Tests", item 2 (pool of 3 pages of 2 rows)."""
    pt = PT(3, 2)
    pt.new(0)
    raised = False
    try:
        for i in range(10):
            pt.append(0, (i, i))
    except OutOfPages:
        raised = True
    P = []
    if not raised:
        P.append("no OutOfPages when the pool is exhausted")
    if pt.length[0] != 6:
        P.append(f"a failed append changed the length ({pt.length[0]})")
    return P


def check_paged_equals_plain(PT):
    """Chapter 15, section "Tests", item 4: rows through the table == a plain list."""
    P = []
    for W, page in ((None, 4), (8, 4), (6, 2), (4, 4), (3, 1)):
        pt = PT(64, page)
        pt.new(0)
        plain = []
        for L in range(1, 25):
            nc = L if W is None else min(L, W)
            lo = L - nc
            if pt.rows(0, lo, L - 1) != plain[lo:L - 1]:
                P.append(f"W={W} page={page} step {L}: paged gather differs from the plain list")
                break
            row = (L, -L)
            pt.append(0, row)
            plain.append(row)
            if W is not None:
                pt.trim(0, max(0, L + 1 - W))
    return P


# ---------------------------------------------------------------------------
# Running example B (chapter 15): prefix sharing and admission tables.
# ---------------------------------------------------------------------------
def check_prefix_sharing(PT):
    P = []
    for ln in _lines("ch15_prefix_sharing.txt"):
        prompt, page, want_c, want_s, want_cow = (int(x) for x in ln.split())
        pc, ps = PT(400, page), PT(400, page)
        for i in range(8):
            pc.new(i)
            for _ in range(prompt + 40):
                pc.append(i, None)
        ps.new("base")
        for _ in range(prompt):
            ps.append("base", None)
        cow = 0
        for i in range(8):
            ps.fork("base", i)
            for _ in range(40):
                u0 = ps.used()
                ps.append(i, None)
                cow += (ps.used() - u0 > 0 and (ps.length[i] - 1) % page != 0)
        ps.release("base")
        got = (pc.used(), ps.used(), cow)
        if got != (want_c, want_s, want_cow):
            P.append(f"prompt {prompt} page {page}: {got}, page prints {(want_c, want_s, want_cow)}")
    return P


def admission_lengths():
    R = random.Random(11)
    return [min(2048, max(16, int(R.lognormvariate(5.2, 0.9)))) for _ in range(400)]


def check_admission(PT, OutOfPages):
    P = []
    lines = _lines("ch15_admission.txt")
    lens = admission_lengths()
    stats = dict(kv.split("=") for kv in lines[0].split()[1:])
    got = {"mean": f"{sum(lens) / len(lens):.0f}", "median": str(sorted(lens)[200]), "max": str(max(lens))}
    if got != stats:
        P.append(f"length sample {got}, page prints {stats}")
    CAP = 8192
    for ln in lines[1:]:
        scheme, page, want_n, want_u, want_r = ln.split()
        page, want = int(page), (int(want_n), int(want_u), int(want_r))
        if scheme == "contiguous":
            n = used = 0
            for L in lens:
                if (n + 1) * page > CAP:
                    break
                n += 1
                used += L
            res = (n, used, n * page)
        else:
            pt = PT(CAP // page, page)
            n = used = 0
            for i, L in enumerate(lens):
                pt.new(i)
                try:
                    for _ in range(L):
                        pt.append(i, None)
                except OutOfPages:
                    pt.release(i)
                    break
                n += 1
                used += L
            res = (n, used, pt.used() * page)
        if res != want:
            P.append(f"{scheme} page {page}: {res}, page prints {want}")
    return P


def all_bookkeeping_problems(PT, OutOfPages, shadow_seeds=range(6)):
    P = []
    P += check_example_a(PT, OutOfPages)
    P += check_pages_in_use(PT)
    P += check_exact_counts(PT)
    for s in shadow_seeds:
        P += check_shadow(PT, OutOfPages, s)
    P += check_exhaustion(PT, OutOfPages)
    P += check_paged_equals_plain(PT)
    P += check_prefix_sharing(PT)
    P += check_admission(PT, OutOfPages)
    return P
