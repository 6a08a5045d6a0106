"""Host-side checks of the C library: it loads, exports every declared symbol, and the planner's
tables (tile -> job map, packed rank windows, work lists) are complete and consistent.  No GPU:
plans are built with MLORA_PLAN_HOST_ONLY, which makes no CUDA call."""
import os
import re

import numpy as np
import pytest

from adapter_gemm_packed_gb300 import _mlora as M
from adapter_gemm_packed_gb300 import workloads as W
from adapter_gemm_packed_gb300.layer import host_plan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from adapter_gemm_packed_gb300 import build
    build.build()


def test_header_symbols_exported():
    hdr = open(os.path.join(ROOT, "include", "mlora.h")).read()
    declared = set(re.findall(r"\b(mlora_[a-z0-9_]+)\s*\(", hdr))
    assert declared == set(M.EXPORTS)
    L = M.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert M.mlora_version() >= 100
    assert M.mlora_status_string(M.MLORA_ERR_TIMEOUT) == "device wait timed out"


def _tables(plan):
    s = M.mlora_plan_describe(plan, M.MLORA_Q_SUMMARY)
    keys = ["N", "d_in", "d_out", "n_segs", "n_mtiles", "C_total", "n_chunks", "n_images", "n_win", "n_da", "n_db",
            "ws"]
    summ = dict(zip(keys, s))
    mt = np.array(M.mlora_plan_describe(plan, M.MLORA_Q_MTILES)).reshape(-1, 5)
    cols = np.array(M.mlora_plan_describe(plan, M.MLORA_Q_COLUMNS)).reshape(-1, 2)
    win = np.array(M.mlora_plan_describe(plan, M.MLORA_Q_WINDOW)).reshape(-1, 5)
    da = np.array(M.mlora_plan_describe(plan, M.MLORA_Q_WGRAD_A)).reshape(-1, 9)
    db = np.array(M.mlora_plan_describe(plan, M.MLORA_Q_WGRAD_B)).reshape(-1, 9)
    return summ, mt, cols, win, da, db


CASES = {
    "qproj": (4096, 4096, [8, 8, 16, 16, 32, 32, 64, 64], [2048] * 8),
    "ragged": (512, 640, [1, 7, 64, 256], [200, 56, 300, 17]),
    "tiny_segments": (256, 256, [1, 2, 4, 8, 16, 32, 64, 128, 256, 3], [16, 16, 32, 16, 48, 16, 16, 64, 16, 5]),
    "one_token": (64, 64, [5], [1]),
    "many_small": None,
    "mlp_up": None,
}


def _case(name):
    if name == "many_small":
        wl = W.llama70b_down_many_small()
        return wl.d_in, wl.d_out, wl.ranks, wl.n_tokens
    if name == "mlp_up":
        wl = W.mlp_up_lognormal()
        return wl.d_in, wl.d_out, wl.ranks, wl.n_tokens
    return CASES[name]


@pytest.mark.parametrize("name", sorted(CASES))
def test_planner_tables(name):
    _check_tables(*_case(name))


def _random_case(seed):
    g = np.random.default_rng(1000 + seed)
    n_jobs = int(g.integers(1, 24))
    ranks = [int(r) for r in g.choice([1, 2, 3, 5, 8, 16, 24, 32, 48, 64, 100, 128, 200, 256], size=n_jobs)]
    ns = [int(n) for n in g.choice([1, 5, 17, 64, 100, 127, 128, 129, 250, 256, 300, 700], size=n_jobs)]
    d_in = 8 * int(g.integers(8, 160))
    d_out = 8 * int(g.integers(8, 160))
    return d_in, d_out, ranks, ns


@pytest.mark.parametrize("seed", range(40))
def test_planner_tables_random(seed):
    """The same invariants on seeded random job tables (ranks 1-256, jobs of 1-700 tokens,
    ragged d_in / d_out), plus the CTA-pair window items."""
    d_in, d_out, ranks, ns = _random_case(seed)
    _check_tables(d_in, d_out, ranks, ns)
    plan, _ = host_plan(d_in, d_out, ranks, ns)
    try:
        mt = _describe(plan, M.MLORA_Q_MTILES).reshape(-1, 5)
        shrink, dh = _pair_entries(plan)
    finally:
        M.mlora_plan_destroy(plan)
    _check_pair_pieces(shrink, lambda t, q: (0, -(-d_in // 64)))
    _check_pair_pieces(dh, lambda t, q: (0, -(-d_out // 64)))
    for items in (shrink, dh):
        items = items[items[:, 6] == 0]          # one entry per item: its first piece
        items = items[np.lexsort((items[:, 2], items[:, 1]))]
        for p in range((len(mt) + 1) // 2):
            q_lo, nch = mt[2 * p, 2], mt[2 * p, 3]
            got = [q for row in items[items[:, 1] == p] for q in range(row[2], row[2] + row[3])]
            assert got[:nch] == list(range(q_lo, q_lo + nch)) and len(got) - nch in (0, 1)


def _pair_entries(plan):
    """The CTA-pair schedules as (shrink entries, dH entries), each row: pair, 256-token pair of
    tiles, first chunk, chunks, first K slice, K slices, piece, pieces."""
    d = _describe(plan, M.MLORA_Q_WINDOW_PAIRS)[1:].reshape(-1, 9)
    return d[d[:, 0] == 0][:, 1:], d[d[:, 0] == 1][:, 1:]


def _check_pair_pieces(items, kslices):
    """One product's CTA-pair schedule: the list runs pair by pair; the pieces of an item sit on
    distinct pairs, numbered 0..S-1, and in that order tile the item's K range exactly once (all
    of it: kslices(first chunk) gives its first slice and count), each piece of a cut item keeping
    at least 16 slices (the planner cuts at shares of 16 slices, rounded down: 15 or more)."""
    assert (np.diff(items[:, 0]) >= 0).all()
    groups = {}
    for row in items:
        groups.setdefault((row[1], row[2]), []).append(row)
    for (tile, q0), rows in groups.items():
        rows.sort(key=lambda r: r[6])
        S = rows[0][7]
        assert [r[6] for r in rows] == list(range(S)) and all(r[7] == S for r in rows)
        assert len({r[0] for r in rows}) == S and len({r[3] for r in rows}) == 1
        k0, n = kslices(tile, q0)
        for r in rows:
            assert r[4] == k0 and r[5] >= (15 if S > 1 else 1)
            k0 += r[5]
        assert k0 == kslices(tile, q0)[0] + n
    return groups


def _check_tables(d_in, d_out, ranks, ns):
    plan, ws = host_plan(d_in, d_out, ranks, ns)
    try:
        summ, mt, cols, win, da, db = _tables(plan)
        pw_shrink, pw_dh = _pair_entries(plan)
    finally:
        M.mlora_plan_destroy(plan)
    N = sum(ns)
    offs = np.cumsum([0] + ns)[:-1]
    assert summ["N"] == N and summ["n_segs"] == len(ranks)
    # packed rank space: windows in job order, 16-aligned, wide enough, no overlap
    c = 0
    for i, r in enumerate(ranks):
        assert cols[i, 0] == c and cols[i, 1] % 16 == 0 and r <= cols[i, 1] < r + 16
        c += cols[i, 1]
    assert summ["C_total"] == c and summ["n_chunks"] == -(-c // 64)
    # token tiles: every row covered once, and the tile's job range is exactly the jobs it touches;
    # its staged chunk range is the union over its 256-token pair (the CTA-pair GEMM tile)
    assert summ["n_mtiles"] == -(-N // 128) == len(mt)
    seg_of = np.repeat(np.arange(len(ns)), ns)
    img = 0
    for t in range(len(mt)):
        rows = np.arange(128 * t, min(N, 128 * t + 128))
        jobs = np.unique(seg_of[rows])
        f, l, q_lo, nch, img_off = mt[t]
        assert (f, l) == (jobs[0], jobs[-1])
        prow = np.arange(256 * (t // 2), min(N, 256 * (t // 2) + 256))
        pj = np.unique(seg_of[prow])
        lo, hi = cols[pj[0], 0], cols[pj[-1], 0] + cols[pj[-1], 1]
        assert q_lo == lo // 64 and q_lo + nch == -(-hi // 64)
        assert q_lo <= cols[f, 0] // 64 and -(-(cols[l, 0] + cols[l, 1]) // 64) <= q_lo + nch
        assert img_off == img
        img += nch
    assert summ["n_images"] == img
    # window work: each tile's chunks exactly once, <= 4 per item
    seen = {}
    for t, q0, nq, kb0, nkb in win:
        assert 1 <= nq <= 4
        assert (kb0, nkb) == (0, -(-d_out // 64))    # one projection: dH reads all of d_out
        for q in range(q0, q0 + nq):
            assert (t, q) not in seen
            seen[(t, q)] = 1
    want = {(t, q) for t in range(len(mt)) for q in range(mt[t, 2], mt[t, 2] + mt[t, 3])}
    assert set(seen) == want
    # weight-gradient work: per job, its chunk span x row blocks exactly once, its tokens covered
    # exactly once by the parts of each item; the list runs CTA by CTA, each CTA's cut parts first
    wg_units = []
    for items, rows_total in ((da, d_in), (db, d_out)):
        _check_wgrad(items, rows_total, ns, offs, cols)
        wg_units.append(sum(nq for _, _, _, _, _, nq, part, parts, _ in items if parts > 1))
    # workspace = bf16 shadows + the split items' fp32 partial sums (one region: the pair items'
    # or dA's / dB's, whichever is larger) + two image sets
    shadow = -(-c * d_in * 2 // 1024) * 1024 + -(-c * d_out * 2 // 1024) * 1024
    # the pieces of cut pair items, one partial set each (shrink and dH share the region)
    split = max((pw_shrink[:, 7] > 1).sum(), (pw_dh[:, 7] > 1).sum())
    partials = max(split * 2 * 128 * 256 * 4, max(wg_units) * 256 * 64 * 4)
    assert ws == shadow + -(-partials // 1024) * 1024 + 2 * img * 16384


def _check_wgrad(items, rows_total, ns, offs, cols):
    cover = {}
    parts_of = {}
    for row0, j, ga, gb, q0, nq, part, parts, cta in items:
        assert row0 % 256 == 0 and 0 <= row0 < rows_total and 1 <= nq <= 2
        assert 0 <= part < parts and ga < gb
        parts_of.setdefault((row0, j, q0, nq), []).append((part, parts, ga, gb, cta))
    for (row0, j, q0, nq), ps in parts_of.items():
        ps.sort()
        S = ps[0][1]
        assert [p[0] for p in ps] == list(range(S)) and all(p[1] == S for p in ps)
        # the parts' token ranges tile the job's half-tiles in order, each on its own CTA
        assert ps[0][2] * 64 <= offs[j] < (ps[0][2] + 1) * 64
        assert (ps[-1][3] - 1) * 64 < offs[j] + ns[j] <= ps[-1][3] * 64
        assert all(ps[k][3] == ps[k + 1][2] for k in range(S - 1))
        assert len({p[4] for p in ps}) == S
        if S > 1:
            assert all(p[3] - p[2] >= 4 for p in ps)   # no part shorter than 256 tokens
        for q in range(q0, q0 + nq):
            key = (row0, j, q)
            assert key not in cover
            cover[key] = 1
    want = set()
    for j in range(len(ns)):
        qa, qb = cols[j, 0] // 64, -(-(cols[j, 0] + cols[j, 1]) // 64)
        want |= {(r0, j, q) for r0 in range(0, rows_total, 256) for q in range(qa, qb)}
    assert set(cover) == want
    ctas = items[:, 8]
    assert list(ctas) == sorted(ctas) and set(ctas) == set(range(ctas.max() + 1 if len(ctas) else 0))
    for c in set(ctas):
        split = items[ctas == c][:, 7] > 1
        assert list(split) == sorted(split, reverse=True)   # cut parts first


def _status_of(fn):
    try:
        fn()
    except M.MloraError as e:
        return e.status
    return M.MLORA_OK


@pytest.mark.parametrize("bad,status", [
    (dict(offsets=[0, 5]), M.MLORA_ERR_INVALID),            # overlap (second job should start at 10)
    (dict(offsets=[0, 12]), M.MLORA_ERR_INVALID),           # gap
    (dict(n_total=25), M.MLORA_ERR_INVALID),                # rows not covered
    (dict(ranks=[0, 4]), M.MLORA_ERR_INVALID),
    (dict(ranks=[257, 4]), M.MLORA_ERR_UNSUPPORTED),
    (dict(d_in=100), M.MLORA_ERR_UNSUPPORTED),              # not a multiple of 8 (bf16)
    (dict(n_tokens=[0, 10]), M.MLORA_ERR_INVALID),
])
def test_plan_rejects_bad_tables(bad, status):
    args = dict(d_in=128, d_out=64, ranks=[4, 8], n_tokens=[10, 10])
    args.update(bad)
    assert _status_of(lambda: M.mlora_plan_destroy(host_plan(**args)[0])) == status


def test_plan_rejects_an_empty_pack():
    """A pack with no jobs (and no tokens) is an invalid table, reported with a message."""
    assert _status_of(lambda: host_plan(64, 64, [], [])) == M.MLORA_ERR_INVALID
    assert b"n_segs" in M.lib().mlora_last_error()


def test_plan_rejects_null_and_misaligned_adapters():
    ok = M.mlora_segment(0, 4, 2, 1.0, 0x1000, 0x2000, 0, 0, 0, 0, 0, 0)
    prob = M.mlora_problem(4, 64, 64, M.MLORA_BF16, M.MLORA_PLAN_HOST_ONLY)
    h, _ = M.mlora_plan(prob, [ok])
    M.mlora_plan_destroy(h)
    for field, val in (("At", 0), ("Bt", 0), ("At", 0x1004), ("dBt", 0x2008)):
        s = M.mlora_segment(0, 4, 2, 1.0, 0x1000, 0x2000, 0, 0, 0, 0, 0, 0)
        setattr(s, field, val)
        assert _status_of(lambda: M.mlora_plan(prob, [s])) == M.MLORA_ERR_INVALID


def test_host_only_plan_refuses_execution():
    plan, _ = host_plan(128, 64, [4], [10])
    try:
        st = M.lib().mlora_forward(plan, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, None)
        assert st == M.MLORA_ERR_INVALID
        assert "HOST_ONLY" in M.lib().mlora_last_error().decode()
    finally:
        M.mlora_plan_destroy(plan)


def test_h_elems_is_sum_n_r():
    plan, _ = host_plan(128, 64, [4, 8, 3], [10, 7, 5])
    try:
        assert M.mlora_h_elems(plan) == 4 * 10 + 8 * 7 + 3 * 5
    finally:
        M.mlora_plan_destroy(plan)


def test_w4_workspace_holds_the_expansion_unless_fused():
    """A 4-bit-base plan's workspace adds the bf16 expansion of W (2 d_in d_out bytes, 1 KB
    aligned) to the bf16 plan's; with MLORA_W4_FUSED it is the bf16 plan's."""
    d_in, d_out, ranks, ns = 512, 384, [8, 64], [300, 100]
    h16, ws16 = host_plan(d_in, d_out, ranks, ns)
    h4, ws4 = host_plan(d_in, d_out, ranks, ns, dtype="bf16_w4")
    hf, wsf = host_plan(d_in, d_out, ranks, ns, dtype="bf16_w4", flags=M.MLORA_W4_FUSED)
    for h in (h16, h4, hf):
        M.mlora_plan_destroy(h)
    assert wsf == ws16
    assert ws4 == -(-ws16 // 1024) * 1024 + 2 * d_in * d_out


@pytest.mark.parametrize("flags,status", [
    (0, M.MLORA_OK),
    (M.MLORA_GEMM_SINGLE_CTA, M.MLORA_OK),
    (M.MLORA_W4_FUSED, M.MLORA_OK),
    (M.MLORA_W4_FUSED | M.MLORA_GEMM_SINGLE_CTA, M.MLORA_ERR_UNSUPPORTED),
])
def test_w4_plan_flags(flags, status):
    assert _status_of(lambda: M.mlora_plan_destroy(
        host_plan(512, 384, [8], [100], dtype="bf16_w4", flags=flags)[0])) == status
    # d_in must hold whole 64-wide scale groups
    assert _status_of(lambda: M.mlora_plan_destroy(
        host_plan(520, 384, [8], [100], dtype="bf16_w4", flags=flags)[0])) == M.MLORA_ERR_UNSUPPORTED


# ---------------------------------------------------------------- shared-input packs

def _describe(plan, what):
    return np.array(M.mlora_plan_describe(plan, what), dtype=np.int64)


def test_grouped_plan_tables():
    """A job's adapters sit side by side in its window (no padding between them, the window
    padded to 16); H holds sum_g r_jg columns per job; dB items cover exactly the chunks of the
    adapters whose output range meets their 256-row block; dA items cover the whole window."""
    from adapter_gemm_packed_gb300.layer import host_plan_grouped
    d_in, widths = 512, [256, 64, 320]
    ranks_jg = [[8, 8, 8], [64, 16, 1], [3, 128, 32], [16, 16, 16]]
    ns = [200, 56, 300, 17]
    plan, ws = host_plan_grouped(d_in, widths, ranks_jg, ns)
    try:
        ad = _describe(plan, M.MLORA_Q_ADAPTERS).reshape(-1, 5)
        cols = _describe(plan, M.MLORA_Q_COLUMNS).reshape(-1, 2)
        wa = _describe(plan, M.MLORA_Q_WGRAD_A).reshape(-1, 9)
        wb = _describe(plan, M.MLORA_Q_WGRAD_B).reshape(-1, 9)
        h = M.mlora_h_elems(plan)
    finally:
        M.mlora_plan_destroy(plan)
    offs = [0, 256, 320]
    c, k = 0, 0
    for j, rj in enumerate(ranks_jg):
        assert cols[j][0] == c and cols[j][1] == -(-sum(rj) // 16) * 16
        t = c
        for g, r in enumerate(rj):
            assert list(ad[k]) == [j, t, r, offs[g], offs[g] + widths[g]]
            t += r
            k += 1
        c += cols[j][1]
    assert h == sum(n * sum(rj) for n, rj in zip(ns, ranks_jg))
    d_out = sum(widths)
    for j, rj in enumerate(ranks_jg):
        sub = ad[ad[:, 0] == j]
        for r0 in range(0, d_out, 256):
            meets = sub[(sub[:, 3] < r0 + 256) & (sub[:, 4] > r0)]
            got = sorted(q for row0, job, ga, gb, q0, nq, part, *_ in wb if job == j and row0 == r0 and part == 0
                         for q in range(q0, q0 + nq))
            if len(meets) == 0:
                assert got == []
                continue
            lo, hi = meets[:, 1].min(), (meets[:, 1] + meets[:, 2]).max()
            assert got == list(range(lo // 64, -(-hi // 64)))
        for r0 in range(0, d_in, 256):
            got = sorted(q for row0, job, ga, gb, q0, nq, part, *_ in wa if job == j and row0 == r0 and part == 0
                         for q in range(q0, q0 + nq))
            lo, hi = cols[j][0], cols[j][0] + sum(rj)
            assert got == list(range(lo // 64, -(-hi // 64)))


def test_grouped_memory_model_counts_each_adapters_own_width():
    from adapter_gemm_packed_gb300.layer import host_plan_grouped
    d_in, widths = 512, [256, 64, 320]
    ranks_jg = [[8, 8, 8], [64, 16, 1]]
    plan, _ = host_plan_grouped(d_in, widths, ranks_jg, [100, 30])
    try:
        m = M.mlora_memory_estimate(plan)
    finally:
        M.mlora_plan_destroy(plan)
    params = sum(r * (d_in + w) for rj in ranks_jg for r, w in zip(rj, widths))
    assert m["lora_params"] == 4 * params


@pytest.mark.parametrize("bad,status", [
    (dict(widths_off=[(0, 256), (200, 128)]), M.MLORA_ERR_INVALID),       # groups overlap
    (dict(widths_off=[(0, 256), (256, 0)]), M.MLORA_ERR_INVALID),         # zero width
    (dict(widths_off=[(0, 256), (256, 64)]), M.MLORA_ERR_INVALID),        # do not reach d_out
    (dict(rows=[(0, 10), (0, 11)]), M.MLORA_ERR_INVALID),                 # a job's entries disagree
    (dict(drop_last=True), M.MLORA_ERR_INVALID),                          # not n_jobs x n_groups
    (dict(dtype=M.MLORA_F32), M.MLORA_ERR_UNSUPPORTED),                   # fp32 has one group only
    (dict(rank=257), M.MLORA_ERR_UNSUPPORTED),
])
def test_grouped_plan_rejects(bad, status):
    d_out = 384
    groups = bad.get("widths_off", [(0, 256), (256, 128)])
    rows = bad.get("rows", [(0, 10), (0, 10)])
    segs = []
    for j in range(2):
        for g in range(2):
            o, n = rows[g] if j == 0 else (10, 5)
            segs.append(M.mlora_segment(o, n, bad.get("rank", 4) if (j, g) == (1, 1) else 4, 1.0,
                                        *[0x100000 * (1 + 16 * (2 * j + g) + u) for u in range(8)]))
    if bad.get("drop_last"):
        segs = segs[:3]
    prob = M.mlora_problem(15, 128, d_out, bad.get("dtype", M.MLORA_BF16), M.MLORA_PLAN_HOST_ONLY)
    assert _status_of(lambda: M.mlora_plan_destroy(M.mlora_plan_grouped(prob, groups, segs)[0])) == status


def test_grouped_pair_dh_pieces_stay_in_their_slices():
    """A shared-input pack on CTA pairs: job 0's window (ranks 256, 64, 64: six chunks) makes a pair
    item of chunks 0-3 that holds only q columns and one of chunks 4-5 with only k / v columns;
    their dH K ranges are those projections' d_out slices (0..31 and 32..63), and each item's
    pieces tile exactly its range."""
    from adapter_gemm_packed_gb300.layer import host_plan_grouped
    plan, _ = host_plan_grouped(4096, [2048, 1024, 1024], [[256, 64, 64], [32, 16, 16], [16, 8, 8]],
                                [256, 200, 250], flags=M.MLORA_WINDOW_PAIRS)
    try:
        shrink, dh = _pair_entries(plan)
    finally:
        M.mlora_plan_destroy(plan)
    whole = {(0, 0): (0, 32), (0, 4): (32, 32), (1, 6): (0, 64), (2, 7): (0, 64)}
    _check_pair_pieces(shrink, lambda t, q: (0, 64))
    groups = _check_pair_pieces(dh, lambda t, q: whole[(t, q)])
    assert set(groups) == set(whole) and all(rows[0][7] >= 2 for rows in groups.values())


def test_grouped_dh_items_read_only_their_projections_slices():
    """A dH item of a shared-input pack streams only the d_out slices covered by the adapters
    that own its chunks' columns: chunks holding only k columns read only k's slice of dY."""
    from adapter_gemm_packed_gb300.layer import host_plan_grouped
    widths = [4096, 1024, 1024]
    ranks_jg = [[128, 128, 128], [8, 8, 8]]
    plan, _ = host_plan_grouped(512, widths, ranks_jg, [256, 256])
    try:
        ad = _describe(plan, M.MLORA_Q_ADAPTERS).reshape(-1, 5)
        win = _describe(plan, M.MLORA_Q_WINDOW).reshape(-1, 5)
    finally:
        M.mlora_plan_destroy(plan)
    for t, q0, nq, kb0, nkb in win:
        lo, hi = 1 << 30, 0
        for job, c0, r, o_lo, o_hi in ad:
            if c0 < (q0 + nq) * 64 and c0 + r > q0 * 64:
                lo, hi = min(lo, o_lo), max(hi, o_hi)
        assert (kb0, nkb) == (lo // 64, -(-hi // 64) - lo // 64)
    # job 0 (rank 128 per projection) spans chunks 0-5: q in 0-1, k in 2-3, v in 4-5
    by_q0 = {q0: (kb0, nkb) for t, q0, nq, kb0, nkb in win if t == 0}
    assert by_q0[0] == (0, 64) and by_q0[2] == (64, 16) and by_q0[4] == (80, 16)


# ---------------------------------------------------------------- shrink / dH on CTA pairs

@pytest.mark.parametrize("name", ["ragged", "tiny_segments", "one_token", "qproj", "many_small"])
def test_pair_window_items(name):
    """Pair items cover each 256-token pair's shared chunk range exactly once, in groups of at most
    four chunks padded to an even count (the padding chunk sits right after the range), in both
    products' schedules; the shrink reads all of d_in and dH all of d_out (one projection)."""
    d_in, d_out, ranks, ns = _case(name)
    plan, _ = host_plan(d_in, d_out, ranks, ns)
    try:
        mt = _describe(plan, M.MLORA_Q_MTILES).reshape(-1, 5)
        shrink, dh = _pair_entries(plan)
    finally:
        M.mlora_plan_destroy(plan)
    for items, K in ((shrink, -(-d_in // 64)), (dh, -(-d_out // 64))):
        groups = _check_pair_pieces(items, lambda t, q: (0, K))
        for p in range((len(mt) + 1) // 2):
            q_lo, nch = mt[2 * p, 2], mt[2 * p, 3]
            got = []
            for (tile, q0), rows in sorted(groups.items()):
                if tile == p:
                    assert rows[0][3] in (2, 4)
                    got.extend(range(q0, q0 + rows[0][3]))
            assert got[:nch] == list(range(q_lo, q_lo + nch)) and len(got) - nch in (0, 1)


def _pair_loads(items):
    """Modelled per-pair load of one product's CTA-pair schedule, as the planner counts it (KB
    per CTA)."""
    loads = np.zeros(items[:, 0].max() + 1)
    for row in items:
        nq, S = row[3], row[7]
        loads[row[0]] += row[5] * (16 + 8 * (nq // 2)) + 32 + 16 * nq + (64 * nq if S > 1 else 0)
    return loads


@pytest.mark.parametrize("name, bound", [("many_small", 1.12), ("mlp_up", 1.12), ("qproj", 1.0),
                                         ("layer_q", 1.05), ("layer_gate", 1.05), ("layer_down", 1.05)])
def test_pair_schedule_balances_the_pairs(name, bound):
    """Each product's per-pair lists (host plans assume 148 SMs: 74 pairs) keep every pair near the
    average modelled load: whole items first while they fit, then the rest cut along K across the
    least loaded pairs.  A round robin left these packs at 1.10-1.41x the average (the
    many-small-jobs pack 1.37, mlp_up 1.41, q_proj's 64 items on 64 of 74 pairs).  q_proj stays
    whole: cutting its 64 items over 74 pairs would save less than the pieces' partial sums cost."""
    if name.startswith("layer_"):
        wl = W.llama8b_layer(["q", "k", "v", "o", "gate", "up", "down"].index(name[6:]))
        d_in, d_out, ranks, ns = wl.d_in, wl.d_out, wl.ranks, wl.n_tokens
    else:
        d_in, d_out, ranks, ns = _case(name)
    plan, _ = host_plan(d_in, d_out, ranks, ns, flags=M.MLORA_WINDOW_PAIRS)
    try:
        shrink, dh = _pair_entries(plan)
    finally:
        M.mlora_plan_destroy(plan)
    for items, K in ((shrink, -(-d_in // 64)), (dh, -(-d_out // 64))):
        _check_pair_pieces(items, lambda t, q: (0, K))
        loads = _pair_loads(items)
        assert len(loads) <= 74
        if name == "qproj":
            assert (items[:, 7] == 1).all() and len(loads) == len(items) == 64
        else:
            assert len(loads) == 74 and (items[:, 7] > 1).any()
            assert loads.max() <= bound * loads.sum() / 74


def test_pair_schedule_hand_worked():
    """Three items of 64 K slices each way (d_in = d_out = 4096, one 256-token pair per job, two
    chunks) on 74 pairs: an item costs 64 x 24 + 32 + 32 = 1600 KB per CTA and the average over 74
    pairs is far below one item, so the greedy phase takes none and McNaughton's rule cuts every
    item into pieces of the smallest share, 16 of its 64 slices: four pieces each, on 12 distinct
    pairs, in both products."""
    plan, _ = host_plan(4096, 4096, [128, 128, 128], [256, 256, 256], flags=M.MLORA_WINDOW_PAIRS)
    try:
        shrink, dh = _pair_entries(plan)
    finally:
        M.mlora_plan_destroy(plan)
    for items in (shrink, dh):
        groups = _check_pair_pieces(items, lambda t, q: (0, 64))
        assert len(groups) == 3
        for rows in groups.values():
            assert [(r[4], r[5]) for r in rows] == [(0, 16), (16, 16), (32, 16), (48, 16)]
        assert sorted(items[:, 0]) == list(range(12))


def test_window_engine_choice():
    """Pairs when the token tiles' windows average more than 1.25 chunks, unless a flag says."""
    def pairs(ranks, ns, flags=0):
        plan, _ = host_plan(512, 256, ranks, ns, flags=flags)
        try:
            return _describe(plan, M.MLORA_Q_WINDOW_PAIRS)[0] == 1
        finally:
            M.mlora_plan_destroy(plan)
    assert not pairs([8, 8], [1024, 1024])                   # both windows in chunk 0: one chunk per tile
    assert pairs([8, 64], [1024, 1024])                      # the second window [16, 80) spans two chunks
    assert pairs([128, 256], [1024, 1024])                   # 2 and 4 chunks per tile
    assert pairs([8, 8], [1024, 1024], M.MLORA_WINDOW_PAIRS)
    assert not pairs([128, 256], [1024, 1024], M.MLORA_WINDOW_SINGLE)


def _gemm_list(plan, what):
    v = M.mlora_plan_describe(plan, what)
    head, items = v[:5], v[5:]
    return head, [tuple(items[i:i + 3]) for i in range(0, len(items), 3)]


@pytest.mark.parametrize("d_in,d_out,n_tokens", [
    (4096, 4096, [2048] * 8),            # q_proj: the whole weight fits the L2 budget
    (4096, 14336, [1024] * 20),          # MLP up / gate
    (14336, 4096, [1024] * 20),          # down: K = 14336, small groups
    (512, 384, [300, 100, 150, 77]),     # ragged, less than one wave (split tail)
    (1024, 640, [130, 500, 333]),        # odd number of 128-token tiles
])
def test_base_gemm_work_list_covers_every_output_tile_once(d_in, d_out, n_tokens):
    """The CTA-pair GEMMs' work list, decoded exactly as the kernels decode it, covers every
    (256-token pair, output column) once, with full tiles first and half tiles only in a split
    last wave; the raster keeps its resident panels inside the L2 budget."""
    plan, _ = host_plan(d_in, d_out, [16] * len(n_tokens), n_tokens)
    try:
        for what, K, width in ((M.MLORA_Q_GEMM_FWD, d_in, d_out), (M.MLORA_Q_GEMM_BWD, d_out, d_in)):
            (raster_n, group, n_items, n_full, n_pairs), items = _gemm_list(plan, what)
            assert len(items) == n_items and 1 <= n_pairs <= 74
            m_pairs = (-(-sum(n_tokens) // 128) + 1) // 2
            n_tiles = -(-width // 256)
            cover = np.zeros((m_pairs, n_tiles * 2), dtype=int)     # 128-column halves
            for i, (mp, col0, w) in enumerate(items):
                assert (w == 256) == (i < n_full) and col0 % 128 == 0
                cover[mp, col0 // 128:(col0 + w) // 128] += 1
            assert (cover == 1).all()
            # resident panels: group x 256 x K bf16 within the 48 MiB budget (or a group of one)
            assert raster_n in (0, 1) and 1 <= group <= (n_tiles if raster_n else m_pairs)
            assert group == 1 or group * 256 * K * 2 <= 48 << 20
    finally:
        M.mlora_plan_destroy(plan)


def test_base_gemm_raster_keeps_the_weight_resident():
    """q_proj: the whole weight (16 output tiles, 32 MiB) is one resident group; the MLP's 56 output
    tiles split into three equal groups of 19; the down projection's K = 14336 panels allow 6."""
    for d_in, d_out, want in ((4096, 4096, (1, 16)), (4096, 14336, (1, 19)), (14336, 4096, (1, 6))):
        plan, _ = host_plan(d_in, d_out, [16] * 20, [1024] * 20)
        try:
            (raster_n, group, *_), _ = _gemm_list(plan, M.MLORA_Q_GEMM_FWD)
            assert (raster_n, group) == want
        finally:
            M.mlora_plan_destroy(plan)


def test_wgrad_schedule_balances_mixed_job_lengths():
    """dA / dB on the Llama-3-8B k projection's pack (32 jobs of 1-8 sequences of 1024 tokens, d_out
    1024: four 256-row blocks, so a few long jobs' items would dominate a one-item-per-CTA
    schedule): the wrap-around schedule cuts the long items into parts of at least 256 tokens and
    no CTA's modelled load is more than 10 % above the mean (the planner's cost: 32 + 8 nq KB per
    64-token half-tile; per piece 32 plus 1 per column of the job's rank window inside the piece's
    chunks, and 128 nq more for a piece of a cut item)."""
    part = W.llama8b_layer_all().parts[1]
    assert (part.d_in, part.d_out) == (4096, 1024)
    plan, _ = host_plan(part.d_in, part.d_out, part.ranks, part.n_tokens)
    try:
        got = [_describe(plan, w).reshape(-1, 9) for w in (M.MLORA_Q_WGRAD_A, M.MLORA_Q_WGRAD_B)]
        cols = _describe(plan, M.MLORA_Q_COLUMNS).reshape(-1, 2)
    finally:
        M.mlora_plan_destroy(plan)
    for items in got:
        load = np.zeros(items[:, 8].max() + 1)
        for _, j, ga, gb, q0, nq, _, parts, c in items:
            inside = max(0, min(cols[j, 0] + part.ranks[j], 64 * (q0 + nq)) - max(cols[j, 0], 64 * q0))
            load[c] += (gb - ga) * (32 + 8 * nq) + 32 + inside + (128 * nq if parts > 1 else 0)
        assert len(load) == 148                      # a host plan models a 148-SM part
        assert load.max() <= 1.10 * load.mean()
    assert got[1][:, 7].max() >= 2                   # dB: long jobs' items were cut
