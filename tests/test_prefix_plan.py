"""Host planner of the shared-prefix (cascade) attention, checked by brute force.

"Faster fuzzy minds" ("When scheduler does the work"): with a radix prefix
cache, requests sharing a prompt prefix point at the same physical pages.
rlt_plan_prefix must find, for every request, exactly the leading 128-token
tiles it shares page-for-page with at least one other request, group them into
segments of one member set, and number each request's partial slots 0..n-1.
The brute-force reference compares every pair of requests tile by tile.
"""
import numpy as np
import pytest

import paged_kv_looped_gb300 as rlt
import workloads as W

TILE = 128


def copies(members, G):
    """Copies of a segment's query rows in the tensor-core kernel: its first member block's
    rows spread over the four TMEM lane quarters (4 copies of <= 8 rows, 2 of <= 64)."""
    rows = min(members, 128 // G) * G
    return 4 if rows <= 8 else 2 if rows <= 64 else 1


def tile_key(pt, b, t, ps):
    tok = t * TILE
    if ps <= TILE:
        return tuple(pt[b, (tok + j * ps) // ps] for j in range(TILE // ps))
    return (pt[b, tok // ps], tok % ps)


def common_tiles(pt, sl, ps, b, c):
    n = min(int(sl[b]) // TILE, int(sl[c]) // TILE)
    t = 0
    while t < n and tile_key(pt, b, t, ps) == tile_key(pt, c, t, ps):
        t += 1
    return t


def common_pages(pt, sl, ps, b, c):
    """Leading pages b and c map alike, each page whole inside both requests."""
    n = min(int(sl[b]), int(sl[c])) // ps
    j = 0
    while j < n and pt[b, j] == pt[c, j]:
        j += 1
    return j


def check_plan(case, chunk_tiles=4, G=1, exact_pages=True):
    """exact_pages: every request's pages shared with others form one chain (a radix tree over
    one prompt), so its covered prefix is exactly its longest page-for-page run with another
    request; otherwise it lies between its longest whole-tile run and that."""
    pt, sl, ps = case.page_table, case.seq_lens, case.page_size
    plan = rlt.rlt_plan_prefix(pt, sl, ps, chunk_tiles, False, G)
    per_block = 128 // G
    assert plan.max_rest_len == max(int(sl[b]) - int(plan.request_prefix[b, 0]) for b in range(case.batch))
    B = case.batch
    cp = np.zeros((B, B), int)
    cpg = np.zeros((B, B), int)
    for b in range(B):
        for c in range(B):
            if b != c:
                cp[b, c] = common_tiles(pt, sl, ps, b, c)
                cpg[b, c] = common_pages(pt, sl, ps, b, c)
    # each request's covered prefix: its longest shared run of whole 128-token tiles with any
    # other request, continued page by page (pages below a tile) while it still shares them
    for b in range(B):
        cov = int(plan.request_prefix[b, 0])
        tiles = TILE * (cp[b].max() if B > 1 else 0)
        pages = ps * (cpg[b].max() if B > 1 else 0) if ps < TILE else tiles
        assert cov % min(ps, TILE) == 0 and tiles <= cov <= max(tiles, pages), b
        if exact_pages:
            assert cov == max(tiles, pages), b
    # segments: at tile t the members whose limit lies past t share its pages below their
    # limit with the page row
    seg_of_tile = {}
    for s in range(plan.num_segments):
        first, n, base, mb, mc, row, end, work = plan.segments[s]
        assert (first + n - 1) * TILE < end <= (first + n) * TILE
        mem = plan.members[mb: mb + mc]
        lim = plan.member_limit[mb: mb + mc]
        assert mc >= 2 and row in mem and lim[-1] == end
        assert list(lim) == sorted(lim) and len(set(mem)) == mc
        assert all(first * TILE < x <= end and x % min(ps, TILE) == 0 for x in lim)
        if len(set(lim)) > 1:
            assert mc <= per_block                 # a merged chain fits one member block
        for t in range(first, first + n):
            live = {int(b) for b, x in zip(mem, lim) if x > t * TILE}
            # every request sharing the row's whole tile t is a live member
            assert {c for c in range(B) if c != row and cp[row, c] >= t + 1} <= live, (s, t)
            for b, x in zip(mem, lim):
                if x <= t * TILE:
                    continue
                if ps >= TILE:
                    assert tile_key(pt, b, t, ps) == tile_key(pt, row, t, ps)
                else:
                    for j in range(t * TILE // ps, min(x, (t + 1) * TILE) // ps):
                        assert pt[b, j] == pt[row, j], (s, t, b, j)
                seg_of_tile.setdefault(int(b), []).append((t, s))
    # along each request's path: tiles 0..n-1 in order, partial slots contiguous from 0
    for b in range(B):
        tiles = sorted(seg_of_tile.get(b, []))
        assert [t for t, _ in tiles] == list(range(-(-int(plan.request_prefix[b, 0]) // TILE)))
        slots = []
        for s in dict.fromkeys(s for _, s in tiles):
            first, n, base = plan.segments[s][:3]
            slots += list(range(base, base + -(-n // chunk_tiles) * copies(int(plan.segments[s][4]), G)))
        assert slots == list(range(len(slots))) and len(slots) == plan.request_prefix[b, 1]
    assert plan.max_prefix_slots == (plan.request_prefix[:, 1].max() if B else 0)
    # work units: chunks x member blocks per segment, numbered in segment order
    units = 0
    for s in range(plan.num_segments):
        assert plan.segments[s][7] == units
        units += -(-int(plan.segments[s][1]) // chunk_tiles) * -(-int(plan.segments[s][4]) // per_block)
    assert plan.work_units == units
    return plan


@pytest.mark.parametrize("name", ["huginn", "longctx", "ouro", "tiny"])
def test_plan_of_workloads(name):
    case = W.config(name)
    plan = check_plan(case, G=case.group)
    if name in ("huginn", "longctx"):
        # one prompt chain that requests leave one by one: a single segment with limits
        assert plan.num_segments == 1
        assert plan.segments[0][4] == case.batch
    else:
        assert plan.num_segments == 0              # nothing shared


@pytest.mark.parametrize("G", [1, 8, 32, 64])
def test_chain_merge_respects_member_blocks(G):
    # 5 requests on one prompt chain, leaving it at different tiles: the chain is merged
    # from the first link whose members fit one block of 128 / G; links with more
    # members stay segments of their own, every member reading all their tiles
    case = W.custom(B=5, Hq=8, Hkv=8, D=128, ps=16, seq_lens=[3000, 2600, 4100, 1700, 2222], shared_frac=0.8,
                    seed=11)
    # (limits go on page by page only in segments of one member block)
    plan = check_plan(case, 2, G, exact_pages=5 <= 128 // G)
    if 5 <= 128 // G:
        assert plan.num_segments == 1
    else:
        assert plan.num_segments > 1
        for s in range(plan.num_segments):
            mb, mc = plan.segments[s][3], plan.segments[s][4]
            if mc > 128 // G:
                assert len(set(plan.member_limit[mb: mb + mc])) == 1


@pytest.mark.parametrize("chunk_tiles", [1, 3, 32])
def test_plan_chunking(chunk_tiles):
    check_plan(W.config("huginn"), chunk_tiles)


def test_plan_of_two_trees_and_loners():
    # requests 0-3 share one 700-token prompt, 4-6 another, 7 and 8 share nothing
    rng = np.random.default_rng(3)
    ps = 16
    lens = [900, 1300, 751, 2000, 1500, 1600, 1501, 999, 3000]
    P = 2000
    perm = iter(rng.permutation(P))
    max_pages = -(-max(lens) // ps)
    pt = np.full((len(lens), max_pages), -1, np.int32)
    a = [next(perm) for _ in range(700 // ps)]
    bprefix = [next(perm) for _ in range(1400 // ps)]
    for r, L in enumerate(lens):
        n = -(-L // ps)
        shared = a if r < 4 else bprefix if r < 7 else []
        k = min(len(shared), n - 1)
        pt[r, :k] = shared[:k]
        pt[r, k:n] = [next(perm) for _ in range(n - k)]
    case = W.PagedCase(name="trees", num_layers=1, num_planes=1, recurrent=np.zeros(1, np.uint8), batch=len(lens),
                       num_q_heads=8, num_kv_heads=8, head_dim=128, page_size=ps, num_pages=P,
                       seq_lens=np.array(lens, np.int32), page_table=pt, new_slots=np.zeros(len(lens), np.int64))
    plan = check_plan(case)
    assert plan.request_prefix[7, 0] == 0 and plan.request_prefix[8, 0] == 0
    # the shared prompts end mid-tile: every whole page of them is covered (700 tokens -> 43
    # pages of 16 = 5 whole tiles and 3 pages; 1400 -> 87 pages = 10 tiles and 7 pages)
    assert plan.request_prefix[0, 0] == 43 * ps
    assert plan.request_prefix[4, 0] == 87 * ps


@pytest.mark.parametrize("ps", [32, 64, 128, 256])
def test_plan_page_sizes(ps):
    case = W.custom(B=5, Hq=8, Hkv=8, D=128, ps=ps, seq_lens=[3000, 2600, 4100, 1700, 2222], shared_frac=0.8,
                    seed=ps)
    check_plan(case)


def test_plan_rejects_page_size_not_aligned_to_tiles():
    case = W.custom(B=2, Hq=2, Hkv=2, D=128, ps=48, seq_lens=[300, 300], shared_frac=0.5)
    with pytest.raises(rlt.RltError):
        rlt.rlt_plan_prefix(case.page_table, case.seq_lens, 48)


@pytest.mark.parametrize("name", ["huginn", "longctx", "gqa", "tiny"])
def test_private_tails_cover_every_token(name):
    case = W.config(name)
    pt, sl, ps = case.page_table, case.seq_lens, case.page_size
    shared = rlt.rlt_plan_prefix(pt, sl, ps, 4)
    plan = rlt.rlt_plan_prefix(pt, sl, ps, 4, private_tails=True)
    assert plan.max_rest_len == 0
    assert np.array_equal(plan.request_prefix[:, 0], sl)
    # the shared segments are those of the plan without tails, cut back to whole tiles (a
    # tail starts on a tile); one tail per request follows them
    n = shared.num_segments
    assert np.array_equal(plan.segments[:n, [0, 3, 4, 5]], shared.segments[:, [0, 3, 4, 5]])
    assert np.all(plan.segments[:n, 6] % TILE == 0) and np.all(plan.segments[:n, 6] <= shared.segments[:, 6])
    covered = {}                                  # each request's shared tokens, whole tiles
    for first, ntiles, base, mb, mc, row, end, work in plan.segments[:n]:
        for b, lim in zip(plan.members[mb: mb + mc], plan.member_limit[mb: mb + mc]):
            covered[int(b)] = max(covered.get(int(b), 0), int(lim))
            assert lim % TILE == 0
    tails = plan.segments[n:]
    assert len(tails) == sum(1 for b in range(case.batch) if sl[b] > covered.get(b, 0))
    for first, ntiles, base, mb, mc, row, end, work in tails:
        b = int(plan.members[mb])
        assert mc == 1 and row == b and end == sl[b]
        assert first * TILE == covered.get(b, 0) == shared.request_prefix[b, 0] // TILE * TILE
        assert (first + ntiles) * TILE >= end > (first + ntiles - 1) * TILE
        assert plan.request_prefix[b, 1] == base + -(-ntiles // 4) * copies(1, 1)


@pytest.mark.parametrize("G,chunk_tiles", [(1, 1), (4, 2), (8, 3)])
def test_extend_plan_by_brute_force(G, chunk_tiles):
    lens = [300, 50, 1000, 128, 129, 7]
    new = [40, 50, 0, 128, 1, 7]
    plan = rlt.rlt_plan_extend(lens, new, 16, chunk_tiles, G)
    per_block = 128 // G
    ct = chunk_tiles * TILE
    assert plan.num_rows == sum(new) and plan.num_segments == sum(1 for n in new if n)
    row, units, s = 0, 0, 0
    for b, (L, n) in enumerate(zip(lens, new)):
        if n == 0:
            continue
        first, tiles, base, mb, mc, page_row, end, work = plan.segments[s]
        assert (first, tiles, base, mc, page_row, end, work) == (0, -(-L // TILE), 0, n, b, L, units)
        assert mb == row
        for i in range(n):
            assert plan.members[row + i] == row + i                     # packed q row of the token
            assert plan.member_limit[row + i] == L - n + i + 1          # causal key count
            assert plan.row_len[row + i] == L - n + i + 1
            block_last = min(n, (i // per_block + 1) * per_block) - 1
            assert plan.row_prefix[row + i, 0] == L - n + i + 1
            assert plan.row_prefix[row + i, 1] == -(-(L - n + block_last + 1) // ct) * copies(n, G)
        units += -(-tiles // chunk_tiles) * -(-n // per_block)
        row += n
        s += 1
    assert plan.work_units == units
    assert plan.max_slots == max(-(-(-(-L // TILE)) // chunk_tiles) * copies(n, G) for L, n in zip(lens, new) if n)


def test_extend_plan_rejects_more_new_tokens_than_the_sequence():
    with pytest.raises(rlt.RltError):
        rlt.rlt_plan_extend([10], [11], 16)


# ---------------------------------------------------------------- work-item size

def busiest_cta(case, chunk, tails, ctas, sub_us=1.55, run_us=4.7):
    """Brute-force estimate of the tensor-core kernel's busiest CTA for one chunk size: items
    (kv head, segment, member block, chunk) in the kernel's order, contiguous equal-count runs of
    them per CTA, each CTA paying its tiles and one hand-over per change of (head, segment, block)."""
    plan = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, chunk, tails, case.group)
    per_block = 128 // case.group
    units = []
    for si, seg in enumerate(plan.segments):
        n, mc = int(seg[1]), int(seg[4])
        for mb in range(-(-mc // per_block)):
            for c in range(max(1, -(-n // chunk))):
                units.append((si, mb, min(chunk, n - c * chunk)))
    items = [(g,) + u for g in range(case.num_kv_heads) for u in units]
    n = len(items)
    ctas = min(ctas, n)
    worst = 0.0
    for c in range(ctas):
        run, runs, tiles = None, 0, 0
        for it in items[c * n // ctas:(c + 1) * n // ctas]:
            tiles += it[3]
            if it[:3] != run:
                run, runs = it[:3], runs + 1
        worst = max(worst, tiles * sub_us + runs * run_us)
    return worst


@pytest.mark.parametrize("name,ctas", [("longctx", 152), ("longctx", 100), ("huginn", 152), ("huginn", 37)])
def test_choose_chunk_tiles_private_tails_minimises_the_busiest_cta(name, ctas):
    case = W.config(name)
    got = rlt.rlt_choose_chunk_tiles(case.page_table, case.seq_lens, case.page_size, case.group, True,
                                     case.num_kv_heads, ctas)
    costs = {c: busiest_cta(case, c, True, ctas) for c in range(4, 17)}
    best = min(costs.values())
    assert costs[got] <= best + 1e-6
    # the larger on a tie, no larger than the longest segment
    longest = max(int(s[1]) for s in rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, 1, True,
                                                         case.group).segments)
    assert got == min(max(c for c, v in costs.items() if v <= best + 1e-6), longest)


@pytest.mark.parametrize("G", [1, 4, 8])
def test_choose_chunk_tiles_custom_batches(G):
    case = W.custom(B=7, Hq=8 * G, Hkv=8, D=128, ps=16, seq_lens=[3000, 2600, 4100, 1700, 2222, 900, 5000],
                    shared_frac=0.8, seed=40 + G)
    for ctas in (19, 152):
        got = rlt.rlt_choose_chunk_tiles(case.page_table, case.seq_lens, case.page_size, G, True, 8, ctas)
        costs = {c: busiest_cta(case, c, True, ctas) for c in range(4, 17)}
        longest = max(int(s[1]) for s in rlt.rlt_plan_prefix(case.page_table, case.seq_lens, 16, 1, True, G).segments)
        best = min(costs.values())
        want = min(max(c for c, v in costs.items() if v <= best + 1e-6), longest)
        assert got == want
        # without private tails: the chunk (2..16, at most the longest segment) with the fewest
        # sub-tiles on the busiest tensor-core CTA when the CTAs are the SMs' share the call
        # gives that kernel beside the split-K rest, items spread evenly; the larger on a tie
        got2 = rlt.rlt_choose_chunk_tiles(case.page_table, case.seq_lens, case.page_size, G, False, 8, ctas)
        p1 = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, 16, 1, False, G)
        longest2 = max([int(s[1]) for s in p1.segments] + [1])
        loads = {}
        for c in range(2, min(16, longest2) + 1):
            pc = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, 16, c, False, G)
            items = 8 * pc.work_units
            share = min(1.0, 2.25 * pc.work_units * c * 128 / (pc.work_units * c * 128 + 0.75 * case.batch
                                                                 * pc.max_rest_len))
            n = max(1, min(ctas - 1, int(np.ceil(ctas * share))))
            per = -(-items // n)
            n = max(1, -(-items // per))
            loads[c] = -(-items // n) * c
        assert got2 == max(c for c, v in loads.items() if v == min(loads.values()))


def test_choose_chunk_tiles_rejects_bad_arguments():
    case = W.config("tiny")
    with pytest.raises(rlt.RltError):
        rlt.rlt_choose_chunk_tiles(case.page_table, case.seq_lens, case.page_size, 1, True, 0, 152)
    with pytest.raises(rlt.RltError):
        rlt.rlt_choose_chunk_tiles(case.page_table, case.seq_lens, 48, 1, True, 2, 152)
