"""Host-side tests of libpkv (no GPU): exports, block pool, lowering, work list, scheduler.

The library's host code is checked against the pages' worked examples and
against the oracle (slot mapping recomputed independently; the scheduler's
plans against the oracle's own replay of the same trace).
"""

import ctypes

import numpy as np
import pytest

import oracle
from continuous_batching_paged_pkv_gb300 import binding as B
from continuous_batching_paged_pkv_gb300 import build as libbuild
from continuous_batching_paged_pkv_gb300 import scheduler as S
from continuous_batching_paged_pkv_gb300 import workloads as W
from oracle import churn
from tests.conftest import golden


@pytest.fixture(scope="module", autouse=True)
def built():
    libbuild.build()


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(B.LIB_PATH)
    names = B.declared_functions()
    assert {"pkv_cache_write", "pkv_attention", "pkv_plan_lower", "pkv_plan_work"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/pkv.h but not exported"
    assert B.pkv_version() > 0
    assert B.pkv_status_string(7) == "not enough free KV blocks"


# ---- block pool ---------------------------------------------------------------

def test_pool_block_table_example_from_the_page():
    """A [7,2,9,4], B [1,8], free [0,3,5,6]; B finishes; its blocks go to a new request; A stays."""
    g = golden("block_table_example.json")
    pool = B.Pool(10, 16, 3, 4)
    pool.admit_blocks(0, g["tables"]["A"])
    pool.admit_blocks(1, g["tables"]["B"])
    assert pool.stats().free_blocks == len(g["free_pool"])
    before = pool.block_tables()[0].copy()
    pool.release(1)
    assert pool.admit(2, 2 * 16) == B.PKV_OK
    bt = pool.block_tables()
    assert sorted(bt[2, :2]) == sorted(g["released_when_B_finishes"])
    assert list(bt[2, :2]) == g["tables"]["B"]  # last released first block is on top
    np.testing.assert_array_equal(bt[0], before)


def test_pool_admission_is_all_or_nothing():
    pool = B.Pool(8, 16, 4, 8)
    assert pool.admit(0, 5 * 16) == B.PKV_OK
    before = pool.block_tables().copy()
    assert pool.admit(1, 4 * 16) == B.PKV_ERR_NO_BLOCKS
    assert pool.stats().free_blocks == 3 and pool.slot_blocks(1) == -1
    np.testing.assert_array_equal(pool.block_tables(), before)
    assert pool.admit(1, 3 * 16) == B.PKV_OK
    assert pool.stats().free_blocks == 0


def test_pool_rejects_double_release_and_owned_blocks():
    pool = B.Pool(8, 16, 2, 8)
    pool.admit_blocks(0, [3, 5])
    with pytest.raises(B.PkvError):
        pool.admit_blocks(1, [5])
    pool.release(0)
    with pytest.raises(B.PkvError):
        pool.release(0)


def test_pool_each_block_owned_once():
    rng = np.random.default_rng(0)
    pool = B.Pool(200, 16, 16, 64, free_order=rng.permutation(200).astype(np.int32))
    live = set()
    for step in range(300):
        slot = int(rng.integers(16))
        if slot in live and rng.random() < 0.5:
            pool.release(slot)
            live.discard(slot)
        elif slot not in live:
            if pool.admit(slot, int(rng.integers(1, 400))) == B.PKV_OK:
                live.add(slot)
        bt = pool.block_tables()
        used = bt[bt >= 0]
        assert len(used) == len(set(used.tolist()))
        st = pool.stats()
        assert st.free_blocks + st.owned_blocks == 200


# ---- prefix adoption and copy-on-write -------------------------------------------

def _check_accounting(pool, total):
    st = pool.stats()
    assert st.free_blocks + st.owned_blocks == total
    bt = pool.block_tables()
    used = bt[bt >= 0]
    for b in np.unique(used):
        assert pool.block_refs(int(b)) == int((used == b).sum())


def test_adopt_shares_blocks_and_copies_on_first_append():
    """mlxcel manual, §Paged KV cache and prefix sharing: adopt by reference, copy on divergence."""
    pool = B.Pool(64, 16, 4, 16)
    assert pool.admit(0, 100) == B.PKV_OK
    pool.lower([(0, 100)])
    a_blocks = pool.block_tables()[0, :7].copy()
    free0 = pool.stats().free_blocks
    # B adopts 70 tokens (blocks 0..4, the last one partly filled) and reserves room for 90
    assert pool.adopt(1, 0, 70, 90) == B.PKV_OK
    assert pool.slot_length(1) == 70 and pool.slot_blocks(1) == 6
    assert list(pool.block_tables()[1, :5]) == list(a_blocks[:5])
    assert pool.stats().free_blocks == free0 - 1 and pool.stats().shared_blocks == 5
    assert [pool.block_refs(int(b)) for b in a_blocks[:6]] == [2, 2, 2, 2, 2, 1]
    _check_accounting(pool, 64)
    # B's first append lands in shared block 4: it gets a copy, A keeps the original
    low = pool.lower([(1, 20)])
    cp = pool.take_copies()
    b_blocks = pool.block_tables()[1]
    assert cp.shape == (1, 2) and cp[0, 0] == a_blocks[4] and cp[0, 1] == b_blocks[4] != a_blocks[4]
    assert pool.block_refs(int(a_blocks[4])) == 1 and pool.block_refs(int(b_blocks[4])) == 1
    pos = np.arange(70, 90)
    assert np.array_equal(low.slot_mapping, b_blocks[pos // 16].astype(np.int64) * 16 + pos % 16)
    assert pool.take_copies().shape == (0, 2)  # handed over once
    # later appends into B's own blocks copy nothing; A's appends never touch B's blocks
    pool.lower([(1, 1), (0, 1)])
    assert pool.take_copies().shape == (0, 2)
    assert list(pool.block_tables()[0, :7]) == list(a_blocks)
    _check_accounting(pool, 64)


def test_adopt_on_a_block_boundary_never_copies():
    pool = B.Pool(64, 16, 4, 16)
    assert pool.admit(0, 100) == B.PKV_OK
    pool.lower([(0, 100)])
    assert pool.adopt(2, 0, 64, 0) == B.PKV_OK  # four full blocks, no reserve: the next block is grown
    pool.lower([(2, 3)])
    assert pool.take_copies().shape == (0, 2) and pool.slot_blocks(2) == 5
    _check_accounting(pool, 64)


def test_donor_append_into_a_shared_block_copies_for_the_donor():
    pool = B.Pool(64, 16, 4, 16)
    assert pool.admit(0, 100) == B.PKV_OK
    pool.lower([(0, 100)])
    a6 = int(pool.block_tables()[0, 6])
    assert pool.adopt(1, 0, 100, 0) == B.PKV_OK  # shares all seven blocks, the last partly filled
    pool.lower([(0, 1)])
    cp = pool.take_copies()
    assert cp.tolist() == [[a6, int(pool.block_tables()[0, 6])]] and pool.block_tables()[1, 6] == a6
    _check_accounting(pool, 64)


def test_release_keeps_shared_blocks_until_the_last_holder():
    pool = B.Pool(32, 16, 4, 8)
    assert pool.admit(0, 64) == B.PKV_OK
    pool.lower([(0, 64)])
    assert pool.adopt(1, 0, 64, 64) == B.PKV_OK  # a prefix-cache slot holding A's four blocks
    shared = pool.block_tables()[0, :4].copy()
    pool.release(0)
    assert pool.stats().free_blocks == 28 and all(pool.block_refs(int(b)) == 1 for b in shared)
    # a new request adopts from the cache slot, then the cache entry is evicted
    assert pool.adopt(2, 1, 40, 80) == B.PKV_OK
    pool.release(1)
    assert pool.stats().free_blocks == 32 - 5  # slot 2: prefix blocks 0..2 and two fresh blocks
    assert [pool.block_refs(int(b)) for b in shared] == [1, 1, 1, 0]
    pool.release(2)
    assert pool.stats().free_blocks == 32 and pool.stats().shared_blocks == 0
    _check_accounting(pool, 32)


def test_adopt_is_all_or_nothing_and_validated():
    pool = B.Pool(8, 16, 4, 8)
    assert pool.admit(0, 64) == B.PKV_OK
    pool.lower([(0, 40)])
    before = pool.block_tables().copy()
    assert pool.adopt(1, 0, 40, 16 * 8) == B.PKV_ERR_NO_BLOCKS  # needs 5 fresh, 4 free
    assert np.array_equal(pool.block_tables(), before) and pool.slot_length(1) == -1
    assert [pool.block_refs(int(b)) for b in before[0, :4]] == [1, 1, 1, 1]
    for args in ((1, 0, 41, 0), (1, 3, 10, 0), (0, 0, 10, 0)):  # past the donor, donor not live, slot live
        assert pool.adopt(*args) != B.PKV_OK
    # a lowering that needs a copy counts the copy's block: all or nothing
    assert pool.adopt(1, 0, 40, 0) == B.PKV_OK
    assert pool.admit(2, 64) == B.PKV_OK  # takes the last four free blocks
    with pytest.raises(B.PkvError):
        pool.lower([(1, 1)])
    assert pool.slot_length(1) == 40 and pool.take_copies().shape == (0, 2)
    _check_accounting(pool, 8)


# ---- lowering ----------------------------------------------------------------

def test_lowering_packing_example_from_the_page():
    g = golden("packing_example.json")
    pool = B.Pool(1000, 16, 8, 64)
    plan = []
    for i, seg in enumerate(g["segments"]):
        assert pool.admit(i, 600) == B.PKV_OK
        if seg["kind"] == "decode":
            pool.lower([(i, 30)])  # some history before the decode row
        plan.append((i, seg["rows"]))
    low = pool.lower(plan)
    np.testing.assert_array_equal(np.diff(low.cu_seqlens_q), [s["rows"] for s in g["segments"]])
    assert low.cu_seqlens_q[-1] == len(low.slot_mapping) == 1206
    np.testing.assert_array_equal(low.seq_slot, np.arange(5))


def _oracle_mapping(pool, plan, ctx_before):
    segs = [(s, n, ctx_before[s] + n) for s, n in plan]
    p = oracle.pack(segs)
    return oracle.slot_mapping(pool.block_tables(), p.token_slot, p.token_pos, pool.block_size, pool.num_blocks)


@pytest.mark.parametrize("bs", [16, 32, 64])
def test_lowering_slot_mapping_matches_oracle(bs):
    rng = np.random.default_rng(bs)
    pool = B.Pool(4096, bs, 12, 128, free_order=rng.permutation(4096).astype(np.int32))
    lens = {}
    for slot in range(12):
        assert pool.admit(slot, int(rng.integers(1, 300))) == B.PKV_OK
        lens[slot] = 0
    for step in range(25):
        slots = rng.permutation(12)[: int(rng.integers(1, 12))]
        plan = [(int(s), int(rng.integers(0, 70)) if rng.random() < 0.4 else 1) for s in slots]
        before = dict(lens)
        low = pool.lower(plan)
        np.testing.assert_array_equal(low.slot_mapping, _oracle_mapping(pool, plan, before))
        for s, n in plan:
            lens[s] += n
            assert low.context_lens[s] == lens[s] == pool.slot_length(s)
        assert len(set(low.slot_mapping.tolist())) == len(low.slot_mapping)


def test_lowering_grows_blocks_at_boundaries_and_is_all_or_nothing():
    pool = B.Pool(4, 16, 2, 4)
    assert pool.admit(0, 16) == B.PKV_OK and pool.admit(1, 16) == B.PKV_OK
    pool.lower([(0, 16), (1, 15)])
    assert pool.slot_blocks(0) == 1 and pool.stats().free_blocks == 2
    pool.lower([(0, 1), (1, 1)])  # slot 0 opens block 1; slot 1 fills row 15
    assert pool.slot_blocks(0) == 2 and pool.slot_blocks(1) == 1
    with pytest.raises(B.PkvError) as e:
        pool.lower([(0, 40), (1, 20)])  # needs 2 + 2 blocks, only 1 free
    assert e.value.status == B.PKV_ERR_NO_BLOCKS
    assert pool.slot_length(0) == 17 and pool.slot_length(1) == 16 and pool.stats().free_blocks == 1


def test_lowering_rejects_bad_plans():
    pool = B.Pool(64, 16, 4, 8)
    assert pool.admit(0, 10) == B.PKV_OK
    for plan in ([(0, 1), (0, 1)], [(1, 1)], [(9, 1)], [(0, -1)], [(0, 200)]):
        with pytest.raises(B.PkvError):
            pool.lower(plan)
    assert pool.slot_length(0) == 0


# ---- work list ---------------------------------------------------------------

def _work(cu, slots, ctx, **kw):
    args = dict(max_slots=8, max_blocks_per_slot=64, block_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128)
    args.update(kw)
    return B.pkv_plan_work(np.array(cu), np.array(slots), np.array(ctx), **args)


def test_long_merge_rows_come_first_and_are_counted():
    """Rows of more than 64 spans are counted in num_long_combine_items and lead the merge list
    (the merge launch gives exactly those rows four lanes per column)."""
    S = B.PKV_SPLIT_KEYS
    ctx = np.zeros(8, np.int32)
    ctx[[0, 1, 2, 3, 4]] = [3 * S, 65 * S, 64 * S, 100 * S + 7, 2 * S]  # spans 3, 65, 64, 101, 2
    cu = [0, 1, 2, 3, 4, 5]
    work, info = B.pkv_plan_work(np.array(cu), np.array([0, 1, 2, 3, 4]), ctx, max_slots=8,
                                 max_blocks_per_slot=2048, block_size=16, num_q_heads=32, num_kv_heads=8,
                                 head_dim=128)
    assert info.num_combine_items == 5 and info.num_long_combine_items == 2
    items = work.reshape(-1, 4)
    comb = items[info.num_decode_items + info.num_prefill_items:][:info.num_combine_items]
    spans = [int(c[2]) & 0xFFFF for c in comb]
    assert spans == sorted(spans, reverse=True) and spans[:2] == [101, 65]


def test_work_list_items():
    S = B.PKV_SPLIT_KEYS
    ctx = np.zeros(8, np.int32)
    ctx[[3, 1, 6, 2]] = [1536, 2 * S + 1, 2 * S, 1]
    work, info = _work([0, 512, 513, 514, 515], [3, 1, 6, 2], ctx, max_blocks_per_slot=128)
    # decode spans: 3 for slot 1 (S, S, 1 keys), 2 for slot 6, 1 for slot 2; the chunk has 16 tiles,
    # run as 8 pairs at head_dim 128
    assert (info.num_decode_items, info.num_prefill_items, info.num_combine_items) == (6, 8, 2)
    items = work.reshape(-1, 4)
    assert len(items) == 17 and info.num_scratch_items == 1
    dec, pre, comb, scr = items[:6], items[6:14], items[14:16], items[16:]
    # the chunk's history (1536 keys) as 96 scratch blocks for the 8-bit pool's chunk path
    assert scr.tolist() == [[0, 3, 0, 96]] and info.scratch_blocks == 96
    assert [list(c) for c in comb] == [[1, 1, 3, 0], [2, 6, 2, 3]]  # (seg, slot, spans, partial base)
    assert sorted(map(tuple, dec[:, :3].tolist())) == [(1, 1, 0), (1, 1, 1), (1, 1, 2), (2, 6, 0), (2, 6, 1),
                                                        (3, 2, 0)]
    full = {(1, 1, 0), (1, 1, 1), (2, 6, 0), (2, 6, 1)}
    assert {tuple(x) for x in dec[:4, :3].tolist()} == full      # full spans first
    assert [tuple(x) for x in dec[4:, :3].tolist()] == [(1, 1, 2), (3, 2, 0)]  # 1-key spans, stable
    bases = {tuple(x[:3]): x[3] for x in dec.tolist()}
    assert bases[(1, 1, 0)] == bases[(1, 1, 1)] == bases[(1, 1, 2)] == 0
    assert bases[(2, 6, 0)] == bases[(2, 6, 1)] == 3 and bases[(3, 2, 0)] == -1
    assert info.num_partials == 5
    assert sorted(pre[:, 2].tolist()) == list(range(0, 16, 2)) and (pre[:, :2] == [0, 3]).all()
    assert (pre[:, 3] == 2).all()
    assert pre[0, 2] == 14  # the pair that sees the most keys first
    a256 = lambda x: (x + 255) // 256 * 256
    assert info.workspace_bytes == a256(5 * 32 * 128 * 4) + a256(5 * 32 * 2 * 4) + 256  # + the task counter
    assert info.workspace_bytes_q8 == info.workspace_bytes + 2 * a256(96 * 8 * 16 * 128 * 2) + a256(8 * 128 * 4)


def _model_work_list(cu, slots, ctx, group, head_dim, block_size):
    """The work list's rules restated: decode segments (at most 16 / group rows) cut into
    PKV_SPLIT_KEYS-key spans, full spans in segment order and then each segment's shorter last
    span, longest first; chunk tiles of 128 / group rows (pairs at head_dim 128), the pair
    that sees the most keys first; one merge item per row of a multi-span segment, rows of the
    most spans first; one scratch item per chunk segment. Equal costs keep their order."""
    S = B.PKV_SPLIT_KEYS
    decode_rows, rpt, step = max(1, 16 // group), 128 // group, 2 if head_dim == 128 else 1
    full, tails, pre, rows, scr = [], [], [], [], []
    partials = scratch = 0
    for s in range(len(slots)):
        n, slot = cu[s + 1] - cu[s], slots[s]
        L = int(ctx[slot])
        if n == 0:
            continue
        if n <= decode_rows:
            spans = -(-L // S)
            base = partials if spans > 1 else -1
            full += [[s, slot, sp, base] for sp in range(L // S)]
            if L % S:
                tails.append((L % S, s, [s, slot, L // S, base]))
            if spans > 1:
                rows.append((spans, s, [[s, slot, spans | (i << 16) | ((n - 1) << 24), base + i] for i in range(n)]))
                partials += spans * n
        else:
            nblk = -(-L // block_size)
            scr.append([s, slot, scratch, nblk])
            scratch += nblk
            tiles = -(-n // rpt)
            for t in range(0, tiles, step):
                count = min(step, tiles - t)
                pre.append((L - n + min(n, (t + count) * rpt), len(pre), [s, slot, t, count]))
    order = lambda x: (-x[0], x[1])
    dec = full + [t[2] for t in sorted(tails, key=order)]
    comb = [r for _, _, rr in sorted(rows, key=order) for r in rr]
    return dec, [p[2] for p in sorted(pre, key=order)], comb, scr, partials, scratch


def test_work_list_matches_its_rules_on_random_steps():
    rng = np.random.default_rng(7)
    for _ in range(300):
        hkv = int(rng.choice([1, 2, 8]))
        group = int(rng.choice([1, 2, 4, 5, 8, 16]))
        head_dim, bs = int(rng.choice([64, 128])), int(rng.choice([16, 32, 64]))
        max_slots, mbps = 24, 512
        nseg = int(rng.integers(0, 12))
        slots = [int(x) for x in rng.permutation(max_slots)[:nseg]]
        kind = rng.random(nseg)
        n = np.where(kind < 0.55, 1, np.where(kind < 0.8, rng.integers(1, 17, nseg), rng.integers(17, 600, nseg)))
        n = np.where(rng.random(nseg) < 0.05, 0, n).astype(int)
        ctx = np.zeros(max_slots, np.int32)
        for i, slot in enumerate(slots):
            L = int(rng.integers(max(int(n[i]), 1), min(mbps * bs, 40000) + 1))
            whole = (L // 256) * 256  # some contexts end on a span boundary
            ctx[slot] = whole if whole >= max(int(n[i]), 1) and rng.random() < 0.3 else L
        cu = [0] + np.cumsum(n).tolist()
        work, info = _work(cu, slots, ctx, max_slots=max_slots, max_blocks_per_slot=mbps, block_size=bs,
                           num_q_heads=hkv * group, num_kv_heads=hkv, head_dim=head_dim)
        dec, pre, comb, scr, partials, scratch = _model_work_list(cu, slots, ctx, group, head_dim, bs)
        items = np.asarray(work)[:int(info.work_words)].reshape(-1, 4).tolist()
        assert items == dec + pre + comb + scr
        assert (info.num_decode_items, info.num_prefill_items, info.num_combine_items, info.num_scratch_items) == \
            (len(dec), len(pre), len(comb), len(scr))
        assert info.num_partials == partials and info.scratch_blocks == scratch
        assert info.num_long_combine_items == sum((c[2] & 0xFFFF) > 64 for c in comb)
        decode_n = [x for x in n if 0 < x <= max(1, 16 // group)]
        assert info.decode_rows_max == (max(decode_n) if decode_n else 0)


@pytest.mark.parametrize("cu,slots,ctx_pairs,err", [
    ([0, 5], [0], {0: 4}, B.STATUS_NAMES[1]),            # rows > context
    ([0, 1, 2], [1, 1], {1: 9}, B.STATUS_NAMES[1]),      # duplicate slot
    ([0, 1], [9], {}, B.STATUS_NAMES[2]),                # slot out of range
    ([1, 2], [0], {0: 3}, B.STATUS_NAMES[1]),            # cu does not start at 0
    ([0, 1], [0], {0: 64 * 16 + 1}, B.STATUS_NAMES[2]),  # context beyond the table
])
def test_work_list_validation(cu, slots, ctx_pairs, err):
    ctx = np.zeros(8, np.int32)
    for k, v in ctx_pairs.items():
        ctx[k] = v
    with pytest.raises(B.PkvError, match=err):
        _work(cu, slots, ctx)


def test_work_list_tile_pairs():
    """head_dim 128 pairs consecutive tiles; an odd tile count leaves a single at the end; head_dim 64 does not pair."""
    ctx = np.zeros(8, np.int32)
    ctx[[0, 1]] = [100, 90]
    # group 4: 32 rows per tile; 80 and 70 rows are 3 tiles each: a pair and a single
    work, info = _work([0, 80, 150], [0, 1], ctx)
    pre = work.reshape(-1, 4)[:info.num_prefill_items]
    assert info.num_prefill_items == 4 and info.num_scratch_items == 2 and info.scratch_blocks == 7 + 6
    by_seg = {}
    for seg, slot, t, c in pre.tolist():
        by_seg.setdefault(seg, []).append((t, c))
    assert sorted(by_seg[0]) == [(0, 2), (2, 1)]          # 80 rows: 3 tiles
    assert sorted(by_seg[1]) == [(0, 2), (2, 1)]          # 70 rows: 3 tiles
    work64, info64 = _work([0, 80, 150], [0, 1], ctx, head_dim=64)
    assert info64.num_prefill_items == 6 and (work64.reshape(-1, 4)[:6, 3] == 1).all()


def test_work_list_verify_rows():
    """Segments of up to 16 / group rows take the decode path; the merge runs one item per row."""
    S = B.PKV_SPLIT_KEYS
    ctx = np.zeros(8, np.int32)
    ctx[[2, 5, 7]] = [2 * S + 88, 100, 40]
    # group 4: 3 rows over 3 spans, 4 rows in one span, 5 rows (a chunk)
    work, info = _work([0, 3, 7, 12], [2, 5, 7], ctx)
    assert (info.num_decode_items, info.num_prefill_items, info.num_combine_items) == (4, 1, 3)
    assert info.decode_rows_max == 4 and info.num_partials == 9 and info.num_scratch_items == 1
    items = work.reshape(-1, 4)
    dec, pre, comb = items[:4], items[4:5], items[5:8]
    assert items[8:].tolist() == [[2, 7, 0, 3]]
    assert sorted(map(tuple, dec.tolist())) == [(0, 2, 0, 0), (0, 2, 1, 0), (0, 2, 2, 0), (1, 5, 0, -1)]
    assert pre.tolist() == [[2, 7, 0, 1]]
    # spans | row << 16 | (rows - 1) << 24, and the row's entry for span 0 (span s: + s * rows)
    assert comb.tolist() == [[0, 2, 3 | (i << 16) | (2 << 24), i] for i in range(3)]
    # group 1: 16 rows still fit; 17 do not. group 16: every multi-row segment is a chunk.
    ctx[[0, 1]] = [600, 600]
    _, i1 = _work([0, 16, 33], [0, 1], ctx, num_q_heads=8, num_kv_heads=8)
    assert (i1.num_prefill_items, i1.decode_rows_max, i1.num_partials) == (1, 16, 48)
    _, i16 = _work([0, 1, 3], [0, 1], ctx, num_q_heads=16, num_kv_heads=1)
    assert (i16.num_prefill_items, i16.decode_rows_max, i16.num_partials) == (1, 1, 3)


def test_work_list_unsupported_shapes():
    ctx = np.array([5] + [0] * 7, np.int32)
    for kw in (dict(head_dim=96), dict(block_size=8), dict(num_q_heads=34 * 8, num_kv_heads=8)):
        with pytest.raises(B.PkvError, match="UNSUPPORTED"):
            _work([0, 1], [0], ctx, **kw)


# ---- host-staged step ------------------------------------------------------------

def test_stage_layout_offsets():
    T, S, ms, mb, hq, hkv, d = 516, 5, 8, 200, 32, 8, 128
    lay = B.pkv_stage_layout_init(T, S, ms, mb, hq, hkv, d)
    sizes = {"q": T * hq * d * 2, "k_new": T * hkv * d * 2, "v_new": T * hkv * d * 2, "slot_mapping": T * 8,
             "cu_seqlens_q": (S + 1) * 4, "seq_slot": S * 4, "context_lens": ms * 4, "block_tables": ms * mb * 4}
    order = list(sizes)
    offs = [getattr(lay, n) for n in order] + [lay.work]
    assert all(o % 256 == 0 for o in offs)
    for i, n in enumerate(order):  # in order, each field fits before the next
        assert offs[i] + sizes[n] <= offs[i + 1] < offs[i] + sizes[n] + 256
    assert (lay.total_q, lay.num_seqs, lay.max_slots, lay.max_blocks_per_slot) == (T, S, ms, mb)
    with pytest.raises(B.PkvError, match="INVALID_ARG"):
        B.pkv_stage_layout_init(-1, S, ms, mb, hq, hkv, d)


def _aligned_bytes(n):
    raw = np.zeros(n + 256, np.uint8)
    off = (-raw.ctypes.data) % 256
    return raw[off:off + n]


def test_step_rejects_bad_staging_before_any_device_work():
    """Every check here fails on the host, before pkv_step enqueues anything (no GPU needed)."""
    ctx = np.zeros(8, np.int32)
    ctx[[0, 1]] = [600, 40]
    lay = B.pkv_stage_layout_init(2, 2, 8, 64, 32, 8, 128)
    host = _aligned_bytes(lay.work + 4096)
    def put(name, a):
        a = np.ascontiguousarray(a)
        host[getattr(lay, name):getattr(lay, name) + a.nbytes] = a.reshape(-1).view(np.uint8)
    put("cu_seqlens_q", np.array([0, 1, 2], np.int32))
    put("seq_slot", np.array([0, 1], np.int32))
    put("context_lens", ctx)
    # host stand-ins for the device pointers: pkv_step must return before using any of them
    pools = _aligned_bytes(4 * 8 * 16 * 128 * 2)
    out = _aligned_bytes(2 * 32 * 128 * 2)
    dev = _aligned_bytes(lay.work + 4096)
    p = lambda a: ctypes.c_void_p(a.ctypes.data)

    def call(h, d_, ws=None):
        info = B.WorkInfo()
        rc = B._lib().pkv_step(ctypes.byref(lay), p(h), h.nbytes, p(d_), d_.nbytes, p(pools), p(pools), 4, 16,
                               0.0, None if ws is None else p(ws), 0 if ws is None else ws.nbytes, p(out), None,
                               None, None, ctypes.byref(info), 0)
        return B.STATUS_NAMES[rc], info

    # workspace missing: slot 0 has 3 spans, so partials are needed
    rc, info = call(host, dev)
    assert rc == "PKV_ERR_WORKSPACE_TOO_SMALL" and info.num_partials == 3 and info.workspace_bytes > 0
    # no room for the work list in the host buffer
    rc, info = call(host[:lay.work + 8], dev)
    assert rc == "PKV_ERR_WORKSPACE_TOO_SMALL" and info.work_words == 4 * (3 + 1 + 1)  # 3 + 1 spans, 1 merge row
    # device stage too small for the staged bytes
    assert call(host, dev[:lay.work], _aligned_bytes(1 << 20))[0] == "PKV_ERR_WORKSPACE_TOO_SMALL"
    # device stage not 256-byte aligned; cu_seqlens_q not ending at total_q
    assert call(host, dev[1:])[0] == "PKV_ERR_INVALID_ARG"
    put("cu_seqlens_q", np.array([0, 1, 3], np.int32))
    assert call(host, dev)[0] == "PKV_ERR_INVALID_ARG"


# ---- scheduler vs the oracle's replay -------------------------------------------

def _compare_trace(reqs, spec_steps, num_blocks, max_slots, bs=16, **policy):
    pool = B.Pool(num_blocks, bs, max_slots + policy.get("prefix_cache", 0), 1024,
                  free_order=W.churn_free_order(0, num_blocks))
    sch = S.ChurnScheduler(reqs, pool, **policy)
    ref = churn.ChurnReplay(reqs, max_slots=max_slots, num_blocks=num_blocks, block_size=bs, **policy)
    for step in range(spec_steps):
        rows = sch.plan()
        want = ref.plan()
        assert [(r.rid, r.begin, r.n, r.prefill) for r in rows] == \
               [(r.rid, r.begin, r.n, r.prefill) for r in want], f"step {step}"
        assert sch.preempted == ref.preempted, f"step {step}: preemptions differ"
        assert sch.preempt_reasons == ref.preempt_reasons, f"step {step}: preemption reasons differ"
        assert sch.cache_events == ref.cache_events, f"step {step}: prefix cache events differ"
        low = pool.lower([(r.slot, r.n) for r in rows])
        assert len(low.slot_mapping) == sum(r.n for r in rows)
        assert len(pool.take_copies()) == 0  # only whole blocks are ever shared: nothing to copy
        assert sch.commit(rows) == ref.commit(want)
        assert pool.stats().free_blocks == ref.free_blocks
    return sch


# 300 blocks (4800 tokens) and 16 slots for ~100 requests of 64-1024 prompt tokens: the pool, not the
# slots, limits admission, decode rows run out of blocks, and 30% of requests carry priority 1.
PRESSURE = W.ChurnSpec(num_steps=200, arrival_rate=0.5, prompt_min=64, prompt_max=1024, output_mean=96.0,
                       output_max=400, high_priority=0.3)


@pytest.mark.parametrize("policy", [dict(), dict(watermark=0.01), dict(watermark=0.01, preemption="longest-first"),
                                    dict(watermark=0.01, preemption="lowest-priority")])
def test_budgeted_scheduler_matches_oracle_under_pool_pressure(policy):
    """Small pool: watermark admission, priority preemption and decode-headroom preemption all fire."""
    reqs = W.churn_trace(5, PRESSURE)
    sch = _compare_trace(reqs, PRESSURE.num_steps, 300, 16, **policy)
    assert len(sch.preempted) > 0  # the budget rules were exercised, not just the happy path
    if policy.get("preemption"):
        assert "priority" in sch.preempt_reasons and "headroom" in sch.preempt_reasons
    else:
        assert set(sch.preempt_reasons) == {"headroom"}


def test_watermark_reduces_decode_preemptions():
    """The pages' reason for the watermark: keeping free blocks at admission leaves decode headroom."""
    reqs = W.churn_trace(5, PRESSURE)
    counts = [len(_compare_trace(reqs, PRESSURE.num_steps, 300, 16, watermark=f).preempted) for f in (0.0, 0.05)]
    assert counts[1] < counts[0]


PREFIXED = W.ChurnSpec(num_steps=200, arrival_rate=0.5, prompt_min=64, prompt_max=1024, output_mean=96.0,
                       output_max=400, high_priority=0.3, prefix_groups=5, prefix_share=0.6, prefix_min=100,
                       prefix_max=600)


def test_prefix_cache_scheduler_matches_oracle_under_pool_pressure():
    """Shared prompt prefixes, a 4-entry prefix cache and a tight pool: donations, adoptions and every
    kind of cache eviction happen, and the library (real refcounted pool) agrees with the replay."""
    reqs = W.churn_trace(6, PREFIXED)
    sch = _compare_trace(reqs, PREFIXED.num_steps, 300, 16, watermark=0.01, preemption="lowest-priority",
                         prefix_cache=4)
    kinds = {e[1] for e in sch.cache_events}
    assert kinds == {"donate", "adopt", "drop-capacity", "drop-admission", "drop-headroom"}
    assert sch.preempted
    # an adopter's first prefill row starts after the cached prefix
    assert sum(1 for e in sch.cache_events if e[1] == "adopt") >= 3


def test_prefix_cache_off_leaves_plans_unchanged():
    reqs = W.churn_trace(6, PREFIXED)
    a = _compare_trace(reqs, 120, 300, 16, watermark=0.01, preemption="lowest-priority")
    assert a.cache_events == []


def test_scheduler_matches_oracle_replay_on_churn_trace():
    spec = W.ChurnSpec(num_steps=120)
    reqs = W.churn_trace(0, spec)
    sch = _compare_trace(reqs, 120, spec.num_blocks, spec.max_slots)
    assert sch.step_index == 120


def test_scheduler_matches_oracle_under_pool_pressure():
    """Small pool: admission is limited by KV capacity, FIFO head-of-line blocking shows up."""
    spec = W.ChurnSpec(num_steps=80, prompt_max=3000)
    reqs = W.churn_trace(3, spec)
    _compare_trace(reqs, 80, 900, 16)


def test_scheduler_fifo_example_from_the_page():
    g = golden("fifo_admission_example.json")
    d_tokens = g["queue"][0]["blocks"] * 16 - 1
    e_tokens = g["queue"][1]["blocks"] * 16 - 1
    reqs = [W.Request(0, 0, d_tokens, 1), W.Request(1, 0, e_tokens, 1)]
    pool = B.Pool(g["free_blocks"], 16, 4, 200)
    sch = S.ChurnScheduler(reqs, pool)
    assert sch.plan() == [] and len(sch.queue) == 2 and pool.stats().free_blocks == g["free_blocks"]
