"""The physical block pool behind the block tables (host-side C++ through the C ABI).

No GPU involved: the pool lives in host memory. Also checks that the append calls
validate their arguments on the host before anything is launched.
"""
import numpy as np
import pytest

from paged_kv_cache_61_gb300 import build, pda


@pytest.fixture(scope="module", autouse=True)
def built_library():
    import os
    if not os.path.exists(pda.LIB_PATH):
        build.build()
    return pda.lib()


def _row(n=8):
    return np.full(n, -1, dtype=np.int32)


def test_grow_assigns_pages_in_order_and_only_new_ones():
    pool = pda.BlockPool(10)
    r = _row()
    pool.grow(r, 16, 0, 1)              # 1 token -> 1 page
    assert r.tolist()[:2] == [0, -1] and pool.num_free == 9
    pool.grow(r, 16, 1, 16)             # still one page: nothing new
    assert pool.num_free == 9
    pool.grow(r, 16, 16, 17)            # token 16 opens page 1
    assert r.tolist()[:3] == [0, 1, -1] and pool.num_free == 8
    pool.grow(r, 16, 17, 64)
    assert r.tolist()[:5] == [0, 1, 2, 3, -1] and pool.num_free == 6


def test_every_block_is_handed_out_once_until_released():
    pool = pda.BlockPool(12)
    rows = [_row(4) for _ in range(3)]
    for r in rows:
        pool.grow(r, 16, 0, 64)
    ids = np.concatenate(rows)
    assert sorted(ids.tolist()) == list(range(12)) and pool.num_free == 0
    with pytest.raises(pda.PdaError) as e:
        pool.grow(_row(4), 16, 0, 1)
    assert e.value.status == pda.PDA_ERR_OUT_OF_BLOCKS


def test_grow_is_all_or_nothing():
    pool = pda.BlockPool(3)
    r = _row(8)
    pool.grow(r, 16, 0, 16)
    before = r.copy()
    with pytest.raises(pda.PdaError) as e:
        pool.grow(r, 16, 16, 16 * 5)      # needs 4 more, 2 free
    assert e.value.status == pda.PDA_ERR_OUT_OF_BLOCKS
    np.testing.assert_array_equal(r, before)
    assert pool.num_free == 2


def test_release_returns_blocks_and_clears_entries():
    pool = pda.BlockPool(6)
    a, b = _row(4), _row(4)
    pool.grow(a, 16, 0, 40)               # 3 pages
    pool.grow(b, 16, 0, 20)               # 2 pages
    got = a[:3].tolist()
    pool.release(a, 16, 40)
    assert a.tolist() == [-1] * 4 and pool.num_free == 4
    c = _row(4)
    pool.grow(c, 16, 0, 48)               # the released blocks come back in page order
    assert c[:3].tolist() == got


def test_release_refuses_foreign_double_and_duplicate_ids_without_changes():
    pool = pda.BlockPool(6)
    a = _row(4)
    pool.grow(a, 16, 0, 32)
    for bad in ([7, 1], [-1, 1], [0, 0]):
        r = np.array(bad + [-1, -1], dtype=np.int32)
        with pytest.raises(pda.PdaError) as e:
            pool.release(r, 16, 32)
        assert e.value.status == pda.PDA_ERR_INVALID_ARG
        assert r.tolist()[:2] == bad
    assert pool.num_free == 4
    pool.release(a, 16, 32)
    with pytest.raises(pda.PdaError):     # released twice
        pool.release(np.array([0, 1], dtype=np.int32), 16, 32)
    assert pool.num_free == 6


def test_grow_and_release_validate_sizes():
    pool = pda.BlockPool(4)
    for args in ((16, 10, 5), (16, -1, 5), (0, 0, 5), (16, 0, 16 * 9)):
        with pytest.raises(pda.PdaError) as e:
            pool.grow(_row(8), *args)
        assert e.value.status == pda.PDA_ERR_INVALID_ARG
    with pytest.raises(pda.PdaError):
        pda.BlockPool(0)


def test_serving_churn_keeps_the_pool_consistent():
    # sequences start, grow a token at a time and finish; at every point the in-use
    # blocks are exactly the distinct entries of the live tables
    rng = np.random.default_rng(4)
    pool = pda.BlockPool(64)
    live = {}
    for step in range(400):
        if live and rng.random() < 0.1:
            k = list(live)[rng.integers(len(live))]
            row, n = live.pop(k)
            pool.release(row, 16, n)
        elif len(live) < 6 and rng.random() < 0.2:
            live[step] = (_row(16), 0)
        for k, (row, n) in list(live.items()):
            try:
                pool.grow(row, 16, n, n + 1)
                live[k] = (row, n + 1)
            except pda.PdaError as err:
                assert err.status == pda.PDA_ERR_OUT_OF_BLOCKS
        used = [int(x) for row, n in live.values() for x in row[: (n + 15) // 16]]
        assert len(used) == len(set(used)) and pool.num_free == 64 - len(used)


def _plan(**kw):
    args = dict(kind=pda.PDA_KIND_GQA, dtype=pda.PDA_FP16, batch=2, num_q_heads=8, num_kv_heads=2,
                head_dim_qk=64, head_dim_v=64, page_size=16, max_blocks_per_seq=4, num_blocks=8,
                context_lens=[5, 64], num_sms=152)
    args.update(kw)
    return pda.Plan(**args)


def test_append_calls_validate_before_launch():
    p, f8 = _plan(), _plan(kv_format=pda.PDA_KV_FP8_E4M3)
    ok = dict(k_new=4096, v_new=4096, k_cache=8192, v_cache=8192, tables=64, ctx=128, ws=1 << 20)
    for key, val in (("k_new", 0), ("v_cache", 0), ("k_new", 4100), ("ws", 0), ("ws", 4096 + 8)):
        a = dict(ok, **{key: val})
        with pytest.raises(pda.PdaError) as e:
            pda.kv_append(a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["tables"],
                          a["ctx"], p, a["ws"], stream=0)
        assert e.value.status in (pda.PDA_ERR_INVALID_ARG, pda.PDA_ERR_WORKSPACE)
    with pytest.raises(pda.PdaError):      # fp8 plan, 16-bit call and the other way round
        pda.kv_append(4096, 4096, 8192, 8192, 64, 128, f8, 1 << 20, stream=0)
    with pytest.raises(pda.PdaError):
        pda.kv_append_fp8(4096, 4096, 8192, 8192, 1.0, 1.0, 64, 128, p, 1 << 20, stream=0)
    with pytest.raises(pda.PdaError):      # a zero scale cannot be divided by
        pda.kv_append_fp8(4096, 4096, 8192, 8192, 0.0, 1.0, 64, 128, f8, 1 << 20, stream=0)
    with pytest.raises(pda.PdaError):      # kind mismatch
        pda.mla_append(4096, 8192, 64, 128, p, 1 << 20, stream=0)
    pda.kv_append(0, 0, 0, 0, 0, 0, _plan(batch=0, context_lens=[]), 0, stream=0)   # no-op
