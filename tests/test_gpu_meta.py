"""Metadata on the GPU must equal the oracle's bit for bit."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300 import lora as L
from gpu_util import long_short_tiles, tile_keyn, tiles_from_groups
from oracle_pins_util import load_golden

pytestmark = pytest.mark.gpu


def _dense_pool(Lk, ranks, enabled=None):
    d = L.PoolDesc()
    d.max_loras, d.max_rank, d.in_dim, d.n_slices = Lk, 64, 64, 1
    d.out_dims[0] = 64
    pool = L.lora_pool_create(d)
    for a in range(Lk):
        r = int(ranks[a])
        if r and (enabled is None or enabled[a]):
            L.lora_set(pool, a, r, 1.0, [np.zeros((r, 64), np.uint16)], [np.zeros((64, r), np.uint16)])
    return pool


def _check_dense(idx, Lk, ranks, enabled):
    T = len(idx)
    pool = _dense_pool(Lk, ranks, enabled)
    try:
        mb = H.MetaBuffer(max(T, 1), Lk)
        L.lora_build_meta(pool, torch.from_numpy(np.asarray(idx, np.int32)).cuda(), T, None, 1, mb.meta)
        got = mb.read()
        en = np.array([1 if (ranks[a] and (enabled is None or enabled[a])) else 0 for a in range(Lk)], np.int32)
        ref = oracle.dense_meta(idx, Lk, en, ranks)
        assert np.array_equal(got["sorted"], ref.sorted_tok)
        assert got["n_active"] == ref.n_active
        assert got["n_groups"] == ref.n_seg
        assert got["n_bad"] == ref.n_bad
        assert np.array_equal(got["key_count"], ref.slot_count)
        assert np.array_equal(got["key_offset"], np.concatenate([[0], np.cumsum(ref.slot_count)]))
        assert np.array_equal(got["group_key"], ref.seg_slot)
        assert np.array_equal(got["group_start"], ref.seg_start)
        assert np.array_equal(got["key_group"], ref.slot_seg)
        tg, tr = tiles_from_groups(ref.seg_start)
        assert got["n_tiles"] == len(tg)
        assert np.array_equal(got["tile_group"], tg) and np.array_equal(got["tile_row0"], tr)
        assert np.array_equal(got["tile_keyn"], tile_keyn(tg, tr, ref.seg_slot, ref.seg_start))
        lt, st = long_short_tiles(ref.seg_slot, ref.seg_start, ref.sorted_tok)
        assert got["n_ltiles"] == len(lt) and got["n_stiles"] == len(st)
        if lt:
            assert np.array_equal(got["ltile_row0"], [x[0] for x in lt])
            assert np.array_equal(got["ltile_keyn"], [x[1] for x in lt])
            assert np.array_equal(got["ltile_tok0"], [x[2] for x in lt])
        if st:
            assert np.array_equal(got["stile_row0"], [x[0] for x in st])
            assert np.array_equal(got["stile_keyn"], [x[1] for x in st])
        st = L.lora_get_device_status(pool)
        assert st == (L.CODE["LORA_ERR_DEVICE_INDEX"] if ref.n_bad else 0)
    finally:
        L.lora_pool_destroy(pool)


@pytest.mark.parametrize("preset", [1, 2, 3, 4])
def test_dense_meta_presets(preset):
    c = {1: gen.tiny, 2: gen.decode_qkv, 3: lambda: gen.prefill_gate_up(permuted=True),
         4: gen.many_adapter_down}[preset]() if preset != 4 else None
    if preset == 4:
        # ranks and idx of the many-adapter preset without drawing its 2 GB pool
        rng = np.random.Generator(np.random.PCG64(1004))
        ranks = rng.choice(np.array([8, 16, 32, 64], np.int32), size=1024).astype(np.int32)
        idx = rng.choice(1024, size=2048, p=gen.zipf_pmf(1024, 1.2)).astype(np.int32)
        _check_dense(idx, 1024, ranks, None)
    else:
        _check_dense(c.idx, c.L, np.minimum(c.ranks, 64), None)


@pytest.mark.parametrize("case", ["all_none", "one_token", "empty", "single_slot", "bad_and_disabled",
                                  "big_skewed", "huge_uncached"])
def test_dense_meta_edges(case):
    rng = np.random.default_rng(7)
    Lk, ranks, en = 16, np.full(16, 8, np.int32), None
    if case == "all_none":
        idx = np.full(300, -1, np.int32)
    elif case == "one_token":
        idx = np.array([3], np.int32)
    elif case == "empty":
        idx = np.zeros(0, np.int32)
    elif case == "single_slot":
        idx = np.full(1000, 5, np.int32)
    elif case == "bad_and_disabled":
        idx = rng.integers(-3, 20, size=777).astype(np.int32)
        ranks = rng.choice([0, 8, 16], size=16).astype(np.int32)
        en = (rng.random(16) < 0.7)
    elif case == "big_skewed":
        idx = rng.choice(16, size=20000, p=gen.zipf_pmf(16, 1.5)).astype(np.int32)
    else:  # more rows than the key cache holds: keys are recomputed in the scatter pass
        idx = rng.integers(-1, 16, size=70000).astype(np.int32)
    _check_dense(idx, Lk, ranks, en)


def test_moe_meta_preset_and_small():
    for c in (gen.moe(), gen.moe_case(T=77, K=3, E=5, D=16, F=16, L=4, R=8, seed=3, p_none=0.2,
                                      ranks=(8, 0, 8, 8))):
        run = H.MoERun(c)
        try:
            run.build_meta()
            got = run.mb.read()
            ref = oracle.moe_meta(c.topk_ids, c.idx, c.L, c.E, c.enabled, c.ranks)
            assert np.array_equal(got["sorted"], ref.sorted_pair)
            assert got["n_active"] == ref.n_active and got["n_groups"] == ref.n_groups
            assert got["n_bad"] == ref.n_bad
            assert np.array_equal(got["key_count"], ref.key_count)
            assert np.array_equal(got["key_offset"], ref.key_offset)
            assert np.array_equal(got["group_key"], ref.group_key)
            assert np.array_equal(got["group_start"], ref.group_start)
            tg, tr = tiles_from_groups(ref.group_start)
            assert np.array_equal(got["tile_group"], tg) and np.array_equal(got["tile_row0"], tr)
            assert np.array_equal(got["tile_keyn"], tile_keyn(tg, tr, ref.group_key, ref.group_start))
            assert got["n_ltiles"] == 0   # pairs of one (slot, expert) are never a contiguous run
            lt, st = long_short_tiles(ref.group_key, ref.group_start, ref.sorted_pair, dense=False)
            assert got["n_stiles"] == len(st)
        finally:
            run.close()


def _check_moe_meta(c, expect):
    """GPU MoE metadata of case c against the oracle (and, if given, against
    the expected arrays of a hand-worked case)."""
    run = H.MoERun(c)
    try:
        run.build_meta()
        got = run.mb.read()
        st = run.status()
    finally:
        run.close()
    ref = oracle.moe_meta(c.topk_ids, c.idx, c.L, c.E, c.enabled, c.ranks)
    assert np.array_equal(got["sorted"], ref.sorted_pair)
    assert (got["n_active"], got["n_groups"], got["n_bad"]) == (ref.n_active, ref.n_groups, ref.n_bad)
    assert np.array_equal(got["key_count"], ref.key_count)
    assert np.array_equal(got["key_offset"], ref.key_offset)
    assert np.array_equal(got["group_key"], ref.group_key)
    assert np.array_equal(got["group_start"], ref.group_start)
    tg, tr = tiles_from_groups(ref.group_start)
    assert np.array_equal(got["tile_group"], tg) and np.array_equal(got["tile_row0"], tr)
    assert np.array_equal(got["tile_keyn"], tile_keyn(tg, tr, ref.group_key, ref.group_start))
    assert st == (L.CODE["LORA_ERR_DEVICE_INDEX"] if ref.n_bad else 0)
    if expect is not None:
        assert got["sorted"].tolist() == expect["sorted_pair"]
        assert got["key_count"].tolist() == expect["key_count"]
        assert got["group_key"].tolist() == expect["group_key"]
        assert got["group_start"].tolist() == expect["group_start"]
        assert got["n_bad"] == expect["n_bad"]


def test_moe_meta_out_of_range_ids_hand_case():
    # the hand-worked case of the oracle pins: expert ids -1, E, E+1 and -3,
    # slot id L, an idx -1 token with a bad expert id
    g = load_golden("moe_meta_bad_ids_by_hand.json")
    c = gen.moe_case(T=g["T"], K=g["K"], E=g["E"], D=16, F=16, L=g["L"], R=4, seed=5, n13=1)
    c.idx[:] = np.asarray(g["idx"], np.int32)
    c.topk_ids[:] = np.asarray(g["topk_ids"], np.int32)
    _check_moe_meta(c, g)


@pytest.mark.parametrize("seed", [0, 1])
def test_moe_meta_out_of_range_ids_random(seed):
    rng = np.random.default_rng(70 + seed)
    c = gen.moe_case(T=300, K=4, E=7, D=16, F=16, L=5, R=8, seed=seed, n13=1, ranks=(8, 0, 8, 8, 8),
                     p_none=0.1)
    bad = rng.random(c.topk_ids.shape) < 0.1
    c.topk_ids[bad] = rng.choice(np.array([-2, -1, 7, 8, 100], np.int32), size=int(bad.sum()))
    tb = rng.random(c.T) < 0.05
    c.idx[tb] = rng.choice(np.array([-7, 5, 6], np.int32), size=int(tb.sum()))
    _check_moe_meta(c, None)


def test_meta_is_deterministic_across_runs():
    c = gen.decode_qkv()
    pool = _dense_pool(c.L, np.full(c.L, 16, np.int32))
    try:
        mb = H.MetaBuffer(c.T, c.L)
        d_idx = torch.from_numpy(c.idx).cuda()
        outs = []
        for _ in range(3):
            L.lora_build_meta(pool, d_idx, c.T, None, 1, mb.meta)
            outs.append(mb.read()["sorted"].copy())
        assert all(np.array_equal(outs[0], o) for o in outs[1:])
    finally:
        L.lora_pool_destroy(pool)


def test_long_tiles_need_one_contiguous_run():
    """Slot 0: one run of 300 tokens (long tiles); slot 1: two runs of 100
    (short tiles); slot 2: 40 tokens (too few, short tiles)."""
    idx = np.full(700, -1, np.int32)
    idx[0:300] = 0
    idx[300:400] = 1
    idx[450:550] = 1
    idx[600:640] = 2
    _check_dense(idx, 4, np.full(4, 16, np.int32), None)


@pytest.mark.parametrize("bm", [4, 16, 64])
def test_moe_align_padded_matches_oracle(bm):
    for c in (gen.moe(), gen.moe_case(T=57, K=3, E=7, D=16, F=16, L=4, R=8, seed=9, p_none=0.2,
                                      ranks=(8, 0, 8, 8))):
        run = H.MoERun(c)
        try:
            run.build_meta()
            P = c.T * c.K
            cap = ((P + c.E * (bm - 1) + bm - 1) // bm) * bm
            ds = torch.empty((c.L, cap), dtype=torch.int32, device="cuda")
            de = torch.empty((c.L, cap // bm), dtype=torch.int32, device="cuda")
            dn = torch.empty(c.L, dtype=torch.int32, device="cuda")
            L.lora_moe_align_padded(run.pool, run.mb.meta, bm, cap, ds, de, dn)
            got_s, got_e, got_n = ds.cpu().numpy(), de.cpu().numpy(), dn.cpu().numpy()
        finally:
            run.close()
        ref = oracle.moe_align_padded(c.topk_ids, c.idx, c.L, c.E, c.enabled, c.ranks, bm, cap)
        assert np.array_equal(got_n, ref.npp)
        assert np.array_equal(got_s, ref.sorted)
        assert np.array_equal(got_e, ref.expert)
