"""The persistent tile scheduler's work items, on the host (no GPU).

gemm_schedule_model lists the items each unit of a launch runs -- built by
the same code as a launch's parameters (fill_schedule) and the kernel's own
item functions, compiled for the host.  For many shapes, every division the
plan offers (the model's own, whole tiles, last-arriver splits, early
partials, half-width items, stream-K, the CTA-pair split) and two device
sizes, the items of all units must cover the output exactly once: every
tile's K blocks once across its pieces, or each of its two column halves
once over the whole K; pieces of a divided tile carry consistent roles and
split indices; early partials run first on their units and their owners
last; the tile order is a bijection onto the tile grid.
"""
import pytest

import tensor_core_dense_tma_gb300 as tc
from tensor_core_dense_tma_gb300 import build as tcbuild

ROLE_WHOLE, ROLE_SPLIT, ROLE_EARLY, ROLE_OWNER, ROLE_PAIR = 0, 1, 2, 3, 4


@pytest.fixture(scope="module", autouse=True)
def built():
    tcbuild.build()


def schedule(sms, *args, division="auto", splits=0, **kw):
    """All units' items: {unit: [items]}; None when the division does not fit."""
    try:
        n_units, first = tc.gemm_schedule_model(sms, *args, division=division, splits=splits, unit=0, **kw)
    except tc.GemmError as e:
        if e.status == 2:   # GEMM_ERR_UNSUPPORTED: the pinned division does not fit this problem
            return None
        raise
    out = {0: first}
    for u in range(1, n_units):
        out[u] = tc.gemm_schedule_model(sms, *args, division=division, splits=splits, unit=u, **kw)[1]
    return out


def check(units):
    pieces = {}
    coords = {}
    for u, items in units.items():
        roles = [x["role"] for x in items]
        # early partials run before the unit's other items, owners after them
        for k, r in enumerate(roles):
            if r == ROLE_EARLY:
                assert all(rr in (ROLE_WHOLE, ROLE_EARLY) for rr in roles[:k]), (u, roles)
            if r == ROLE_OWNER:
                assert k == len(roles) - 1, (u, roles)
        for x in items:
            assert 0 <= x["kb0"] < x["kb1"], x
            pieces.setdefault(x["tile"], []).append(x)
            c = (x["tile_row"], x["tile_col"])
            assert coords.setdefault(x["tile"], c) == c
    # the tile order is a bijection onto the grid
    tiles = sorted(pieces)
    assert tiles == list(range(len(tiles)))
    rows = 1 + max(c[0] for c in coords.values())
    cols = 1 + max(c[1] for c in coords.values())
    assert rows * cols == len(tiles) and len(set(coords.values())) == len(tiles)
    kb = max(x["kb1"] for ps in pieces.values() for x in ps)
    for t, ps in pieces.items():
        halves = [x for x in ps if x["half"] >= 0]
        if halves:
            # two half-width items, each over the whole K
            assert len(halves) == len(ps) == 2 and sorted(x["half"] for x in ps) == [0, 1], ps
            assert all(x["kb0"] == 0 and x["kb1"] == kb and x["role"] == ROLE_WHOLE for x in ps), ps
            continue
        ps = sorted(ps, key=lambda x: x["kb0"])
        # the K ranges partition [0, kb)
        assert ps[0]["kb0"] == 0 and ps[-1]["kb1"] == kb, ps
        assert all(a["kb1"] == b["kb0"] for a, b in zip(ps, ps[1:])), ps
        roles = sorted(x["role"] for x in ps)
        if len(ps) == 1:
            assert roles == [ROLE_WHOLE], ps
            continue
        s = len(ps)
        assert all(x["nsplit"] == s for x in ps) and [x["split"] for x in ps] == list(range(s)), ps
        assert (roles == [ROLE_SPLIT] * s or roles == [ROLE_EARLY] * (s - 1) + [ROLE_OWNER]
                or roles == [ROLE_PAIR] * 2), ps
        if roles[-1] == ROLE_OWNER:
            assert ps[0]["role"] == ROLE_OWNER, ps   # the owner holds split 0, the first K range
    return len(tiles)


SHAPES = [
    ("f16", 4096, 4096, 4096), ("f16", 8192, 8192, 8192), ("f16", 4097, 2055, 1000, "row", "col"),
    ("f16", 256, 256, 256), ("f16", 3000, 5000, 2000), ("f16", 1024, 1024, 16384), ("f16", 300, 600, 328),
    ("f16", 2300, 2290, 800), ("f16", 5000, 300, 4000), ("bf16", 16, 8192, 8192, "row", "row", "f32", "bf16"),
    ("bf16", 48, 1024, 4096, "row", "row", "f32", "bf16"), ("bf16", 64, 20000, 512, "row", "row", "f32", "bf16"),
    ("f16", 1, 300, 64), ("f16", 9000, 700, 64), ("f16", 4096, 4096, 4096, "row", "col", "f16", "f16"),
    ("e4m3", 8192, 8192, 8192, "row", "col", "f32", "bf16"), ("tf32", 4096, 4096, 4096, "row", "col"),
]
DIVISIONS = [("auto", 0), ("whole", 0), ("split", 0), ("split", 3), ("early_split", 0), ("early_split", 2),
             ("early_split", 4), ("halves", 0), ("stream_k", 0), ("pair_split", 0)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "_".join(map(str, s)))
@pytest.mark.parametrize("sms", [152, 38])
def test_every_division_covers_the_output_once(shape, sms):
    ran = 0
    for division, splits in DIVISIONS:
        units = schedule(sms, *shape, division=division, splits=splits)
        if units is None:
            continue
        check(units)
        ran += 1
    assert ran >= 2   # the model's own choice and whole tiles always fit


def test_random_shapes_model_choice():
    import numpy as np
    rng = np.random.default_rng(123)
    for _ in range(60):
        M, N, K = (int(v) for v in (rng.integers(1, 6000), rng.integers(1, 6000), rng.integers(8, 9000) // 8 * 8))
        for division in ("auto", "early_split", "stream_k"):
            units = schedule(int(rng.choice([16, 76, 152])), "f16", M, N, K, "row", "col", division=division)
            if units is not None:
                check(units)


def test_arguments():
    # empty problems run no tile kernel
    assert tc.gemm_schedule_model(152, "f16", 0, 64, 64) == (0, [])
    assert tc.gemm_schedule_model(152, "f16", 64, 64, 0) == (0, [])
    with pytest.raises(tc.GemmError) as e:   # a unit beyond the launch
        tc.gemm_schedule_model(152, "f16", 4096, 4096, 4096, unit=76)
    assert e.value.status == 1
    with pytest.raises(tc.GemmError) as e:
        tc.gemm_schedule_model(1, "f16", 64, 64, 64)
    assert e.value.status == 1
    with pytest.raises(tc.GemmError) as e:   # stream-K needs two whole waves
        tc.gemm_schedule_model(152, "f16", 512, 512, 1024, division="stream_k")
    assert e.value.status == 2


def test_the_check_notices_mistakes():
    """Plausible scheduler mistakes, planted in a real schedule, fail the check."""
    import copy
    base = schedule(152, "f16", 4096, 4096, 4096)            # 3 whole waves + early partials
    assert check(base) == 256

    def fails(mutate):
        units = copy.deepcopy(base)
        mutate(units)
        with pytest.raises(AssertionError):
            check(units)

    fails(lambda u: u[5].pop(0))                               # a tile left out
    fails(lambda u: u[5].append(dict(u[6][0])))                # a tile run twice
    fails(lambda u: u[0][-1].update(kb1=u[0][-1]["kb1"] - 1))  # a K block left out of a split
    fails(lambda u: u[0].reverse())                            # the owner before the unit's whole tiles
    fails(lambda u: u[0][-1].update(role=ROLE_SPLIT))          # mixed reductions on one tile
    fails(lambda u: u[3][0].update(tile_col=u[4][0]["tile_col"], tile_row=u[4][0]["tile_row"]))   # two tiles, one place
