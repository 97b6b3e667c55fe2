"""The launch plans of mxfp4_linear, checked on the host (no GPU): which
kernel a shape gets (the packed-E2M1 tensor-core kernel when k % 512 == 0
and t <= 8, or t <= 16 when each CTA's tiles fit one batch; the E4M3-split
tensor-core kernel for the other k % 512 == 0 shapes; else the streaming
engine with whole K per CTA, K walked in parts or a cluster split of K),
and the invariants every plan must keep for the kernel's indexing to
hold."""
import math

import pytest

import mxfp4_weight_streaming_gb300 as mx

SMS, SMEM = 152, 232448  # GB300: SMs and opt-in shared memory per block


@pytest.fixture(scope="module", autouse=True)
def lib():
    from mxfp4_weight_streaming_gb300 import build
    build.build()
    mx.load()


def consumer_warps(t):
    return 14 if t <= 8 else (12 if t <= 16 else 8)


@pytest.mark.parametrize("t,k,n,cluster,ctas,rows,tiles", [
    (4, 7168, 7168, 2, 150, 96, 1),       # verify: 75 clusters of 96 rows, K in halves
    (8, 7168, 7168, 2, 150, 96, 1),
    (1, 1024, 1024, 2, 128, 16, 1),       # 64 clusters of 16 rows
    (1, 7168, 18432, 1, 144, 128, 1),     # FFN up: one 128-row tile per CTA
    (4, 7168, 18432, 1, 144, 128, 1),
    (8, 7168, 18432, 2, 150, 248, 2),     # t > 4: K in halves, two tiles (128 + 120 rows) per CTA
    (5, 7168, 18432, 2, 150, 248, 2),
    (4, 7168, 129280, 1, 152, 856, 7),    # LM head: 6 tiles of 128 rows and one of 88 per CTA
    (6, 7168, 129280, 1, 152, 856, 7),    # t > 4, but 14 tiles per cluster would not fit TMEM: lone CTAs
    (8, 7168, 129280, 1, 152, 856, 7),
    (3, 512, 64, 1, 8, 8, 1),             # one stage: no K split, 8-row groups
    (6, 512, 64, 1, 8, 8, 1),
    (9, 7168, 7168, 2, 150, 96, 1),       # t = 9-16: 128 MMA columns, x converted once per CTA
    (16, 7168, 18432, 2, 150, 248, 2),
    (16, 7168, 4900, 2, 138, 72, 1),
])
def test_packed_e2m1_plans(t, k, n, cluster, ctas, rows, tiles):
    p = mx.linear_plan(t, k, n, SMS, SMEM)
    assert p["mode"] == 4, p
    assert (p["cluster"], p["ctas"], p["group_rows"], p["batch_units"]) == (cluster, ctas, rows, tiles), p
    assert p["stage_steps"] == 2 and p["part_steps"] == 0 and p["ring_slots"] >= 2, p


@pytest.mark.parametrize("t", [1, 2, 3, 4])
def test_packed_e2m1_residency_ffn_width(t):
    """FFN-up width (N = 18432, one 128-row tile per CTA): at t <= 2 three
    32 KB weight slots and two activation buffers fit half the SM, so two
    CTAs share it; at t = 3-4 they do not, and one CTA runs per SM."""
    p = mx.linear_plan(t, 7168, 18432, SMS, SMEM)
    half = (SMEM + 1024) // 2 - 1024
    assert p["mode"] == 4 and (p["smem_bytes"] <= half) == (t <= 2), p


@pytest.mark.parametrize("t,two_per_sm", [(1, True), (2, True), (3, True), (4, True), (5, False), (8, False)])
def test_packed_e2m1_residency(t, two_per_sm):
    """Verify width (K = N = 7168): up to 32 MMA columns (t <= 4) a plan
    within half the SM's shared memory (the next call's CTA shares the SM);
    wider, one CTA per SM with the weight ring first (at least 5 slots)."""
    p = mx.linear_plan(t, 7168, 7168, SMS, SMEM)
    assert p["mode"] == 4, p
    half = (SMEM + 1024) // 2 - 1024
    if two_per_sm:
        assert p["smem_bytes"] <= half and p["ring_slots"] >= 3, p
    else:
        assert p["smem_bytes"] > half and p["ring_slots"] >= 5, p


@pytest.mark.parametrize("t,k,n,cluster,ctas", [
    (24, 7168, 7168, 2, 112),       # 56 tiles of 128 rows, K split over 2-CTA clusters
    (20, 1024, 1024, 2, 16),
    (17, 7168, 18432, 1, 144),      # FFN up: one tile per CTA
    (32, 7168, 18432, 1, 144),
    (12, 7168, 129280, 1, 152),     # LM-head width at t <= 16: the packed-E2M1 kernel would need 7 tiles in one batch
    (17, 7168, 4900, 2, 78),
])
def test_tensor_core_plans(t, k, n, cluster, ctas):
    p = mx.linear_plan(t, k, n, SMS, SMEM)
    assert p["mode"] == 3, p
    assert (p["cluster"], p["ctas"]) == (cluster, ctas), p
    tiles = -(-n // 128)
    per_cta = -(-tiles // (ctas // cluster))
    assert p["batch_units"] == per_cta and p["part_steps"] == 0, p


@pytest.mark.parametrize("t,k,n,mode,stage,chunk,part,batch", [
    (4, 7200, 7168, 0, 1, 1, 0, 0),      # k % 512 != 0: 29 K steps (prime): 1-step stages
    (1, 1056, 1024, 0, 1, 1, 0, 0),      # 5 K steps, the last one block long
    (4, 7424, 7168, 0, 1, 1, 0, 0),      # 29 K steps of 256
    (1, 7424, 18432, 0, 1, 1, 0, 0),
    (8, 6176, 18432, 0, 5, 5, 0, 0),     # 25 K steps: whole 5-step stage chunks
    (2, 6400, 129280, 0, 5, 5, 0, 0),    # 25 K steps, LM-head width
    (32, 7200, 18432, 1, 1, 1, 1, 8),    # activations of all of K fill shared memory: K in parts
    (32, 7200, 4900, 1, 1, 1, 1, 3),     # 29 K steps (prime): one-step parts
])
def test_streaming_engine_plans(t, k, n, mode, stage, chunk, part, batch):
    p = mx.linear_plan(t, k, n, SMS, SMEM)
    assert (p["mode"], p["stage_steps"], p["chunk_steps"], p["part_steps"], p["batch_units"]) == \
        (mode, stage, chunk, part, batch), p
    assert p["cluster"] == 1 and p["ctas"] == min(SMS, (n + 15) // 16)


def test_cluster_only_for_single_row_group_ctas():
    p = mx.linear_plan(16, 7200, 130, SMS, SMEM)
    assert p["mode"] == 2 and p["cluster"] == 2 and p["ctas"] == 2 * 9
    p = mx.linear_plan(16, 7200, 4900, SMS, SMEM)  # 2-3 row groups per CTA
    assert p["mode"] == 1


def grid():
    for t in (1, 2, 3, 4, 5, 8, 9, 12, 16, 17, 23, 24, 32):
        for k in (32, 96, 1024, 1056, 2048, 4096, 7168, 7200, 14336, 16384, 30720, 6176):
            for n in (1, 17, 130, 1024, 4900, 18432, 129280):
                yield t, k, n


def test_plan_invariants_over_shapes():
    seen = set()
    for t, k, n in grid():
        try:
            p = mx.linear_plan(t, k, n, SMS, SMEM)
        except mx.Mxfp4Error as e:
            assert e.status == mx.MXFP4_ERR_SHAPE
            continue
        seen.add(p["mode"])
        where = f"t={t} k={k} n={n}: {p}"
        assert p["smem_bytes"] <= SMEM, where
        if p["mode"] == 4:
            # packed-E2M1 kernel: t <= 8, k % 512; groups of a multiple of 8
            # rows covering n, one per CTA or per 2-CTA cluster (K halves,
            # when K has >= 2 stages and lone CTAs would get < 96 rows, or
            # t > 4 and the cluster's tiles fit one TMEM batch)
            assert k % 512 == 0 and t <= 16, where
            rows, cl = p["group_rows"], p["cluster"]
            lone_rows = -(-(-(-n // SMS)) // 8) * 8
            if k >= 1024 and lone_rows < 96:
                assert cl == 2, where
            elif k < 1024 or t <= 4:
                assert cl == 1, where
            else:
                assert cl in (1, 2), where
            assert rows % 8 == 0 and rows >= 8 and p["ctas"] == cl * -(-n // rows) <= SMS, where
            assert p["ctas"] // cl * rows >= n > (p["ctas"] // cl - 1) * rows, where
            assert p["batch_units"] == (1 if rows <= 128 else rows // 128 + (rows % 128 != 0)), where
            assert p["stage_steps"] == 2 and p["ring_slots"] >= 2, where
            continue
        if p["mode"] == 3:
            # tensor-core kernel: t >= 5, k % 512, 128-row tiles, one tile
            # per 2-CTA cluster or a tile range per CTA, 2- or 4-atom stages
            tiles = -(-n // 128)
            assert k % 512 == 0 and t >= 9, where
            assert p["stage_steps"] in (1, 2) and p["ring_slots"] >= 2, where
            if p["cluster"] == 2:
                assert p["ctas"] == 2 * tiles and 2 * tiles <= SMS and p["batch_units"] == 1, where
            else:
                assert p["cluster"] == 1 and p["ctas"] == min(SMS, tiles), where
            continue
        assert k % 512 != 0, where
        nkb = -(-k // 256)
        n_rg = -(-n // 16)
        upc = -(-n_rg // min(SMS, n_rg))
        ncw = consumer_warps(t)
        assert p["stage_steps"] >= 1 and p["stage_steps"] % p["chunk_steps"] == 0, where
        assert p["ring_slots"] >= 2, where
        if p["mode"] == 0:
            assert p["cluster"] == 1 and p["ctas"] == min(SMS, n_rg), where
            assert nkb % p["stage_steps"] == 0, where
            # whole-stage chunks unless some warp would get none
            if p["chunk_steps"] < p["stage_steps"]:
                bigger = [g for g in range(p["chunk_steps"] + 1, p["stage_steps"] + 1) if p["stage_steps"] % g == 0]
                assert all(upc * (nkb // g) < ncw for g in bigger), where
        elif p["mode"] == 1:
            assert p["cluster"] == 1 and p["ctas"] == min(SMS, n_rg), where
            assert p["part_steps"] % p["stage_steps"] == 0 and nkb % p["part_steps"] == 0, where
            assert p["chunk_steps"] == p["stage_steps"], where
            assert 1 <= p["batch_units"] <= min(ncw, upc, 16), where
        else:
            cl = p["cluster"]
            assert cl in (2, 4, 8) and p["ctas"] % cl == 0 and p["ctas"] <= SMS, where
            # the stage divides every rank's share of the K steps
            share = -(-nkb // cl)
            steps = [min(nkb, (r + 1) * share) - min(nkb, r * share) for r in range(cl)]
            assert all(s % p["stage_steps"] == 0 for s in steps), where
            assert p["part_steps"] == 0 and p["batch_units"] == 0, where
    assert seen == {0, 1, 2, 3, 4}


def test_plan_argument_errors():
    for args, status in [((33, 64, 8), mx.MXFP4_ERR_SHAPE), ((1, 48, 8), mx.MXFP4_ERR_SHAPE),
                         ((0, 64, 8), mx.MXFP4_ERR_INVALID_ARG), ((1, 64, 0), mx.MXFP4_ERR_INVALID_ARG)]:
        with pytest.raises(mx.Mxfp4Error) as e:
            mx.linear_plan(*args, SMS, SMEM)
        assert e.value.status == status
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.linear_plan(4, 7168, 7168, 0, SMEM)
    assert e.value.status == mx.MXFP4_ERR_INVALID_ARG


def test_smaller_devices_still_plan_or_refuse():
    """With less shared memory the planner falls back (parts, clusters) or
    reports MXFP4_ERR_SHAPE; it never returns a plan that does not fit."""
    for smem in (101376, 166912):
        for t, k, n in [(4, 7168, 7168), (32, 7168, 18432), (8, 14336, 4096), (1, 1024, 1024)]:
            try:
                p = mx.linear_plan(t, k, n, 132, smem)
            except mx.Mxfp4Error as e:
                assert e.status == mx.MXFP4_ERR_SHAPE
                continue
            assert p["smem_bytes"] <= smem and math.gcd(p["stage_steps"], p["chunk_steps"]) == p["chunk_steps"]


def test_every_token_count_plans_up_to_k_262144():
    """The header's promise: on GB300 every t <= 32 and n plans for k up to
    262144 (the limit is a row group's k/2 scale bytes on chip)."""
    for t in range(1, 33):
        for n in (1, 17, 1000, 40000, 129280):
            for k in (262144, 262144 - 32, 131104):
                p = mx.linear_plan(t, k, n, SMS, SMEM)
                assert p["smem_bytes"] <= SMEM

