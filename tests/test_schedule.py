"""CPU checks of the tensor-core kernel's schedule (host arithmetic behind DG_OPT_SCHEDULE and
DG_OPT_SPLITS), through dg_attn_schedule_info, which touches no device.

The stream-K run arithmetic is restated here independently (unit u of U belongs to CTA c when
floor(c*U/C) <= u < floor((c+1)*U/C)) and the library's figures are checked against it."""
import random

import pytest

from gqa_canvas_attention_gb300 import binding as B
from gqa_canvas_attention_gb300 import build as build_mod

NK = {64: 128, 128: 64, 256: 64}          # keys per score tile of the tensor-core kernel


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.load()


def geometry(T, ctx, nh, nkv, hd):
    G = nh // nkv
    n_tiles = -(-(ctx + T) // NK[hd])
    pairs = -(-(T * G) // 128) * nkv
    return n_tiles, pairs


def runs(U, C):
    return [(c * U // C, (c + 1) * U // C) for c in range(C)]


def pieces_per_pair(U, C, n_tiles, pairs):
    owners = [set() for _ in range(pairs)]
    for c, (a, b) in enumerate(runs(U, C)):
        for u in range(a, b):
            owners[u // n_tiles].add(c)
    return [len(o) for o in owners]


def test_bench_geometry_uses_four_clustered_partitions():
    # the 48-step workload on 152 SMs: 32 (query tile, kv group) pairs x 136 key tiles
    sched, parts, ctas, run = B.dg_attn_schedule_info(8, 4, 256, 8192, 512, 152)
    assert (sched, parts, ctas, run) == (B.DG_SCHEDULE_SPLIT, 4, 128, 34)


def test_forced_stream_k_on_the_bench_geometry():
    sched, kmax, ctas, run = B.dg_attn_schedule_info(8, 4, 256, 8192, 512, 152,
                                                     schedule=B.DG_SCHEDULE_STREAM_K)
    n_tiles, pairs = geometry(512, 8192, 8, 4, 256)
    U = n_tiles * pairs
    assert sched == B.DG_SCHEDULE_STREAM_K
    assert ctas == 152 and run == -(-U // 152)
    assert kmax == max(pieces_per_pair(U, ctas, n_tiles, pairs)) == 6


def test_forced_split_reports_the_split_schedule():
    sched, parts, ctas, run = B.dg_attn_schedule_info(8, 4, 256, 8192, 512, 152,
                                                      schedule=B.DG_SCHEDULE_SPLIT)
    assert sched == B.DG_SCHEDULE_SPLIT and parts == 4


@pytest.mark.parametrize("seed", range(6))
def test_schedules_cover_every_key_tile_of_every_pair(seed):
    rnd = random.Random(seed)
    for _ in range(40):
        hd = rnd.choice([64, 128, 256])
        nkv = rnd.choice([1, 2, 4, 8])
        nh = nkv * rnd.choice([1, 2, 4, 8])
        T = rnd.randint(1, 1200)
        ctx = rnd.choice([0, rnd.randint(1, 9000)])
        sms = rnd.choice([8, 64, 152])
        n_tiles, pairs = geometry(T, ctx, nh, nkv, hd)
        for req in (B.DG_SCHEDULE_AUTO, B.DG_SCHEDULE_SPLIT, B.DG_SCHEDULE_STREAM_K):
            sched, k, ctas, run = B.dg_attn_schedule_info(nh, nkv, hd, ctx, T, sms, schedule=req)
            if req == B.DG_SCHEDULE_SPLIT:
                assert sched == B.DG_SCHEDULE_SPLIT
            if sched == B.DG_SCHEDULE_SPLIT:
                # k partitions of `run` tiles: none empty, all tiles covered
                assert 1 <= k <= 64 and ctas == pairs * k
                assert k * run >= n_tiles > (k - 1) * run
            else:
                U = pairs * n_tiles
                assert pairs <= ctas <= min(sms, U)
                assert run == -(-U // ctas)
                per_pair = pieces_per_pair(U, ctas, n_tiles, pairs)
                assert k == max(per_pair) <= 16
                # a run covers at most two pairs (the kernel holds two pieces)
                for a, b in runs(U, ctas):
                    assert b > a and (b - 1) // n_tiles - a // n_tiles <= 1


def test_clusters_that_do_not_fit_change_the_choice():
    # With no cluster fitting, 2..8 partitions lose their in-kernel merge and would go through
    # the combine kernel as well; the cost model then prefers stream-K on the bench geometry.
    # Forced split still leaves no partition empty.
    n_tiles, pairs = geometry(512, 8192, 8, 4, 256)
    sched, k, ctas, run = B.dg_attn_schedule_info(8, 4, 256, 8192, 512, 152,
                                                  max_clusters=[0] * 9)
    assert sched == B.DG_SCHEDULE_STREAM_K and ctas == 152
    sched, parts, ctas, run = B.dg_attn_schedule_info(8, 4, 256, 8192, 512, 152,
                                                      max_clusters=[0] * 9,
                                                      schedule=B.DG_SCHEDULE_SPLIT)
    assert sched == B.DG_SCHEDULE_SPLIT
    assert parts * run >= n_tiles > (parts - 1) * run


def test_bad_arguments_are_rejected():
    for args in [(6, 4, 256, 0, 8, 152), (4, 2, 32, 0, 8, 152), (4, 2, 64, -1, 8, 152),
                 (4, 2, 64, 0, 0, 152), (4, 2, 64, 0, 8, 0)]:
        with pytest.raises(B.DgAttnError):
            B.dg_attn_schedule_info(*args)
    with pytest.raises(B.DgAttnError):
        B.dg_attn_schedule_info(4, 2, 64, 0, 8, 152, schedule=7)
