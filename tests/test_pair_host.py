"""Host-only checks of the FFN pair kernel's planner (q8mv_pair_choose_config), no GPU.

The one-launch pair kernel needs every CTA resident: each product's items (128-column
tiles x K ranges) must fit the resident CTAs, the grid is the larger product's items,
every K range holds at least one block, and a wanted split is honoured or refused.
"""
import itertools
import random

import pytest


@pytest.fixture(scope="module")
def q8():
    import q8_matrix_vector_gb300 as q8mv

    return q8mv


def ceil_div(a, b):
    return (a + b - 1) // b


def check(info, K, Nm, No, sms, cps):
    slots = sms * cps
    for phase, (k, n) in (("up", (K, Nm)), ("down", (Nm, No))):
        kb = ceil_div(k, 32)
        tiles, split = info[f"tiles_{phase}"], info[f"split_{phase}"]
        assert tiles == ceil_div(n, 128), phase
        assert 1 <= split <= 64 and tiles * split <= slots, phase
        bps = ceil_div(kb, split)
        assert (split - 1) * bps < kb, f"{phase}: an empty K range"
        assert split * bps >= kb, phase
    assert info["grid"] == max(info["tiles_up"] * info["split_up"], info["tiles_down"] * info["split_down"])
    assert info["grid"] <= slots
    assert info["one_launch"] == 1


def test_7b_ffn_pair_plan(q8):
    info = q8.choose_pair_config(4096, 11008, 4096, 152, 2)
    # 86 up tiles x 3 ranges and 32 down tiles x 9 ranges within 304 resident CTAs
    assert (info["tiles_up"], info["split_up"], info["tiles_down"], info["split_down"]) == (86, 3, 32, 9)
    assert info["grid"] == 288 and info["threads_per_cta"] == 256
    check(info, 4096, 11008, 4096, 152, 2)
    info = q8.choose_pair_config(4096, 11008, 4096, 152, 4, cta_threads=128)
    assert info["threads_per_cta"] == 128 and (info["split_up"], info["split_down"]) == (7, 19)
    check(info, 4096, 11008, 4096, 152, 4)


def test_pair_plans_hold_their_invariants():
    import q8_matrix_vector_gb300 as q8

    rng = random.Random(7)
    for _ in range(300):
        K = rng.randint(1, 20000)
        Nm = 8 * rng.randint(1, 4000)
        No = 8 * rng.randint(1, 4000)
        sms = rng.choice([1, 8, 76, 132, 152])
        cps = rng.randint(1, 4)
        if ceil_div(Nm, 128) > sms * cps or ceil_div(No, 128) > sms * cps:
            with pytest.raises(q8.Q8mvError):
                q8.choose_pair_config(K, Nm, No, sms, cps)
            continue
        check(q8.choose_pair_config(K, Nm, No, sms, cps), K, Nm, No, sms, cps)


@pytest.mark.parametrize("split_up,split_down", [(1, 1), (2, 7), (7, 2), (15, 22)])
def test_wanted_splits_are_honoured(q8, split_up, split_down):
    info = q8.choose_pair_config(4100, 1376, 1024, 152, 2, split_up=split_up, split_down=split_down)
    assert (info["split_up"], info["split_down"]) == (split_up, split_down)
    check(info, 4100, 1376, 1024, 152, 2)


def test_shapes_and_splits_the_kernel_cannot_take(q8):
    for K, Nm, No in ((0, 256, 256), (256, 0, 256), (256, 204, 64), (256, 256, 60)):
        with pytest.raises(q8.Q8mvError):
            q8.choose_pair_config(K, Nm, No, 152, 2)
    with pytest.raises(q8.Q8mvError):  # 16 ranges of 129 blocks leave a range empty (9 blocks each: 15 used)
        q8.choose_pair_config(4100, 1376, 1024, 152, 2, split_up=16)
    with pytest.raises(q8.Q8mvError):  # more items than resident CTAs
        q8.choose_pair_config(4096, 11008, 4096, 152, 2, split_up=4)
    with pytest.raises(q8.Q8mvError):
        q8.choose_pair_config(4096, 11008, 4096, 152, 2, cta_threads=64)
    with pytest.raises(q8.Q8mvError):
        q8.choose_pair_config(4096, 11008, 4096, 0, 2)
