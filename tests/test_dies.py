"""Host logic of the grid kernels' die placement, without a GPU.

The grid kernels put each batch group's CTAs on one of the GPU's two dies and
its step counter in a 1 KB block of the workspace homed on that die. On a GPU
the inputs come from L2 flag round trips; rnn_die_plan_for takes them as
stated numbers, so the decisions (which SMs form die 0, which blocks are
homed where, how the groups split over the dies, which block holds each
group's counter) are checked here on the CPU.
"""
import random

import pytest

from recurrent_networks_gb300 import _lib

FAST, SLOW = 1000, 1800  # round trips in cycles: same die / across the dies


def sm_lat(n0, n1, fast=FAST, slow=SLOW):
    # entry 0 is the measuring CTA itself (its own round trip is not measured)
    return [0] + [fast] * (n0 - 1) + [slow] * n1


def test_two_dies_two_groups():
    blk = [FAST, SLOW] * 8
    assert _lib.rnn_die_plan_for(2, 64, sm_lat(72, 80), blk) == (72, 80, 1, [0, 256])


def test_counter_blocks_follow_their_homes():
    # block 0 is homed on die 1, blocks 1.. alternate starting with die 0
    blk = [SLOW] + [FAST, SLOW] * 7 + [FAST]
    d0, d1, g0, words = _lib.rnn_die_plan_for(2, 64, sm_lat(76, 76), blk)
    assert (d0, d1, g0) == (76, 76, 1)
    assert words == [1 * 256, 0]  # group 0 (die 0): first fast block; group 1: first slow one


def test_the_measuring_cta_counts_on_die_0():
    # even with every other CTA far, the measuring CTA's own SM is on die 0
    assert _lib.rnn_die_plan_for(1, 1, [0, SLOW, SLOW, FAST], [FAST, SLOW])[:2] == (2, 2)


@pytest.mark.parametrize("lat", [sm_lat(76, 76, FAST, FAST), sm_lat(76, 76, FAST, int(FAST * 1.25))])
def test_untrusted_sm_split(lat):
    # fast/slow ratio under 1.3: no two-die structure is trusted
    assert _lib.rnn_die_plan_for(2, 64, lat, [FAST, SLOW] * 8) is None


def test_untrusted_block_split():
    assert _lib.rnn_die_plan_for(2, 64, sm_lat(72, 80), [FAST] * 16) is None


def test_no_split_fits():
    # two groups of 76 CTAs: neither die holds one next to the other
    assert _lib.rnn_die_plan_for(2, 76, sm_lat(72, 80), [FAST, SLOW] * 8) is None
    # one group larger than either die
    assert _lib.rnn_die_plan_for(1, 81, sm_lat(72, 80), [FAST, SLOW] * 8) is None


def test_one_group_goes_where_it_fits():
    # 76 CTAs fit die 1 (80 SMs) only
    assert _lib.rnn_die_plan_for(1, 76, sm_lat(72, 80), [FAST, SLOW] * 8)[2:] == (0, [256])


def test_too_few_blocks_homed_on_a_die():
    blk = [FAST] * 15 + [SLOW]
    # four groups of 32 split 2 + 2, but only one block is homed on die 1
    assert _lib.rnn_die_plan_for(4, 32, sm_lat(76, 76), blk) is None
    # three groups split 1 + 2 also need two
    assert _lib.rnn_die_plan_for(3, 32, sm_lat(76, 76), blk) is None
    assert _lib.rnn_die_plan_for(2, 32, sm_lat(76, 76), blk)[2:] == (1, [0, 15 * 256])


@pytest.mark.parametrize("args", [
    (0, 64, sm_lat(72, 80), [FAST, SLOW]),
    (17, 8, sm_lat(72, 80), [FAST, SLOW]),
    (2, 0, sm_lat(72, 80), [FAST, SLOW]),
    (2, 64, [0], [FAST, SLOW]),
    (2, 64, sm_lat(72, 80), []),
    (2, 64, sm_lat(72, 80), [FAST, SLOW] * 9),
])
def test_invalid_arguments(args):
    with pytest.raises(_lib.RnnError) as e:
        _lib.rnn_die_plan_for(*args)
    assert e.value.status == _lib.RNN_EINVAL


def brute_force_split(groups, C, n0, n1):
    """Every k groups on die 0 that fits, the one closest to an even split
    (the smallest such k on a tie), or None."""
    fits = [k for k in range(groups + 1) if k * C <= n0 and (groups - k) * C <= n1]
    return min(fits, key=lambda k: (abs(2 * k - groups), k)) if fits else None


def test_split_and_counters_against_brute_force():
    rng = random.Random(7)
    for _ in range(400):
        n0, n1 = rng.randint(1, 100), rng.randint(1, 100)
        groups, C = rng.randint(1, 16), rng.randint(1, 80)
        nblocks = rng.randint(2, 16)
        homes = [rng.randint(0, 1) for _ in range(nblocks)]
        homes[rng.randrange(nblocks)] = 0
        homes[rng.randrange(nblocks)] = 1  # both dies present, so the block split is trusted
        blk = [FAST if h == 0 else SLOW for h in homes]
        got = _lib.rnn_die_plan_for(groups, C, sm_lat(n0, n1), blk)
        k = brute_force_split(groups, C, n0, n1)
        need = [k, groups - k] if k is not None else None
        if k is None or need[0] > homes.count(0) or need[1] > homes.count(1):
            assert got is None, (groups, C, n0, n1, homes)
            continue
        d0, d1, g0, words = got
        assert (d0, d1, g0) == (n0, n1, k)
        # each group in the first unused block homed on its die, in group order
        free = {0: [i for i, h in enumerate(homes) if h == 0], 1: [i for i, h in enumerate(homes) if h == 1]}
        want = [free[0 if g < k else 1].pop(0) * 256 for g in range(groups)]
        assert words == want
