"""Host logic of the tensor-core planner's segment length (no GPU): the library's
choice through la_test_segment_plan against an independent simulation of the
block schedule it models, and against the one-wave rule it replaces.

The schedule: a sequence of nchunks chunks is cut into segments of L chunks (the
last one shorter); every (segment, head) pair is one block; blocks are taken
longest first, each on the SM that frees up first, and each costs its chunks plus
one chunk of set-up.  The planner keeps the L with the earliest finish among those
giving half a wave to two waves of blocks.
"""
import heapq
import math

import pytest


@pytest.fixture(scope="module")
def la():
    import kernelized_linear_attention_gb300 as m
    import os
    if not os.path.exists(m.library_path()):
        from kernelized_linear_attention_gb300 import build
        build.build()
    m.load_library()
    return m


def makespan(nchunks, pairs, nsm, lc):
    """Independent restatement: list every block, longest first, onto a heap of SM free times."""
    segs = math.ceil(nchunks / lc)
    sizes = [lc] * ((segs - 1) * pairs) + [nchunks - (segs - 1) * lc] * pairs
    sizes.sort(reverse=True)
    free = [0] * nsm
    end = 0
    for s in sizes:
        t = heapq.heappop(free) + s + 1
        end = max(end, t)
        heapq.heappush(free, t)
    return end


def one_wave_chunks(nchunks, pairs, nsm):
    per = max(1, nsm // pairs)
    return math.ceil(math.ceil(nchunks * 128 / per) / 128)


@pytest.mark.parametrize("nchunks,pairs,want", [(512, 16, 54), (128, 32, 29), (32, 64, 14)])
def test_bench_workloads_on_152_sms(la, nchunks, pairs, want):
    # B1 H16 N65536, B4 H8 N16384, B8 H8 N4096
    lc, ms = la.la_test_segment_plan(nchunks, pairs, 152)
    assert lc == want
    assert ms == makespan(nchunks, pairs, 152, lc)
    assert ms < makespan(nchunks, pairs, 152, one_wave_chunks(nchunks, pairs, 152))


def test_headline_schedule_in_detail(la):
    # 144 blocks of 54 chunks and 16 of 26: 152 start at once, the last eight short blocks
    # where the first eight end (27 + 27 chunk times), so the 54-chunk blocks finish last
    assert la.la_test_segment_plan(512, 16, 152, 54) == (54, 55)
    assert la.la_test_segment_plan(512, 16, 152, 57) == (57, 58)
    assert la.la_test_segment_plan(512, 16, 152, 53)[1] == makespan(512, 16, 152, 53) == 72


@pytest.mark.parametrize("nsm", [8, 37, 152])
def test_choice_is_the_best_candidate_and_never_worse_than_one_wave(la, nsm):
    for nchunks in (1, 2, 3, 7, 16, 33, 64, 100, 257):
        for pairs in (1, 2, 3, 5, 16, 40, 64):
            lc, ms = la.la_test_segment_plan(nchunks, pairs, nsm)
            base = one_wave_chunks(nchunks, pairs, nsm)
            cands = [L for L in range(1, nchunks + 1)
                     if math.ceil(nchunks / L) * pairs <= 2 * nsm
                     and math.ceil(nchunks / L) >= max(1, math.ceil(nsm / (2 * pairs)))]
            if lc == 0:
                # no length gives half a wave to two waves: the call keeps the one-wave rule
                assert not cands
                continue
            assert 1 <= lc <= nchunks
            assert ms == makespan(nchunks, pairs, nsm, lc)
            best = min(makespan(nchunks, pairs, nsm, L) for L in cands)
            assert ms == best
            # ties go to the longest such length
            assert lc == max(L for L in cands if makespan(nchunks, pairs, nsm, L) == best)
            if math.ceil(nchunks / base) * pairs <= 2 * nsm and base in cands:
                assert ms <= makespan(nchunks, pairs, nsm, base)


def test_rejects_empty_arguments(la):
    with pytest.raises(ValueError):
        la.la_test_segment_plan(0, 1, 152)
    with pytest.raises(ValueError):
        la.la_test_segment_plan(4, 0, 152)
