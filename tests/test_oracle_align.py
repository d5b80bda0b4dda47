"""Pins of the oracle's align step (no GPU): the expert_offsets invariants, a
brute-force sort, capacity bounds and the grouped-launch validation vectors."""
import json
import os

import numpy as np
import pytest

import oracle as orc
from conftest import GOLDEN
from mixture_experts_grouped_gb300.synth import random_ids


def check_align_invariants(ids, E, bs, res, max_padded):
    """Properties that pin an align result without recomputing it."""
    ids = np.asarray(ids).reshape(-1)
    P = ids.shape[0]
    off = res.expert_offsets.astype(np.int64)
    assert off.shape == (E + 1,)
    assert off[0] == 0 and np.all(np.diff(off) >= 0)                 # non-negative, non-decreasing
    assert off[E] == res.total_tokens_post_pad <= max_padded          # last entry is the padded total
    assert np.all(off % bs == 0)                                      # every span a bs multiple
    st = res.sorted_token_ids
    assert st.shape == (max_padded,)
    valid = (ids >= 0) & (ids < E)
    real = st[st != P]
    assert sorted(real.tolist()) == np.nonzero(valid)[0].tolist()     # a permutation of the kept pairs
    assert np.all(st[res.total_tokens_post_pad:] == P)
    for e in range(E):
        seg = st[off[e]:off[e + 1]]
        n = int(np.sum(ids == e))
        assert off[e + 1] - off[e] == -(-n // bs) * bs
        assert np.all(ids[seg[:n]] == e) and np.all(np.diff(seg[:n]) > 0)   # stable
        assert np.all(seg[n:] == P)
        assert np.all(res.expert_ids[off[e] // bs: off[e + 1] // bs] == e)
    assert np.all(res.expert_ids[res.total_tokens_post_pad // bs:] == -1)
    p2r = res.pair_to_row
    for p in range(P):
        if valid[p]:
            assert st[p2r[p]] == p
        else:
            assert p2r[p] == -1


@pytest.mark.parametrize("P,E,bs,skew", [
    (0, 4, 16, 0), (1, 1, 1, 0), (7, 3, 1, 0), (32, 8, 16, 0), (100, 8, 16, 1.5),
    (500, 128, 64, 1.1), (1000, 256, 16, 0), (4096, 8, 64, 0), (3000, 64, 16, 2.0),
    (257, 2, 256, 0),
])
def test_invariants(P, E, bs, skew):
    ids = random_ids(P + E, P, E, skew)
    cap = orc.align_capacity(P, E, bs)
    res = orc.align_block_size(ids, E, bs, cap)
    check_align_invariants(ids, E, bs, res, cap)
    assert res.err == 0


def test_brute_force_tiny():
    ids = np.array([3, 0, 3, 1, 0, 3, 3, 2, 0, 3], np.int32)
    res = orc.align_block_size(ids, 5, 4, 32)
    P = 10
    # expert 0: pairs 1, 4, 8 + 1 pad; expert 1: pair 3 + 3 pads; expert 2: pair 7 + 3 pads;
    # expert 3: pairs 0, 2, 5, 6, 9 + 3 pads; expert 4: empty
    want = [1, 4, 8, P, 3, P, P, P, 7, P, P, P, 0, 2, 5, 6, 9, P, P, P]
    assert res.sorted_token_ids[:20].tolist() == want
    assert res.sorted_token_ids[20:].tolist() == [P] * 12
    assert res.expert_offsets.tolist() == [0, 4, 8, 12, 20, 20]
    assert res.total_tokens_post_pad == 20
    assert res.expert_ids.tolist() == [0, 1, 2, 3, 3, -1, -1, -1]
    assert res.pair_to_row.tolist() == [12, 0, 13, 4, 1, 14, 15, 8, 2, 16]


def test_block_size_one_has_no_padding():
    ids = random_ids(9, 300, 16, 1.0)
    res = orc.align_block_size(ids, 16, 1)
    assert res.total_tokens_post_pad == 300
    assert np.all(res.sorted_token_ids[:300] != 300)
    # bs = 1 is a plain stable sort by expert
    assert res.sorted_token_ids[:300].tolist() == np.argsort(ids, kind="stable").tolist()


def test_capacity_is_tight_for_one_pair_per_expert():
    E, bs = 16, 8
    ids = np.arange(E, dtype=np.int32)
    cap = orc.align_capacity(E, E, bs)
    res = orc.align_block_size(ids, E, bs, cap)
    assert res.total_tokens_post_pad == cap == E * bs
    # and never exceeded on random skewed routings
    for seed in range(20):
        P, E2, bs2 = 50 + 37 * seed, 1 + seed * 13 % 200, [1, 4, 16, 64][seed % 4]
        ids = random_ids(seed, P, E2, 1.2 * (seed % 3))
        assert orc.align_block_size(ids, E2, bs2).total_tokens_post_pad <= orc.align_capacity(P, E2, bs2)


def test_out_of_range_ids_are_dropped_and_flagged():
    ids = np.array([0, 5, 1, -1, 1], np.int32)
    res = orc.align_block_size(ids, 2, 2)
    assert res.err == 1
    assert res.pair_to_row.tolist()[1] == -1 and res.pair_to_row.tolist()[3] == -1
    check_align_invariants(ids, 2, 2, res, orc.align_capacity(5, 2, 2))


def test_too_small_buffer_rejected():
    with pytest.raises(ValueError):
        orc.align_block_size(np.arange(8, dtype=np.int32), 8, 4, 16)


def test_group_array_vectors():
    with open(os.path.join(GOLDEN, "group_arrays_vectors.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        args = ("t", c["num_experts"], [tuple(p) for p in c["per_expert"]], c["offsets"])
        if c["ok"]:
            orc.ensure_group_arrays(*args)
        else:
            with pytest.raises(orc.GroupArrayError) as ei:
                orc.ensure_group_arrays(*args)
            if "message_contains" in c:
                assert c["message_contains"] in str(ei.value)


def test_align_output_passes_group_array_rules():
    ids = random_ids(3, 999, 40, 1.0)
    res = orc.align_block_size(ids, 40, 16)
    orc.ensure_group_arrays("align", 40, [], res.expert_offsets.tolist())
