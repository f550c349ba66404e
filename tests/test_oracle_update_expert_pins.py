"""Pins of the MoeUpdateExpert oracle ("MoeUpdateExpert", 功能说明 and
参数说明): logical -> physical mapping through the EPLB table, pruning by
threshold, the active mask."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

TABLE = np.array([[1, 7, 0, 0],     # expert 0: one instance, 7
                  [2, 3, 5, 0],     # expert 1: instances 3, 5
                  [3, 1, 4, 6]],    # expert 2: instances 1, 4, 6
                 np.int32)


def test_hand_worked_by_rank_and_by_token():
    ids = np.array([[0, 1, 2], [2, 1, 0]], np.int32)
    # by rank, localRankId 4: expert 0 -> 4 % 1 = 0 -> 7; expert 1 -> 4 % 2 = 0 -> 3;
    # expert 2 -> 4 % 3 = 1 -> 4
    o = oracle.update_expert(ids, TABLE, local_rank=4, balance_mode=0)
    assert o["balancedExpertIds"].tolist() == [[7, 3, 4], [4, 3, 7]]
    assert o["balancedActiveMask"] is None
    # by token: token 0 -> index 0 of each row, token 1 -> 1 % count
    o = oracle.update_expert(ids, TABLE, local_rank=4, balance_mode=1)
    assert o["balancedExpertIds"].tolist() == [[7, 3, 1], [4, 5, 7]]
    # int64 ids keep their dtype
    o = oracle.update_expert(ids.astype(np.int64), TABLE, local_rank=1, balance_mode=0)
    assert o["balancedExpertIds"].dtype == np.int64
    assert o["balancedExpertIds"].tolist() == [[7, 5, 4], [4, 5, 7]]


def test_invalid_ids_and_counts_give_minus_one():
    ids = np.array([[-1, 3, 1]], np.int32)
    bad = TABLE.copy()
    bad[1, 0] = 4                       # count larger than the F - 1 columns
    o = oracle.update_expert(ids, bad, local_rank=0, balance_mode=0)
    assert o["balancedExpertIds"].tolist() == [[-1, -1, -1]]


def test_pruning_by_hand():
    ids = np.array([[0, 1, 2], [2, 1, 0], [1, 2, 0]], np.int32)
    scales = np.array([[0.6, 0.3, 0.1], [0.5, 0.25, 0.25], [0.9, 0.06, 0.04]], np.float32)
    thr = np.array([0.2, 0.25, 0.1], np.float32)
    active = np.array([True, True, False])
    o = oracle.update_expert(ids, TABLE, local_rank=0, balance_mode=0, scales=scales, scales_dtype=3,
                             threshold=thr, active=active)
    # 0.3 >= 0.25 kept, 0.1 >= 0.1 kept (not below), 0.25 >= 0.25 kept; token 2 inactive
    assert o["balancedActiveMask"].tolist() == [[True, True, True], [True, True, True],
                                                [False, False, False]]
    thr = np.array([0.2, 0.26, 0.3], np.float32)
    o = oracle.update_expert(ids, TABLE, local_rank=0, balance_mode=0, scales=scales, scales_dtype=3,
                             threshold=thr, active=None)
    assert o["balancedActiveMask"].tolist() == [[True, True, False], [True, False, False],
                                                [True, False, False]]


@pytest.mark.parametrize("mode,seed,sdt", [(0, 0, 3), (1, 1, 1), (0, 2, 0), (1, 3, 3)])
def test_invariants_on_generated_inputs(mode, seed, sdt):
    inp = w.make_update_expert(BS=128, K=8, moe_expert_num=64, world_size=16, place_per_rank=8,
                               scales_dtype=sdt, seed=seed)
    t = inp["table"]
    o = oracle.update_expert(inp["expert_ids"], t, local_rank=5, balance_mode=mode,
                             scales=inp["scales"], scales_dtype=sdt, threshold=inp["threshold"],
                             active=inp["active"])
    bal = o["balancedExpertIds"]
    ids = inp["expert_ids"]
    for b in range(ids.shape[0]):
        for k in range(ids.shape[1]):
            e = ids[b, k]
            inst = t[e, 1:1 + t[e, 0]]
            assert bal[b, k] in inst
            c = (5 if mode == 0 else b) % t[e, 0]
            assert bal[b, k] == inst[c]
    # instance ids are never shared between logical experts, so the mapping is invertible
    owner = {int(i): e for e in range(t.shape[0]) for i in t[e, 1:1 + t[e, 0]]}
    assert all(owner[int(bal[b, k])] == ids[b, k] for b in range(ids.shape[0]) for k in range(ids.shape[1]))
    # pruning against torch's comparison of the fp32 scales; a prefix per token
    sc = torch.from_numpy(inp["scales"].view(np.int16)).view(
        {0: torch.float16, 1: torch.bfloat16}[sdt]).float().numpy() if sdt != 3 else inp["scales"]
    ref = inp["active"][:, None] & ~(sc < inp["threshold"][None, :])
    assert np.array_equal(o["balancedActiveMask"], ref)
    m = o["balancedActiveMask"].astype(np.int8)
    assert np.all(np.diff(m, axis=1) <= 0)
