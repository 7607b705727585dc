"""Pins of the oracle's slot-stable packed buffer (CPU only).

The reading pinned here (the pages fix no slot rule): an update frees every
slot whose id left I_t, then the ids of I_t that hold no slot take the free
slots in ascending id order, lowest slot first.  Hand-worked tables
(tests/golden/slot_toys.json), a brute-force search over every assignment on
tiny cases, the invariants that characterise the rule, and equality of the
top-k with the full-repack path on a whole synthetic stream.
"""

import itertools
import json
import os
import random

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden", "slot_toys.json")
with open(GOLD) as f:
    SLOTS = json.load(f)


def _bf16(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("toy", SLOTS["toys"], ids=lambda t: t["name"])
def test_slot_toys(toy):
    table = [-1] * toy["W_max"]
    for st in toy["steps"]:
        table, pairs = O.slot_update(table, st["I"])
        assert table.tolist() == st["table"]
        assert [list(p) for p in pairs] == st["pairs"]
        assert O.slot_high_water(table) == st["hw"]


def test_slot_projection_ties_go_to_the_smaller_id():
    pj = SLOTS["projection"]
    W = _bf16([[x, 1.0] for x in range(pj["V"])])
    table = np.array(pj["table"], dtype=np.int32)
    rows = np.zeros((len(table), 2), dtype=np.uint16)
    rows = O.slot_gather(rows, W, [(s, x) for s, x in enumerate(table) if x >= 0])
    logits, ids, vals = O.slot_project_topk(_bf16(pj["hidden"]), rows, table, pj["k"])
    assert ids.tolist() == pj["ids"]
    assert vals.tolist() == pj["vals"]
    assert logits.shape == (2, len(table))
    assert logits[0].tolist() == [float(x) for x in table]


def _brute_force(table, I):
    """The assignment the rule describes, found by search: among every
    injective map of the unplaced ids onto free slots, the one whose slots,
    listed for the ids in ascending order, are lexicographically smallest."""
    I = set(I)
    t = [x if x in I else -1 for x in table]
    new = sorted(I - set(t))
    free = [s for s, x in enumerate(t) if x < 0]
    best = min(itertools.permutations(free, len(new)))
    for s, x in zip(best, new):
        t[s] = x
    return t


def test_slot_update_brute_force_tiny():
    rng = random.Random(7)
    for _ in range(300):
        W_max = rng.randint(1, 6)
        table = [-1] * W_max
        for _ in range(6):
            I = sorted(rng.sample(range(10), rng.randint(0, W_max)))
            want = _brute_force(table, I)
            table, _ = O.slot_update(table, I)
            assert table.tolist() == want


def test_slot_invariants_random_sequences():
    rng = random.Random(11)
    for _ in range(100):
        W_max, V = rng.randint(1, 12), 24
        table = np.full(W_max, -1, dtype=np.int32)
        prev = set()
        for _ in range(10):
            I = sorted(rng.sample(range(V), rng.randint(0, W_max)))
            old = table.copy()
            table, pairs = O.slot_update(table, I)
            occ = [int(x) for x in table if x >= 0]
            assert sorted(occ) == I                                 # every active id holds exactly one slot
            for s in range(W_max):                                   # survivors keep their slot
                if old[s] >= 0 and old[s] in set(I):
                    assert table[s] == old[s]
            assert [x for _, x in pairs] == sorted(set(I) - prev)    # only newly active rows are gathered
            freed = [s for s in range(W_max) if old[s] < 0 or old[s] not in set(I)]
            assert [s for s, _ in pairs] == freed[:len(pairs)]       # lowest free slots, in order
            hw = O.slot_high_water(table)
            assert all(x < 0 for x in table[hw:]) and (hw == 0 or table[hw - 1] >= 0)
            prev = set(I)


def test_slot_update_rejects_overfull():
    with pytest.raises(ValueError):
        O.slot_update([-1, -1], [1, 2, 3])


def test_slot_path_equals_full_repack_on_a_stream():
    from synth import Workload, get_config

    cfg = get_config("toy_v4096_h256")
    wl = Workload(cfg)
    W = wl.w_head()
    st = O.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
    st.init(wl.prompt(0), wl.prefill_logits(0))
    sl = O.OracleSlots(cfg.W_max, cfg.H)
    trees = wl.trees(0)
    prev = None
    copied = 0
    for t in range(cfg.steps):
        if t > 0:
            st.append(trees[t - 1], wl.verify_logits(0, t - 1), wl.verify_row(0, t - 1))
        I = st.active()
        pairs = sl.update(I, W)
        copied += len(pairs)
        if prev is None:  # the first update lays I_1 out ascending, like the full repack
            assert sl.slot_id[:len(I)].tolist() == I.tolist()
        else:
            assert len(pairs) == len(set(I.tolist()) - set(prev.tolist()))
        occ = np.flatnonzero(sl.slot_id >= 0)
        assert np.array_equal(sl.rows[occ], W[sl.slot_id[occ]])     # every occupied slot holds its row
        hid = wl.hiddens(0, t)
        _, logits, ids, vals = O.sub_head_step(hid, W, I, cfg.k)
        slogits, sids, svals = sl.project_topk(hid, cfg.k)
        assert np.array_equal(sids, ids) and np.array_equal(svals, vals)
        col = {int(x): j for j, x in enumerate(I)}
        for s in occ:
            assert np.array_equal(slogits[:, s], logits[:, col[int(sl.slot_id[s])]])
        prev = I
    assert copied < cfg.steps * cfg.W_max  # far fewer rows than one full repack per step
