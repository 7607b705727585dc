"""Pins of the oracle's batched shared gather (CPU only): one packed buffer
holding the union of several sequences' I_t, each sequence ranking only its
own columns.  Hand-worked cases (tests/golden/union_toys.json), invariants,
and equality with each sequence's own sub-head step on a synthetic batch.
"""

import json
import os

import numpy as np

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden", "union_toys.json")
with open(GOLD) as f:
    UNION = json.load(f)


def _bf16(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_union_golden():
    g = UNION["union"]
    U, M = O.union_vocab(g["I"])
    assert U.tolist() == g["U"]
    assert M.astype(int).tolist() == g["M"]


def test_union_projection_ranks_own_columns_only():
    g = UNION["projection"]
    W = _bf16([[x, 1.0] for x in range(g["V"])])
    hid = [_bf16([[1.0, 0.0]]) for _ in g["I"]]
    U, M, packed, logits, ids, vals = O.union_sub_head_step(hid, W, g["I"], g["k"])
    assert U.tolist() == [2, 5, 9]
    assert np.array_equal(packed, W[U])
    for b in range(len(g["I"])):
        assert ids[b].tolist() == g["ids"][b]
        assert [float(v) for v in vals[b][0]] == [float(v) for v in g["vals"][b][0]]
        assert logits[b].tolist() == [[2.0, 5.0, 9.0]]


def test_union_equals_each_sequence_alone():
    from synth import Workload, get_config

    cfg = get_config("toy_v4096_h256").with_(batch=3, steps=4)
    wl = Workload(cfg)
    W = wl.w_head()
    streams = []
    for b in range(cfg.batch):
        o = O.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        o.init(wl.prompt(b), wl.prefill_logits(b))
        streams.append(o)
    trees = [wl.trees(b) for b in range(cfg.batch)]
    for t in range(cfg.steps):
        for b, o in enumerate(streams):
            o.append(trees[b][t], wl.verify_logits(b, t), wl.verify_row(b, t))
        I_list = [o.active() for o in streams]
        hid = [wl.hiddens(b, t) for b in range(cfg.batch)]
        U, M, packed, logits, ids, vals = O.union_sub_head_step(hid, W, I_list, cfg.k)
        assert np.all(np.diff(U) > 0)                                   # ascending, no repeats
        assert set(U.tolist()) == set().union(*[set(I.tolist()) for I in I_list])
        assert M.sum(axis=1).tolist() == [len(I) for I in I_list]
        assert len(U) < sum(len(I) for I in I_list)                     # the sequences share rows
        assert np.array_equal(packed, W[U])
        for b, I in enumerate(I_list):
            _, lb, ib, vb = O.sub_head_step(hid[b], W, I, cfg.k)
            assert np.array_equal(ids[b], ib) and np.array_equal(vals[b], vb)
            assert np.array_equal(logits[b][:, M[b]], lb)
