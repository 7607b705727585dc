"""GPU parity of the slot-stable buffer (incremental gather of the rows of
newly active ids) through the C ABI, against the oracle's OracleSlots.

Every checked step compares bit-exactly the slot table, the high-water mark,
the (slot, id) list of the rows the update copied and every occupied slot's
row against W_head; the logits of occupied slots within 1e-2 * max|oracle
logit| per row; and the top-k by the same rule as the full repack (ids and
values must be those of the canonical path on the same I_t).
"""

import numpy as np
import pytest
import torch

import oracle
from synth import Workload, WorkloadConfig, get_config

from parity import check_logits, check_state, check_topk, dev_bf16, dev_f32, dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import speculative_decoding_draft_stream_gb300 as p
    from speculative_decoding_draft_stream_gb300 import build

    build.build()
    p.load_library()
    return p


def _handle(pkg, cfg, max_prompt):
    return pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=max(cfg.n_tree, 1), max_k=cfg.k,
                      batch=1, max_prompt=max_prompt)


def check_slots(h, seq, osl: oracle.OracleSlots, pairs, W_bits, full=True):
    slot_id, meta, new_slots, new_ids, rows = h.get_slots(seq)
    table = slot_id.cpu().numpy()
    assert np.array_equal(table, osl.slot_id), "slot table differs"
    meta = meta.cpu().numpy()
    assert int(meta[0]) == oracle.slot_high_water(osl.slot_id), "high-water mark differs"
    assert int(meta[1]) == len(pairs), "number of copied rows differs"
    n = len(pairs)
    assert new_slots[:n].cpu().numpy().tolist() == [p[0] for p in pairs], "copied slots differ"
    assert new_ids[:n].cpu().numpy().tolist() == [p[1] for p in pairs], "copied ids differ"
    occ = np.flatnonzero(table >= 0)
    if full or n:
        got = rows.cpu().numpy().view(np.uint16)
        want_rows = occ if full else np.array([p[0] for p in pairs], dtype=np.int64)
        assert np.array_equal(got[want_rows], W_bits[table[want_rows]]), "slot rows differ"
    return table


def check_slot_projection(logits_dev, ids_dev, vals_dev, hid_bits, osl: oracle.OracleSlots, I, k):
    """Logits of occupied slots, and the top-k against the canonical rule."""
    table = osl.slot_id
    occ = np.flatnonzero(table >= 0)
    want_slots, _, _ = osl.project_topk(hid_bits, k)
    got = logits_dev.cpu().numpy()
    if len(occ) == 0:
        assert np.all(ids_dev.cpu().numpy() == -1)
        return
    tol = check_logits(got[:, occ], want_slots[:, occ])
    col = {int(x): j for j, x in enumerate(np.asarray(I).tolist())}
    want_by_I = np.empty((want_slots.shape[0], len(I)), dtype=np.float32)
    for s in occ:
        want_by_I[:, col[int(table[s])]] = want_slots[:, s]
    check_topk(ids_dev.cpu().numpy(), vals_dev.cpu().numpy(), want_by_I, I, k, tol)


def _run(pkg, cfg: WorkloadConfig, fused: bool, steps=None, logit_steps=None, one_launch=False):
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    seq = 0
    with _handle(pkg, cfg, wl.prompt_len(seq)) as h:
        prompt = wl.prompt(seq)
        Z = wl.prefill_logits(seq) if cfg.K_pre > 0 else None
        ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        ost.init(prompt, Z)
        osl = oracle.OracleSlots(cfg.W_max, cfg.H)
        h.stream_init(seq, dev_i32(prompt), dev_f32(Z) if Z is not None else None)
        h.build_active_vocab(seq)
        # the update right after init lays I_1 out ascending
        h.gather_new_head_rows(seq, W_dev)
        I = ost.active()
        pairs = osl.update(I, W)
        check_slots(h, seq, osl, pairs, W)
        logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        trees = wl.trees(seq)
        for t in range(cfg.steps if steps is None else steps):
            vb = wl.verify_logits(seq, t) if cfg.K_ver > 0 else None
            vr = wl.verify_row(seq, t)
            hid = wl.hiddens(seq, t)
            tree_d, hid_d = dev_i32(trees[t]), dev_bf16(hid)
            vb_d = dev_f32(vb) if vb is not None else None
            if fused:
                if one_launch:  # the table matches the window: ns_step_slots is the one-launch kernel
                    assert h.step_slots_fused(seq) == 1
                ids, vals = h.step_slots(seq, tree_d, vb_d, vr, W_dev, hid_d, cfg.k, logits=logits)
            else:
                h.state_update(seq, tree_d, vb_d, vr)
                h.gather_new_head_rows(seq, W_dev)
                ids, vals = h.slot_lm_head_logits_topk(seq, hid_d, cfg.k, logits=logits)
            ost.append(trees[t], vb, vr)
            I = check_state(h, seq, ost, full=False)
            pairs = osl.update(I, W)
            sampled = logit_steps is None or t in logit_steps
            check_slots(h, seq, osl, pairs, W, full=sampled)
            if sampled:
                check_slot_projection(logits, ids, vals, hid, osl, I, cfg.k)
        assert h.get_error() == 0


TOY = get_config("toy_v4096_h256")
MID = WorkloadConfig(name="mid", V=20011, H=1024, W_max=1000, K_pre=3, K_ver=3, prompt_len=700, self_copy=0.4,
                     zipf_s=1.05, steps=12, n_tree=60, tree_local=0.7, tree_recent=256, n_verify=4)
WIDE = WorkloadConfig(name="h4096", V=30011, H=4096, W_max=700, K_pre=3, K_ver=3, prompt_len=500, self_copy=0.4,
                      zipf_s=1.05, steps=6, n_tree=60, tree_local=0.7, tree_recent=256, n_verify=2)
EDGE = [
    WorkloadConfig(name="tiny", V=64, H=64, W_max=4, K_pre=1, K_ver=2, prompt_len=9, self_copy=0.3, zipf_s=1.0,
                   steps=10, n_tree=5, tree_local=0.5, tree_recent=4, n_verify=3),
    WorkloadConfig(name="w1", V=300, H=128, W_max=1, K_pre=2, K_ver=1, prompt_len=20, self_copy=0.2, zipf_s=1.1,
                   steps=6, n_tree=7, tree_local=0.5, tree_recent=8, n_verify=1),
    WorkloadConfig(name="wide", V=5000, H=192, W_max=8192, K_pre=3, K_ver=3, prompt_len=100, self_copy=0.5,
                   zipf_s=1.1, steps=5, n_tree=30, tree_local=0.5, tree_recent=64, n_verify=2),
    WorkloadConfig(name="noK", V=1001, H=64, W_max=50, K_pre=0, K_ver=0, prompt_len=40, self_copy=0.3, zipf_s=1.0,
                   steps=6, n_tree=12, tree_local=0.6, tree_recent=16, n_verify=1),
    WorkloadConfig(name="n1", V=2048, H=256, W_max=130, K_pre=3, K_ver=3, prompt_len=50, self_copy=0.3,
                   zipf_s=1.1, steps=4, n_tree=1, tree_local=0.5, tree_recent=16, n_verify=1, k=7),
]


@pytest.mark.parametrize("fused", [False, True], ids=["separate_calls", "step_slots"])
@pytest.mark.parametrize("cfg", [TOY, MID, WIDE] + EDGE, ids=lambda c: c.name)
def test_slots_every_step(pkg, cfg, fused):
    _run(pkg, cfg, fused, one_launch=fused and cfg in (TOY, MID, WIDE))


def test_slots_full_size_llama(pkg):
    """The Llama-3-8B-shaped head (V=128256, H=4096, W_max=3072): slot state
    on 40 one-launch steps, logits and top-k on a sample of them."""
    cfg = get_config("llama3_8b_v128256_h4096")
    _run(pkg, cfg, True, steps=40, logit_steps={0, 1, 2, 3, 17, 39}, one_launch=True)


def test_step_slots_paths_interleave(pkg):
    """ns_step_slots is one launch only while the slot table matches the
    window: a canonical step, an append with a rebuild, or a state update in
    between send it down the multi-launch chain once, which puts the table
    back in step.  Every step of the mix is checked against the oracle."""
    cfg = MID
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    # what runs at each step: the slot step, or a window change without a slot update first
    plan = ["slots", "slots", "step", "slots", "slots", "append", "slots", "update", "slots", "slots", "slots",
            "slots"]
    assert len(plan) <= cfg.steps
    with _handle(pkg, cfg, wl.prompt_len(0)) as h:
        ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        osl = oracle.OracleSlots(cfg.W_max, cfg.H)
        prompt, Z = wl.prompt(0), wl.prefill_logits(0)
        ost.init(prompt, Z)
        h.stream_init(0, dev_i32(prompt), dev_f32(Z))
        h.build_active_vocab(0)
        assert h.step_slots_fused(0) == 0  # the table is empty, the window is not
        trees = wl.trees(0)
        logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        for t, what in enumerate(plan):
            vb, vr, hid = wl.verify_logits(0, t), wl.verify_row(0, t), wl.hiddens(0, t)
            tree_d, vb_d, hid_d = dev_i32(trees[t]), dev_f32(vb), dev_bf16(hid)
            ost.append(trees[t], vb, vr)
            if what == "slots":
                expect = 0 if t == 0 or plan[t - 1] != "slots" else 1
                assert h.step_slots_fused(0) == expect, (t, what)
                ids, vals = h.step_slots(0, tree_d, vb_d, vr, W_dev, hid_d, cfg.k, logits=logits)
                assert h.step_slots_fused(0) == 1
                I = check_state(h, 0, ost, full=False)
                pairs = osl.update(I, W)
                check_slots(h, 0, osl, pairs, W)
                check_slot_projection(logits, ids, vals, hid, osl, I, cfg.k)
            else:
                if what == "step":
                    h.step(0, tree_d, vb_d, vr, W_dev, hid_d, cfg.k)
                elif what == "append":
                    h.stream_append(0, tree_d, vb_d, vr)
                    h.build_active_vocab(0)
                else:
                    h.state_update(0, tree_d, vb_d, vr)
                assert h.step_slots_fused(0) == 0, (t, what)
                check_state(h, 0, ost, full=False)
        assert h.get_error() == 0


def test_slots_follow_any_update_schedule(pkg):
    """Slot updates skipped for several canonical steps, then one update:
    the table moves straight from the old active set to the current one; a
    re-initialised stream empties it."""
    cfg = MID
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    with _handle(pkg, cfg, wl.prompt_len(0)) as h:
        ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        osl = oracle.OracleSlots(cfg.W_max, cfg.H)
        prompt, Z = wl.prompt(0), wl.prefill_logits(0)
        ost.init(prompt, Z)
        h.stream_init(0, dev_i32(prompt), dev_f32(Z))
        h.build_active_vocab(0)
        h.gather_new_head_rows(0, W_dev)
        check_slots(h, 0, osl, osl.update(ost.active(), W), W)
        trees = wl.trees(0)
        for t in range(cfg.steps):
            vb, vr, hid = wl.verify_logits(0, t), wl.verify_row(0, t), wl.hiddens(0, t)
            h.step(0, dev_i32(trees[t]), dev_f32(vb), vr, W_dev, dev_bf16(hid), cfg.k)
            ost.append(trees[t], vb, vr)
            if t % 4 == 3:  # a slot update every fourth step only
                h.gather_new_head_rows(0, W_dev)
                I = ost.active()
                check_slots(h, 0, osl, osl.update(I, W), W)
                logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
                ids, vals = h.slot_lm_head_logits_topk(0, dev_bf16(hid), cfg.k, logits=logits)
                check_slot_projection(logits, ids, vals, hid, osl, I, cfg.k)
        # re-initialisation empties the table; the next update lays I_1 out ascending
        ost.init(prompt, Z)
        osl = oracle.OracleSlots(cfg.W_max, cfg.H)
        h.stream_init(0, dev_i32(prompt), dev_f32(Z))
        slot_id, meta, _, _, _ = h.get_slots(0)
        assert np.all(slot_id.cpu().numpy() == -1) and meta.cpu().numpy().tolist() == [0, 0]
        h.build_active_vocab(0)
        h.gather_new_head_rows(0, W_dev)
        check_slots(h, 0, osl, osl.update(ost.active(), W), W)
        assert h.get_error() == 0


def _draft_phase(pkg, cfg, steps, depth=6):
    """An EAGLE-style draft phase on the slot buffer: per step one state
    update and one slot gather, then `depth` projections of the same I_t
    with different hidden rows (one per level of the draft tree), each
    against the oracle."""
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    with _handle(pkg, cfg, wl.prompt_len(0)) as h:
        prompt, Z = wl.prompt(0), wl.prefill_logits(0)
        ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        ost.init(prompt, Z)
        osl = oracle.OracleSlots(cfg.W_max, cfg.H)
        h.stream_init(0, dev_i32(prompt), dev_f32(Z))
        h.build_active_vocab(0)
        h.gather_new_head_rows(0, W_dev)
        osl.update(ost.active(), W)
        logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        trees = wl.trees(0)
        for t in range(steps):
            vb, vr = wl.verify_logits(0, t), wl.verify_row(0, t)
            h.state_update(0, dev_i32(trees[t]), dev_f32(vb), vr)
            h.gather_new_head_rows(0, W_dev)
            ost.append(trees[t], vb, vr)
            I = check_state(h, 0, ost, full=False)
            pairs = osl.update(I, W)
            check_slots(h, 0, osl, pairs, W, full=False)
            for d in range(depth):
                hid = wl.hiddens(0, cfg.steps + t * depth + d)
                ids, vals = h.slot_lm_head_logits_topk(0, dev_bf16(hid), cfg.k, logits=logits)
                check_slot_projection(logits, ids, vals, hid, osl, I, cfg.k)
        assert h.get_error() == 0


def test_one_gather_serves_a_draft_phase(pkg):
    _draft_phase(pkg, MID, steps=6)


def test_one_gather_serves_a_draft_phase_full_size(pkg):
    _draft_phase(pkg, get_config("llama3_8b_v128256_h4096"), steps=3)
