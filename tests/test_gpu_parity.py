"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Small workloads are compared element by element on every step (state, packed
sub-head, logits, top-k); they still span several 128-row tiles of the fused
kernel, H split over the CTAs of a cluster, and ragged tails.  Edge cases cover the degenerate windows, empty appends, bad
ids, padding, the scalar (V % 4 != 0) paths and the largest K and k.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import Workload, WorkloadConfig, get_config

from parity import (check_logits, check_packed, check_projection, check_state, check_topk, dev_bf16, dev_f32,
                    dev_i32)

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


def _handle(pkg, cfg, batch=1, max_prompt=None, max_k=None):
    return pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=max(cfg.n_tree, 1),
                      max_k=max_k or cfg.k, batch=batch, max_prompt=max_prompt or 4096)


# How a decode step is issued: the five calls of the problem statement, ns_step
# (one cooperative launch where the device holds its grid), or its two halves.
MODES = ["separate_calls", "fused_step", "two_launch"]


def _run_workload(pkg, cfg: WorkloadConfig, mode: str, logit_steps=None, seq=0, h=None,
                  W_dev=None, wl=None):
    """Init + every decode step; returns the oracle stream.

    I_t, its count, the bitmap and |S| are compared on every step.  Ring,
    window counts, packed rows, logits and top-k are compared on every step
    when logit_steps is None, else on those steps only."""
    wl = wl or Workload(cfg)
    W = wl.w_head()
    W_dev = W_dev if W_dev is not None else dev_bf16(W)
    own = h is None
    h = h or _handle(pkg, cfg, max_prompt=wl.prompt_len(seq))
    try:
        prompt = wl.prompt(seq)
        Z = wl.prefill_logits(seq) if cfg.K_pre > 0 else None
        ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        ost.init(prompt, Z)
        h.stream_init(seq, dev_i32(prompt), dev_f32(Z) if Z is not None else None)
        h.build_active_vocab(seq)
        check_state(h, seq, ost, full=True)
        trees = wl.trees(seq)
        logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        for t in range(cfg.steps):
            vb = wl.verify_logits(seq, t) if cfg.K_ver > 0 else None
            vr = wl.verify_row(seq, t)
            hid = wl.hiddens(seq, t)
            tree_d = dev_i32(trees[t])
            vb_d = dev_f32(vb) if vb is not None else None
            hid_d = dev_bf16(hid)
            if mode == "fused_step":
                ids, vals = h.step(seq, tree_d, vb_d, vr, W_dev, hid_d, cfg.k, logits=logits)
            elif mode == "two_launch":
                h.state_update(seq, tree_d, vb_d, vr)
                ids, vals = h.gather_sub_lm_head_topk(seq, W_dev, hid_d, cfg.k, logits=logits)
            else:
                h.stream_append(seq, tree_d, vb_d, vr)
                h.build_active_vocab(seq)
                h.gather_head_rows(seq, W_dev)
                ids, vals = h.sub_lm_head_logits_topk(seq, hid_d, cfg.k, logits=logits)
            ost.append(trees[t], vb, vr)
            sampled = logit_steps is None or t in logit_steps
            I = check_state(h, seq, ost, full=sampled)
            if sampled:
                check_packed(h, seq, W, I)
                if len(I):
                    check_projection(logits, ids, vals, hid, W, I, cfg.k)
        assert h.get_error() == 0
        return ost
    finally:
        if own:
            h.close()


TOY = get_config("toy_v4096_h256")


@pytest.mark.parametrize("mode", MODES)
def test_toy_every_step(pkg, mode):
    _run_workload(pkg, TOY, mode)


# A mid-size head: several row tiles, a ragged last tile, H split over a cluster,
# H = 1024 (16 k-slices) and V not a multiple of 32.
MID = WorkloadConfig(name="mid", V=20011, H=1024, W_max=1000, K_pre=3, K_ver=3, prompt_len=700, self_copy=0.4,
                     zipf_s=1.05, steps=12, n_tree=60, tree_local=0.7, tree_recent=256, n_verify=4)


@pytest.mark.parametrize("mode", MODES)
def test_mid_every_step(pkg, mode):
    _run_workload(pkg, MID, mode)


# Full-width heads on a small vocabulary: H = 4096 and 3584 give every CTA of
# the fused kernel more k slices than its stage ring holds, so stages are
# reused (the Llama-3 and Qwen-2.5 widths), with ragged last tiles.
WIDE = [
    WorkloadConfig(name="h4096", V=30011, H=4096, W_max=700, K_pre=3, K_ver=3, prompt_len=500, self_copy=0.4,
                   zipf_s=1.05, steps=6, n_tree=60, tree_local=0.7, tree_recent=256, n_verify=2),
    WorkloadConfig(name="h3584", V=9001, H=3584, W_max=333, K_pre=3, K_ver=3, prompt_len=200, self_copy=0.4,
                   zipf_s=1.05, steps=5, n_tree=45, tree_local=0.7, tree_recent=128, n_verify=1),
]


@pytest.mark.parametrize("cfg", WIDE, ids=lambda c: c.name)
@pytest.mark.parametrize("mode", ["fused_step", "two_launch"])
def test_wide_heads_every_step(pkg, cfg, mode):
    _run_workload(pkg, cfg, mode)


EDGE = [
    # tiny vocabulary and window; |I_t| < k pads the top-k
    WorkloadConfig(name="tiny", V=64, H=64, W_max=4, K_pre=1, K_ver=2, prompt_len=9, self_copy=0.3, zipf_s=1.0,
                   steps=10, n_tree=5, tree_local=0.5, tree_recent=4, n_verify=3),
    # window of one entry
    WorkloadConfig(name="w1", V=300, H=128, W_max=1, K_pre=2, K_ver=1, prompt_len=20, self_copy=0.2, zipf_s=1.1,
                   steps=6, n_tree=7, tree_local=0.5, tree_recent=8, n_verify=1),
    # window longer than the whole stream: every id ever seen stays active
    WorkloadConfig(name="wide", V=5000, H=192, W_max=8192, K_pre=3, K_ver=3, prompt_len=100, self_copy=0.5,
                   zipf_s=1.1, steps=5, n_tree=30, tree_local=0.5, tree_recent=64, n_verify=2),
    # V not a multiple of 4 (scalar Top-K loads), no prefill or verify candidates
    WorkloadConfig(name="noK", V=1001, H=64, W_max=50, K_pre=0, K_ver=0, prompt_len=40, self_copy=0.3, zipf_s=1.0,
                   steps=6, n_tree=12, tree_local=0.6, tree_recent=16, n_verify=1),
    # odd V with the largest K and k
    WorkloadConfig(name="bigK", V=3001, H=128, W_max=300, K_pre=16, K_ver=16, prompt_len=30, self_copy=0.2,
                   zipf_s=1.0, steps=4, n_tree=64, tree_local=0.5, tree_recent=32, n_verify=2, k=32),
    # single hidden row, window not a multiple of the tile
    WorkloadConfig(name="n1", V=2048, H=256, W_max=130, K_pre=3, K_ver=3, prompt_len=50, self_copy=0.3,
                   zipf_s=1.1, steps=4, n_tree=1, tree_local=0.5, tree_recent=16, n_verify=1, k=7),
]


@pytest.mark.parametrize("cfg", EDGE, ids=lambda c: c.name)
@pytest.mark.parametrize("mode", MODES)
def test_edge_configs(pkg, cfg, mode):
    _run_workload(pkg, cfg, mode)


def test_empty_tree_and_reinit(pkg):
    cfg = TOY.with_(steps=2)
    wl = Workload(cfg)
    with _handle(pkg, cfg, max_prompt=256) as h:
        prompt, Z = wl.prompt(0), wl.prefill_logits(0)
        for _ in range(2):  # a second init resets the sequence
            ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
            ost.init(prompt, Z)
            h.stream_init(0, dev_i32(prompt), dev_f32(Z))
            h.build_active_vocab(0)
            check_state(h, 0, ost)
            vb = wl.verify_logits(0, 0)
            h.stream_append(0, None, dev_f32(vb), 5)
            h.build_active_vocab(0)
            ost.append([], vb, 5)
            check_state(h, 0, ost)
            h.stream_append(0, dev_i32(wl.trees(0)[1]), dev_f32(vb), 2)
            h.build_active_vocab(0)
            ost.append(wl.trees(0)[1], vb, 2)
            check_state(h, 0, ost)


def _special_rows(V, base):
    """Verify rows that exercise the ranking order: NaN never ranks, -0.0 ties
    +0.0, infinities are ordered, ties go to the smaller id, the best values
    sit in the last (ragged) slots."""
    rows = {}
    r = base.copy()
    r[[V - 1, V - 2, V - 3]] = [100.0, 99.0, 98.0]
    rows["best_at_the_end"] = r
    r = base.copy()
    r[np.argsort(-base, kind="stable")[:5]] = np.nan
    r[::97] = np.nan
    rows["nan_where_the_best_was"] = r
    r = -np.abs(base)
    r[[7, 3, V - 2, 11]] = [-0.0, 0.0, 0.0, -0.0]
    rows["signed_zero_ties"] = r
    rows["all_equal"] = np.full(V, 1.5, np.float32)
    r = np.full(V, -np.inf, np.float32)
    r[[V // 2, 9]] = [-3.0, 2.0]
    rows["minus_inf_fill"] = r
    r = base.copy()
    r[V // 3] = np.inf
    rows["plus_inf"] = r
    rows["all_nan"] = np.full(V, np.nan, np.float32)
    return rows


@pytest.mark.parametrize("V", [4099, 4100], ids=["scalar", "float4"])
def test_verify_rows_with_special_values(pkg, V):
    cfg = WorkloadConfig(name=f"special{V}", V=V, H=64, W_max=64, K_pre=2, K_ver=3, prompt_len=12, self_copy=0.2,
                         zipf_s=1.1, steps=1, n_tree=8, tree_local=0.5, tree_recent=8, n_verify=1)
    wl = Workload(cfg)
    prompt, Z, tree = wl.prompt(0), wl.prefill_logits(0), wl.trees(0)[0]
    with _handle(pkg, cfg, max_prompt=64) as h:
        for name, row in _special_rows(V, wl.verify_logits(0, 0)[0]).items():
            ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
            ost.init(prompt, Z)
            h.stream_init(0, dev_i32(prompt), dev_f32(Z))
            h.stream_append(0, dev_i32(tree), dev_f32(row[None, :]), 0)
            h.build_active_vocab(0)
            ost.append(tree, row[None, :], 0)
            check_state(h, 0, ost)
            flags = h.get_error(clear=True)
            short = len(oracle.top_k(row, cfg.K_ver)) < cfg.K_ver
            assert bool(flags & pkg.FLAG_BAD_ID) == short, name
            assert flags & ~pkg.FLAG_BAD_ID == 0, name


def test_bad_ids_are_skipped_and_flagged(pkg):
    cfg = WorkloadConfig(name="bad", V=500, H=64, W_max=40, K_pre=2, K_ver=2, prompt_len=30, self_copy=0.2,
                         zipf_s=1.0, steps=1, n_tree=10, tree_local=0.5, tree_recent=8, n_verify=1)
    wl = Workload(cfg)
    with _handle(pkg, cfg, max_prompt=64) as h:
        prompt = wl.prompt(0).copy()
        prompt[[3, 17]] = [-1, 500]
        Z = wl.prefill_logits(0)
        h.stream_init(0, dev_i32(prompt), dev_f32(Z))
        h.build_active_vocab(0)
        assert h.get_error(clear=True) & pkg.FLAG_BAD_ID
        assert h.get_error() == 0
        good = [int(x) for x in prompt if 0 <= x < cfg.V]
        L = len(prompt)
        # invalid prompt ids are dropped; the union still ranks every prefill row
        union = oracle.stream_init([0] * L, Z, cfg.K_pre)[L:]
        ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        ost.S = good + union
        check_state(h, 0, ost)
        tree = np.array([7, -5, 7, 499, 1 << 30, 3], np.int32)
        vb = wl.verify_logits(0, 0)
        h.stream_append(0, dev_i32(tree), dev_f32(vb), 0)
        h.build_active_vocab(0)
        assert h.get_error(clear=True) & pkg.FLAG_BAD_ID
        ost.append([7, 7, 499, 3], vb, 0)
        check_state(h, 0, ost)


def test_host_argument_errors(pkg):
    cfg = TOY
    with _handle(pkg, cfg, max_prompt=256) as h:
        tree = dev_i32(np.zeros(4, np.int32))
        vb = dev_f32(np.zeros((2, cfg.V), np.float32))
        with pytest.raises(pkg.NanoSpecError) as e:
            h.stream_append(0, tree, vb, 0)  # before init
        assert e.value.status == -5
        prompt = dev_i32(np.arange(10, dtype=np.int32))
        Z = dev_f32(np.zeros((10, cfg.V), np.float32))
        h.stream_init(0, prompt, Z)
        for bad in [lambda: h.stream_append(0, tree, vb, 2),          # verify_row out of range
                    lambda: h.stream_append(1, tree, vb, 0),          # no such sequence
                    lambda: h.stream_append(0, dev_i32(np.zeros(17, np.int32)), vb, 0),  # n_tree > max_tree
                    lambda: h.stream_init(0, dev_i32(np.zeros(257, np.int32)), Z)]:   # L > max_prompt
            with pytest.raises(pkg.NanoSpecError) as e:
                bad()
            assert e.value.status == -1
        hid = dev_bf16(np.zeros((65, cfg.H), np.uint16))
        with pytest.raises(pkg.NanoSpecError):
            h.sub_lm_head_logits_topk(0, hid, 5)  # n > 64
        hid = dev_bf16(np.zeros((4, cfg.H), np.uint16))
        with pytest.raises(pkg.NanoSpecError):
            h.sub_lm_head_logits_topk(0, hid, cfg.k + 1)  # k > max_k
        assert h.get_error() == 0


def test_sequences_are_independent(pkg):
    cfg = TOY.with_(steps=5)
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    B = 3
    with _handle(pkg, cfg, batch=B, max_prompt=256) as h:
        osts = []
        for b in range(B):
            p, Z = wl.prompt(b), wl.prefill_logits(b)
            o = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
            o.init(p, Z)
            h.stream_init(b, dev_i32(p), dev_f32(Z))
            osts.append(o)
        logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        for t in range(cfg.steps):
            for b in reversed(range(B)):  # interleave sequences
                tr, vb, vr, hid = wl.trees(b)[t], wl.verify_logits(b, t), wl.verify_row(b, t), wl.hiddens(b, t)
                ids, vals = h.step(b, dev_i32(tr), dev_f32(vb), vr, W_dev, dev_bf16(hid), cfg.k, logits=logits)
                osts[b].append(tr, vb, vr)
                I = check_state(h, b, osts[b])
                check_packed(h, b, W, I)
                check_projection(logits, ids, vals, hid, W, I, cfg.k)


def test_copy_stream_overlap(pkg):
    """Gather on a copy stream, stand-in backbone GEMM on the compute stream,
    which waits on the gather's event only before the projection."""
    cfg = MID.with_(steps=3)
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    copy_s = torch.cuda.Stream()
    comp_s = torch.cuda.Stream()
    x = torch.randn(2048, 2048, device="cuda", dtype=torch.bfloat16)
    with _handle(pkg, cfg, max_prompt=cfg.prompt_len) as h:
        p, Z = wl.prompt(0), wl.prefill_logits(0)
        o = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        o.init(p, Z)
        h.stream_init(0, dev_i32(p), dev_f32(Z))
        torch.cuda.synchronize()
        logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        for t in range(cfg.steps):
            tr, vb, vr, hid = wl.trees(0)[t], wl.verify_logits(0, t), wl.verify_row(0, t), wl.hiddens(0, t)
            tr_d, vb_d, hid_d = dev_i32(tr), dev_f32(vb), dev_bf16(hid)
            torch.cuda.synchronize()
            state_done = torch.cuda.Event()
            gathered = torch.cuda.Event()
            with torch.cuda.stream(comp_s):
                h.stream_append(0, tr_d, vb_d, vr, stream=comp_s)
                h.build_active_vocab(0, stream=comp_s)
                state_done.record(comp_s)
            copy_s.wait_event(state_done)
            h.gather_head_rows(0, W_dev, copy_stream=copy_s, done=gathered)
            with torch.cuda.stream(comp_s):
                for _ in range(4):
                    y = x @ x  # stand-in draft backbone
                comp_s.wait_event(gathered)
                ids, vals = h.sub_lm_head_logits_topk(0, hid_d, cfg.k, logits=logits, stream=comp_s)
            torch.cuda.synchronize()
            del y
            o.append(tr, vb, vr)
            I = check_state(h, 0, o)
            check_packed(h, 0, W, I)
            check_projection(logits, ids, vals, hid, W, I, cfg.k)


@pytest.mark.parametrize("rows", [4096, 1000, 37])
def test_dense_head_toy(pkg, rows):
    cfg = TOY
    wl = Workload(cfg)
    W = wl.w_head()
    hid = wl.hiddens(0, 3)
    with _handle(pkg, cfg) as h:
        logits = torch.zeros((cfg.n_tree, cfg.V), dtype=torch.float32, device="cuda")
        ids, vals = h.dense_lm_head_topk(dev_bf16(W), rows, dev_bf16(hid), cfg.k, logits=logits)
        want = oracle.dense_logits(hid, W[:rows])
        tol = check_logits(logits[:, :rows].cpu().numpy(), want)
        check_topk(ids.cpu().numpy(), vals.cpu().numpy(), want, np.arange(rows), cfg.k, tol)


def test_dense_head_mid(pkg):
    cfg = MID
    wl = Workload(cfg)
    W = wl.w_head()
    hid = wl.hiddens(0, 0)
    with _handle(pkg, cfg) as h:
        ids, vals = h.dense_lm_head_topk(dev_bf16(W), cfg.V, dev_bf16(hid), cfg.k)
        logits = torch.zeros((cfg.n_tree, cfg.V), dtype=torch.float32, device="cuda")
        ids2, vals2 = h.dense_lm_head_topk(dev_bf16(W), cfg.V, dev_bf16(hid), cfg.k, logits=logits)
        want = oracle.dense_logits(hid, W)
        tol = check_logits(logits.cpu().numpy(), want)
        check_topk(ids.cpu().numpy(), vals.cpu().numpy(), want, np.arange(cfg.V), cfg.k, tol)
        assert torch.equal(ids, ids2) and torch.equal(vals, vals2)


def test_trace_events_bracket_the_step(pkg):
    """ns_trace_events records the step's kernel boundaries and leaves results unchanged."""
    cfg = TOY.with_(steps=3)
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    with _handle(pkg, cfg, max_prompt=256) as h:
        p, Z = wl.prompt(0), wl.prefill_logits(0)
        o = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        o.init(p, Z)
        h.stream_init(0, dev_i32(p), dev_f32(Z))
        logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        for t in range(cfg.steps):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]  # not yet created by torch
            h.trace_events(evs)
            tr, vb, vr, hid = wl.trees(0)[t], wl.verify_logits(0, t), wl.verify_row(0, t), wl.hiddens(0, t)
            ids, vals = h.step(0, dev_i32(tr), dev_f32(vb), vr, W_dev, dev_bf16(hid), cfg.k, logits=logits)
            h.trace_events(None)
            torch.cuda.synchronize()
            spans = [evs[i].elapsed_time(evs[i + 1]) for i in range(3)]
            assert all(s >= 0 for s in spans) and sum(spans) > 0
            o.append(tr, vb, vr)
            I = check_state(h, 0, o)
            check_projection(logits, ids, vals, hid, W, I, cfg.k)
        assert h._lib.ns_trace_events(h._h, None, 3) == -1  # wrong event count


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_step_host_equals_step(pkg, pinned):
    """ns_step_host (inputs and outputs in host memory: pinned buffers read and
    written in place by the kernel, pageable ones through copies) gives
    ns_step's window, I_t and top-k, bit for bit, on every step."""
    cfg = MID

    def host(t):
        return t.pin_memory() if pinned else t.clone()
    wl = Workload(cfg)
    W_dev = dev_bf16(wl.w_head())
    k = cfg.k
    with _handle(pkg, cfg) as ha, _handle(pkg, cfg) as hb:
        prompt, Z = wl.prompt(0), wl.prefill_logits(0)
        for h in (ha, hb):
            h.stream_init(0, dev_i32(prompt), dev_f32(Z))
            h.build_active_vocab(0)
        ids_h = host(torch.empty((cfg.n_tree, k), dtype=torch.int32))
        vals_h = host(torch.empty((cfg.n_tree, k), dtype=torch.float32))
        for t in range(cfg.steps):
            tree, vb, vr, hid = wl.trees(0)[t], wl.verify_logits(0, t), wl.verify_row(0, t), wl.hiddens(0, t)
            ids_b, vals_b = hb.step(0, dev_i32(tree), dev_f32(vb), vr, W_dev, dev_bf16(hid), k)
            # the host inputs stay alive until the stream has passed the step
            tree_h = host(torch.from_numpy(np.ascontiguousarray(tree)))
            verify_h = host(torch.from_numpy(np.ascontiguousarray(vb[vr])))
            hid_h = host(torch.from_numpy(np.ascontiguousarray(hid).view(np.int16)))
            ha.step_host(0, tree_h, verify_h, W_dev, hid_h, k, ids_h, vals_h)
            torch.cuda.synchronize()
            assert torch.equal(ids_h, ids_b.cpu()), f"step {t}: top-k ids"
            assert torch.equal(vals_h, vals_b.cpu()), f"step {t}: top-k values"
            ia, ca, ba, _ = ha.get_active(0)
            ib, cb, bb, _ = hb.get_active(0)
            m = int(ca.item())
            assert m == int(cb.item()) and torch.equal(ia[:m], ib[:m]) and torch.equal(ba, bb), f"step {t}: I_t"
        assert ha.get_error() == 0 and hb.get_error() == 0
        with pytest.raises(ValueError):  # device tensors are not host buffers
            ha.step_host(0, dev_i32(wl.trees(0)[0]), None, W_dev, dev_bf16(wl.hiddens(0, 0)), k, ids_h, vals_h)
