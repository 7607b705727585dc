"""GPU parity on values where the ranking order alone decides the result.

The sub-head top-k and the verify Top-K break ties toward the smaller id, rank
+inf and -inf like any value and never rank NaN (the orders the oracle
defines).  These cases have exact answers, so ids and values are compared
exactly, through each way of issuing a step: the five separate calls,
ns_step (one launch where the device holds its grid) and its two halves.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import Workload, WorkloadConfig

from parity import check_state, dev_bf16, dev_f32, dev_i32

pytestmark = pytest.mark.gpu

MODES = ["separate_calls", "fused_step", "two_launch"]
BF16_POS_INF = 0x7F80

CFG = WorkloadConfig(name="edge_values", V=6007, H=256, W_max=700, K_pre=3, K_ver=3, prompt_len=600,
                     self_copy=0.3, zipf_s=1.05, steps=2, n_tree=48, tree_local=0.6, tree_recent=64, n_verify=2)


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import speculative_decoding_draft_stream_gb300 as p
    from speculative_decoding_draft_stream_gb300 import build

    build.build()
    p.load_library()
    return p


def _step(h, mode, tree_d, vb_d, vr, W_dev, hid_d, k, logits):
    if mode == "fused_step":
        return h.step(0, tree_d, vb_d, vr, W_dev, hid_d, k, logits=logits)
    if mode == "two_launch":
        h.state_update(0, tree_d, vb_d, vr)
        return h.gather_sub_lm_head_topk(0, W_dev, hid_d, k, logits=logits)
    h.stream_append(0, tree_d, vb_d, vr)
    h.build_active_vocab(0)
    h.gather_head_rows(0, W_dev)
    return h.sub_lm_head_logits_topk(0, hid_d, k, logits=logits)


def _exact_topk(logits, I, k):
    """The oracle's top-k on logits it computed itself."""
    ids, vals = oracle.topk_remap(logits, I, k)
    return np.asarray(ids), np.asarray(vals)


@pytest.mark.parametrize("mode", MODES)
def test_equal_and_infinite_logits(pkg, mode):
    """Zero hidden rows give all-zero logits (every id ties: the k smallest
    ids of I_t win); a row with one +inf element gives +inf, -inf or NaN
    logits by the sign of W_head's column (the +inf ties again go to the
    smaller ids, NaN never ranks)."""
    wl = Workload(CFG)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    k = 10
    with pkg.Handle(CFG.V, CFG.H, CFG.W_max, CFG.K_pre, CFG.K_ver, max_tree=CFG.n_tree, max_k=k,
                    max_prompt=CFG.prompt_len) as h:
        prompt, Z = wl.prompt(0), wl.prefill_logits(0)
        ost = oracle.OracleStream(CFG.V, CFG.W_max, CFG.K_pre, CFG.K_ver)
        ost.init(prompt, Z)
        h.stream_init(0, dev_i32(prompt), dev_f32(Z))
        h.build_active_vocab(0)
        logits = torch.zeros((CFG.n_tree, CFG.W_max), dtype=torch.float32, device="cuda")
        for t in range(CFG.steps):
            hid = wl.hiddens(0, t).copy()
            hid[: CFG.n_tree // 2] = 0  # all-equal logits
            hid[CFG.n_tree // 2:, 17] = BF16_POS_INF  # one +inf element per row
            tree, vb, vr = wl.trees(0)[t], wl.verify_logits(0, t), wl.verify_row(0, t)
            ids, vals = _step(h, mode, dev_i32(tree), dev_f32(vb), vr, W_dev, dev_bf16(hid), k, logits)
            ost.append(tree, vb, vr)
            I = check_state(h, 0, ost)
            want = oracle.project(hid, oracle.gather_rows(W, I))
            o_ids, o_vals = _exact_topk(want, I, k)
            assert np.array_equal(ids.cpu().numpy(), o_ids), "top-k ids"
            got_v = vals.cpu().numpy()
            assert np.array_equal(np.isposinf(got_v), np.isposinf(o_vals))
            fin = np.isfinite(o_vals)
            assert np.array_equal(got_v[fin], o_vals[fin].astype(np.float32)), "top-k values"
            # the equal rows: the first k ids of I_t, value 0
            assert np.array_equal(ids.cpu().numpy()[: CFG.n_tree // 2], np.tile(I[:k], (CFG.n_tree // 2, 1)))
            # logits: infinities and NaNs where the oracle has them, exact zeros on the equal rows
            g = logits[:, : len(I)].cpu().numpy()
            assert np.array_equal(np.isnan(g), np.isnan(want)) and np.array_equal(np.isinf(g), np.isinf(want))
            assert np.all(g[: CFG.n_tree // 2] == 0)
        assert h.get_error() == 0


def _special_rows(V, base):
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
def test_special_verify_rows_through_the_step(pkg, V):
    """The verify Top-K inside ns_step (the one-launch path ranks the row in
    slices over every CTA and merges them after its grid barrier)."""
    cfg = WorkloadConfig(name=f"special_step{V}", V=V, H=64, W_max=64, K_pre=2, K_ver=3, prompt_len=12,
                         self_copy=0.2, zipf_s=1.1, steps=1, n_tree=8, tree_local=0.5, tree_recent=8, n_verify=1)
    wl = Workload(cfg)
    prompt, Z, tree = wl.prompt(0), wl.prefill_logits(0), wl.trees(0)[0]
    W_dev = dev_bf16(wl.w_head())
    hid_d = dev_bf16(wl.hiddens(0, 0))
    with pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=cfg.n_tree, max_k=cfg.k,
                    max_prompt=64) as h:
        for name, row in _special_rows(V, wl.verify_logits(0, 0)[0]).items():
            ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
            ost.init(prompt, Z)
            h.stream_init(0, dev_i32(prompt), dev_f32(Z))
            h.build_active_vocab(0)
            h.step(0, dev_i32(tree), dev_f32(row[None, :]), 0, W_dev, hid_d, cfg.k)
            ost.append(tree, row[None, :], 0)
            check_state(h, 0, ost)
            flags = h.get_error(clear=True)
            short = len(oracle.top_k(row, cfg.K_ver)) < cfg.K_ver
            assert bool(flags & pkg.FLAG_BAD_ID) == short, name
            assert flags & ~pkg.FLAG_BAD_ID == 0, name
