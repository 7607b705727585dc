"""GPU parity of the vocabulary policies and the indexed product of NanoSpec's
ablation (evaluation, Table 5) through the C ABI, against the oracle.

* Ctx-only: the stream is the prefill S^(0) and nothing is appended while
  decoding (a handle with K_ver = 0 stepped with empty draft trees): I_t is
  the window of S^(0) at every step.
* Ext-only: the stream starts empty (ns_stream_init with L = 0), so I_t holds
  draft-tree and verify candidates only.
* The indexed product: logits and top-k straight from W_head through I_t with
  no packed copy (ns_sub_lm_head_indexed_topk); the packed buffer is left as
  it was.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import Workload, WorkloadConfig, get_config

from parity import check_projection, check_state, dev_bf16, dev_f32, dev_i32

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


MID = WorkloadConfig(name="mid", V=20011, H=1024, W_max=1000, K_pre=3, K_ver=3, prompt_len=700, self_copy=0.4,
                     zipf_s=1.05, steps=8, n_tree=60, tree_local=0.7, tree_recent=256, n_verify=4)


@pytest.mark.parametrize("cfg", [get_config("toy_v4096_h256"), MID], ids=lambda c: c.name)
def test_ctx_only(pkg, cfg):
    cfg = cfg.with_(K_ver=0)
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    with pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, 0, max_tree=cfg.n_tree, max_k=cfg.k,
                    max_prompt=cfg.prompt_len) as h:
        prompt, Z = wl.prompt(0), wl.prefill_logits(0)
        o = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, 0)
        o.init(prompt, Z)
        h.stream_init(0, dev_i32(prompt), dev_f32(Z))
        I0 = o.active()
        logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        for t in range(cfg.steps):
            hid = wl.hiddens(0, t)
            ids, vals = h.step(0, None, None, 0, W_dev, dev_bf16(hid), cfg.k, logits=logits)
            o.append([], None, 0)
            I = check_state(h, 0, o, full=True)
            assert np.array_equal(I, I0)  # nothing enters or leaves
            check_projection(logits, ids, vals, hid, W, I, cfg.k)
        assert h.get_error() == 0


@pytest.mark.parametrize("cfg", [get_config("toy_v4096_h256"), MID], ids=lambda c: c.name)
def test_ext_only(pkg, cfg):
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    with pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=cfg.n_tree, max_k=cfg.k,
                    max_prompt=16) as h:
        o = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        o.init([], None)
        h.stream_init(0, None, None)
        h.build_active_vocab(0)
        I = check_state(h, 0, o, full=True)
        assert len(I) == 0
        trees = wl.trees(0)
        logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        for t in range(cfg.steps):
            vb, vr, hid = wl.verify_logits(0, t), wl.verify_row(0, t), wl.hiddens(0, t)
            ids, vals = h.step(0, dev_i32(trees[t]), dev_f32(vb), vr, W_dev, dev_bf16(hid), cfg.k, logits=logits)
            o.append(trees[t], vb, vr)
            I = check_state(h, 0, o, full=True)
            assert set(I.tolist()) <= set(np.concatenate([trees[u] for u in range(t + 1)]).tolist()) | \
                set(x for u in range(t + 1) for x in oracle.top_k(wl.verify_logits(0, u)[wl.verify_row(0, u)],
                                                                  cfg.K_ver))
            check_projection(logits, ids, vals, hid, W, I, cfg.k)
        assert h.get_error() == 0


@pytest.mark.parametrize("cfg", [get_config("toy_v4096_h256"), MID], ids=lambda c: c.name)
def test_indexed_product(pkg, cfg):
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    with pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=cfg.n_tree, max_k=cfg.k,
                    max_prompt=cfg.prompt_len) as h:
        prompt, Z = wl.prompt(0), wl.prefill_logits(0)
        o = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        o.init(prompt, Z)
        h.stream_init(0, dev_i32(prompt), dev_f32(Z))
        trees = wl.trees(0)
        logits = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        _, _, _, packed = h.get_active(0)
        for t in range(cfg.steps):
            vb, vr, hid = wl.verify_logits(0, t), wl.verify_row(0, t), wl.hiddens(0, t)
            h.state_update(0, dev_i32(trees[t]), dev_f32(vb), vr)
            before = packed.clone()
            ids, vals = h.sub_lm_head_indexed_topk(0, W_dev, dev_bf16(hid), cfg.k, logits=logits)
            o.append(trees[t], vb, vr)
            I = check_state(h, 0, o, full=False)
            check_projection(logits, ids, vals, hid, W, I, cfg.k)
            assert torch.equal(packed, before)  # nothing packed
        assert h.get_error() == 0
