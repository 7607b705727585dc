"""GPU parity of the batched step (ns_step_batch: every sequence of a handle
stepped by one state-update launch and one grouped fused launch) against the
oracle, sequence by sequence.

State (I_t, count, bitmap, |S|) is compared on every step of every sequence;
ring, counts, packed sub-head, logits and top-k on every step of the small
workloads and on sampled steps of the 16-sequence Llama-3-shaped one.  One
workload has 35 sequences, so the call splits into two launches of each kind.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import Workload, WorkloadConfig, get_config

from parity import check_packed, check_projection, check_state, dev_bf16, dev_f32, dev_i32

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


def _run_batch(pkg, cfg, steps, sample=None):
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    B = cfg.batch
    max_prompt = max(wl.prompt_len(b) for b in range(B))
    with pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=cfg.n_tree, max_k=cfg.k, batch=B,
                    max_prompt=max_prompt) as h:
        osts, trees = [], []
        for b in range(B):
            prompt, Z = wl.prompt(b), wl.prefill_logits(b)
            o = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
            o.init(prompt, Z)
            h.stream_init(b, dev_i32(prompt), dev_f32(Z))
            h.build_active_vocab(b)
            osts.append(o)
            trees.append(wl.trees(b))
        logits = torch.zeros((B, cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        for t in range(steps):
            tree_t = np.stack([trees[b][t] for b in range(B)])
            vb = np.stack([wl.verify_logits(b, t) for b in range(B)])
            vr = [wl.verify_row(b, t) for b in range(B)]
            hid = np.stack([wl.hiddens(b, t) for b in range(B)])
            ids, vals = h.step_batch(dev_i32(tree_t), dev_f32(vb), vr, W_dev, dev_bf16(hid), cfg.k, logits=logits)
            full = sample is None or t in sample
            for b in range(B):
                osts[b].append(trees[b][t], vb[b], vr[b])
                I = check_state(h, b, osts[b], full=full)
                if full:
                    check_packed(h, b, W, I)
                    check_projection(logits[b], ids[b], vals[b], hid[b], W, I, cfg.k)
        assert h.get_error() == 0


SMALL = WorkloadConfig(name="batch5", V=20011, H=1024, W_max=1000, K_pre=3, K_ver=3, prompt_len=0,
                       prompt_len_min=200, prompt_len_max=700, self_copy=0.4, zipf_s=1.05, steps=8, n_tree=60,
                       tree_local=0.7, tree_recent=256, n_verify=4, batch=5)
MANY = WorkloadConfig(name="batch35", V=2053, H=256, W_max=130, K_pre=2, K_ver=3, prompt_len=0, prompt_len_min=40,
                      prompt_len_max=100, self_copy=0.3, zipf_s=1.1, steps=3, n_tree=16, tree_local=0.6,
                      tree_recent=32, n_verify=2, batch=35, k=7)


@pytest.mark.parametrize("cfg", [SMALL, MANY], ids=lambda c: c.name)
def test_batch_every_step(pkg, cfg):
    _run_batch(pkg, cfg, cfg.steps)


def test_batch_full_size_16_sequences(pkg):
    cfg = get_config("batched16_v128256_h4096")
    _run_batch(pkg, cfg, 12, sample={0, 1, 2, 3, 11})


def test_batch_argument_errors(pkg):
    cfg = SMALL
    wl = Workload(cfg)
    W_dev = dev_bf16(wl.w_head())
    B, n, H = 3, cfg.n_tree, cfg.H
    with pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=n, max_k=cfg.k, batch=B,
                    max_prompt=1024) as h:
        tree = torch.zeros((B, n), dtype=torch.int32, device="cuda")
        vb = torch.zeros((B, 2, cfg.V), dtype=torch.float32, device="cuda")
        hid = torch.zeros((B, n, H), dtype=torch.int16, device="cuda")
        with pytest.raises(pkg.NanoSpecError) as e:  # no sequence initialised yet
            h.step_batch(tree, vb, [0] * B, W_dev, hid, cfg.k)
        assert "NS_ERR_STATE" in str(e.value)
        for b in range(B):
            p = dev_i32(wl.prompt(b)[:100])
            h.stream_init(b, p, torch.zeros((100, cfg.V), dtype=torch.float32, device="cuda"))
        with pytest.raises(pkg.NanoSpecError):  # verify row outside the block
            h.step_batch(tree, vb, [0, 2, 0], W_dev, hid, cfg.k)
        with pytest.raises(pkg.NanoSpecError):  # more sequences than the handle holds
            h.step_batch(torch.zeros((B + 1, n), dtype=torch.int32, device="cuda"),
                         torch.zeros((B + 1, 2, cfg.V), dtype=torch.float32, device="cuda"), [0] * (B + 1), W_dev,
                         torch.zeros((B + 1, n, H), dtype=torch.int16, device="cuda"), cfg.k)
        assert h.get_error() == 0
