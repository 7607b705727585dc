"""GPU parity of the batched step with one shared gather (ns_step_batch_union)
against the oracle's union step (oracle.union_sub_head_step).

Per step: every sequence's state (I_t, bitmap, |S|; ring and counts on full
steps), the union U bit-exact, the membership of each U column in each
sequence's window (from the sequence's bitmap) equal to the oracle's M, the
union's packed rows W_head[U, :] byte-exact, each sequence's logits over all
of U within 1e-2 * max|oracle logit| of its row, and each sequence's top-k
over its own columns by the top-k rule.  The 35-sequence workload splits the
state updates and the projection into two launches each.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import Workload, WorkloadConfig, get_config

from parity import check_logits, check_state, check_topk, dev_bf16, dev_f32, dev_i32

pytestmark = pytest.mark.gpu

SMALL = WorkloadConfig(name="union5", V=20011, H=1024, W_max=1000, K_pre=3, K_ver=3, prompt_len=0,
                       prompt_len_min=200, prompt_len_max=700, self_copy=0.4, zipf_s=1.05, steps=8, n_tree=60,
                       tree_local=0.7, tree_recent=256, n_verify=4, batch=5)
MANY = WorkloadConfig(name="union35", V=2053, H=256, W_max=130, K_pre=2, K_ver=3, prompt_len=0, prompt_len_min=40,
                      prompt_len_max=100, self_copy=0.3, zipf_s=1.1, steps=3, n_tree=16, tree_local=0.6,
                      tree_recent=32, n_verify=2, batch=35, k=7)


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import speculative_decoding_draft_stream_gb300 as p
    from speculative_decoding_draft_stream_gb300 import build

    build.build()
    p.load_library()
    return p


def _run_union(pkg, cfg, steps, sample=None):
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
        u_ids, u_cnt, u_bm, u_packed, cap = h.get_union()
        assert cap == min(B * cfg.W_max, cfg.V)
        logits = torch.zeros((B, cfg.n_tree, cap), dtype=torch.float32, device="cuda")
        for t in range(steps):
            tree_t = np.stack([trees[b][t] for b in range(B)])
            vb = np.stack([wl.verify_logits(b, t) for b in range(B)])
            vr = [wl.verify_row(b, t) for b in range(B)]
            hid = np.stack([wl.hiddens(b, t) for b in range(B)])
            ids, vals = h.step_batch_union(dev_i32(tree_t), dev_f32(vb), vr, W_dev, dev_bf16(hid), cfg.k,
                                           logits=logits)
            full = sample is None or t in sample
            I_list = []
            for b in range(B):
                osts[b].append(trees[b][t], vb[b], vr[b])
                I_list.append(check_state(h, b, osts[b], full=full))
            m = int(u_cnt.item())
            U_gpu = u_ids[:m].cpu().numpy()
            U, M = oracle.union_vocab(I_list)
            assert np.array_equal(U_gpu, U), "union differs"
            assert np.array_equal(u_bm.cpu().numpy().view(np.uint32), oracle.bitmap_words(U, cfg.V)), "union bitmap"
            # membership of every union column in every sequence's window, read from the GPU's bitmaps
            for b in range(B):
                bm = h.get_active(b)[2].cpu().numpy().view(np.uint32)
                member = ((bm[U_gpu >> 5] >> (U_gpu & 31)) & 1).astype(bool)
                assert np.array_equal(member, M[b]), f"membership of sequence {b}"
            if not full:
                continue
            assert np.array_equal(u_packed[:m].cpu().numpy().view(np.uint16), oracle.gather_rows(W, U)), "packed union"
            _, _, _, want_logits, o_ids, _ = oracle.union_sub_head_step(list(hid), W, I_list, cfg.k)
            got_logits = logits[:, :, :m].cpu().numpy()
            for b in range(B):
                tol = check_logits(got_logits[b], want_logits[b])
                cols = np.flatnonzero(M[b])
                check_topk(ids[b].cpu().numpy(), vals[b].cpu().numpy(), want_logits[b][:, cols], U[cols], cfg.k, tol)
        assert h.get_error() == 0


@pytest.mark.parametrize("cfg", [SMALL, MANY], ids=lambda c: c.name)
def test_union_every_step(pkg, cfg):
    _run_union(pkg, cfg, cfg.steps)


def test_union_full_size_16_sequences(pkg):
    cfg = get_config("batched16_v128256_h4096")
    _run_union(pkg, cfg, 12, sample={0, 1, 11})


def test_union_needs_a_batch_handle(pkg):
    cfg = SMALL
    wl = Workload(cfg)
    with pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=cfg.n_tree, max_k=cfg.k, batch=1,
                    max_prompt=1024) as h:
        with pytest.raises(pkg.NanoSpecError) as e:
            h.get_union()
        assert e.value.status == -5
        h.stream_init(0, dev_i32(wl.prompt(0)[:50]), dev_f32(np.zeros((50, cfg.V), np.float32)))
        with pytest.raises(pkg.NanoSpecError) as e:
            h.step_batch_union(dev_i32(np.zeros((1, 4), np.int32)), dev_f32(np.zeros((1, 1, cfg.V), np.float32)),
                               [0], dev_bf16(wl.w_head()), dev_bf16(np.zeros((1, 4, cfg.H), np.uint16)), 5)
        assert e.value.status == -5
        assert h.get_error() == 0
