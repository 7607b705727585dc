"""GPU parity at the library's size limits: V = 524288 (the largest
vocabulary a handle takes) and H = 8192 (the widest hidden size).

V = 524288 makes the window bitmap 64 KB, more than the one-launch step keeps
in shared memory, so ns_step takes its two-launch path there; H = 8192 runs
the one-launch step with 128 k slices split over each cluster.  Both go
through the five separate calls and ns_step, every step against the oracle
(state, packed rows, logits and top-k with k = 32), and the dense head at
H = 8192 against the oracle's dense logits.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import Workload, WorkloadConfig

from parity import check_logits, check_topk, dev_bf16
from test_gpu_parity import _run_workload

pytestmark = pytest.mark.gpu

LIMIT_V = WorkloadConfig(name="limit_v524288", V=524288, H=256, W_max=4096, K_pre=3, K_ver=3, prompt_len=200,
                         self_copy=0.3, zipf_s=1.05, steps=4, n_tree=64, tree_local=0.6, tree_recent=64, n_verify=1,
                         k=32)
LIMIT_H = WorkloadConfig(name="limit_h8192", V=20011, H=8192, W_max=2048, K_pre=3, K_ver=3, prompt_len=700,
                         self_copy=0.3, zipf_s=1.05, steps=4, n_tree=64, tree_local=0.6, tree_recent=64, n_verify=1,
                         k=32)


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import speculative_decoding_draft_stream_gb300 as p
    from speculative_decoding_draft_stream_gb300 import build

    build.build()
    p.load_library()
    return p


@pytest.mark.parametrize("cfg", [LIMIT_V, LIMIT_H], ids=lambda c: c.name)
@pytest.mark.parametrize("mode", ["separate_calls", "fused_step"])
def test_limits_every_step(pkg, cfg, mode):
    _run_workload(pkg, cfg, mode)


def test_dense_head_at_h8192(pkg):
    cfg = LIMIT_H
    wl = Workload(cfg)
    W = wl.w_head()
    hid = wl.hiddens(0, 0)
    rows, k = 9000, 32
    with pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=cfg.n_tree, max_k=k) as h:
        logits = torch.zeros((cfg.n_tree, rows), dtype=torch.float32, device="cuda")
        ids, vals = h.dense_lm_head_topk(dev_bf16(W), rows, dev_bf16(hid), k, logits=logits)
        want = oracle.dense_logits(hid, W[:rows])
        tol = check_logits(logits.cpu().numpy(), want)
        check_topk(ids.cpu().numpy(), vals.cpu().numpy(), want, np.arange(rows), k, tol)
        assert h.get_error() == 0
