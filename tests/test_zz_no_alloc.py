"""The no-allocation dense head matches the handle-based one and the oracle.

ns_dense_lm_head_topk_noalloc exists for callers that cannot allocate device
memory (and so cannot create a handle): it keeps its scratch in a fixed
array inside the library.  These checks call it through the C ABI twice in a
row (the second call finds the first call's leftovers in the scratch) and
compare it with ns_dense_lm_head_topk on the same inputs and with the CPU
oracle's dense logits and top-k rule.  The two CUDA paths run the same
kernels, so their logits and top-k must be equal bit for bit.  This file
sorts last so that a run stopping at the first failure has run everything
else.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import Workload, WorkloadConfig

from parity import check_logits, check_topk, dev_bf16

pytestmark = pytest.mark.gpu

CFG = WorkloadConfig(name="noalloc", V=20011, H=1024, W_max=64, K_pre=3, K_ver=3, prompt_len=16, self_copy=0.0,
                     zipf_s=1.1, steps=2, n_tree=60, tree_local=0.5, tree_recent=8, n_verify=1)


@pytest.fixture(scope="module")
def ns():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import speculative_decoding_draft_stream_gb300 as p
    from speculative_decoding_draft_stream_gb300 import build, nanospec

    build.build()
    p.load_library()
    return nanospec


# 1000 rows: a partial last row tile and a single, partial top-k slice;
# 17000 rows: several slices, the last one partial.
@pytest.mark.parametrize("rows", [1000, 17000])
def test_noalloc_matches_handle_path_twice(ns, rows):
    wl = Workload(CFG)
    W = wl.w_head()
    W_d = dev_bf16(W)
    k = 10
    with ns.Handle(CFG.V, CFG.H, 64, 3, 3, max_tree=60, max_k=k) as h:
        for call in range(2):
            hid = wl.hiddens(0, call)
            hid_d = dev_bf16(hid)
            ref_logits = torch.zeros((CFG.n_tree, rows), dtype=torch.float32, device="cuda")
            ref_ids, ref_vals = h.dense_lm_head_topk(W_d, rows, hid_d, k, logits=ref_logits)
            # logits kept in the scratch (n * rows fits) and, second, in a caller buffer
            if CFG.n_tree * rows <= ns.NOALLOC_MAX_LOGITS:
                ids0, vals0 = ns.dense_lm_head_topk_noalloc(W_d, rows, hid_d, k)
            else:
                ids0, vals0 = None, None
            out_logits = torch.zeros((CFG.n_tree, rows), dtype=torch.float32, device="cuda")
            ids1, vals1 = ns.dense_lm_head_topk_noalloc(W_d, rows, hid_d, k, logits=out_logits)
            torch.cuda.synchronize()
            got = out_logits.cpu().numpy()
            ref = ref_logits.cpu().numpy()
            # against the handle's dense head: the same kernels, the same bits
            assert np.array_equal(got, ref), "logits differ from the handle's dense head"
            tol_ref = check_logits(got, ref)
            # against the oracle: logits, and the top-k rule on its logits
            want = oracle.dense_logits(hid, W[:rows])
            tol = check_logits(got, want)
            for ids, vals in ((ids0, vals0), (ids1, vals1)):
                if ids is None:
                    continue
                check_topk(ids.cpu().numpy(), vals.cpu().numpy(), want, np.arange(rows), k, tol)
                check_topk(ids.cpu().numpy(), vals.cpu().numpy(), ref, np.arange(rows), k, tol_ref)
                assert torch.equal(ids, ref_ids) and torch.equal(vals, ref_vals), "top-k differs from the handle's"
        assert h.get_error() == 0


def test_noalloc_rejects_logits_beyond_its_scratch(ns):
    wl = Workload(CFG)
    W_d = dev_bf16(wl.w_head())
    hid_d = dev_bf16(wl.hiddens(0, 0))
    rows = ns.NOALLOC_MAX_LOGITS // CFG.n_tree + 1  # n * rows just over the scratch
    lib = ns.load_library()
    ids = torch.empty((CFG.n_tree, 10), dtype=torch.int32, device="cuda")
    vals = torch.empty((CFG.n_tree, 10), dtype=torch.float32, device="cuda")
    st = lib.ns_dense_lm_head_topk_noalloc(W_d.data_ptr(), rows, CFG.H, hid_d.data_ptr(), CFG.n_tree, 10, None, 0,
                                           ids.data_ptr(), vals.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == -1
    with pytest.raises(ns.NanoSpecError):
        ns.dense_lm_head_topk_noalloc(W_d, rows, hid_d, 10, ids=ids, vals=vals)
