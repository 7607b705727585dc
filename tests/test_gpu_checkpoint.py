"""GPU tests of checkpoint and resume (ns_state_export / ns_state_import)
through the C ABI.

A sequence decoded for a few steps is exported; a second handle imports the
checkpoint and both decode the same further steps.  Their states and
outputs must be equal bit for bit, and both must match the oracle stream
that never stopped.  The checkpoint's bytes are the header the header file
describes followed by the window's entries, oldest first; a malformed one is
refused.
"""

import struct

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
                     zipf_s=1.05, steps=12, n_tree=60, tree_local=0.7, tree_recent=256, n_verify=4)


def _handle(pkg, cfg, max_prompt):
    return pkg.Handle(cfg.V, cfg.H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=max(cfg.n_tree, 1), max_k=cfg.k,
                      max_prompt=max(max_prompt, 1))


def _step_inputs(wl, cfg, t):
    vb = wl.verify_logits(0, t) if cfg.K_ver > 0 else None
    return wl.trees(0)[t], vb, wl.verify_row(0, t), wl.hiddens(0, t)


def _header(blob):
    magic, version, V, W_max, length, n, _ = struct.unpack("<4sIiiqii", blob[:32])
    return magic, version, V, W_max, length, n


@pytest.mark.parametrize("cfg", [get_config("toy_v4096_h256"), MID], ids=lambda c: c.name)
def test_resume_continues_the_stream(pkg, cfg):
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    split = cfg.steps // 2
    prompt = wl.prompt(0)
    Z = wl.prefill_logits(0) if cfg.K_pre > 0 else None
    ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
    ost.init(prompt, Z)
    with _handle(pkg, cfg, len(prompt)) as a, _handle(pkg, cfg, len(prompt)) as b:
        a.stream_init(0, dev_i32(prompt), dev_f32(Z) if Z is not None else None)
        a.build_active_vocab(0)
        for t in range(split):
            tree, vb, vr, hid = _step_inputs(wl, cfg, t)
            a.step(0, dev_i32(tree), dev_f32(vb) if vb is not None else None, vr, W_dev, dev_bf16(hid), cfg.k)
            ost.append(tree, vb, vr)
        blob = a.state_export(0)
        magic, version, V, W_max, length, n = _header(blob)
        assert (magic, version, V, W_max) == (b"NSST", 1, cfg.V, cfg.W_max)
        assert length == len(ost.S) and n == min(len(ost.S), cfg.W_max) and len(blob) == 32 + 4 * n
        window = np.frombuffer(blob[32:], dtype="<i4")
        assert np.array_equal(window, np.asarray(ost.S[len(ost.S) - n:], dtype=np.int32)), "window entries"

        b.state_import(0, blob)
        check_state(b, 0, ost, full=True)  # ring, |S|, counts, bitmap and I_t as the stream that went on
        assert b.state_export(0) == blob, "export of the import"

        logits_a = torch.zeros((cfg.n_tree, cfg.W_max), dtype=torch.float32, device="cuda")
        logits_b = torch.zeros_like(logits_a)
        for t in range(split, cfg.steps):
            tree, vb, vr, hid = _step_inputs(wl, cfg, t)
            args = (dev_i32(tree), dev_f32(vb) if vb is not None else None, vr, W_dev, dev_bf16(hid), cfg.k)
            ids_a, vals_a = a.step(0, *args, logits=logits_a)
            ids_b, vals_b = b.step(0, *args, logits=logits_b)
            ost.append(tree, vb, vr)
            I = check_state(b, 0, ost, full=True)
            check_state(a, 0, ost, full=True)
            assert torch.equal(ids_a, ids_b) and torch.equal(vals_a, vals_b), f"step {t}: top-k differ"
            assert torch.equal(logits_a[:, : len(I)], logits_b[:, : len(I)]), f"step {t}: logits differ"
            check_projection(logits_b, ids_b, vals_b, hid, W, I, cfg.k)
        assert a.get_error() == 0 and b.get_error() == 0


def test_resume_an_empty_stream_and_the_slot_step(pkg):
    """An empty stream's checkpoint holds no entries; after an import the
    slot table is empty, so the next ns_step_slots takes the multi-launch
    chain, which lays I_t out in the slots."""
    cfg = MID
    wl = Workload(cfg)
    W = wl.w_head()
    W_dev = dev_bf16(W)
    with _handle(pkg, cfg, 1) as a, _handle(pkg, cfg, 1) as b:
        a.stream_init(0, None, None)
        a.build_active_vocab(0)
        blob = a.state_export(0)
        assert _header(blob)[4:] == (0, 0) and len(blob) == 32
        b.state_import(0, blob)
        ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        ost.init([], None)
        osl = oracle.OracleSlots(cfg.W_max, cfg.H)
        check_state(b, 0, ost, full=True)
        for t in range(3):
            tree, vb, vr, hid = _step_inputs(wl, cfg, t)
            assert b.step_slots_fused(0) == (0 if t == 0 else 1)
            ids, vals = b.step_slots(0, dev_i32(tree), dev_f32(vb), vr, W_dev, dev_bf16(hid), cfg.k)
            ost.append(tree, vb, vr)
            I = check_state(b, 0, ost, full=False)
            osl.update(I, W)
            slot_id, _, _, _, _ = b.get_slots(0)
            assert np.array_equal(slot_id.cpu().numpy(), osl.slot_id), "slot table"
        assert b.get_error() == 0


def test_malformed_checkpoints_are_refused(pkg):
    cfg = get_config("toy_v4096_h256")
    wl = Workload(cfg)
    prompt, Z = wl.prompt(0), wl.prefill_logits(0)
    with _handle(pkg, cfg, len(prompt)) as a, _handle(pkg, cfg.with_(W_max=cfg.W_max + 1), len(prompt)) as other:
        a.stream_init(0, dev_i32(prompt), dev_f32(Z))
        blob = a.state_export(0)
        n = _header(blob)[5]
        assert n > 0
        bad = [
            b"XXXX" + blob[4:],                                   # magic
            blob[:4] + struct.pack("<I", 2) + blob[8:],           # version
            blob[:-4],                                            # truncated
            blob[:32 + 4 * (n - 1)] + struct.pack("<i", cfg.V),  # an id outside [0, V)
            blob[:24] + struct.pack("<i", n + 1) + blob[28:],     # n that does not match |S|
        ]
        for data in bad:
            with pytest.raises(pkg.NanoSpecError) as e:
                a.state_import(0, data)
            assert e.value.status == -1
        with pytest.raises(pkg.NanoSpecError) as e:
            other.state_import(0, blob)  # another W_max
        assert e.value.status == -1
        # the refused imports left the sequence as it was
        ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
        ost.init(prompt, Z)
        a.build_active_vocab(0)
        check_state(a, 0, ost, full=True)
        assert a.get_error() == 0
