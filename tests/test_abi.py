"""The C-ABI library builds, loads without a GPU and exports every declared entry point."""

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for hdr in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(ns_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib_path():
    from speculative_decoding_draft_stream_gb300 import build

    return build.build()


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("ns_stream_init", "ns_stream_append", "ns_build_active_vocab", "ns_gather_head_rows",
                     "ns_sub_lm_head_logits_topk"):
        assert required in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_binding_covers_every_declared_symbol():
    from speculative_decoding_draft_stream_gb300.nanospec import EXPORTED

    assert sorted(EXPORTED) == _declared()


def test_status_strings_without_gpu(lib_path):
    from speculative_decoding_draft_stream_gb300.nanospec import load_library

    lib = load_library(lib_path)
    assert lib.ns_status_string(0) == b"ok"
    assert lib.ns_status_string(-1) == b"invalid argument"
    assert lib.ns_status_string(-5) == b"call out of order"


def test_create_rejects_bad_config_before_touching_the_gpu(lib_path):
    from speculative_decoding_draft_stream_gb300.nanospec import load_library, ns_config

    lib = load_library(lib_path)
    h = ctypes.c_void_p()
    bad = [
        ns_config(0, 256, 16, 3, 3, 16, 10, 1, 16),      # V = 0
        ns_config(100, 100, 16, 3, 3, 16, 10, 1, 16),    # H not a multiple of 64
        ns_config(100, 256, 0, 3, 3, 16, 10, 1, 16),     # W_max = 0
        ns_config(100, 256, 16, 17, 3, 16, 10, 1, 16),   # K_pre too large
        ns_config(100, 256, 16, 3, 3, 65, 10, 1, 16),    # max_tree too large
        ns_config(100, 256, 16, 3, 3, 16, 33, 1, 16),    # max_k too large
        ns_config(100, 256, 16, 3, 3, 16, 10, 0, 16),    # batch = 0
        ns_config(2, 256, 16, 3, 3, 16, 10, 1, 16),      # K_pre > V
    ]
    for cfg in bad:
        assert lib.ns_create(ctypes.byref(cfg), ctypes.byref(h)) == -1
    assert lib.ns_create(None, ctypes.byref(h)) == -1
    assert lib.ns_destroy(None) == -1
    assert lib.ns_stream_init(None, 0, None, 1, None, None) == -1
    assert lib.ns_get_error(None, None, 0) == -1


def test_every_entry_point_rejects_a_null_handle(lib_path):
    """Each call that takes a handle returns NS_ERR_ARG for NULL before
    touching the GPU (the argument checks run on the host first)."""
    from speculative_decoding_draft_stream_gb300.nanospec import load_library

    lib = load_library(lib_path)
    z = None
    calls = {
        "ns_stream_append": (z, 0, z, 0, z, 0, 0, z),
        "ns_build_active_vocab": (z, 0, z),
        "ns_gather_head_rows": (z, 0, z, z, z),
        "ns_sub_lm_head_logits_topk": (z, 0, z, 1, 1, z, 0, z, z, z),
        "ns_step": (z, 0, z, 0, z, 0, 0, z, z, 1, 1, z, 0, z, z, z),
        "ns_state_update": (z, 0, z, 0, z, 0, 0, z),
        "ns_gather_sub_lm_head_topk": (z, 0, z, z, 1, 1, z, 0, z, z, z),
        "ns_sub_lm_head_indexed_topk": (z, 0, z, z, 1, 1, z, 0, z, z, z),
        "ns_dense_lm_head_topk": (z, z, 1, z, 1, 1, z, 0, z, z, z),
        "ns_gather_new_head_rows": (z, 0, z, z, z),
        "ns_slot_lm_head_logits_topk": (z, 0, z, 1, 1, z, 0, z, z, z),
        "ns_step_slots": (z, 0, z, 0, z, 0, 0, z, z, 1, 1, z, 0, z, z, z),
        "ns_step_batch": (z, 1, z, 0, z, 0, z, z, z, 1, 1, z, 0, z, z, z),
        "ns_get_active": (z, 0, z, z, z, z),
        "ns_get_state": (z, 0, z, z, z),
        "ns_get_slots": (z, 0, z, z, z, z, z),
        "ns_trace_events": (z, z, 0),
    }
    for name, args in calls.items():
        assert getattr(lib, name)(*args) == -1, name
