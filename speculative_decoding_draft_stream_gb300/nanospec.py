"""ctypes binding of libnanospec.so (include/nanospec.h), same names as the C ABI.

This module only marshals arguments: torch tensors become device pointers and
CUDA stream/event handles, and status codes become exceptions.  Every step of
the method runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or cannot be loaded, loading raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libnanospec.so")

NS_OK = 0
STATUS_NAMES = {0: "NS_OK", -1: "NS_ERR_ARG", -2: "NS_ERR_CUDA", -3: "NS_ERR_OOM", -4: "NS_ERR_TIMEOUT",
                -5: "NS_ERR_STATE"}
FLAG_BAD_ID = 0x1
FLAG_OVERFLOW = 0x2
FLAG_TIMEOUT = 0x4
FLAG_INTERNAL = 0x8
MAX_SELECT_K = 16
MAX_TOPK = 32
MAX_ROWS = 64

# Every entry point declared in include/nanospec.h.
EXPORTED = (
    "ns_status_string", "ns_create", "ns_destroy", "ns_device_bytes", "ns_stream_init", "ns_stream_append",
    "ns_build_active_vocab", "ns_gather_head_rows", "ns_sub_lm_head_logits_topk", "ns_step",
    "ns_dense_lm_head_topk", "ns_get_active", "ns_get_state", "ns_get_error", "ns_state_update",
    "ns_gather_sub_lm_head_topk", "ns_trace_events", "ns_dense_lm_head_topk_noalloc", "ns_gather_new_head_rows",
    "ns_slot_lm_head_logits_topk", "ns_step_slots", "ns_get_slots", "ns_step_batch", "ns_sub_lm_head_indexed_topk",
    "ns_step_launches", "ns_step_batch_union", "ns_get_union", "ns_set_copy_ctas", "ns_step_host",
    "ns_step_slots_fused", "ns_state_export_bytes", "ns_state_export", "ns_state_import",
)
NOALLOC_MAX_LOGITS = 1 << 20


class NanoSpecError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class ns_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("V", "H", "W_max", "K_pre", "K_ver", "max_tree", "max_k", "batch", "max_prompt")]


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the library (once).  Raises OSError when it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} not found: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P, I32, I64, U16P = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    sig = {
        "ns_status_string": (ctypes.c_char_p, [I32]),
        "ns_create": (I32, [ctypes.POINTER(ns_config), ctypes.POINTER(P)]),
        "ns_destroy": (I32, [P]),
        "ns_device_bytes": (I64, [P]),
        "ns_step_launches": (I32, [P]),
        "ns_step_slots_fused": (I32, [P, I32]),
        "ns_state_export_bytes": (I64, [P]),
        "ns_state_export": (I32, [P, I32, P, I64, ctypes.POINTER(I64), P]),
        "ns_state_import": (I32, [P, I32, P, I64, P]),
        "ns_set_copy_ctas": (I32, [P, I32]),
        "ns_step_host": (I32, [P, I32, P, I32, P, U16P, P, I32, I32, P, P, P]),
        "ns_stream_init": (I32, [P, I32, P, I32, P, P]),
        "ns_stream_append": (I32, [P, I32, P, I32, P, I32, I32, P]),
        "ns_build_active_vocab": (I32, [P, I32, P]),
        "ns_gather_head_rows": (I32, [P, I32, U16P, P, P]),
        "ns_sub_lm_head_logits_topk": (I32, [P, I32, U16P, I32, I32, P, I32, P, P, P]),
        "ns_step": (I32, [P, I32, P, I32, P, I32, I32, U16P, U16P, I32, I32, P, I32, P, P, P]),
        "ns_dense_lm_head_topk": (I32, [P, U16P, I32, U16P, I32, I32, P, I32, P, P, P]),
        "ns_get_active": (I32, [P, I32, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P),
                                ctypes.POINTER(P)]),
        "ns_get_state": (I32, [P, I32, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P)]),
        "ns_get_error": (I32, [P, ctypes.POINTER(ctypes.c_uint32), I32]),
        "ns_state_update": (I32, [P, I32, P, I32, P, I32, I32, P]),
        "ns_gather_sub_lm_head_topk": (I32, [P, I32, U16P, U16P, I32, I32, P, I32, P, P, P]),
        "ns_trace_events": (I32, [P, ctypes.POINTER(P), I32]),
        "ns_dense_lm_head_topk_noalloc": (I32, [U16P, I32, I32, U16P, I32, I32, P, I32, P, P, P]),
        "ns_gather_new_head_rows": (I32, [P, I32, U16P, P, P]),
        "ns_slot_lm_head_logits_topk": (I32, [P, I32, U16P, I32, I32, P, I32, P, P, P]),
        "ns_step_slots": (I32, [P, I32, P, I32, P, I32, I32, U16P, U16P, I32, I32, P, I32, P, P, P]),
        "ns_get_slots": (I32, [P, I32] + [ctypes.POINTER(P)] * 5),
        "ns_sub_lm_head_indexed_topk": (I32, [P, I32, U16P, U16P, I32, I32, P, I32, P, P, P]),
        "ns_step_batch": (I32, [P, I32, P, I32, P, I32, ctypes.POINTER(I32), U16P, U16P, I32, I32, P, I32, P, P,
                                P]),
        "ns_step_batch_union": (I32, [P, I32, P, I32, P, I32, ctypes.POINTER(I32), U16P, U16P, I32, I32, P, I32, P,
                                      P, P]),
        "ns_get_union": (I32, [P] + [ctypes.POINTER(P)] * 4 + [ctypes.POINTER(I64)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str) -> None:
    if status != NS_OK:
        raise NanoSpecError(status, where)


def _ptr(t: Optional[torch.Tensor], dtype=None, what: str = "tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{what} has dtype {t.dtype}, expected {dtype}")
    return t.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        s = torch.cuda.current_stream()
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)


class _DevView:
    """Object exposing a raw device pointer through __cuda_array_interface__."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def _view(ptr: int, shape, typestr: str, device) -> torch.Tensor:
    return torch.as_tensor(_DevView(ptr, shape, typestr), device=device)


class Handle:
    """One ns_handle: the device state of `batch` independent sequences."""

    def __init__(self, V: int, H: int, W_max: int, K_pre: int = 3, K_ver: int = 3, max_tree: int = 64,
                 max_k: int = 16, batch: int = 1, max_prompt: int = 4096):
        self._lib = load_library()
        self.cfg = ns_config(V, H, W_max, K_pre, K_ver, max_tree, max_k, batch, max_prompt)
        self.device = torch.device("cuda", torch.cuda.current_device())
        h = ctypes.c_void_p()
        _check(self._lib.ns_create(ctypes.byref(self.cfg), ctypes.byref(h)), "ns_create")
        self._h = h

    # -- lifetime --------------------------------------------------------------
    def close(self) -> None:
        if self._h:
            _check(self._lib.ns_destroy(self._h), "ns_destroy")
            self._h = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            if self._h:
                self._lib.ns_destroy(self._h)
        except Exception:
            pass

    @property
    def device_bytes(self) -> int:
        return int(self._lib.ns_device_bytes(self._h))

    @property
    def step_launches(self) -> int:
        """Kernel launches of one ns_step on this handle (1: the one-launch step)."""
        return int(self._lib.ns_step_launches(self._h))

    def state_export(self, seq: int, stream=None) -> bytes:
        """The checkpoint of `seq` (synchronises the stream)."""
        n = self._lib.ns_state_export_bytes(self._h)
        buf = ctypes.create_string_buffer(int(n))
        written = ctypes.c_int64(0)
        _check(self._lib.ns_state_export(self._h, seq, buf, n, ctypes.byref(written), _stream(stream)),
               "ns_state_export")
        return buf.raw[: written.value]

    def state_import(self, seq: int, data: bytes, stream=None) -> None:
        """Continue `seq` from a checkpoint made by state_export."""
        buf = ctypes.create_string_buffer(bytes(data), len(data))
        _check(self._lib.ns_state_import(self._h, seq, buf, len(data), _stream(stream)), "ns_state_import")

    def step_slots_fused(self, seq: int) -> int:
        """1 when the next ns_step_slots on `seq` is one launch (the slot table matches the window)."""
        return int(self._lib.ns_step_slots_fused(self._h, seq))

    # -- the C ABI -------------------------------------------------------------
    def stream_init(self, seq: int, prompt: Optional[torch.Tensor], prefill_logits: Optional[torch.Tensor],
                    stream=None) -> None:
        """prompt None (or empty) starts an empty stream."""
        L = 0 if prompt is None else prompt.numel()
        if L == 0:
            prompt = None
        _check(self._lib.ns_stream_init(self._h, seq, _ptr(prompt, torch.int32, "prompt"), L,
                                        _ptr(prefill_logits, torch.float32, "prefill_logits"), _stream(stream)),
               "ns_stream_init")

    def stream_append(self, seq: int, tree_ids: Optional[torch.Tensor], verify_logits: Optional[torch.Tensor],
                      verify_row: int = 0, stream=None) -> None:
        n_tree = 0 if tree_ids is None else tree_ids.numel()
        n_v = 0 if verify_logits is None else (verify_logits.shape[0] if verify_logits.dim() == 2 else 1)
        _check(self._lib.ns_stream_append(self._h, seq, _ptr(tree_ids, torch.int32, "tree_ids"), n_tree,
                                          _ptr(verify_logits, torch.float32, "verify_logits"), n_v, verify_row,
                                          _stream(stream)), "ns_stream_append")

    def build_active_vocab(self, seq: int, stream=None) -> None:
        _check(self._lib.ns_build_active_vocab(self._h, seq, _stream(stream)), "ns_build_active_vocab")

    def gather_head_rows(self, seq: int, W_head: torch.Tensor, copy_stream=None,
                         done: Optional[torch.cuda.Event] = None) -> None:
        ev = done.cuda_event if done is not None else None
        _check(self._lib.ns_gather_head_rows(self._h, seq, _ptr(W_head, _BF16, "W_head"), _stream(copy_stream), ev),
               "ns_gather_head_rows")

    def _outputs(self, n, k, ids, vals):
        if ids is None:
            ids = torch.empty((n, k), dtype=torch.int32, device=self.device)
        if vals is None:
            vals = torch.empty((n, k), dtype=torch.float32, device=self.device)
        return ids, vals

    def sub_lm_head_logits_topk(self, seq: int, hidden: torch.Tensor, k: int, logits: Optional[torch.Tensor] = None,
                                ids: Optional[torch.Tensor] = None, vals: Optional[torch.Tensor] = None,
                                stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        n = hidden.shape[0]
        ids, vals = self._outputs(n, k, ids, vals)
        ld = logits.shape[1] if logits is not None else 0
        _check(self._lib.ns_sub_lm_head_logits_topk(self._h, seq, _ptr(hidden, _BF16, "hidden"), n, k,
                                                    _ptr(logits, torch.float32, "logits"), ld,
                                                    _ptr(ids, torch.int32, "ids"), _ptr(vals, torch.float32, "vals"),
                                                    _stream(stream)), "ns_sub_lm_head_logits_topk")
        return ids, vals

    def step(self, seq: int, tree_ids: Optional[torch.Tensor], verify_logits: Optional[torch.Tensor],
             verify_row: int, W_head: torch.Tensor, hidden: torch.Tensor, k: int,
             logits: Optional[torch.Tensor] = None, ids: Optional[torch.Tensor] = None,
             vals: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        n_tree = 0 if tree_ids is None else tree_ids.numel()
        n_v = 0 if verify_logits is None else (verify_logits.shape[0] if verify_logits.dim() == 2 else 1)
        n = hidden.shape[0]
        ids, vals = self._outputs(n, k, ids, vals)
        ld = logits.shape[1] if logits is not None else 0
        _check(self._lib.ns_step(self._h, seq, _ptr(tree_ids, torch.int32, "tree_ids"), n_tree,
                                 _ptr(verify_logits, torch.float32, "verify_logits"), n_v, verify_row,
                                 _ptr(W_head, _BF16, "W_head"), _ptr(hidden, _BF16, "hidden"), n, k,
                                 _ptr(logits, torch.float32, "logits"), ld, _ptr(ids, torch.int32, "ids"),
                                 _ptr(vals, torch.float32, "vals"), _stream(stream)), "ns_step")
        return ids, vals

    def step_host(self, seq: int, tree_ids: Optional[torch.Tensor], verify_row: Optional[torch.Tensor],
                  W_head: torch.Tensor, hidden: torch.Tensor, k: int, ids: torch.Tensor, vals: torch.Tensor,
                  stream=None) -> None:
        """ns_step_host: tree_ids int32 [n_tree], verify_row fp32 [V] and hidden bf16 [n, H] in (pinned) host
        memory, ids int32 / vals fp32 [n, k] host outputs, valid once the stream synchronises."""
        def host(t, what):
            if t is None:
                return None
            if t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{what} must be a contiguous host tensor")
            return t.data_ptr()
        n_tree = 0 if tree_ids is None else tree_ids.numel()
        _check(self._lib.ns_step_host(self._h, seq, host(tree_ids, "tree_ids"), n_tree, host(verify_row, "verify_row"),
                                      _ptr(W_head, _BF16, "W_head"), host(hidden, "hidden"), hidden.shape[0], k,
                                      host(ids, "ids"), host(vals, "vals"), _stream(stream)), "ns_step_host")

    def step_batch(self, tree_ids: Optional[torch.Tensor], verify_logits: Optional[torch.Tensor], verify_rows,
                   W_head: torch.Tensor, hidden: torch.Tensor, k: int, logits: Optional[torch.Tensor] = None,
                   ids: Optional[torch.Tensor] = None, vals: Optional[torch.Tensor] = None,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        """ns_step_batch for sequences 0 .. B-1: tree_ids [B, n_tree], verify_logits [B, n_verify, V],
        verify_rows (B ints), hidden [B, n, H]; returns ids, vals [B, n, k]."""
        B, n = hidden.shape[0], hidden.shape[1]
        n_tree = 0 if tree_ids is None else tree_ids.shape[1]
        n_v = 0 if verify_logits is None else verify_logits.shape[1]
        rows = (ctypes.c_int32 * B)(*[int(x) for x in verify_rows]) if verify_logits is not None else None
        if ids is None:
            ids = torch.empty((B, n, k), dtype=torch.int32, device=self.device)
        if vals is None:
            vals = torch.empty((B, n, k), dtype=torch.float32, device=self.device)
        ld = logits.shape[-1] if logits is not None else 0
        _check(self._lib.ns_step_batch(self._h, B, _ptr(tree_ids, torch.int32, "tree_ids"), n_tree,
                                       _ptr(verify_logits, torch.float32, "verify_logits"), n_v, rows,
                                       _ptr(W_head, _BF16, "W_head"), _ptr(hidden, _BF16, "hidden"), n, k,
                                       _ptr(logits, torch.float32, "logits"), ld, _ptr(ids, torch.int32, "ids"),
                                       _ptr(vals, torch.float32, "vals"), _stream(stream)), "ns_step_batch")
        return ids, vals

    def step_batch_union(self, tree_ids: Optional[torch.Tensor], verify_logits: Optional[torch.Tensor], verify_rows,
                         W_head: torch.Tensor, hidden: torch.Tensor, k: int, logits: Optional[torch.Tensor] = None,
                         ids: Optional[torch.Tensor] = None, vals: Optional[torch.Tensor] = None,
                         stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        """ns_step_batch_union for sequences 0 .. B-1 (shapes as step_batch; logits [B, n, >= union capacity])."""
        B, n = hidden.shape[0], hidden.shape[1]
        n_tree = 0 if tree_ids is None else tree_ids.shape[1]
        n_v = 0 if verify_logits is None else verify_logits.shape[1]
        rows = (ctypes.c_int32 * B)(*[int(x) for x in verify_rows]) if verify_logits is not None else None
        if ids is None:
            ids = torch.empty((B, n, k), dtype=torch.int32, device=self.device)
        if vals is None:
            vals = torch.empty((B, n, k), dtype=torch.float32, device=self.device)
        ld = logits.shape[-1] if logits is not None else 0
        _check(self._lib.ns_step_batch_union(self._h, B, _ptr(tree_ids, torch.int32, "tree_ids"), n_tree,
                                             _ptr(verify_logits, torch.float32, "verify_logits"), n_v, rows,
                                             _ptr(W_head, _BF16, "W_head"), _ptr(hidden, _BF16, "hidden"), n, k,
                                             _ptr(logits, torch.float32, "logits"), ld, _ptr(ids, torch.int32, "ids"),
                                             _ptr(vals, torch.float32, "vals"), _stream(stream)),
               "ns_step_batch_union")
        return ids, vals

    def get_union(self):
        """Views (ids int32 [cap], count int32 [1], bitmap int32 [ceil(V/32)], packed int16 [cap, H]) and cap."""
        p = [ctypes.c_void_p() for _ in range(4)]
        cap = ctypes.c_int64()
        _check(self._lib.ns_get_union(self._h, *[ctypes.byref(x) for x in p], ctypes.byref(cap)), "ns_get_union")
        c, m = self.cfg, int(cap.value)
        nwords = (c.V + 31) // 32
        return (_view(p[0].value, (m,), "<i4", self.device), _view(p[1].value, (1,), "<i4", self.device),
                _view(p[2].value, (nwords,), "<i4", self.device), _view(p[3].value, (m, c.H), "<i2", self.device), m)

    def state_update(self, seq: int, tree_ids: Optional[torch.Tensor], verify_logits: Optional[torch.Tensor],
                     verify_row: int = 0, stream=None) -> None:
        n_tree = 0 if tree_ids is None else tree_ids.numel()
        n_v = 0 if verify_logits is None else (verify_logits.shape[0] if verify_logits.dim() == 2 else 1)
        _check(self._lib.ns_state_update(self._h, seq, _ptr(tree_ids, torch.int32, "tree_ids"), n_tree,
                                         _ptr(verify_logits, torch.float32, "verify_logits"), n_v, verify_row,
                                         _stream(stream)), "ns_state_update")

    def gather_sub_lm_head_topk(self, seq: int, W_head: torch.Tensor, hidden: torch.Tensor, k: int,
                                logits: Optional[torch.Tensor] = None, ids: Optional[torch.Tensor] = None,
                                vals: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        n = hidden.shape[0]
        ids, vals = self._outputs(n, k, ids, vals)
        ld = logits.shape[1] if logits is not None else 0
        _check(self._lib.ns_gather_sub_lm_head_topk(self._h, seq, _ptr(W_head, _BF16, "W_head"),
                                                    _ptr(hidden, _BF16, "hidden"), n, k,
                                                    _ptr(logits, torch.float32, "logits"), ld,
                                                    _ptr(ids, torch.int32, "ids"), _ptr(vals, torch.float32, "vals"),
                                                    _stream(stream)), "ns_gather_sub_lm_head_topk")
        return ids, vals

    def set_copy_ctas(self, ctas: int) -> None:
        """CTAs of the copy kernels (0: the default)."""
        _check(self._lib.ns_set_copy_ctas(self._h, ctas), "ns_set_copy_ctas")

    # -- the slot-stable buffer (incremental gather) ---------------------------
    def gather_new_head_rows(self, seq: int, W_head: torch.Tensor, copy_stream=None,
                             done: Optional[torch.cuda.Event] = None) -> None:
        ev = done.cuda_event if done is not None else None
        _check(self._lib.ns_gather_new_head_rows(self._h, seq, _ptr(W_head, _BF16, "W_head"), _stream(copy_stream),
                                                 ev), "ns_gather_new_head_rows")

    def slot_lm_head_logits_topk(self, seq: int, hidden: torch.Tensor, k: int,
                                 logits: Optional[torch.Tensor] = None, ids: Optional[torch.Tensor] = None,
                                 vals: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        n = hidden.shape[0]
        ids, vals = self._outputs(n, k, ids, vals)
        ld = logits.shape[1] if logits is not None else 0
        _check(self._lib.ns_slot_lm_head_logits_topk(self._h, seq, _ptr(hidden, _BF16, "hidden"), n, k,
                                                     _ptr(logits, torch.float32, "logits"), ld,
                                                     _ptr(ids, torch.int32, "ids"), _ptr(vals, torch.float32, "vals"),
                                                     _stream(stream)), "ns_slot_lm_head_logits_topk")
        return ids, vals

    def step_slots(self, seq: int, tree_ids: Optional[torch.Tensor], verify_logits: Optional[torch.Tensor],
                   verify_row: int, W_head: torch.Tensor, hidden: torch.Tensor, k: int,
                   logits: Optional[torch.Tensor] = None, ids: Optional[torch.Tensor] = None,
                   vals: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        n_tree = 0 if tree_ids is None else tree_ids.numel()
        n_v = 0 if verify_logits is None else (verify_logits.shape[0] if verify_logits.dim() == 2 else 1)
        n = hidden.shape[0]
        ids, vals = self._outputs(n, k, ids, vals)
        ld = logits.shape[1] if logits is not None else 0
        _check(self._lib.ns_step_slots(self._h, seq, _ptr(tree_ids, torch.int32, "tree_ids"), n_tree,
                                       _ptr(verify_logits, torch.float32, "verify_logits"), n_v, verify_row,
                                       _ptr(W_head, _BF16, "W_head"), _ptr(hidden, _BF16, "hidden"), n, k,
                                       _ptr(logits, torch.float32, "logits"), ld, _ptr(ids, torch.int32, "ids"),
                                       _ptr(vals, torch.float32, "vals"), _stream(stream)), "ns_step_slots")
        return ids, vals

    def get_slots(self, seq: int):
        """Views (slot_id int32 [W_max], meta int32 [2] = (high-water mark, rows copied by the last update),
        new_slots int32 [W_max], new_ids int32 [W_max], rows int16 [W_max, H])."""
        p = [ctypes.c_void_p() for _ in range(5)]
        _check(self._lib.ns_get_slots(self._h, seq, *[ctypes.byref(x) for x in p]), "ns_get_slots")
        c = self.cfg
        return (_view(p[0].value, (c.W_max,), "<i4", self.device), _view(p[1].value, (2,), "<i4", self.device),
                _view(p[2].value, (c.W_max,), "<i4", self.device), _view(p[3].value, (c.W_max,), "<i4", self.device),
                _view(p[4].value, (c.W_max, c.H), "<i2", self.device))

    def sub_lm_head_indexed_topk(self, seq: int, W_head: torch.Tensor, hidden: torch.Tensor, k: int,
                                 logits: Optional[torch.Tensor] = None, ids: Optional[torch.Tensor] = None,
                                 vals: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        n = hidden.shape[0]
        ids, vals = self._outputs(n, k, ids, vals)
        ld = logits.shape[1] if logits is not None else 0
        _check(self._lib.ns_sub_lm_head_indexed_topk(self._h, seq, _ptr(W_head, _BF16, "W_head"),
                                                     _ptr(hidden, _BF16, "hidden"), n, k,
                                                     _ptr(logits, torch.float32, "logits"), ld,
                                                     _ptr(ids, torch.int32, "ids"), _ptr(vals, torch.float32, "vals"),
                                                     _stream(stream)), "ns_sub_lm_head_indexed_topk")
        return ids, vals

    def trace_events(self, events) -> None:
        """Record ns_step's kernel boundaries on four torch.cuda.Events (None: off)."""
        if events is None:
            _check(self._lib.ns_trace_events(self._h, None, 0), "ns_trace_events")
            self._trace = None
            return
        events = list(events)
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event on its first record
                e.record()
        arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
        _check(self._lib.ns_trace_events(self._h, arr, 4), "ns_trace_events")
        self._trace = (arr, list(events))  # keep the events alive while set

    def dense_lm_head_topk(self, W_head: torch.Tensor, rows: int, hidden: torch.Tensor, k: int,
                           logits: Optional[torch.Tensor] = None, ids: Optional[torch.Tensor] = None,
                           vals: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        n = hidden.shape[0]
        ids, vals = self._outputs(n, k, ids, vals)
        ld = logits.shape[1] if logits is not None else 0
        _check(self._lib.ns_dense_lm_head_topk(self._h, _ptr(W_head, _BF16, "W_head"), rows,
                                               _ptr(hidden, _BF16, "hidden"), n, k,
                                               _ptr(logits, torch.float32, "logits"), ld,
                                               _ptr(ids, torch.int32, "ids"), _ptr(vals, torch.float32, "vals"),
                                               _stream(stream)), "ns_dense_lm_head_topk")
        return ids, vals

    # -- state views (device tensors aliasing library memory) ----------------
    def get_active(self, seq: int):
        """Views (ids int32 [W_max], count int32 [1], bitmap int32 [ceil(V/32)], packed int16 [W_max, H])."""
        p = [ctypes.c_void_p() for _ in range(4)]
        _check(self._lib.ns_get_active(self._h, seq, *[ctypes.byref(x) for x in p]), "ns_get_active")
        c = self.cfg
        nwords = (c.V + 31) // 32
        return (_view(p[0].value, (c.W_max,), "<i4", self.device), _view(p[1].value, (1,), "<i4", self.device),
                _view(p[2].value, (nwords,), "<i4", self.device),
                _view(p[3].value, (c.W_max, c.H), "<i2", self.device))

    def get_state(self, seq: int):
        """Views (ring int32 [W_max], length int64 [1], counts int32 [V])."""
        p = [ctypes.c_void_p() for _ in range(3)]
        _check(self._lib.ns_get_state(self._h, seq, *[ctypes.byref(x) for x in p]), "ns_get_state")
        c = self.cfg
        return (_view(p[0].value, (c.W_max,), "<i4", self.device), _view(p[1].value, (1,), "<i8", self.device),
                _view(p[2].value, (c.V,), "<i4", self.device))

    def get_error(self, clear: bool = False) -> int:
        f = ctypes.c_uint32()
        _check(self._lib.ns_get_error(self._h, ctypes.byref(f), int(clear)), "ns_get_error")
        return int(f.value)


def dense_lm_head_topk_noalloc(W_head: torch.Tensor, rows: int, hidden: torch.Tensor, k: int,
                               logits: Optional[torch.Tensor] = None, ids: Optional[torch.Tensor] = None,
                               vals: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """ns_dense_lm_head_topk_noalloc: the dense head for callers that cannot allocate device memory.

    No handle; the library allocates nothing and uses a fixed scratch array in
    its own image.  Output tensors can be passed in (so nothing is allocated
    here either).  Without `logits`, n * rows must not exceed
    NOALLOC_MAX_LOGITS.  Calls that may overlap on the GPU share the scratch
    and race.
    """
    lib = load_library()
    n, H = hidden.shape
    if ids is None:
        ids = torch.empty((n, k), dtype=torch.int32, device=hidden.device)
    if vals is None:
        vals = torch.empty((n, k), dtype=torch.float32, device=hidden.device)
    if logits is None and n * rows > NOALLOC_MAX_LOGITS:
        raise NanoSpecError(-1, f"ns_dense_lm_head_topk_noalloc: n*rows = {n * rows} exceeds the scratch "
                                f"({NOALLOC_MAX_LOGITS} logits); pass a logits tensor")
    ld = logits.shape[1] if logits is not None else 0
    _check(lib.ns_dense_lm_head_topk_noalloc(_ptr(W_head, _BF16, "W_head"), rows, H, _ptr(hidden, _BF16, "hidden"),
                                             n, k, _ptr(logits, torch.float32, "logits"), ld,
                                             _ptr(ids, torch.int32, "ids"), _ptr(vals, torch.float32, "vals"),
                                             _stream(stream)), "ns_dense_lm_head_topk_noalloc")
    return ids, vals
