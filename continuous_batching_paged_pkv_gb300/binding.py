"""Python binding of libpkv (ctypes). Argument marshalling only.

Every function here forwards to the C-ABI entry point of the same name in
``include/pkv.h``; all computation runs in the library's CUDA kernels or its
host C++ code. If ``libpkv.so`` has not been built the first call raises: there
is no fallback path.

Device tensors are torch tensors (torch provides device memory and streams);
host-side metadata is numpy.
"""

from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv.so")
HEADER_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pkv.h")

PKV_OK = 0
STATUS_NAMES = {
    0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_OUT_OF_RANGE", 3: "PKV_ERR_UNSUPPORTED",
    4: "PKV_ERR_WORKSPACE_TOO_SMALL", 5: "PKV_ERR_CUDA", 6: "PKV_ERR_DEVICE_TIMEOUT",
    7: "PKV_ERR_NO_BLOCKS", 8: "PKV_ERR_DEVICE_INDEX",
}
PKV_ERR_WORKSPACE_TOO_SMALL = 4
PKV_ERR_NO_BLOCKS = 7
PKV_SPLIT_KEYS = 256
PKV_NO_ALLOC_SCRATCH_BYTES = 32 << 20
PKV_WORK_WORDS_PER_ITEM = 4
PKV_STEP_IN_PLACE = 1
PKV_STEP_IN_PLACE_MAX_BYTES = 1 << 20


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({_lib().pkv_status_string(status).decode()})")


class WorkInfo(ctypes.Structure):
    _fields_ = [("num_decode_items", ctypes.c_int32), ("num_prefill_items", ctypes.c_int32),
                ("num_combine_items", ctypes.c_int32), ("num_partials", ctypes.c_int32),
                ("work_words", ctypes.c_int64), ("workspace_bytes", ctypes.c_uint64),
                ("decode_rows_max", ctypes.c_int32), ("num_scratch_items", ctypes.c_int32),
                ("scratch_blocks", ctypes.c_int64), ("workspace_bytes_q8", ctypes.c_uint64),
                ("num_long_combine_items", ctypes.c_int32)]


class StageLayout(ctypes.Structure):
    _fields_ = [("total_q", ctypes.c_int64), ("num_seqs", ctypes.c_int32), ("max_slots", ctypes.c_int32),
                ("max_blocks_per_slot", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)] + \
              [(n, ctypes.c_uint64) for n in ("q", "k_new", "v_new", "slot_mapping", "cu_seqlens_q", "seq_slot",
                                              "context_lens", "block_tables", "work")]


class PoolStats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("max_slots", ctypes.c_int32), ("free_blocks", ctypes.c_int64),
                ("owned_blocks", ctypes.c_int64), ("live_slots", ctypes.c_int32),
                ("live_tokens", ctypes.c_int64), ("shared_blocks", ctypes.c_int64)]


class Segment(ctypes.Structure):
    _fields_ = [("slot", ctypes.c_int32), ("num_tokens", ctypes.c_int32)]


_L = None


def _lib():
    global _L
    if _L is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(needs the CUDA toolkit); there is no non-CUDA fallback")
        L = ctypes.CDLL(LIB_PATH)
        p, i32, i64, u64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
        sig = {
            "pkv_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "pkv_version": ([], i32),
            "pkv_pool_create": ([i64, i32, i32, i32, p, i64], p),
            "pkv_pool_destroy": ([p], None),
            "pkv_pool_admit": ([p, i32, i64], ctypes.c_int),
            "pkv_pool_admit_blocks": ([p, i32, p, i32], ctypes.c_int),
            "pkv_pool_release": ([p, i32], ctypes.c_int),
            "pkv_pool_slot_length": ([p, i32], i64),
            "pkv_pool_slot_blocks": ([p, i32], i32),
            "pkv_pool_get_stats": ([p, ctypes.POINTER(PoolStats)], ctypes.c_int),
            "pkv_pool_copy_block_tables": ([p, p, i64], ctypes.c_int),
            "pkv_pool_adopt": ([p, i32, i32, i64, i64], ctypes.c_int),
            "pkv_pool_block_refs": ([p, i32], i32),
            "pkv_pool_take_copies": ([p, p, i64, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
            "pkv_copy_blocks": ([p, i64, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int64), i32, i64,
                                 p, p], ctypes.c_int),
            "pkv_plan_lower": ([p, p, i32, p, p, p, p, i64, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
            "pkv_plan_work": ([p, i32, p, p, i32, i32, i32, i32, i32, i32, p, i64, ctypes.POINTER(WorkInfo)],
                              ctypes.c_int),
            "pkv_cache_write": ([p, p, p, i64, p, p, i64, i32, i32, i32, p, p], ctypes.c_int),
            "pkv_attention": ([p, p, i32, i64, p, p, p, i32, i32, i32, p, p, i64, i32, i32, i32, f32, p,
                               ctypes.POINTER(WorkInfo), p, p, u64, p, p], ctypes.c_int),
            "pkv_check_device_status": ([p, p, ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
            "pkv_attention_no_alloc": ([p, p, i32, i64, p, p, p, i32, i32, i32, p, p, i64, i32, i32, i32, f32, p,
                                        ctypes.POINTER(WorkInfo), p, p, p], ctypes.c_int),
            "pkv_cache_write_q8": ([p, p, p, i64, p, p, p, p, i64, i32, i32, i32, p, p], ctypes.c_int),
            "pkv_attention_q8": ([p, p, i32, i64, p, p, p, i32, i32, i32, p, p, p, p, i64, i32, i32, i32, f32, p,
                                  ctypes.POINTER(WorkInfo), p, p, u64, p, p], ctypes.c_int),
            "pkv_cache_write_q4": ([p, p, p, i64, p, p, p, p, i64, i32, i32, i32, p, p], ctypes.c_int),
            "pkv_attention_q4": ([p, p, i32, i64, p, p, p, i32, i32, i32, p, p, p, p, i64, i32, i32, i32, f32, p,
                                  ctypes.POINTER(WorkInfo), p, p, u64, p, p], ctypes.c_int),
            "pkv_stage_layout_init": ([ctypes.POINTER(StageLayout), i64, i32, i32, i32, i32, i32, i32], ctypes.c_int),
            "pkv_step": ([ctypes.POINTER(StageLayout), p, u64, p, u64, p, p, i64, i32, f32, p, u64, p, p, p, p,
                          ctypes.POINTER(WorkInfo), ctypes.c_uint32], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes, fn.restype = args, res
        _L = L
    return _L


def declared_functions() -> list[str]:
    """Names of the functions ``include/pkv.h`` declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def _check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, what)


def _np_ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _t_ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch

        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream))


def pkv_status_string(status: int) -> str:
    return _lib().pkv_status_string(status).decode()


def pkv_version() -> int:
    return _lib().pkv_version()


# ---------------------------------------------------------------------------
# Host: pool, lowering, work list.
# ---------------------------------------------------------------------------

@dataclass
class Lowered:
    cu_seqlens_q: np.ndarray  # int32 [S+1]
    seq_slot: np.ndarray      # int32 [S]
    context_lens: np.ndarray  # int32 [max_slots]
    slot_mapping: np.ndarray  # int64 [T]


class Pool:
    """The library's block pool (``pkv_pool_*``)."""

    def __init__(self, num_blocks: int, block_size: int, max_slots: int, max_blocks_per_slot: int,
                 free_order: np.ndarray | None = None):
        fo = None if free_order is None else np.ascontiguousarray(free_order, dtype=np.int32)
        self._h = _lib().pkv_pool_create(num_blocks, block_size, max_slots, max_blocks_per_slot,
                                         _np_ptr(fo), 0 if fo is None else len(fo))
        if not self._h:
            raise PkvError(1, "pkv_pool_create")
        self.num_blocks, self.block_size = num_blocks, block_size
        self.max_slots, self.max_blocks_per_slot = max_slots, max_blocks_per_slot

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _L is not None:
            _L.pkv_pool_destroy(h)
            self._h = None

    def admit(self, slot: int, reserve_tokens: int) -> int:
        """Returns the status code (PKV_ERR_NO_BLOCKS is an answer, not an error)."""
        return _lib().pkv_pool_admit(self._h, slot, reserve_tokens)

    def admit_blocks(self, slot: int, blocks) -> None:
        b = np.ascontiguousarray(blocks, dtype=np.int32)
        _check(_lib().pkv_pool_admit_blocks(self._h, slot, _np_ptr(b), len(b)), "pkv_pool_admit_blocks")

    def release(self, slot: int) -> None:
        _check(_lib().pkv_pool_release(self._h, slot), "pkv_pool_release")

    def adopt(self, slot: int, donor_slot: int, num_tokens: int, reserve_tokens: int = 0) -> int:
        """``pkv_pool_adopt``; returns the status code (PKV_ERR_NO_BLOCKS is an answer, not an error)."""
        return _lib().pkv_pool_adopt(self._h, slot, donor_slot, num_tokens, reserve_tokens)

    def block_refs(self, block: int) -> int:
        return _lib().pkv_pool_block_refs(self._h, block)

    def take_copies(self) -> np.ndarray:
        """Pending copy-on-write copies as an int32 ``[n, 2]`` array of (source, destination) blocks."""
        n = ctypes.c_int64(0)
        rc = _lib().pkv_pool_take_copies(self._h, None, 0, ctypes.byref(n))
        if rc == PKV_OK and n.value == 0:
            return np.zeros((0, 2), np.int32)
        out = np.empty((n.value, 2), np.int32)
        _check(_lib().pkv_pool_take_copies(self._h, _np_ptr(out), n.value, ctypes.byref(n)), "pkv_pool_take_copies")
        return out

    def slot_length(self, slot: int) -> int:
        return _lib().pkv_pool_slot_length(self._h, slot)

    def slot_blocks(self, slot: int) -> int:
        return _lib().pkv_pool_slot_blocks(self._h, slot)

    def stats(self) -> PoolStats:
        st = PoolStats()
        _check(_lib().pkv_pool_get_stats(self._h, ctypes.byref(st)), "pkv_pool_get_stats")
        return st

    def block_tables(self) -> np.ndarray:
        out = np.empty((self.max_slots, self.max_blocks_per_slot), np.int32)
        _check(_lib().pkv_pool_copy_block_tables(self._h, _np_ptr(out), out.size), "pkv_pool_copy_block_tables")
        return out

    def lower(self, plan) -> Lowered:
        """``plan``: sequence of (slot, num_tokens) in packed order -> ``pkv_plan_lower``."""
        return pkv_plan_lower(self, plan)


def pkv_plan_lower(pool: Pool, plan) -> Lowered:
    segs = (Segment * max(len(plan), 1))(*[Segment(int(s), int(n)) for s, n in plan])
    total = sum(int(n) for _, n in plan)
    cu = np.empty(len(plan) + 1, np.int32)
    ss = np.empty(max(len(plan), 1), np.int32)
    cl = np.empty(pool.max_slots, np.int32)
    sm = np.empty(max(total, 1), np.int64)
    tq = ctypes.c_int64(0)
    _check(_lib().pkv_plan_lower(pool._h, segs, len(plan), _np_ptr(cu), _np_ptr(ss), _np_ptr(cl),
                                 _np_ptr(sm), len(sm), ctypes.byref(tq)), "pkv_plan_lower")
    return Lowered(cu, ss[: len(plan)], cl, sm[: tq.value])


def pkv_plan_work(cu_seqlens_q, seq_slot, context_lens, *, max_slots: int, max_blocks_per_slot: int,
                  block_size: int, num_q_heads: int, num_kv_heads: int, head_dim: int):
    """Returns (work int32 array, WorkInfo)."""
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    ss = np.ascontiguousarray(seq_slot, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    info = WorkInfo()
    args = (_np_ptr(cu), len(cu) - 1, _np_ptr(ss), _np_ptr(cl), max_slots, max_blocks_per_slot, block_size,
            num_q_heads, num_kv_heads, head_dim)
    rc = _lib().pkv_plan_work(*args, None, 0, ctypes.byref(info))
    if rc != PKV_ERR_WORKSPACE_TOO_SMALL:
        _check(rc, "pkv_plan_work")
    work = np.zeros(max(info.work_words, PKV_WORK_WORDS_PER_ITEM), np.int32)
    _check(_lib().pkv_plan_work(*args, _np_ptr(work), len(work), ctypes.byref(info)), "pkv_plan_work")
    return work, info


# ---------------------------------------------------------------------------
# Device calls (torch tensors on the GPU).
# ---------------------------------------------------------------------------

def _need(t, dtype_name: str, what: str):
    if t is None or not t.is_cuda or not t.is_contiguous() or str(t.dtype) != dtype_name:
        raise ValueError(f"{what} must be a contiguous CUDA tensor of {dtype_name}")


def pkv_cache_write(k_new, v_new, slot_mapping, k_pool, v_pool, *, device_status=None, stream=None) -> None:
    _need(k_new, "torch.bfloat16", "k_new")
    _need(v_new, "torch.bfloat16", "v_new")
    _need(slot_mapping, "torch.int64", "slot_mapping")
    _need(k_pool, "torch.bfloat16", "k_pool")
    _need(v_pool, "torch.bfloat16", "v_pool")
    nb, hkv, bs, d = k_pool.shape
    _check(_lib().pkv_cache_write(_t_ptr(k_new), _t_ptr(v_new), _t_ptr(slot_mapping), k_new.shape[0],
                                  _t_ptr(k_pool), _t_ptr(v_pool), nb, bs, hkv, d, _t_ptr(device_status),
                                  _stream(stream)), "pkv_cache_write")


def pkv_attention(q, cu_seqlens_q, seq_slot, context_lens, block_tables, k_pool, v_pool, work,
                  info: WorkInfo, out, workspace=None, *, scale: float = 0.0, device_status=None,
                  stream=None) -> None:
    _need(q, "torch.bfloat16", "q")
    _need(out, "torch.bfloat16", "out")
    for t, nm in ((cu_seqlens_q, "cu_seqlens_q"), (seq_slot, "seq_slot"), (context_lens, "context_lens"),
                  (block_tables, "block_tables"), (work, "work")):
        _need(t, "torch.int32", nm)
    _need(k_pool, "torch.bfloat16", "k_pool")
    _need(v_pool, "torch.bfloat16", "v_pool")
    nb, hkv, bs, d = k_pool.shape
    ms, mbps = block_tables.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().pkv_attention(_t_ptr(q), _t_ptr(cu_seqlens_q), cu_seqlens_q.numel() - 1, q.shape[0],
                                _t_ptr(seq_slot), _t_ptr(context_lens), _t_ptr(block_tables), ms, mbps, bs,
                                _t_ptr(k_pool), _t_ptr(v_pool), nb, q.shape[1], hkv, d, float(scale),
                                _t_ptr(work), ctypes.byref(info), _t_ptr(out), _t_ptr(workspace), ws_bytes,
                                _t_ptr(device_status), _stream(stream)), "pkv_attention")


def pkv_attention_no_alloc(q, cu_seqlens_q, seq_slot, context_lens, block_tables, k_pool, v_pool, work,
                           info: WorkInfo, out, *, scale: float = 0.0, device_status=None, stream=None) -> None:
    """``pkv_attention`` with the library's own fixed scratch array instead of a workspace.

    For callers that cannot allocate device memory; the step's partials must
    fit in PKV_NO_ALLOC_SCRATCH_BYTES. Concurrent calls on one device race.
    """
    _need(q, "torch.bfloat16", "q")
    _need(out, "torch.bfloat16", "out")
    for t, nm in ((cu_seqlens_q, "cu_seqlens_q"), (seq_slot, "seq_slot"), (context_lens, "context_lens"),
                  (block_tables, "block_tables"), (work, "work")):
        _need(t, "torch.int32", nm)
    _need(k_pool, "torch.bfloat16", "k_pool")
    _need(v_pool, "torch.bfloat16", "v_pool")
    nb, hkv, bs, d = k_pool.shape
    ms, mbps = block_tables.shape
    _check(_lib().pkv_attention_no_alloc(_t_ptr(q), _t_ptr(cu_seqlens_q), cu_seqlens_q.numel() - 1, q.shape[0],
                                         _t_ptr(seq_slot), _t_ptr(context_lens), _t_ptr(block_tables), ms, mbps,
                                         bs, _t_ptr(k_pool), _t_ptr(v_pool), nb, q.shape[1], hkv, d, float(scale),
                                         _t_ptr(work), ctypes.byref(info), _t_ptr(out), _t_ptr(device_status),
                                         _stream(stream)), "pkv_attention_no_alloc")


def _need_quant_pool(k_codes, k_scales, v_codes, v_scales, bits: int):
    """Shapes of a block-scaled pool: 8-bit codes int8 [blocks, Hkv, bs, D], 4-bit codes uint8
    [blocks, Hkv, bs, D/2] (two per byte); scales bf16 [blocks, Hkv, bs, D/32]."""
    for t, nm in ((k_codes, "k_codes"), (v_codes, "v_codes")):
        _need(t, "torch.int8" if bits == 8 else "torch.uint8", nm)
    for t, nm in ((k_scales, "k_scales"), (v_scales, "v_scales")):
        _need(t, "torch.bfloat16", nm)
    nb, hkv, bs, w = k_codes.shape
    d = w * 8 // bits
    if tuple(v_codes.shape) != (nb, hkv, bs, w) or tuple(k_scales.shape) != (nb, hkv, bs, d // 32) or \
            tuple(v_scales.shape) != (nb, hkv, bs, d // 32):
        raise ValueError(f"{bits}-bit pool: codes [blocks, Hkv, bs, D*{bits}/8] and scales [blocks, Hkv, bs, D/32] bf16")
    return nb, hkv, bs, d


def _cache_write_quant(bits, k_new, v_new, slot_mapping, k_codes, k_scales, v_codes, v_scales, device_status,
                       stream) -> None:
    _need(k_new, "torch.bfloat16", "k_new")
    _need(v_new, "torch.bfloat16", "v_new")
    _need(slot_mapping, "torch.int64", "slot_mapping")
    nb, hkv, bs, d = _need_quant_pool(k_codes, k_scales, v_codes, v_scales, bits)
    name = f"pkv_cache_write_q{bits}"
    _check(getattr(_lib(), name)(_t_ptr(k_new), _t_ptr(v_new), _t_ptr(slot_mapping), slot_mapping.numel(),
                                 _t_ptr(k_codes), _t_ptr(k_scales), _t_ptr(v_codes), _t_ptr(v_scales), nb, bs, hkv, d,
                                 _t_ptr(device_status), _stream(stream)), name)


def _attention_quant(bits, q, cu_seqlens_q, seq_slot, context_lens, block_tables, k_codes, k_scales, v_codes,
                     v_scales, work, info, out, workspace, scale, device_status, stream) -> None:
    _need(q, "torch.bfloat16", "q")
    _need(out, "torch.bfloat16", "out")
    for t, nm in ((cu_seqlens_q, "cu_seqlens_q"), (seq_slot, "seq_slot"), (context_lens, "context_lens"),
                  (block_tables, "block_tables"), (work, "work")):
        _need(t, "torch.int32", nm)
    nb, hkv, bs, d = _need_quant_pool(k_codes, k_scales, v_codes, v_scales, bits)
    ms, mbps = block_tables.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    name = f"pkv_attention_q{bits}"
    _check(getattr(_lib(), name)(_t_ptr(q), _t_ptr(cu_seqlens_q), cu_seqlens_q.numel() - 1, q.shape[0],
                                 _t_ptr(seq_slot), _t_ptr(context_lens), _t_ptr(block_tables), ms, mbps, bs,
                                 _t_ptr(k_codes), _t_ptr(k_scales), _t_ptr(v_codes), _t_ptr(v_scales), nb,
                                 q.shape[1], hkv, d, float(scale), _t_ptr(work), ctypes.byref(info), _t_ptr(out),
                                 _t_ptr(workspace), ws_bytes, _t_ptr(device_status), _stream(stream)), name)


def pkv_cache_write_q8(k_new, v_new, slot_mapping, k_codes, k_scales, v_codes, v_scales, *, device_status=None,
                       stream=None) -> None:
    _cache_write_quant(8, k_new, v_new, slot_mapping, k_codes, k_scales, v_codes, v_scales, device_status, stream)


def pkv_cache_write_q4(k_new, v_new, slot_mapping, k_codes, k_scales, v_codes, v_scales, *, device_status=None,
                       stream=None) -> None:
    _cache_write_quant(4, k_new, v_new, slot_mapping, k_codes, k_scales, v_codes, v_scales, device_status, stream)


def pkv_attention_q8(q, cu_seqlens_q, seq_slot, context_lens, block_tables, k_codes, k_scales, v_codes, v_scales,
                     work, info: WorkInfo, out, workspace=None, *, scale: float = 0.0, device_status=None,
                     stream=None) -> None:
    _attention_quant(8, q, cu_seqlens_q, seq_slot, context_lens, block_tables, k_codes, k_scales, v_codes, v_scales,
                     work, info, out, workspace, scale, device_status, stream)


def pkv_attention_q4(q, cu_seqlens_q, seq_slot, context_lens, block_tables, k_codes, k_scales, v_codes, v_scales,
                     work, info: WorkInfo, out, workspace=None, *, scale: float = 0.0, device_status=None,
                     stream=None) -> None:
    _attention_quant(4, q, cu_seqlens_q, seq_slot, context_lens, block_tables, k_codes, k_scales, v_codes, v_scales,
                     work, info, out, workspace, scale, device_status, stream)


def pkv_copy_blocks(pairs, arrays, *, device_status=None, stream=None) -> None:
    """Copy whole blocks (source, destination) in every pool array of ``arrays``.

    ``pairs``: int32 device tensor ``[n, 2]``; ``arrays``: device tensors whose
    first dimension is the block (``[num_blocks, ...]``), all with the same
    number of blocks (a bf16 pool's K and V, or an 8-bit pool's four arrays)."""
    _need(pairs, "torch.int32", "pairs")
    if not arrays or len(arrays) > 4:
        raise ValueError("pkv_copy_blocks takes one to four pool arrays")
    nb = arrays[0].shape[0]
    for t in arrays:
        if not t.is_cuda or not t.is_contiguous() or t.shape[0] != nb:
            raise ValueError("pool arrays must be contiguous CUDA tensors with the same number of blocks")
    ptrs = (ctypes.c_void_p * len(arrays))(*[t.data_ptr() for t in arrays])
    sizes = (ctypes.c_int64 * len(arrays))(*[t[0].numel() * t.element_size() for t in arrays])
    _check(_lib().pkv_copy_blocks(_t_ptr(pairs), pairs.shape[0], ptrs, sizes, len(arrays), nb,
                                  _t_ptr(device_status), _stream(stream)), "pkv_copy_blocks")


def pkv_check_device_status(device_status, stream=None) -> int:
    """Synchronises; returns the raw PKV_DEV_* bits (and clears them)."""
    bits = ctypes.c_uint32(0)
    rc = _lib().pkv_check_device_status(_t_ptr(device_status), _stream(stream), ctypes.byref(bits))
    if rc not in (PKV_OK, 6, 8):
        _check(rc, "pkv_check_device_status")
    return bits.value


def pkv_stage_layout_init(total_q: int, num_seqs: int, max_slots: int, max_blocks_per_slot: int,
                          num_q_heads: int, num_kv_heads: int, head_dim: int) -> StageLayout:
    layout = StageLayout()
    _check(_lib().pkv_stage_layout_init(ctypes.byref(layout), total_q, num_seqs, max_slots, max_blocks_per_slot,
                                        num_q_heads, num_kv_heads, head_dim), "pkv_stage_layout_init")
    return layout


def _buf(b):
    """(pointer, bytes) of a torch tensor or numpy array used as a raw byte buffer."""
    if b is None:
        return None, 0
    if isinstance(b, np.ndarray):
        return ctypes.c_void_p(b.ctypes.data), b.nbytes
    return ctypes.c_void_p(b.data_ptr()), b.numel() * b.element_size()


def pkv_step(layout: StageLayout, host_stage, device_stage, k_pool, v_pool, out, workspace=None, *,
             out_host=None, scale: float = 0.0, device_status=None, stream=None, in_place: bool = False) -> WorkInfo:
    """One step from the host staging buffer (see ``include/pkv.h``). Returns the step's work info.

    ``in_place`` passes PKV_STEP_IN_PLACE: the step then writes its output straight into
    ``out_host`` (no copy out), and a small one without prompt chunks also reads its inputs
    from ``host_stage`` in place (no copy in).
    On an error the raised PkvError carries ``info`` (filled where the library got that far).
    """
    _need(out, "torch.bfloat16", "out")
    _need(k_pool, "torch.bfloat16", "k_pool")
    _need(v_pool, "torch.bfloat16", "v_pool")
    nb, hkv, bs, d = k_pool.shape
    hp, hn = _buf(host_stage)
    dp, dn = _buf(device_stage)
    wp, wn = _buf(workspace)
    info = WorkInfo()
    rc = _lib().pkv_step(ctypes.byref(layout), hp, hn, dp, dn, _t_ptr(k_pool), _t_ptr(v_pool), nb, bs, float(scale),
                         wp, wn, _t_ptr(out), _buf(out_host)[0], _t_ptr(device_status), _stream(stream),
                         ctypes.byref(info), PKV_STEP_IN_PLACE if in_place else 0)
    if rc != PKV_OK:
        err = PkvError(rc, "pkv_step")
        err.info = info
        raise err
    return info


class StepCall:
    """``pkv_step`` with its arguments bound once, for a serving loop that reuses the same buffers.

    The constructor takes ``pkv_step``'s arguments and checks them; each call then only
    invokes the library with the marshalled arguments (the staging buffer's contents, which
    the caller refills between steps, are read by the library at the call). The buffers must
    stay alive and in place while the object is used; this object holds references to them.
    """

    def __init__(self, layout: StageLayout, host_stage, device_stage, k_pool, v_pool, out, workspace=None, *,
                 out_host=None, scale: float = 0.0, device_status=None, stream=None, in_place: bool = False):
        _need(out, "torch.bfloat16", "out")
        _need(k_pool, "torch.bfloat16", "k_pool")
        _need(v_pool, "torch.bfloat16", "v_pool")
        nb, hkv, bs, d = k_pool.shape
        hp, hn = _buf(host_stage)
        dp, dn = _buf(device_stage)
        wp, wn = _buf(workspace)
        self.info = WorkInfo()
        self._keep = (layout, host_stage, device_stage, k_pool, v_pool, out, workspace, out_host, device_status)
        self._fn = _lib().pkv_step
        self._args = (ctypes.byref(layout), hp, hn, dp, dn, _t_ptr(k_pool), _t_ptr(v_pool), nb, bs, float(scale),
                      wp, wn, _t_ptr(out), _buf(out_host)[0], _t_ptr(device_status), _stream(stream),
                      ctypes.byref(self.info), PKV_STEP_IN_PLACE if in_place else 0)

    def __call__(self) -> WorkInfo:
        rc = self._fn(*self._args)
        if rc != PKV_OK:
            err = PkvError(rc, "pkv_step")
            err.info = self.info
            raise err
        return self.info
