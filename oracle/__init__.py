"""CPU oracle for the paged-KV attention step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The CUDA library never calls it; the two share no
code. It is a plain, slow statement of what the step computes, in double
precision (see ``pkv_oracle.c`` for the readings of the pages it follows).

Parity pins (tests that tie this oracle to something other than itself) live
in ``tests/test_oracle_pins.py``; every function here is pinned there.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, no fast-math) into a shared object."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC, "-lm"],
                   check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            lib.oracle_slot_mapping.argtypes = [p, i32, i32, i32, i64, p, p, i64, p]
            lib.oracle_cache_write.argtypes = [p, p, p, i64, p, p, i64, i32, i32, i32]
            lib.oracle_attention_paged.argtypes = [p, p, i32, p, p, p, i32, i32, i32, p, p, i64,
                                                   i32, i32, i32, ctypes.c_double, p, p, i32]
            lib.oracle_attention_dense.argtypes = [p, i32, p, p, i32, i32, i32, i32,
                                                   ctypes.c_double, p]
            for f in (lib.oracle_slot_mapping, lib.oracle_cache_write, lib.oracle_attention_paged,
                      lib.oracle_attention_dense):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} rejected its input (code {rc})")


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# Packing: one token axis from an ordered list of (slot, new rows, context).
# Lucebox, "Continuous batching ...", §Packing unequal prompt chunks together:
# segments sit back to back with no padding; segment metadata says where each
# ends and which slot owns it.
# ---------------------------------------------------------------------------

@dataclass
class Packed:
    cu_seqlens_q: np.ndarray  # int32 [S+1]
    seq_slot: np.ndarray      # int32 [S]
    token_slot: np.ndarray    # int32 [T]
    token_pos: np.ndarray     # int32 [T] logical position of each packed row


def pack(segments) -> Packed:
    """``segments``: iterable of (slot, q_len, ctx); rows of a segment sit at ctx-q_len .. ctx-1."""
    cu = [0]
    slots, tslot, tpos = [], [], []
    for slot, q_len, ctx in segments:
        cu.append(cu[-1] + q_len)
        slots.append(slot)
        for i in range(q_len):
            tslot.append(slot)
            tpos.append(ctx - q_len + i)
    return Packed(np.asarray(cu, np.int32), np.asarray(slots, np.int32),
                  np.asarray(tslot, np.int32), np.asarray(tpos, np.int32))


def slot_mapping(block_tables: np.ndarray, token_slot, token_pos, block_size: int,
                 num_blocks: int) -> np.ndarray:
    bt = _c(block_tables, np.int32)
    ts, tp = _c(token_slot, np.int32), _c(token_pos, np.int32)
    out = np.empty(len(ts), np.int64)
    _check(_load().oracle_slot_mapping(_ptr(bt), bt.shape[0], bt.shape[1], block_size, num_blocks,
                                       _ptr(ts), _ptr(tp), len(ts), _ptr(out)), "slot mapping")
    return out


def cache_write(k_pool: np.ndarray, v_pool: np.ndarray, k_new, v_new, mapping) -> None:
    """In place on ``uint16 [num_blocks, Hkv, bs, D]`` pools."""
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    nb, hkv, bs, d = k_pool.shape
    kn, vn, sm = _c(k_new, np.uint16), _c(v_new, np.uint16), _c(mapping, np.int64)
    _check(_load().oracle_cache_write(_ptr(kn), _ptr(vn), _ptr(sm), len(sm), _ptr(k_pool),
                                      _ptr(v_pool), nb, bs, hkv, d), "cache write")


def attention_paged(q, cu_seqlens_q, seq_slot, context_lens, block_tables, k_pool, v_pool,
                    scale: float, *, num_q_heads: int, rows=None, threads: int | None = None):
    """Double-precision ``[T, Hq, D]`` output; rows outside ``rows`` (if given) are NaN."""
    nb, hkv, bs, d = k_pool.shape
    qq = _c(q, np.uint16)
    t = qq.shape[0]
    cu, ss = _c(cu_seqlens_q, np.int32), _c(seq_slot, np.int32)
    cl, bt = _c(context_lens, np.int32), _c(block_tables, np.int32)
    out = np.full((t, num_q_heads, d), np.nan, dtype=np.float64)
    mask = None
    if rows is not None:
        mask = np.zeros(t, np.uint8)
        mask[np.asarray(rows, dtype=np.int64)] = 1
    _check(_load().oracle_attention_paged(
        _ptr(qq), _ptr(cu), len(ss), _ptr(ss), _ptr(cl), _ptr(bt), bt.shape[0], bt.shape[1], bs,
        _ptr(k_pool), _ptr(v_pool), nb, num_q_heads, hkv, d, float(scale), _ptr(mask), _ptr(out),
        threads if threads is not None else default_threads()), "paged attention")
    return out


def attention_dense(q, k, v, scale: float):
    """Causal attention of q ``[n, Hq, D]`` (the last n positions) over k/v ``[L, Hkv, D]``."""
    qq, kk, vv = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    n, hq, d = qq.shape
    L, hkv, _ = kk.shape
    out = np.empty((n, hq, d), np.float64)
    _check(_load().oracle_attention_dense(_ptr(qq), n, _ptr(kk), _ptr(vv), L, hq, hkv, d,
                                          float(scale), _ptr(out)), "dense attention")
    return out


# ---------------------------------------------------------------------------
# A whole step from a workload description (duck-typed: the oracle does not
# import the library package; it only reads plain attributes).
# ---------------------------------------------------------------------------

SENTINEL = 0x7FC1  # quiet bfloat16 NaN in every pool row that was never written


@dataclass
class OracleStep:
    packed: Packed
    context_lens: np.ndarray   # int32 [max_slots]
    block_tables: np.ndarray   # int32 [max_slots, max_blocks_per_slot]
    history_mapping: np.ndarray
    new_mapping: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray


def prepare_step(w, *, sentinel: int = SENTINEL) -> OracleStep:
    """Build the pool as it stands after this step's cache write.

    ``w`` provides: num_blocks, block_size, num_kv_heads, head_dim, max_slots,
    max_blocks_per_slot, segments (slot, q_len, ctx), blocks[slot] (physical
    IDs in logical order) and hist_k/hist_v[slot] ([ctx, Hkv, D] bf16 bits).
    The cached history (positions before the step's rows) is written first,
    then the step's new rows, each through its own slot mapping.
    """
    bs, nb = w.block_size, w.num_blocks
    bt = np.full((w.max_slots, w.max_blocks_per_slot), -1, np.int32)
    for slot, ids in w.blocks.items():
        bt[slot, : len(ids)] = ids
    ctx = np.zeros(w.max_slots, np.int32)
    segs = [(s.slot, s.q_len, s.ctx) for s in w.segments]
    for slot, _, c in segs:
        ctx[slot] = c
    hist = pack([(slot, c - ql, c - ql) for slot, ql, c in segs])
    new = pack(segs)
    hmap = slot_mapping(bt, hist.token_slot, hist.token_pos, bs, nb)
    nmap = slot_mapping(bt, new.token_slot, new.token_pos, bs, nb)
    shape = (nb, w.num_kv_heads, bs, w.head_dim)
    k_pool = np.full(shape, sentinel, np.uint16)
    v_pool = np.full(shape, sentinel, np.uint16)
    hk = [w.hist_k[slot][: c - ql] for slot, ql, c in segs]
    hv = [w.hist_v[slot][: c - ql] for slot, ql, c in segs]
    empty = np.zeros((0, w.num_kv_heads, w.head_dim), np.uint16)
    cache_write(k_pool, v_pool, np.concatenate(hk) if hk else empty,
                np.concatenate(hv) if hv else empty, hmap)
    nk = [w.hist_k[slot][c - ql: c] for slot, ql, c in segs]
    nv = [w.hist_v[slot][c - ql: c] for slot, ql, c in segs]
    cache_write(k_pool, v_pool, np.concatenate(nk) if nk else empty,
                np.concatenate(nv) if nv else empty, nmap)
    return OracleStep(new, ctx, bt, hmap, nmap, k_pool, v_pool)


def step_attention(w, st: OracleStep, *, rows=None, threads=None):
    return attention_paged(w.q, st.packed.cu_seqlens_q, st.packed.seq_slot, st.context_lens,
                           st.block_tables, st.k_pool, st.v_pool, w.scale,
                           num_q_heads=w.num_q_heads, rows=rows, threads=threads)
