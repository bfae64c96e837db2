"""Device-side set-up of one step through the library's own host API.

Given a step description (slots with their physical blocks and key/value
histories, and the packed query rows), this module:

1. creates the library's block pool and hands each slot its blocks
   (``pkv_pool_admit_blocks``);
2. writes each slot's cached history into a sentinel-filled device pool with
   ``pkv_cache_write``, through a slot mapping from ``pkv_plan_lower``;
3. lowers the step plan itself, builds the work list (``pkv_plan_work``) and
   uploads the step's metadata, queries and new keys/values.

``run_cache_write`` and ``run_attention`` then issue the step's two device
calls. ``HostStage`` holds the page-locked staging buffers of the one-call
host path (``pkv_step``). Nothing here computes attention; it only moves
arguments.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import binding as B

SENTINEL_BITS = 0x7FC1  # quiet bfloat16 NaN in pool rows never written


def _bf16_tensor(bits: np.ndarray, device):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def _i32(a, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def _i64(a, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(device)


def empty_pool(num_blocks, num_kv_heads, block_size, head_dim, device):
    import torch

    k = torch.empty((num_blocks, num_kv_heads, block_size, head_dim), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    k.view(torch.int16).fill_(SENTINEL_BITS)
    v.view(torch.int16).fill_(SENTINEL_BITS)
    return k, v


def empty_pool_q8(num_blocks, num_kv_heads, block_size, head_dim, device, bits: int = 8):
    """(k_codes, k_scales, v_codes, v_scales) of an 8-bit (int8 codes) or 4-bit (uint8, two codes per byte)
    pool; codes of rows never written hold the unused code -2^(bits-1), scales NaN."""
    import torch

    if bits == 8:
        codes = [torch.full((num_blocks, num_kv_heads, block_size, head_dim), -128, dtype=torch.int8, device=device)
                 for _ in range(2)]
    else:
        codes = [torch.full((num_blocks, num_kv_heads, block_size, head_dim // 2), 0x88, dtype=torch.uint8,
                            device=device) for _ in range(2)]
    scales = [torch.empty((num_blocks, num_kv_heads, block_size, head_dim // 32), dtype=torch.bfloat16,
                          device=device) for _ in range(2)]
    for t in scales:
        t.view(torch.int16).fill_(SENTINEL_BITS)
    return codes[0], scales[0], codes[1], scales[1]


@dataclass
class DeviceStep:
    w: object                 # the step description (workloads.StepInputs)
    pool: B.Pool
    lowered: B.Lowered        # this step's packed metadata (host)
    k_pool: object
    v_pool: object
    q: object
    k_new: object
    v_new: object
    slot_mapping: object
    cu_seqlens_q: object
    seq_slot: object
    context_lens: object
    block_tables: object
    work: object
    info: B.WorkInfo
    workspace: object
    out: object
    status: object
    kv: str = "bf16"          # pool format: "bf16", "q8" or "q4" (k_pool/v_pool hold the codes)
    k_scales: object = None
    v_scales: object = None

    @property
    def scale(self) -> float:
        return self.w.scale


def prepare(w, device="cuda", *, pools=None, kv: str = "bf16") -> DeviceStep:
    """Build the pool state before the step and upload the step's inputs.

    ``kv="q8"`` / ``kv="q4"`` keep the pool in the 8-bit / 4-bit block-scaled
    format (history written through ``pkv_cache_write_q8`` / ``_q4``)."""
    import torch

    pool = B.Pool(w.num_blocks, w.block_size, w.max_slots, w.max_blocks_per_slot)
    for slot in sorted(w.blocks):
        pool.admit_blocks(slot, w.blocks[slot])
    k_scales = v_scales = None
    if kv in ("q8", "q4"):
        k_pool, k_scales, v_pool, v_scales = pools if pools is not None else empty_pool_q8(
            w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim, device, bits=int(kv[1]))
    elif kv == "bf16":
        k_pool, v_pool = pools if pools is not None else empty_pool(
            w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim, device)
    else:
        raise ValueError(f"unknown pool format {kv!r}")
    status = torch.zeros(1, dtype=torch.int32, device=device)

    # Cached history: every segment's positions before this step's rows.
    hist_plan = [(s.slot, s.ctx - s.q_len) for s in w.segments]
    hist = pool.lower(hist_plan)
    if len(hist.slot_mapping):
        hk = np.concatenate([w.hist_k[s.slot][: s.ctx - s.q_len] for s in w.segments])
        hv = np.concatenate([w.hist_v[s.slot][: s.ctx - s.q_len] for s in w.segments])
        if kv in ("q8", "q4"):
            write = B.pkv_cache_write_q8 if kv == "q8" else B.pkv_cache_write_q4
            write(_bf16_tensor(hk, device), _bf16_tensor(hv, device), _i64(hist.slot_mapping, device),
                  k_pool, k_scales, v_pool, v_scales, device_status=status)
        else:
            B.pkv_cache_write(_bf16_tensor(hk, device), _bf16_tensor(hv, device), _i64(hist.slot_mapping, device),
                              k_pool, v_pool, device_status=status)

    low = pool.lower([(s.slot, s.q_len) for s in w.segments])
    work, info = B.pkv_plan_work(low.cu_seqlens_q, low.seq_slot, low.context_lens, max_slots=w.max_slots,
                                 max_blocks_per_slot=w.max_blocks_per_slot, block_size=w.block_size,
                                 num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim)
    ws = None
    ws_bytes = int(info.workspace_bytes_q8 if kv in ("q8", "q4") else info.workspace_bytes)
    if ws_bytes:
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    out = torch.empty((w.total_q, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=device)
    out.view(torch.int16).fill_(SENTINEL_BITS)
    return DeviceStep(
        w=w, pool=pool, lowered=low, k_pool=k_pool, v_pool=v_pool,
        q=_bf16_tensor(w.q, device), k_new=_bf16_tensor(w.new_k(), device), v_new=_bf16_tensor(w.new_v(), device),
        slot_mapping=_i64(low.slot_mapping, device), cu_seqlens_q=_i32(low.cu_seqlens_q, device),
        seq_slot=_i32(low.seq_slot, device), context_lens=_i32(low.context_lens, device),
        block_tables=_i32(pool.block_tables(), device), work=_i32(work, device), info=info, workspace=ws,
        out=out, status=status, kv=kv, k_scales=k_scales, v_scales=v_scales)


def run_cache_write(ds: DeviceStep, stream=None) -> None:
    if ds.kv in ("q8", "q4"):
        write = B.pkv_cache_write_q8 if ds.kv == "q8" else B.pkv_cache_write_q4
        write(ds.k_new, ds.v_new, ds.slot_mapping, ds.k_pool, ds.k_scales, ds.v_pool, ds.v_scales,
              device_status=ds.status, stream=stream)
    else:
        B.pkv_cache_write(ds.k_new, ds.v_new, ds.slot_mapping, ds.k_pool, ds.v_pool,
                          device_status=ds.status, stream=stream)


def run_attention(ds: DeviceStep, stream=None) -> None:
    if ds.kv in ("q8", "q4"):
        attend = B.pkv_attention_q8 if ds.kv == "q8" else B.pkv_attention_q4
        attend(ds.q, ds.cu_seqlens_q, ds.seq_slot, ds.context_lens, ds.block_tables, ds.k_pool, ds.k_scales,
               ds.v_pool, ds.v_scales, ds.work, ds.info, ds.out, ds.workspace, scale=ds.scale,
               device_status=ds.status, stream=stream)
    else:
        B.pkv_attention(ds.q, ds.cu_seqlens_q, ds.seq_slot, ds.context_lens, ds.block_tables, ds.k_pool,
                        ds.v_pool, ds.work, ds.info, ds.out, ds.workspace, scale=ds.scale,
                        device_status=ds.status, stream=stream)


def split_work(work, info):
    """Two (work, info) pairs from one bf16 step's work list: the prompt-chunk
    items alone (an attention call with them launches the chunk kernel alone),
    and the decode items with their merge items (the decode and merge kernels
    alone). Either is None when the step has no such items. Both compute the
    same output rows as the whole list does for those segments."""
    words = B.PKV_WORK_WORDS_PER_ITEM
    nd, npf, nc = info.num_decode_items, info.num_prefill_items, info.num_combine_items
    chunk = dec = None
    if npf:
        ci = B.WorkInfo()
        ci.num_prefill_items = npf
        ci.work_words = npf * words
        chunk = (work[nd * words:(nd + npf) * words].contiguous(), ci)
    if nd:
        import torch

        di = B.WorkInfo()
        di.num_decode_items, di.num_combine_items = nd, nc
        di.num_long_combine_items = info.num_long_combine_items
        di.num_partials, di.decode_rows_max = info.num_partials, info.decode_rows_max
        di.workspace_bytes = info.workspace_bytes
        di.work_words = (nd + nc) * words
        parts = [work[:nd * words], work[(nd + npf) * words:(nd + npf + nc) * words]]
        dec = (torch.cat(parts).contiguous(), di)
    return chunk, dec


def chunk_only(ds: DeviceStep):
    """(work, info) holding only the step's prompt-chunk items: an attention call
    with them launches the chunk kernel alone, on the same inputs and outputs."""
    return split_work(ds.work, ds.info)[0]


def decode_only(ds: DeviceStep):
    """(work, info) holding only the step's decode and merge items."""
    return split_work(ds.work, ds.info)[1]


def run_chunk_only(ds: DeviceStep, work_info, stream=None) -> None:
    work, info = work_info
    B.pkv_attention(ds.q, ds.cu_seqlens_q, ds.seq_slot, ds.context_lens, ds.block_tables, ds.k_pool,
                    ds.v_pool, work, info, ds.out, None, scale=ds.scale, device_status=ds.status, stream=stream)


def run_decode_only(ds: DeviceStep, work_info, stream=None) -> None:
    work, info = work_info
    B.pkv_attention(ds.q, ds.cu_seqlens_q, ds.seq_slot, ds.context_lens, ds.block_tables, ds.k_pool,
                    ds.v_pool, work, info, ds.out, ds.workspace, scale=ds.scale, device_status=ds.status,
                    stream=stream)


def run_step(ds: DeviceStep, stream=None) -> None:
    run_cache_write(ds, stream)
    run_attention(ds, stream)


def out_f32(ds: DeviceStep) -> np.ndarray:
    import torch

    return ds.out.to(torch.float32).cpu().numpy()


def pool_bits(ds: DeviceStep):
    import torch

    return (ds.k_pool.view(torch.int16).cpu().numpy().view(np.uint16),
            ds.v_pool.view(torch.int16).cpu().numpy().view(np.uint16))


class HostStage:
    """Page-locked host staging buffer for ``pkv_step`` and its device twin.

    One buffer of ``nbytes`` on each side; ``fill`` writes a step's inputs at
    the offsets of its ``pkv_stage_layout`` (the rest of the buffer is the
    work list's room). Reusable across steps of different shapes.
    """

    def __init__(self, nbytes: int, device):
        import torch

        self.nbytes = int(nbytes)
        self.host = torch.empty(self.nbytes, dtype=torch.uint8, pin_memory=True)
        self.device = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self._np = self.host.numpy()

    def _fields(self, layout):
        T, S, ms, mb = layout.total_q, layout.num_seqs, layout.max_slots, layout.max_blocks_per_slot
        hq, hkv, d = layout.num_q_heads, layout.num_kv_heads, layout.head_dim
        return {"q": (np.uint16, (T, hq, d)), "k_new": (np.uint16, (T, hkv, d)), "v_new": (np.uint16, (T, hkv, d)),
                "slot_mapping": (np.int64, (T,)), "cu_seqlens_q": (np.int32, (S + 1,)),
                "seq_slot": (np.int32, (S,)), "context_lens": (np.int32, (ms,)),
                "block_tables": (np.int32, (ms, mb))}

    def fill(self, layout, **arrays) -> None:
        """Write every field of ``layout`` (bf16 tensors as uint16 bit patterns)."""
        if layout.work > self.nbytes:
            raise ValueError(f"staging buffer of {self.nbytes} B is smaller than the layout ({layout.work} B)")
        fields = self._fields(layout)
        if set(arrays) != set(fields):
            raise ValueError(f"fill needs exactly {sorted(fields)}")
        for name, (dtype, shape) in fields.items():
            a = np.asarray(arrays[name])
            if a.dtype != dtype and not (dtype == np.uint16 and a.dtype == np.int16):
                a = a.astype(dtype)
            a = np.ascontiguousarray(a)
            if a.shape != shape:
                raise ValueError(f"{name}: shape {a.shape}, expected {shape}")
            off = getattr(layout, name)
            self._np[off:off + a.nbytes] = a.reshape(-1).view(np.uint8)

    def device_views(self, layout, info):
        """Torch views of the staged inputs and work list in the device buffer (after a ``pkv_step``)."""
        import torch

        tdt = {np.uint16: torch.bfloat16, np.int64: torch.int64, np.int32: torch.int32}
        views = {}
        for name, (dtype, shape) in self._fields(layout).items():
            n = int(np.prod(shape)) * np.dtype(dtype).itemsize
            off = getattr(layout, name)
            raw = self.device[off:off + n]
            views[name] = (raw.view(torch.int16).view(torch.bfloat16) if dtype is np.uint16
                           else raw.view(tdt[dtype])).view(shape)
        nw = int(info.work_words)
        views["work"] = self.device[layout.work:layout.work + 4 * nw].view(torch.int32)
        return views
