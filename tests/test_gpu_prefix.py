"""GPU parity of prefix adoption and copy-on-write blocks.

mlxcel manual, "Continuous batching", §Paged KV cache and prefix sharing:
requests that share a prompt prefix keep its KV blocks once; a request adopts
the donor's blocks by reference instead of prefilling them, a shared block is
copied when a sequence first writes into it, and an adopting request decodes
byte-identically to a cold run.

The trace: A prefills 100 rows; B adopts A's first 70 (the last shared block
is partly filled, so B's first append copies it), C adopts 64 (whole blocks);
then A is released and a new request D takes the freed blocks and writes into
them while B and C keep reading the shared prefix. Each step is checked
* against the oracle: dense attention over each request's own contiguous
  history (the donor's rows for the adopted positions), no pool, no tables;
* bit for bit against a cold run of the same segment in a fresh pool where the
  request prefilled its whole history into blocks of its own.
"""

import numpy as np
import pytest

import oracle
from oracle import kvquant as KQ
from continuous_batching_paged_pkv_gb300 import binding as B
from continuous_batching_paged_pkv_gb300 import build as libbuild
from continuous_batching_paged_pkv_gb300 import runtime as R
from continuous_batching_paged_pkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MAX_REL_L2 = 1e-2
HQ, HKV, D, BS = 32, 8, 128, 16


@pytest.fixture(scope="module", autouse=True)
def cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    oracle.build()
    return torch


class Engine:
    """One pool (bf16 or 8-bit) driven through the library's host and device calls."""

    def __init__(self, kv, num_blocks=256, max_slots=8, mbps=32):
        import torch

        self.kv, self.dev = kv, "cuda"
        self.pool = B.Pool(num_blocks, BS, max_slots, mbps)
        self.max_slots, self.mbps = max_slots, mbps
        if kv == "q8":
            self.arrays = R.empty_pool_q8(num_blocks, HKV, BS, D, self.dev)
        else:
            self.arrays = R.empty_pool(num_blocks, HKV, BS, D, self.dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.copies = 0

    def write(self, low, k, v):
        import torch

        cp = self.pool.take_copies()
        if len(cp):
            self.copies += len(cp)
            B.pkv_copy_blocks(torch.from_numpy(cp).to(self.dev), list(self.arrays), device_status=self.status)
        tk, tv, sm = R._bf16_tensor(k, self.dev), R._bf16_tensor(v, self.dev), R._i64(low.slot_mapping, self.dev)
        if self.kv == "q8":
            kc, ks, vc, vs = self.arrays
            B.pkv_cache_write_q8(tk, tv, sm, kc, ks, vc, vs, device_status=self.status)
        else:
            B.pkv_cache_write(tk, tv, sm, *self.arrays, device_status=self.status)

    def step(self, plan, parts):
        """plan: [(slot, n)], parts: [(k, v, q)] per segment -> float32 output [T, Hq, D]."""
        import torch

        low = self.pool.lower(plan)
        k = np.concatenate([p[0] for p in parts])
        v = np.concatenate([p[1] for p in parts])
        q = np.concatenate([p[2] for p in parts])
        self.write(low, k, v)
        work, info = B.pkv_plan_work(low.cu_seqlens_q, low.seq_slot, low.context_lens, max_slots=self.max_slots,
                                     max_blocks_per_slot=self.mbps, block_size=BS, num_q_heads=HQ,
                                     num_kv_heads=HKV, head_dim=D)
        out = torch.empty((len(q), HQ, D), dtype=torch.bfloat16, device=self.dev)
        nbytes = int(info.workspace_bytes_q8 if self.kv == "q8" else info.workspace_bytes)
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=self.dev)
        args = (R._bf16_tensor(q, self.dev), R._i32(low.cu_seqlens_q, self.dev), R._i32(low.seq_slot, self.dev),
                R._i32(low.context_lens, self.dev), R._i32(self.pool.block_tables(), self.dev))
        if self.kv == "q8":
            B.pkv_attention_q8(*args, *self.arrays, R._i32(work, self.dev), info, out, ws, scale=D ** -0.5,
                               device_status=self.status)
        else:
            B.pkv_attention(*args, *self.arrays, R._i32(work, self.dev), info, out, ws, scale=D ** -0.5,
                            device_status=self.status)
        torch.cuda.synchronize()
        assert B.pkv_check_device_status(self.status) == 0
        return out.float().cpu().numpy(), low


def _history_values(kv, k):
    """The values attention must see for stored rows: bf16 as is, or the 8-bit pool's dequantised
    values (bfloat16 numbers exactly, so they pass through the bf16 oracle unchanged)."""
    if kv == "bf16":
        return k
    deq = KQ.dequantize(*KQ.quantize(k)).astype(np.float32)
    return W.f32_to_bf16_bits(deq)


def _check(kv, got, q, k_hist, v_hist, what):
    ref = oracle.attention_dense(q, _history_values(kv, k_hist), _history_values(kv, v_hist), D ** -0.5)
    assert np.isfinite(got).all(), what
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= MAX_ABS and rel <= MAX_REL_L2, f"{what}: max abs {err:.3e}, rel L2 {rel:.3e}"


def _cold(kv, k_hist, v_hist, n, q, reserve):
    """The same segment (last n rows of the history) in a fresh pool that prefilled everything itself."""
    e = Engine(kv)
    assert e.pool.admit(0, reserve) == B.PKV_OK
    L = len(k_hist)
    if L - n:
        low = e.pool.lower([(0, L - n)])
        e.write(low, k_hist[:L - n], v_hist[:L - n])
    out, _ = e.step([(0, n)], [(k_hist[L - n:], v_hist[L - n:], q)])
    return out


@pytest.mark.parametrize("kv", ["bf16", "q8"])
def test_prefix_adoption_is_cold_identical(kv):
    toks = W.TokenSource(11, HQ, HKV, D)
    e = Engine(kv)
    P = e.pool
    hist_k, hist_v = {}, {}

    def rows(rid, a, b):
        return toks.rows(rid, a, b)

    # step 1: A prefills 100 rows
    ka, va, qa = rows(0, 0, 100)
    assert P.admit(0, 200) == B.PKV_OK
    e.step([(0, 100)], [(ka, va, qa)])
    hist_k[0], hist_v[0] = ka, va

    # B adopts 70 rows (partial last block), C adopts 64 (whole blocks)
    assert P.adopt(1, 0, 70, 120) == B.PKV_OK
    assert P.adopt(2, 0, 64, 100) == B.PKV_OK
    hist_k[1], hist_v[1] = ka[:70], va[:70]
    hist_k[2], hist_v[2] = ka[:64], va[:64]

    # step 2: B appends a 20-row chunk (copy of the shared block first), C and A one row each
    kb, vb, qb = rows(1, 70, 90)
    kc, vc, qc = rows(2, 64, 65)
    ka2, va2, qa2 = rows(0, 100, 101)
    out, low = e.step([(1, 20), (2, 1), (0, 1)], [(kb, vb, qb), (kc, vc, qc), (ka2, va2, qa2)])
    assert e.copies == 1
    hist_k[1], hist_v[1] = np.concatenate([hist_k[1], kb]), np.concatenate([hist_v[1], vb])
    hist_k[2], hist_v[2] = np.concatenate([hist_k[2], kc]), np.concatenate([hist_v[2], vc])
    hist_k[0], hist_v[0] = np.concatenate([hist_k[0], ka2]), np.concatenate([hist_v[0], va2])
    segs = {1: (0, 20, qb), 2: (20, 21, qc), 0: (21, 22, qa2)}
    for slot, (r0, r1, q) in segs.items():
        _check(kv, out[r0:r1], q, hist_k[slot], hist_v[slot], f"step 2 slot {slot}")
        cold = _cold(kv, hist_k[slot], hist_v[slot], r1 - r0, q, 200)
        assert np.array_equal(out[r0:r1], cold), f"step 2 slot {slot}: adopted run differs from the cold run"

    # A retires; D takes freed blocks and writes into them; B and C keep reading the shared prefix
    P.release(0)
    assert P.admit(3, 64) == B.PKV_OK
    kd, vd, qd = rows(3, 0, 40)
    kb2, vb2, qb2 = rows(1, 90, 91)
    kc2, vc2, qc2 = rows(2, 65, 66)
    out, _ = e.step([(3, 40), (1, 1), (2, 1)], [(kd, vd, qd), (kb2, vb2, qb2), (kc2, vc2, qc2)])
    hist_k[1], hist_v[1] = np.concatenate([hist_k[1], kb2]), np.concatenate([hist_v[1], vb2])
    hist_k[2], hist_v[2] = np.concatenate([hist_k[2], kc2]), np.concatenate([hist_v[2], vc2])
    _check(kv, out[:40], qd, kd, vd, "step 3 slot D")
    _check(kv, out[40:41], qb2, hist_k[1], hist_v[1], "step 3 slot B")
    _check(kv, out[41:42], qc2, hist_k[2], hist_v[2], "step 3 slot C")
    assert np.array_equal(out[40:41], _cold(kv, hist_k[1], hist_v[1], 1, qb2, 200))
    assert np.array_equal(out[41:42], _cold(kv, hist_k[2], hist_v[2], 1, qc2, 200))
    st = P.stats()
    assert st.shared_blocks == 4 and st.free_blocks + st.owned_blocks == 256
