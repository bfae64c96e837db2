"""pkv_attention_no_alloc: the attention call for callers that cannot allocate.

A serving process that reserves all device memory in its own arena, or a loop
that may not allocate between steps, calls this entry point instead of
pkv_attention; it keeps the span partials in the library's fixed device array.
These tests drive it through the C ABI and compare it with pkv_attention on
the same step, twice in a row (the array keeps the previous call's contents).
This file is collected last on purpose.
"""

import numpy as np
import pytest

import oracle
from continuous_batching_paged_pkv_gb300 import binding as B
from continuous_batching_paged_pkv_gb300 import build as libbuild
from continuous_batching_paged_pkv_gb300 import runtime as R
from continuous_batching_paged_pkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MAX_REL_L2 = 1e-2


@pytest.fixture(scope="module", autouse=True)
def cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    oracle.build()
    return torch


def _close(got, ref):
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert np.isfinite(got).all()
    assert err.max() <= MAX_ABS and rel <= MAX_REL_L2, (err.max(), rel)


def _many_decode_tasks():
    """128 one-row decode slots at contexts of 4-8 key spans, 64 q / 8 kv heads:
    about 6,000 (span, kv head) tasks, more than three rounds for every warp of
    a 152-SM grid, so the decode kernel hands out the rest from the task
    counter that lives in the scratch array; its partials (~26 MB) still fit."""
    ctx = np.random.default_rng(11).integers(1024, 2049, size=128)
    return W.random_step(11, [(1, int(c)) for c in ctx], num_q_heads=64, num_kv_heads=8, head_dim=128)


CASES = {
    "decode x5": lambda: W.decode5(0),
    "mixed": lambda: W.mixed(0),
    "ragged": lambda: W.random_step(3, [(1, 3000), (40, 333), (1, 70)], num_q_heads=32, num_kv_heads=8,
                                    head_dim=128),
    "many decode tasks": _many_decode_tasks,
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_no_alloc_matches_pkv_attention_bit_for_bit_twice(cuda, case):
    """Same kernels, same work list: the outputs must be the same bits as
    pkv_attention's, on two calls in a row (the second finds the scratch array,
    task counter included, as the first left it)."""
    torch = cuda
    w = CASES[case]()
    ds = R.prepare(w)
    assert 0 < ds.info.workspace_bytes <= B.PKV_NO_ALLOC_SCRATCH_BYTES or ds.info.workspace_bytes == 0
    R.run_step(ds)
    torch.cuda.synchronize()
    assert B.pkv_check_device_status(ds.status) == 0
    ref_bits = ds.out.view(torch.int16).clone()
    # the reference itself is checked against the oracle once
    st = oracle.prepare_step(w)
    _close(R.out_f32(ds), oracle.step_attention(w, st))
    for _ in range(2):
        out = torch.empty_like(ds.out)
        out.view(torch.int16).fill_(R.SENTINEL_BITS)
        B.pkv_attention_no_alloc(ds.q, ds.cu_seqlens_q, ds.seq_slot, ds.context_lens, ds.block_tables, ds.k_pool,
                                 ds.v_pool, ds.work, ds.info, out, scale=w.scale, device_status=ds.status)
        torch.cuda.synchronize()
        assert B.pkv_check_device_status(ds.status) == 0
        assert torch.equal(out.view(torch.int16), ref_bits), "no-alloc output differs from pkv_attention's"


def test_no_alloc_rejects_a_step_larger_than_its_array(cuda):
    torch = cuda
    w = W.tiny(0)
    ds = R.prepare(w)
    big = B.WorkInfo()
    ctypes_fields = ("num_decode_items", "num_prefill_items", "num_combine_items", "num_partials", "work_words")
    for f in ctypes_fields:
        setattr(big, f, getattr(ds.info, f))
    big.workspace_bytes = B.PKV_NO_ALLOC_SCRATCH_BYTES + 256
    with pytest.raises(B.PkvError, match="WORKSPACE_TOO_SMALL"):
        B.pkv_attention_no_alloc(ds.q, ds.cu_seqlens_q, ds.seq_slot, ds.context_lens, ds.block_tables, ds.k_pool,
                                 ds.v_pool, ds.work, big, ds.out, scale=w.scale)
    torch.cuda.synchronize()
