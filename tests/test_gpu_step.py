"""GPU parity of the one-call host path (``pkv_step``).

The step's inputs go through a page-locked host staging buffer, one copy in,
the cache write, attention and one copy out. Its output (read back into host
memory) must be bit-identical to the separate device calls on the same inputs,
and within the attention tolerance of the oracle.
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


@pytest.mark.parametrize("name", ["tiny", "decode5", "mixed"])
def test_host_staged_step_matches_device_calls_and_oracle(name):
    import torch

    w = W.make_step(name, 0)
    ds = R.prepare(w)
    R.run_step(ds)
    torch.cuda.synchronize()
    assert B.pkv_check_device_status(ds.status) == 0
    want_bits = ds.out.view(torch.int16).cpu().numpy()
    check_pool = name == "tiny"  # the other steps hold multi-GiB pools
    if check_pool:
        pool_k, pool_v = R.pool_bits(ds)

    low = ds.lowered
    lay = B.pkv_stage_layout_init(w.total_q, len(w.segments), w.max_slots, w.max_blocks_per_slot, w.num_q_heads,
                                  w.num_kv_heads, w.head_dim)
    stage = R.HostStage(lay.work + 4 * int(ds.info.work_words) + 4096, "cuda")
    stage.fill(lay, q=w.q, k_new=w.new_k(), v_new=w.new_v(), slot_mapping=low.slot_mapping,
               cu_seqlens_q=low.cu_seqlens_q, seq_slot=low.seq_slot, context_lens=low.context_lens,
               block_tables=ds.pool.block_tables())
    out = torch.empty_like(ds.out)
    out.view(torch.int16).fill_(R.SENTINEL_BITS)
    out_host = torch.empty(out.shape, dtype=torch.bfloat16, pin_memory=True)
    info = B.pkv_step(lay, stage.host, stage.device, ds.k_pool, ds.v_pool, out, ds.workspace, out_host=out_host,
                      scale=w.scale, device_status=ds.status)
    torch.cuda.synchronize()
    assert B.pkv_check_device_status(ds.status) == 0
    assert (info.num_decode_items, info.num_prefill_items, info.num_combine_items) == \
           (ds.info.num_decode_items, ds.info.num_prefill_items, ds.info.num_combine_items)

    # the staged copy on the device is what was staged on the host
    nbytes = lay.work + 4 * int(info.work_words)
    assert torch.equal(stage.device[:nbytes].cpu(), stage.host[:nbytes])
    got_bits = out_host.view(torch.int16).numpy()
    assert np.array_equal(got_bits, want_bits), "host-staged step differs from the separate calls"
    if check_pool:  # rewriting the same rows leaves the pool as it was
        k2, v2 = R.pool_bits(ds)
        assert np.array_equal(k2, pool_k) and np.array_equal(v2, pool_v)

    # the same call with its arguments bound once, twice in a row, gives the same bits
    call = B.StepCall(lay, stage.host, stage.device, ds.k_pool, ds.v_pool, out, ds.workspace, out_host=out_host,
                      scale=w.scale, device_status=ds.status)
    for _ in range(2):
        out_host.view(torch.int16).fill_(R.SENTINEL_BITS)
        call()
        torch.cuda.synchronize()
        assert np.array_equal(out_host.view(torch.int16).numpy(), want_bits), "bound step call differs"
    assert B.pkv_check_device_status(ds.status) == 0

    st = oracle.prepare_step(w)
    ref = oracle.step_attention(w, st)
    got = out_host.float().numpy()
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert np.isfinite(got).all() and err <= MAX_ABS and rel <= MAX_REL_L2, (err, rel)


@pytest.mark.parametrize("name", ["decode5", "tiny"])
def test_in_place_step_matches_device_calls(name):
    """PKV_STEP_IN_PLACE: a small step without prompt chunks reads the staging buffer in place
    and writes its output straight to out_host (the device stage and `out` stay untouched), bit
    for bit the same as the separate device calls; a step with a prompt chunk (tiny) copies its
    inputs in and also writes its output straight to out_host."""
    import torch

    w = W.make_step(name, 0)
    ds = R.prepare(w)
    R.run_step(ds)
    torch.cuda.synchronize()
    assert B.pkv_check_device_status(ds.status) == 0
    want_bits = ds.out.view(torch.int16).cpu().numpy()
    low = ds.lowered
    lay = B.pkv_stage_layout_init(w.total_q, len(w.segments), w.max_slots, w.max_blocks_per_slot, w.num_q_heads,
                                  w.num_kv_heads, w.head_dim)
    stage = R.HostStage(lay.work + 4 * int(ds.info.work_words) + 4096, "cuda")
    stage.fill(lay, q=w.q, k_new=w.new_k(), v_new=w.new_v(), slot_mapping=low.slot_mapping,
               cu_seqlens_q=low.cu_seqlens_q, seq_slot=low.seq_slot, context_lens=low.context_lens,
               block_tables=ds.pool.block_tables())
    stage.device.fill_(0x5A)
    out = torch.empty_like(ds.out)
    out.view(torch.int16).fill_(R.SENTINEL_BITS)
    out_host = torch.empty(out.shape, dtype=torch.bfloat16, pin_memory=True)
    call = B.StepCall(lay, stage.host, stage.device, ds.k_pool, ds.v_pool, out, ds.workspace, out_host=out_host,
                      scale=w.scale, device_status=ds.status, in_place=True)
    for _ in range(2):  # twice: nothing left over from the first call decides the second
        out_host.view(torch.int16).fill_(R.SENTINEL_BITS)
        info = call()
        torch.cuda.synchronize()
        assert B.pkv_check_device_status(ds.status) == 0
        assert np.array_equal(out_host.view(torch.int16).numpy(), want_bits), "in-place step differs"
    copied = info.num_prefill_items > 0
    assert copied == (name == "tiny")
    assert bool((stage.device[:64] != 0x5A).any()) == copied, "the device stage is written only by the copy"
    assert (out.view(torch.int16) == R.SENTINEL_BITS).all(), "`out` is never written"


def test_host_staged_step_views_feed_the_device_calls():
    """The device views of a staged step drive pkv_cache_write / pkv_attention to the same bits."""
    import torch

    w = W.make_step("mixed", 0)
    ds = R.prepare(w)
    low = ds.lowered
    lay = B.pkv_stage_layout_init(w.total_q, len(w.segments), w.max_slots, w.max_blocks_per_slot, w.num_q_heads,
                                  w.num_kv_heads, w.head_dim)
    stage = R.HostStage(lay.work + 4 * int(ds.info.work_words), "cuda")
    stage.fill(lay, q=w.q, k_new=w.new_k(), v_new=w.new_v(), slot_mapping=low.slot_mapping,
               cu_seqlens_q=low.cu_seqlens_q, seq_slot=low.seq_slot, context_lens=low.context_lens,
               block_tables=ds.pool.block_tables())
    out = torch.empty_like(ds.out)
    info = B.pkv_step(lay, stage.host, stage.device, ds.k_pool, ds.v_pool, out, ds.workspace, scale=w.scale,
                      device_status=ds.status)
    v = stage.device_views(lay, info)
    out2 = torch.empty_like(out)
    B.pkv_cache_write(v["k_new"], v["v_new"], v["slot_mapping"], ds.k_pool, ds.v_pool, device_status=ds.status)
    B.pkv_attention(v["q"], v["cu_seqlens_q"], v["seq_slot"], v["context_lens"], v["block_tables"], ds.k_pool,
                    ds.v_pool, v["work"], info, out2, ds.workspace, scale=w.scale, device_status=ds.status)
    torch.cuda.synchronize()
    assert B.pkv_check_device_status(ds.status) == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("name", ["verify4", "mixed", "verify16"])
def test_in_place_output_of_larger_steps(name):
    """PKV_STEP_IN_PLACE on steps above the in-place input size: each copies its inputs in
    and writes its output rows straight into out_host, so `out` keeps its sentinel; the decode
    and merge kernels (verify4, 2 MiB of queries) store rows as they go, the chunk kernel
    (mixed: a 512-row chunk beside decode rows; verify16: many short chunk segments) stages
    its rows in shared memory first. Bit for bit the same as the separate device calls."""
    import torch

    w = W.make_step(name, 0)
    ds = R.prepare(w)
    R.run_step(ds)
    torch.cuda.synchronize()
    assert B.pkv_check_device_status(ds.status) == 0
    want_bits = ds.out.view(torch.int16).cpu().numpy()
    low = ds.lowered
    lay = B.pkv_stage_layout_init(w.total_q, len(w.segments), w.max_slots, w.max_blocks_per_slot, w.num_q_heads,
                                  w.num_kv_heads, w.head_dim)
    assert lay.work > B.PKV_STEP_IN_PLACE_MAX_BYTES
    stage = R.HostStage(lay.work + 4 * int(ds.info.work_words) + 4096, "cuda")
    stage.fill(lay, q=w.q, k_new=w.new_k(), v_new=w.new_v(), slot_mapping=low.slot_mapping,
               cu_seqlens_q=low.cu_seqlens_q, seq_slot=low.seq_slot, context_lens=low.context_lens,
               block_tables=ds.pool.block_tables())
    stage.device.fill_(0x5A)
    out = torch.empty_like(ds.out)
    out.view(torch.int16).fill_(R.SENTINEL_BITS)
    out_host = torch.empty(out.shape, dtype=torch.bfloat16, pin_memory=True)
    call = B.StepCall(lay, stage.host, stage.device, ds.k_pool, ds.v_pool, out, ds.workspace, out_host=out_host,
                      scale=w.scale, device_status=ds.status, in_place=True)
    for _ in range(2):
        out_host.view(torch.int16).fill_(R.SENTINEL_BITS)
        info = call()
        torch.cuda.synchronize()
        assert B.pkv_check_device_status(ds.status) == 0
        assert np.array_equal(out_host.view(torch.int16).numpy(), want_bits), "in-place output differs"
    chunked = info.num_prefill_items > 0
    assert chunked == (name != "verify4")
    assert bool((stage.device[:64] != 0x5A).any()), "inputs above the in-place size are copied in"
    assert (out.view(torch.int16) == R.SENTINEL_BITS).all(), "`out` is never written"
