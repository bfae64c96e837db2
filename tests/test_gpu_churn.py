"""GPU parity over the 200-step continuous-batching churn trace.

Every step of the seeded trace (Poisson arrivals, prompts cut into chunks,
decode rows, retirements whose blocks are reused at once) goes through the
library's scheduler, block pool, lowering, cache write and attention on the
GPU. The oracle replays the same trace with its own admission rules and keeps
each request's keys and values as one contiguous array, with no pool and no
block tables; a wrong block table, slot mapping or row-to-slot map therefore
shows up as a wrong output. Per step, the cache write is checked bit for bit on
the rows it wrote and a sample of output rows against the oracle (the last row
of every prompt chunk and a few random rows), within the attention tolerance.
"""

import numpy as np
import pytest

import oracle
from oracle import churn
from continuous_batching_paged_pkv_gb300 import binding as B
from continuous_batching_paged_pkv_gb300 import build as libbuild
from continuous_batching_paged_pkv_gb300 import runtime as R
from continuous_batching_paged_pkv_gb300 import scheduler as S
from continuous_batching_paged_pkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MAX_REL_L2 = 1e-2


def _replay(spec, seed, num_blocks, max_slots, **policy):
    """Run the trace through the library and the oracle side by side; returns what it saw."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    oracle.build()

    reqs = W.churn_trace(seed, spec)
    bs, hq, hkv, d = spec.block_size, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    mbps = -(-(spec.prompt_max + 2 * spec.output_max + 1) // bs) + 1  # re-prefill covers generated tokens too
    pool = B.Pool(num_blocks, bs, max_slots + policy.get("prefix_cache", 0), mbps,
                  free_order=W.churn_free_order(seed, num_blocks))
    sch = S.ChurnScheduler(reqs, pool, **policy)
    ref = churn.ChurnReplay(reqs, max_slots=max_slots, num_blocks=num_blocks, block_size=bs, **policy)
    hist = churn.ContiguousHistory()
    toks = W.TokenSource(0, hq, hkv, d, requests=reqs)
    scale = 1.0 / np.sqrt(d)
    dev = "cuda"
    k_pool, v_pool = R.empty_pool(num_blocks, hkv, bs, d, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pick = np.random.default_rng(7)

    checked_rows = steps_with_rows = max_ctx = adopted_rows = 0
    saw_prefill_and_decode = saw_retire = False
    refilled = set()
    for step in range(spec.num_steps):
        n_pre = len(sch.preempted)
        rows = sch.plan()
        want = ref.plan()
        assert [(r.rid, r.begin, r.n, r.prefill) for r in rows] == \
               [(r.rid, r.begin, r.n, r.prefill) for r in want], f"step {step}: plans differ"
        assert sch.preempted == ref.preempted, f"step {step}: preemptions differ"
        for rid in sch.preempted[n_pre:]:
            hist.drop(rid)  # its KV is gone; it re-prefills when admitted again
        refilled |= {r.rid for r in rows if r.prefill and r.rid in sch.preempted}
        for r in rows:  # an adopter starts after the cached prefix: its history holds the shared rows
            if r.prefill and r.begin > 0 and hist.len.get(r.rid, 0) == 0:
                pk, pv, _ = toks.rows(r.rid, 0, r.begin)
                hist.append(r.rid, pk, pv)
                adopted_rows += r.n
        if rows:
            steps_with_rows += 1
            low = pool.lower([(r.slot, r.n) for r in rows])
            parts = [toks.rows(r.rid, r.begin, r.begin + r.n) for r in rows]
            k_new = np.concatenate([p[0] for p in parts])
            v_new = np.concatenate([p[1] for p in parts])
            q = np.concatenate([p[2] for p in parts])
            work, info = B.pkv_plan_work(low.cu_seqlens_q, low.seq_slot, low.context_lens,
                                         max_slots=pool.max_slots, max_blocks_per_slot=mbps, block_size=bs,
                                         num_q_heads=hq, num_kv_heads=hkv, head_dim=d)
            t_k, t_v, t_q = (R._bf16_tensor(x, dev) for x in (k_new, v_new, q))
            t_sm = R._i64(low.slot_mapping, dev)
            out = torch.empty((len(q), hq, d), dtype=torch.bfloat16, device=dev)
            ws = torch.empty(max(int(info.workspace_bytes), 1), dtype=torch.uint8, device=dev)
            B.pkv_cache_write(t_k, t_v, t_sm, k_pool, v_pool, device_status=status)
            B.pkv_attention(t_q, R._i32(low.cu_seqlens_q, dev), R._i32(low.seq_slot, dev),
                            R._i32(low.context_lens, dev), R._i32(pool.block_tables(), dev), k_pool, v_pool,
                            R._i32(work, dev), info, out, ws, scale=scale, device_status=status)
            assert B.pkv_check_device_status(status) == 0, f"step {step}: device status"

            # the rows this step wrote, bit for bit
            sm = torch.from_numpy(low.slot_mapping).to(dev)
            blk, row = sm // bs, sm % bs
            got_k, got_v = k_pool[blk, :, row, :], v_pool[blk, :, row, :]  # [T, Hkv, D]
            assert np.array_equal(got_k.view(torch.int16).cpu().numpy().view(np.uint16), k_new), f"step {step}: K"
            assert np.array_equal(got_v.view(torch.int16).cpu().numpy().view(np.uint16), v_new), f"step {step}: V"

            got = out.float().cpu().numpy()
            start = 0
            decode_rows = [i for i, r in enumerate(rows) if not r.prefill]
            sampled_decode = set(pick.choice(decode_rows, min(3, len(decode_rows)), replace=False).tolist()) \
                if decode_rows else set()
            saw_prefill_and_decode |= bool(decode_rows) and any(r.prefill for r in rows)
            for i, (r, (kk, vv, qq)) in enumerate(zip(rows, parts)):
                hist.append(r.rid, kk, vv)
                max_ctx = max(max_ctx, hist.len[r.rid])
                if r.prefill:
                    keep = sorted({r.n - 1, *pick.integers(0, r.n, 2).tolist()})
                elif i in sampled_decode:
                    keep = [0]
                else:
                    keep = []
                if keep:
                    ref_rows = hist.attend(r.rid, qq, scale, keep=keep)
                    g = got[start:start + r.n][keep]
                    e = ref_rows[keep]
                    assert np.isfinite(g).all(), f"step {step} rid {r.rid}: non-finite output"
                    err = np.abs(g - e).max()
                    rel = np.linalg.norm(g - e) / max(np.linalg.norm(e), 1e-30)
                    assert err <= MAX_ABS and rel <= MAX_REL_L2, \
                        f"step {step} rid {r.rid} rows {keep}: max abs {err:.3e}, rel L2 {rel:.3e}"
                    checked_rows += len(keep)
                start += r.n
        done = sch.commit(rows)
        assert done == ref.commit(want), f"step {step}: retirements differ"
        saw_retire |= bool(done)
        for rid in done:
            hist.drop(rid)
        assert pool.stats().free_blocks == ref.free_blocks, f"step {step}: free blocks"

    return dict(steps_with_rows=steps_with_rows, checked_rows=checked_rows, max_ctx=max_ctx,
                saw_prefill_and_decode=saw_prefill_and_decode, saw_retire=saw_retire,
                preempted=list(sch.preempted), reasons=list(sch.preempt_reasons), refilled=refilled,
                cache_events=list(sch.cache_events), adopted_rows=adopted_rows)


def test_churn_trace_matches_contiguous_oracle():
    spec = W.ChurnSpec()
    seen = _replay(spec, 0, spec.num_blocks, spec.max_slots)
    # the trace exercised what it is for
    assert seen["steps_with_rows"] >= spec.num_steps - 5 and seen["checked_rows"] > 300
    assert seen["saw_prefill_and_decode"] and seen["saw_retire"] and seen["max_ctx"] > 2048
    assert not seen["preempted"]


# 300 blocks (4,800 tokens) and 16 slots for ~100 requests of 64-1024 prompt tokens, 30% at priority 1
PRESSURE = W.ChurnSpec(num_steps=200, arrival_rate=0.5, prompt_min=64, prompt_max=1024, output_mean=96.0,
                       output_max=400, high_priority=0.3)


def test_churn_under_pool_pressure_with_preemption_matches_oracle():
    """Watermark admission, priority and decode-headroom preemption, and re-prefill of preempted requests:
    the re-prefilled K/V rows land in new blocks and the outputs still match the contiguous replay."""
    seen = _replay(PRESSURE, 5, 300, 16, watermark=0.01, preemption="lowest-priority")
    assert seen["preempted"] and {"priority", "headroom"} <= set(seen["reasons"])
    assert seen["refilled"]  # some preempted request came back and re-prefilled on the GPU
    assert seen["saw_retire"] and seen["checked_rows"] > 100


PREFIXED = W.ChurnSpec(num_steps=200, arrival_rate=0.5, prompt_min=64, prompt_max=1024, output_mean=96.0,
                       output_max=400, high_priority=0.3, prefix_groups=5, prefix_share=0.6, prefix_min=100,
                       prefix_max=600)


def test_churn_with_prefix_cache_matches_oracle():
    """Shared prompt prefixes through a 4-entry prefix cache on a tight pool: adopters attend over
    blocks another request wrote, whose rows the oracle has as part of the adopter's own history."""
    seen = _replay(PREFIXED, 6, 300, 16, watermark=0.01, preemption="lowest-priority", prefix_cache=4)
    kinds = {e[1] for e in seen["cache_events"]}
    assert {"donate", "adopt", "drop-admission", "drop-headroom"} <= kinds
    assert seen["adopted_rows"] > 0 and seen["checked_rows"] > 100 and seen["saw_retire"]
