"""Full-size GPU parity, in the launch configuration of the benchmark: every MoE layer of a
token captured in one CUDA graph and replayed token after token, with the inputs of that
token copied in first.

* decode, 35B-A3B expert shape: 40 layers, H 2048, I 512, 256 experts top-8 + shared
  expert, BF16, 3788 slots (37% of a 64 GB host pool), B_P:B_H = 52.7:77.3, batch 1;
* decode, FP8 large experts: 8 layers, H 7168, I 2048, 256 experts top-8, E4M3 with
  1x128 block scales, 225 slots (11% of a 93 GB host pool), batch 1 and 8.

Every cache decision is checked through the residency table, owners, stamps and counters
after the run (they fold in every decision of every layer-step) and through the decision
trace of the last layer-step; layer outputs are checked against the float64 oracle on
sampled tokens (host-evaluated pairs contribute zero rows on both sides)."""
import gc

import numpy as np
import pytest
import torch

import oracle as O
import synth
from ftharness import GATE_RTOL, OUT_TOL

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g

    g.build()


def _graph_run(w, pool, banks, shared, steps, check, check_layers=None):
    """Run `steps` tokens of workload `w` as graph replays; compare sampled outputs on the way."""
    from serving_router_top_dedupe_gb300 import ftmoe as F

    L, B, H, E, k = w.n_layers, w.batch, w.hidden, w.n_experts, w.top_k
    fp8 = w.wtype == synth.W_FP8_E4M3_B128
    dev = torch.device("cuda:0")
    trace = synth.routing_trace(w, steps=steps)
    cfg = F.make_config(L, H, w.inter, E, k, w.has_shared, w.wtype, B, w.cache_slots, w.bp_gbps, w.bh_gbps)
    h = F.ft_moe_init(cfg, banks, shared)
    try:
        x_s = torch.empty((L, B, H), dtype=torch.int16, device=dev)
        z_s = torch.empty((L, B, E), dtype=torch.float32, device=dev)
        c_s = torch.zeros((L, B, k, H), dtype=torch.float32, device=dev)
        o_s = torch.empty((L, B, H), dtype=torch.float32, device=dev)
        g = F.ft_moe_graph_capture_decode(h, 0, L, B, x_s, z_s, c_s, o_s)
        sim = O.SlotCache(w.cache_slots, w.n_logical)
        bp, bh = O.mbps(w.bp_gbps), O.mbps(w.bh_gbps)
        zero_c = np.zeros((B, k, H), dtype=np.float32)
        max_err, n_checked = 0.0, 0
        last = None
        for s in range(steps):
            xs = np.stack([synth.decode_x(w, s, l) for l in range(L)])
            zs = np.stack([synth.decode_logits(w, s, l, trace) for l in range(L)])
            x_s.copy_(torch.from_numpy(xs.view(np.int16)))
            z_s.copy_(torch.from_numpy(zs))
            F.ft_graph_launch(g)
            torch.cuda.synchronize(dev)
            out = o_s.cpu().numpy() if s in check else None
            for l in range(L):
                sel, gates = O.route(zs[l], k)
                rec = sim.decode_step(l, E, sel, bp, bh)
                last = (rec, sel, gates)
                if out is not None and (check_layers is None or l in check_layers):
                    sh = None if shared is None else {kk: v[l] for kk, v in shared.items()}
                    ref = O.decode_layer_outputs(rec, sel, gates, xs[l], zero_c, pool.expert, shared=sh, fp8=fp8,
                                                 n_experts=E)
                    err = O.rel_err_rows(out[l], ref)
                    max_err = max(max_err, err)
                    n_checked += 1
                    assert err <= OUT_TOL, f"token {s} layer {l}: relative error {err:.3e}"
        # every decision, through the state it leaves behind
        st = F.ft_moe_get_state(h, w.n_logical, w.cache_slots)
        assert st["clock"] == sim.clock
        assert np.array_equal(st["res"], sim.res), "residency table"
        assert np.array_equal(st["owner"], sim.owner), "slot owners"
        assert np.array_equal(st["stamp"].astype(np.int64), sim.stamp), "slot stamps"
        c = sim.cnt
        ss = F.ft_moe_get_stats(h)
        assert (ss.hits, ss.misses, ss.fills, ss.cpu_execs, ss.evictions) == \
            (c.hits, c.misses, c.fills, c.cpu_execs, c.evictions)
        assert ss.error_word == 0
        # and the last layer-step's decisions one by one
        rec, sel, gates = last
        kcap = min(B * k, E)
        gt = F.ft_moe_get_step_trace(h, B, k, kcap)
        assert np.array_equal(gt["sel"], sel)
        np.testing.assert_allclose(gt["gates"], gates, rtol=GATE_RTOL, atol=0)
        assert gt["q"] == rec.q and gt["victims"] == rec.victims
        assert np.array_equal(gt["slot_of_pair"], rec.slot_of_pair)
        F.ft_graph_destroy(g)
        return c, max_err, n_checked
    finally:
        F.ft_moe_destroy(h)


def test_decode_35b_shape_full_size_graph():
    w = synth.decode_bf16()
    pool = synth.ExpertPool(w)
    banks, shared = pool.routed_banks(), pool.shared_banks()
    # 128 tokens: the 3788 slots fill up after ~100 tokens, so evictions are exercised too
    c, err, n = _graph_run(w, pool, banks, shared, steps=128, check={3, 63, 127})
    print(f"35B shape: misses {c.misses} fills {c.fills} host pairs {c.cpu_execs} evictions {c.evictions};"
          f" {n} layer outputs checked, max rel err {err:.2e}")
    assert c.fills > 0 and c.cpu_execs > 0 and c.evictions > 0
    del banks, shared, pool
    gc.collect()


@pytest.fixture(scope="module")
def fp8_pool():
    w = synth.decode_fp8()
    pool = synth.ExpertPool(w)
    banks = pool.routed_banks()
    yield pool, banks
    del banks, pool
    gc.collect()


@pytest.mark.parametrize("batch,steps,check,layers", [(1, 24, {5, 23}, None), (8, 8, {7}, {0, 5})])
def test_decode_fp8_large_experts_full_size_graph(fp8_pool, batch, steps, check, layers):
    pool, banks = fp8_pool
    w = synth.decode_fp8(batch=batch)
    c, err, n = _graph_run(w, pool, banks, None, steps=steps, check=check, check_layers=layers)
    print(f"FP8 B={batch}: misses {c.misses} fills {c.fills} host pairs {c.cpu_execs}; {n} layer outputs checked,"
          f" max rel err {err:.2e}")
    assert c.fills > 0 and c.cpu_execs > 0
