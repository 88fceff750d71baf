"""The sweep workload on the 35B-A3B expert shape (H 2048, I 512, 256 experts top-8 +
shared expert, BF16), reduced to 2 layers so that every point fits a short test: batch 1,
4, 16 and 64 (independent locality traces per sequence) x cache capacity 10/25/37/50/100%
of the routed pool x B_P:B_H in {11.8:47.5, 25:50, 52.7:77.3}.

At every point every decision (routing ids, gates, A/H/M, q, victims, slot rewrites) is
compared with the oracle at every layer-step and the final residency state with the
oracle's, and the layer outputs must be bit-identical to those of a run that keeps every
expert resident: the host-evaluated pairs are given the GPU's own rows from that run, so
where an expert is evaluated must not change a single bit.  Miss rate, fills and host pairs
per point are printed (run with -s)."""
import numpy as np
import pytest

import synth
from ftharness import Run

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LAYERS = 2
STEPS = {1: 48, 4: 24, 16: 12, 64: 8}  # enough tokens for the small caches to evict


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g

    g.build()


@pytest.fixture(scope="module")
def sweep_pool():
    w = synth.sweep_point(1, 1.0, synth.SWEEP_RATIOS[0]).with_(n_layers=LAYERS)
    pool = synth.ExpertPool(w)
    return pool.routed_banks(), pool.shared_banks()


@pytest.mark.parametrize("batch", synth.SWEEP_BATCHES)
def test_sweep_points_identical_outputs(sweep_pool, batch):
    banks, shared = sweep_pool
    steps = STEPS[batch]
    base = synth.sweep_point(batch, 1.0, synth.SWEEP_RATIOS[0]).with_(n_layers=LAYERS, steps=steps)
    tr = synth.routing_trace(base)
    # reference: everything resident and every miss filled (B_P > B_H), so no host pairs
    ref = base.with_(cache_slots=base.n_logical, bp_gbps=80.0, bh_gbps=50.0)  # 100% of the 2-layer pool
    rows, outs = {}, {}
    with Run(ref, banks, shared) as r:
        for s in range(steps):
            for l in range(LAYERS):
                _, _, out, rw = r.step(s, l, tr, rows_out=True)
                rows[s, l], outs[s, l] = rw, out
        r.compare_state()
        assert r.sim.cnt.cpu_execs == 0
    table = []
    for cap in synth.SWEEP_CAPACITIES:
        for ratio in synth.SWEEP_RATIOS:
            w = synth.sweep_point(batch, cap, ratio).with_(
                n_layers=LAYERS, steps=steps, cache_slots=synth.capacity_slots(cap, LAYERS, base.n_experts))
            with Run(w, banks, shared) as r:
                for s in range(steps):
                    for l in range(LAYERS):
                        _, _, out, _ = r.step(s, l, tr, cpart=rows[s, l])
                        np.testing.assert_array_equal(out, outs[s, l], err_msg=f"cap {cap} ratio {ratio} s {s} l {l}")
                r.compare_state()
                c = r.sim.cnt
                acts = c.hits + c.misses
                table.append((cap, ratio, c.misses / max(1, acts), c.fills, c.cpu_execs, c.evictions))
    print(f"\nbatch {batch}: capacity, B_P:B_H, miss rate, fills, host pairs, evictions")
    for cap, ratio, mr, f, cpu, ev in table:
        print(f"  {cap:4.0%}  {ratio[0]:4.1f}:{ratio[1]:4.1f}  {mr:6.3f}  {f:5d}  {cpu:5d}  {ev:5d}")
    # B_H > B_P at every split, so every point leaves misses to the host; the smallest cache
    # evicts at every split
    assert all(t[4] > 0 for t in table)
    assert all(t[5] > 0 for t in table if t[0] == synth.SWEEP_CAPACITIES[0])
