"""GPU parity of block-FP4 experts on the decode path against the float64 oracle: NVFP4
(E2M1 weights packed two per byte, one E4M3 scale per 1x16 block applied after the
block's dot product, one FP32 tensor scale per bank) and MXFP4 (the same elements, one
E8M0 scale per 1x32 block); fills move every bank by the copy kernel and by
cudaMemcpyAsync."""
import numpy as np
import pytest

import synth
from ftharness import Run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g

    g.build()


FP4 = [synth.W_NVFP4, synth.W_MXFP4]


@pytest.mark.parametrize("wtype", FP4)
@pytest.mark.parametrize("batch", [1, 4])
def test_fp4_tiny_every_step(batch, wtype):
    """16 experts top-2, 8 slots, 11.8:47.5: fills, evictions and host pairs."""
    w = synth.tiny().with_(wtype=wtype, batch=batch, steps=10)
    with Run(w) as r:
        for s in range(w.steps):
            for l in range(w.n_layers):
                r.step(s, l, check_out=True)
        r.compare_state()
        print(f"batch {batch}: max rel err {r.max_err:.2e}")
        assert r.sim.cnt.fills > 0 and r.sim.cnt.cpu_execs > 0


@pytest.mark.parametrize("wtype,batch", [(synth.W_NVFP4, 1), (synth.W_NVFP4, 4), (synth.W_MXFP4, 1)])
def test_fp4_35b_expert_shape(wtype, batch):
    """H 2048, I 512, 256 experts top-8 + shared expert, 2 layers, 25% of the pool."""
    w = synth.decode_bf16(batch=batch).with_(wtype=wtype, n_layers=2, steps=8,
                                             cache_slots=synth.capacity_slots(0.25, 2, 256))
    tr = synth.routing_trace(w)
    with Run(w) as r:
        for s in range(w.steps):
            for l in range(w.n_layers):
                r.step(s, l, tr, check_out=(s % 3 == 1))
        r.compare_state()
        print(f"batch {batch}: max rel err {r.max_err:.2e}")


@pytest.mark.parametrize("wtype", FP4)
def test_fp4_memcpy_fill_matches_kernel_fill(wtype):
    w = synth.tiny().with_(wtype=wtype, steps=8)
    pool = synth.ExpertPool(w)
    banks = pool.routed_banks()
    with Run(w, banks, None) as a, Run(w, banks, None, fill_mode=1) as b:
        for s in range(w.steps):
            for l in range(w.n_layers):
                _, _, oa, _ = a.step(s, l, check_out=(s % 2 == 0))
                _, _, ob, _ = b.step(s, l, check_out=(s % 2 == 0))
                np.testing.assert_array_equal(oa, ob)
        a.compare_state()
        b.compare_state()
