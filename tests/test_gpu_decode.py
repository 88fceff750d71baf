"""GPU parity of the decode path (control kernel, fill, SwiGLU GEMV, combine) against
the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from ftharness import OUT_TOL, Run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g

    g.build()


def test_tiny_config_every_step():
    """8 steps x 2 layers, batch 1, 8 slots, 11.8:47.5: every decision, state and output."""
    w = synth.tiny()
    with Run(w) as r:
        for s in range(w.steps):
            for l in range(w.n_layers):
                r.step(s, l, check_out=True)
                r.compare_state()
        assert r.sim.cnt.misses > 0 and r.sim.cnt.cpu_execs > 0 and r.sim.cnt.evictions > 0


@pytest.mark.parametrize("batch,capacity", [(1, 0.37), (1, 0.06), (4, 0.10)])
def test_decode_bf16_shape_reduced_layers(batch, capacity):
    """35B-A3B expert shape (H 2048, I 512, E 256, top-8 + shared), 4 layers."""
    w = synth.decode_bf16(batch=batch).with_(n_layers=4, steps=48)
    w = w.with_(cache_slots=synth.capacity_slots(capacity, 4, 256))
    tr = synth.routing_trace(w)
    with Run(w) as r:
        for s in range(w.steps):
            for l in range(w.n_layers):
                r.step(s, l, tr, check_out=(s % 8 == 3))
        r.compare_state()
        assert r.sim.cnt.cpu_execs > 0
        assert capacity > 0.3 or r.sim.cnt.evictions > 0
        print("max rel err", r.max_err)


def test_decode_batch64_ragged_and_all_experts():
    """Batch 64 (every expert active, ragged tokens per expert), small cache."""
    w = synth.sweep_point(64, 0.10, (25.0, 50.0)).with_(n_layers=2, steps=6, n_experts=64)
    w = w.with_(cache_slots=synth.capacity_slots(0.25, 2, 64))
    tr = synth.routing_trace(w)
    with Run(w) as r:
        for s in range(w.steps):
            for l in range(w.n_layers):
                r.step(s, l, tr, check_out=(s >= 4))
        r.compare_state()


@pytest.mark.parametrize("batch", [1, 8])
def test_decode_fp8_expert_shape(batch):
    """FP8 E4M3 experts with 1x128 block scales at the 7168 x 2048 expert shape (2 layers, 32 experts)."""
    w = synth.decode_fp8(batch=batch).with_(n_layers=2, n_experts=32, steps=10, cache_slots=7)
    tr = synth.routing_trace(w)
    with Run(w) as r:
        for s in range(w.steps):
            for l in range(w.n_layers):
                r.step(s, l, tr, check_out=(s % 3 == 1))
        r.compare_state()
        print("max rel err", r.max_err)


def test_outputs_identical_across_capacity_and_split():
    """Same layer outputs, bit for bit, at every cache size and B_P:B_H split when the
    host rows are the GPU's own rows for those pairs."""
    base = synth.decode_bf16(batch=4).with_(n_layers=3, n_experts=64, steps=10)
    tr = synth.routing_trace(base)
    pool = synth.ExpertPool(base)
    banks, shared = pool.routed_banks(), pool.shared_banks()
    full = base.with_(cache_slots=base.n_logical, bp_gbps=80.0, bh_gbps=50.0)   # everything resident
    rows, outs = {}, {}
    with Run(full, banks, shared) as r:
        for s in range(base.steps):
            for l in range(base.n_layers):
                _, _, out, rw = r.step(s, l, tr, rows_out=True)
                rows[s, l], outs[s, l] = rw, out
    for slots, ratio in [(8, (11.8, 47.5)), (40, (52.7, 77.3)), (19, (25.0, 50.0)), (64, (52.7, 77.3))]:
        w = base.with_(cache_slots=slots, bp_gbps=ratio[0], bh_gbps=ratio[1])
        with Run(w, banks, shared) as r:
            for s in range(base.steps):
                for l in range(base.n_layers):
                    _, _, out, _ = r.step(s, l, tr, cpart=rows[s, l])
                    np.testing.assert_array_equal(out, outs[s, l])
            assert r.sim.cnt.cpu_execs > 0


def test_graph_replay_matches_eager():
    w = synth.decode_bf16(batch=2).with_(n_layers=4, n_experts=64, steps=6, cache_slots=60)
    tr = synth.routing_trace(w)
    pool = synth.ExpertPool(w)
    banks, shared = pool.routed_banks(), pool.shared_banks()
    L, B, H, E, k = w.n_layers, w.batch, w.hidden, w.n_experts, w.top_k
    dev = torch.device("cuda:0")
    x = torch.empty((L, B, H), dtype=torch.int16, device=dev)
    z = torch.empty((L, B, E), dtype=torch.float32, device=dev)
    cp = torch.zeros((L, B, k, H), dtype=torch.float32, device=dev)
    out_e = torch.empty((L, B, H), dtype=torch.float32, device=dev)
    out_g = torch.empty_like(out_e)
    with Run(w, banks, shared) as re, Run(w, banks, shared) as rg:
        F = re.F
        g = F.ft_moe_graph_capture_decode(rg.h, 0, L, B, x, z, cp, out_g)
        for s in range(w.steps):
            for l in range(L):
                xb, zz = re.inputs(s, l, tr)
                x[l].copy_(torch.from_numpy(xb.view(np.int16)))
                z[l].copy_(torch.from_numpy(zz))
            F.ft_moe_decode_layers(re.h, 0, L, B, x, z, cp, out_e)
            F.ft_graph_launch(g)
            F.ft_moe_synchronize(rg.h)
            F.ft_moe_synchronize(re.h)
            assert torch.equal(out_e, out_g)
        se = F.ft_moe_get_state(re.h, w.n_logical, w.cache_slots)
        sg = F.ft_moe_get_state(rg.h, w.n_logical, w.cache_slots)
        for key in ("res", "owner", "stamp"):
            assert np.array_equal(se[key], sg[key])
        F.ft_graph_destroy(g)


def test_memcpy_fill_mode_matches_kernel_fill():
    w = synth.decode_bf16().with_(n_layers=3, n_experts=64, steps=12, cache_slots=20)
    tr = synth.routing_trace(w)
    pool = synth.ExpertPool(w)
    banks, shared = pool.routed_banks(), pool.shared_banks()
    with Run(w, banks, shared) as a, Run(w, banks, shared, fill_mode=1) as b:
        for s in range(w.steps):
            for l in range(w.n_layers):
                _, _, oa, _ = a.step(s, l, tr, check_out=(s % 4 == 0))
                _, _, ob, _ = b.step(s, l, tr, check_out=(s % 4 == 0))
                np.testing.assert_array_equal(oa, ob)
        a.compare_state()
        b.compare_state()


def test_nan_logits_set_the_error_word():
    w = synth.tiny()
    with Run(w) as r:
        F = r.F
        dev = torch.device("cuda:0")
        xb, z = r.inputs(0, 0)
        z[0, 3] = np.nan
        out = torch.empty((1, w.hidden), dtype=torch.float32, device=dev)
        cp = torch.zeros((1, w.top_k, w.hidden), dtype=torch.float32, device=dev)
        F.ft_moe_decode_step(r.h, 0, 1, torch.from_numpy(xb.view(np.int16)).to(dev), torch.from_numpy(z).to(dev),
                             cp, out)
        st = F.ft_moe_get_stats(r.h)
        assert st.error_word & F.FT_DEVERR_NAN_LOGIT
        tr = F.ft_moe_get_step_trace(r.h, 1, w.top_k, w.top_k)
        assert 3 not in tr["sel"][0]


def test_argument_errors_leave_state_untouched():
    w = synth.tiny()
    with Run(w) as r:
        F = r.F
        for bad in [dict(layer=-1), dict(layer=w.n_layers), dict(batch=0), dict(batch=2)]:
            args = dict(layer=0, batch=1)
            args.update(bad)
            with pytest.raises(F.FtError) as e:
                F.ft_moe_decode_step(r.h, args["layer"], args["batch"], 1, 1, 1, 1)
            assert e.value.status == F.FT_ERR_INVALID
        with pytest.raises(F.FtError):   # c_partial NULL while B_H > B_P
            F.ft_moe_decode_step(r.h, 0, 1, 1, 1, None, 1)
        st = F.ft_moe_get_stats(r.h)
        assert st.decode_steps == 0 and st.clock == 0


def test_resize_shrink_and_grow_match_oracle():
    w = synth.decode_bf16(batch=2).with_(n_layers=3, n_experts=32, hidden=512, inter=256, steps=16, cache_slots=40)
    tr = synth.routing_trace(w)
    with Run(w) as r:
        for s in range(8):
            for l in range(w.n_layers):
                r.step(s, l, tr)
        for new in (17, 5, 33):
            r.F.ft_cache_resize(r.h, new)
            r.sim.resize(new)
            r.compare_state()
            for s in range(8, 12) if new != 33 else range(12, 16):
                for l in range(w.n_layers):
                    r.step(s, l, tr, check_out=True)
            r.compare_state()
