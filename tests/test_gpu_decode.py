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


@pytest.mark.parametrize("batch,slots", [(1, 20), (1, 60), (4, 40)])
def test_multilayer_call_matches_per_layer_calls(batch, slots):
    """ft_moe_decode_layers takes the decisions of every layer after the first before the
    control kernel's dependency wait, and starts a fill early when no victim slot belongs to
    the previous layer-step; per-layer ft_moe_decode_step calls take them after the wait.
    Outputs and the residency state must agree bit for bit, with caches small enough that
    victims often belong to the previous layer-step (the fill then takes its ordinary path)."""
    w = synth.decode_bf16(batch=batch).with_(n_layers=5, n_experts=64, steps=8, cache_slots=slots)
    tr = synth.routing_trace(w)
    pool = synth.ExpertPool(w)
    banks, shared = pool.routed_banks(), pool.shared_banks()
    L, B, H, E, k = w.n_layers, w.batch, w.hidden, w.n_experts, w.top_k
    dev = torch.device("cuda:0")
    x = torch.empty((L, B, H), dtype=torch.int16, device=dev)
    z = torch.empty((L, B, E), dtype=torch.float32, device=dev)
    cp = torch.zeros((L, B, k, H), dtype=torch.float32, device=dev)
    out_m = torch.empty((L, B, H), dtype=torch.float32, device=dev)
    out_s = torch.empty_like(out_m)
    with Run(w, banks, shared) as rm, Run(w, banks, shared) as rs:
        F = rm.F
        g = F.ft_moe_graph_capture_decode(rm.h, 0, L, B, x, z, cp, out_m)
        for s in range(w.steps):
            for l in range(L):
                xb, zz = rm.inputs(s, l, tr)
                x[l].copy_(torch.from_numpy(xb.view(np.int16)))
                z[l].copy_(torch.from_numpy(zz))
            F.ft_graph_launch(g)
            F.ft_moe_synchronize(rm.h)
            for l in range(L):
                F.ft_moe_decode_step(rs.h, l, B, x[l], z[l], cp[l], out_s[l])
            F.ft_moe_synchronize(rs.h)
            assert torch.equal(out_m, out_s), f"token {s}"
        sm = F.ft_moe_get_state(rm.h, w.n_logical, w.cache_slots)
        ss = F.ft_moe_get_state(rs.h, w.n_logical, w.cache_slots)
        for key in ("res", "owner", "stamp"):
            assert np.array_equal(sm[key], ss[key]), key
        assert F.ft_moe_get_stats(rm.h).error_word == 0 and F.ft_moe_get_stats(rs.h).error_word == 0
        assert F.ft_moe_get_stats(rm.h).fills > 0


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


def test_host_hook_evaluates_the_c_set_in_step():
    """The in-step host branch: the hook sees the step's routing, computes the C pairs'
    rows (here with the float64 oracle) and the library folds them in.  Decisions match the
    oracle, outputs match the oracle, and they equal bit for bit a run that passes the same
    rows through c_partial; the same holds for a graph replay with the hook as a host node."""
    import oracle as O

    w = synth.decode_bf16().with_(n_layers=2, n_experts=64, steps=6, cache_slots=12)
    tr = synth.routing_trace(w, steps=w.steps + 3)  # 3 more tokens for the graph replays
    pool = synth.ExpertPool(w)
    banks, shared = pool.routed_banks(), pool.shared_banks()
    seen = []

    def rows_for(layer, xb, sel, gates, slot):
        cp = np.zeros((w.batch, w.top_k, w.hidden), dtype=np.float32)
        for t in range(w.batch):
            for r in range(w.top_k):
                if slot[t, r] < 0:
                    cp[t, r] = O.pair_row(pool.expert(layer * w.n_experts + int(sel[t, r])),
                                          O.bf16_to_f64(xb[t]), gates[t, r], False).astype(np.float32)
        return cp

    with Run(w, banks, shared) as hooked, Run(w, banks, shared) as plain:
        F = hooked.F
        xcur, hook_rows = {}, {}

        def hook(layer, batch, sel, gates, slot, rows):
            k = w.top_k
            cp = rows_for(layer, xcur[layer], sel.reshape(batch, k), gates.reshape(batch, k), slot.reshape(batch, k))
            rows.reshape(batch, k, w.hidden)[:] = cp
            hook_rows[layer] = cp
            seen.append((layer, int((slot < 0).sum())))

        F.ft_moe_set_host_hook(hooked.h, hook)
        dev = torch.device("cuda:0")
        for s in range(w.steps):
            for l in range(w.n_layers):
                xb, z = hooked.inputs(s, l, tr)
                xcur[l] = xb
                sel, gates = O.route(z, w.top_k)
                rec = hooked.sim.decode_step(l, w.n_experts, sel, hooked.bp, hooked.bh)
                x_d = torch.from_numpy(xb.view(np.int16)).to(dev)
                z_d = torch.from_numpy(z).to(dev)
                out_d = torch.empty((w.batch, w.hidden), dtype=torch.float32, device=dev)
                F.ft_moe_decode_step(hooked.h, l, w.batch, x_d, z_d, None, out_d)
                F.ft_moe_synchronize(hooked.h)  # the hook runs while this call waits
                gt = F.ft_moe_get_step_trace(hooked.h, w.batch, w.top_k, hooked.kcap)
                hooked.compare(rec, sel, gates, gt)
                cp = rows_for(l, xb, sel, gates, rec.slot_of_pair)
                ref = O.decode_layer_outputs(rec, sel, gates, xb, cp, hooked.expert, shared=hooked.shared_expert(l),
                                             n_experts=w.n_experts)
                out = out_d.cpu().numpy()
                assert O.rel_err_rows(out, ref) <= 1e-2
                # the hook computed its rows from the device's gates: pass exactly those rows
                _, _, out_p, _ = plain.step(s, l, tr, cpart=hook_rows[l])
                np.testing.assert_array_equal(out, out_p)
        hooked.compare_state()
        assert any(n > 0 for _, n in seen)

        # a graph with the hook as a host node, replayed for the next steps
        L, B, H, E, k = w.n_layers, w.batch, w.hidden, w.n_experts, w.top_k
        x = torch.empty((L, B, H), dtype=torch.int16, device=dev)
        z = torch.empty((L, B, E), dtype=torch.float32, device=dev)
        outg = torch.empty((L, B, H), dtype=torch.float32, device=dev)
        g = F.ft_moe_graph_capture_decode(hooked.h, 0, L, B, x, z, None, outg)
        for s in range(w.steps, w.steps + 3):
            for l in range(L):
                xb, zz = hooked.inputs(s, l, tr)
                xcur[l] = xb
                x[l].copy_(torch.from_numpy(xb.view(np.int16)))
                z[l].copy_(torch.from_numpy(zz))
            F.ft_graph_launch(g)
            F.ft_moe_synchronize(hooked.h)
            for l in range(L):
                xb, zz = hooked.inputs(s, l, tr)
                sel, gates = O.route(zz, k)
                rec = hooked.sim.decode_step(l, E, sel, hooked.bp, hooked.bh)
                _, _, out_p, _ = plain.step(s, l, tr, cpart=hook_rows[l])
                np.testing.assert_array_equal(outg[l].cpu().numpy(), out_p)
        hooked.compare_state()
        F.ft_graph_destroy(g)
        F.ft_moe_set_host_hook(hooked.h, None)


def _scaled_x(xb, factor, mixed=False):
    """BF16 activations times `factor` (rounded to BF16); mixed: alternate elements keep
    their N(0, 1) size, so one token spans ~1e5 to ~1e-6 of its largest value."""
    x = O.bf16_to_f64(xb)
    f = np.full(x.shape, float(factor))
    if mixed:
        f[..., 1::2] = 1e-6
    return synth.f32_to_bf16_bits((x * f).astype(np.float32)).reshape(xb.shape)


@pytest.mark.parametrize("wtype,batch", [(synth.W_FP8_E4M3_B128, 1), (synth.W_FP8_E4M3_B128, 4),
                                         (synth.W_NVFP4, 1), (synth.W_MXFP4, 4)])
@pytest.mark.parametrize("factor,mixed", [(1e5, False), (1e-6, False), (1e5, True)])
def test_fp8_fp4_activation_magnitudes(wtype, batch, factor, mixed):
    """FP8 and FP4 products take the activations as F16.  BF16 activations far outside F16's
    range (~1e5 and ~1e-6, and both within one token) still match the oracle: each token is
    scaled by an exact power of two before the narrowing and back after the sum."""
    if wtype == synth.W_FP8_E4M3_B128:
        w = synth.decode_fp8(batch=batch).with_(n_layers=2, n_experts=16, hidden=1024, inter=256, steps=4,
                                                cache_slots=12)
    else:
        w = synth.tiny().with_(wtype=wtype, batch=batch, steps=4)
    tr = synth.routing_trace(w) if w.logits == "trace" else None
    with Run(w) as r:
        for s in range(w.steps):
            for l in range(w.n_layers):
                xb, z = r.inputs(s, l, tr)
                r.step(s, l, tr, check_out=True, xz=(_scaled_x(xb, factor, mixed), z))
        r.compare_state()
        print(f"factor {factor} mixed {mixed}: max rel err {r.max_err:.2e}")
