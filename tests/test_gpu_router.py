"""GPU parity of the router on hidden states: the router kernel's logits against the
oracle's float64 logits (within the FP32 accumulation bound, at every launch shape the
library uses, bitwise reproducible), and the decode and prefill calls that take hidden
states, for each gate function.  The oracle routes on its own float64 logits: every
decision is compared exactly, except that a token whose float64 top-k margin lies inside
twice the logit error bound (a near tie, where either side is correct) takes the kernel's
choice once it is shown to lie inside that band; the tests report how many there were.
Outputs are within the layer tolerance and the final residency is identical.

Edge cases of the top-k itself (equal logits, -0 and +0, -inf, NaN ranked as -inf) run on
given logits through the decode and prefill routers and are compared in full."""
import numpy as np
import pytest
import torch

import synth
from ftharness import Run, prefill_step

pytestmark = pytest.mark.gpu

GATES = (0, 1, 2)  # FT_GATE_SOFTMAX_TOPK, FT_GATE_SOFTMAX_ALL, FT_GATE_SIGMOID_TOPK


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g

    g.build()


@pytest.fixture(scope="module")
def pool35():
    """Expert banks of the 35B-A3B shape reduced to 2 layers, shared by the tests below."""
    w = synth.decode_bf16().with_(n_layers=2)
    p = synth.ExpertPool(w)
    return p.routed_banks(), p.shared_banks()


def _logits(r, layer, xb):
    x_d = torch.from_numpy(xb.view(np.int16)).to(r.dev)
    z_d = torch.empty((xb.shape[0], r.w.n_experts), dtype=torch.float32, device=r.dev)
    torch.cuda.synchronize()
    r.F.ft_moe_router_logits(r.h, layer, xb.shape[0], x_d, z_d)
    r.F.ft_moe_synchronize(r.h)
    return z_d.cpu().numpy()


@pytest.mark.parametrize("shape", ["35B", "wide"])
def test_router_logits_bound_and_launch_shapes(shape, pool35):
    """35B-A3B shape (H 2048, E 256), and H 7168 with 64 experts (the hidden size of the
    FP8 workload: rows run past the 2048 elements held in registers, 4-token tiles).
    Token counts 1, 7, 64 (decode shapes: one row per warp) and 300 (prefill shape: four
    rows per warp, ragged tail)."""
    if shape == "35B":
        w = synth.decode_bf16(batch=64).with_(n_layers=2, cache_slots=synth.capacity_slots(0.25, 2, 256))
        banks, shared = pool35
    else:
        w = synth.decode_bf16(batch=8).with_(n_layers=2, hidden=7168, inter=128, n_experts=64, has_shared=False,
                                             cache_slots=32)
        banks = shared = None
    router = synth.router_weights(w)
    with Run(w, banks, shared, router=router, max_prefill_tokens=300) as r:
        for layer in range(2):
            xb = synth.prefill_x(w, 0, layer, 300)
            z300 = r.gpu_logits(layer, xb)  # checked against the oracle inside
            for T in (1, 7, 64):
                zt = r.gpu_logits(layer, xb[:T].copy())
                # the same token rows give the same bits at every launch shape
                assert np.array_equal(zt, z300[:T]), f"layer {layer} T {T}: launch shape changed bits"
            assert np.array_equal(_logits(r, layer, xb), z300), "repeat call changed bits"


@pytest.mark.parametrize("gate", GATES)
def test_decode_hidden_tiny_every_gate(gate):
    """Tiny config (16 experts, top-2, 8 slots): misses split between fill and host."""
    w = synth.tiny().with_(steps=12)
    router = synth.router_weights(w)
    with Run(w, gate=gate, router=router) as r:
        for s in range(w.steps):
            for l in range(w.n_layers):
                r.step(s, l, check_out=True, hidden=True)
        r.compare_state()
        print(f"gate {gate}: max rel err {r.max_err:.2e}, fills {r.sim.cnt.fills}, host {r.sim.cnt.cpu_execs}, "
              f"near ties {r.near_ties}")
        assert r.sim.cnt.cpu_execs > 0 and r.sim.cnt.fills > 0


@pytest.mark.parametrize("gate,batch", [(0, 1), (2, 1), (1, 4), (2, 16)])
def test_decode_hidden_35b_shape(gate, batch, pool35):
    """35B-A3B expert shape, 2 layers, 25% of the routed pool, the 52.7:77.3 split."""
    w = synth.decode_bf16(batch=batch).with_(n_layers=2, steps=6,
                                             cache_slots=synth.capacity_slots(0.25, 2, 256))
    router = synth.router_weights(w)
    with Run(w, *pool35, gate=gate, router=router) as r:
        for s in range(w.steps):
            for l in range(w.n_layers):
                r.step(s, l, check_out=(s % 2 == 0), hidden=True)
        r.compare_state()
        print(f"gate {gate} batch {batch}: max rel err {r.max_err:.2e}, near ties {r.near_ties}")


def test_decode_gate_functions_on_given_logits(pool35):
    """The gate functions on the logits path (ft_moe_decode_step), trace-driven routing."""
    for gate in (1, 2):
        w = synth.decode_bf16(batch=4).with_(n_layers=2, steps=5, cache_slots=synth.capacity_slots(0.37, 2, 256))
        tr = synth.routing_trace(w)
        with Run(w, *pool35, gate=gate) as r:
            for s in range(w.steps):
                for l in range(w.n_layers):
                    r.step(s, l, tr, check_out=(s == w.steps - 1))
            r.compare_state()


@pytest.mark.parametrize("gate", (0, 2))
def test_prefill_hidden_then_decode_hidden(gate):
    """Prefill of 200 tokens (ragged tiles) through the hidden-state call, 4 layers, 16
    experts top-2, 40 slots; then decode steps on what prefill left resident."""
    w = synth.prefill().with_(n_layers=4, n_experts=16, top_k=2, hidden=256, inter=128, cache_slots=40,
                              prefill_tokens=200)
    router = synth.router_weights(w)
    with Run(w, max_prefill_tokens=256, gate=gate, router=router) as r:
        for l in range(w.n_layers):
            prefill_step(r, 0, l, 200, hidden=True)
        r.w = w.with_(logits="normal")
        for s in range(3):
            for l in range(w.n_layers):
                r.step(s, l, check_out=True, hidden=True)
        r.compare_state()


def test_router_argument_errors():
    w = synth.tiny()
    with Run(w) as r:
        F = r.F
        x = torch.zeros((1, w.hidden), dtype=torch.int16, device=r.dev)
        out = torch.empty((1, w.hidden), dtype=torch.float32, device=r.dev)
        z = torch.empty((1, w.n_experts), dtype=torch.float32, device=r.dev)
        with pytest.raises(F.FtError) as e:  # no router weights yet
            F.ft_moe_decode_step_hidden(r.h, 0, 1, x, None, out)
        assert e.value.status == F.FT_ERR_STATE
        with pytest.raises(F.FtError) as e:
            F.ft_moe_router_logits(r.h, 0, 1, x, z)
        assert e.value.status == F.FT_ERR_STATE
        with pytest.raises(F.FtError) as e:
            F.ft_moe_set_router(r.h, None, 3)
        assert e.value.status == F.FT_ERR_INVALID
        F.ft_moe_set_router(r.h, synth.router_weights(w), 0)
        with pytest.raises(F.FtError) as e:
            F.ft_moe_router_logits(r.h, w.n_layers, 1, x, z)
        assert e.value.status == F.FT_ERR_INVALID
        with pytest.raises(F.FtError) as e:  # beyond max(max_batch, max_prefill_tokens)
            F.ft_moe_router_logits(r.h, 0, 2, x, z)
        assert e.value.status == F.FT_ERR_INVALID
        s = F.ft_moe_get_stats(r.h)
        assert s.error_word == 0


def _edge_logits(B, E, seed):
    """Logits drawn from a few values, so that equal logits are common, with -0 and +0,
    -inf and NaN among them; one finite logit of 3.0 per token keeps the gates defined."""
    rng = np.random.default_rng(seed)
    vals = np.array([0.0, -0.0, 1.0, 1.0, -1.0, 2.5, -np.inf, np.nan], dtype=np.float32)
    z = vals[rng.integers(0, len(vals), size=(B, E))]
    z[np.arange(B), rng.integers(0, E, size=B)] = 3.0
    return np.ascontiguousarray(z)


@pytest.mark.parametrize("shape,batch", [("tiny", 1), ("35B", 1), ("35B", 4)])
def test_router_edge_cases_decode(shape, batch, pool35):
    """Ties go to the lower id, -0 equals +0, NaN ranks as -inf (and sets the NaN error
    bit), a chosen -inf gets gate 0; ids, gates, cache decisions and outputs against the
    oracle at every step."""
    if shape == "tiny":
        w = synth.tiny().with_(steps=6)
        banks = shared = None
    else:
        w = synth.decode_bf16(batch=batch).with_(n_layers=2, steps=4, cache_slots=synth.capacity_slots(0.25, 2, 256))
        banks, shared = pool35
    with Run(w, banks, shared) as r:
        for s in range(w.steps):
            for l in range(w.n_layers):
                xb = synth.decode_x(w, s, l)
                z = _edge_logits(w.batch, w.n_experts, 100 * s + l)
                r.step(s, l, check_out=True, xz=(xb, z))
        st = r.F.ft_moe_get_stats(r.h)
        assert st.error_word == r.F.FT_DEVERR_NAN_LOGIT
        c = r.sim.cnt
        assert (st.hits, st.misses, st.fills, st.cpu_execs, st.evictions) == \
            (c.hits, c.misses, c.fills, c.cpu_execs, c.evictions)


def test_router_edge_cases_prefill():
    """The prefill router on the same kind of logits: 200 tokens, 16 experts top-2."""
    w = synth.prefill().with_(n_layers=2, n_experts=16, top_k=2, hidden=256, inter=128, cache_slots=40,
                              prefill_tokens=200)
    with Run(w, max_prefill_tokens=256) as r:
        for l in range(w.n_layers):
            prefill_step(r, 0, l, 200, z=_edge_logits(200, w.n_experts, 7 + l))
        assert r.F.ft_moe_get_stats(r.h).error_word == r.F.FT_DEVERR_NAN_LOGIT
