"""Lockstep driver for GPU-vs-oracle parity tests.

The library (through the C ABI) and the CPU oracle consume the same seeded
inputs from `synth`; every routing and cache decision is compared exactly, and
layer outputs are compared with the tolerance below.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import synth

# Layer outputs vs the float64 oracle: max over rows of max|y - ref| / max|ref|.
OUT_TOL = 1e-2
GATE_RTOL = 2e-6


def router_tol(xb, wr):
    """Per-logit error bound of the GPU router against the float64 oracle.  BF16 x BF16
    products are exact in FP32; each lane adds H/32 of them in sequence and five xor
    butterfly levels follow, so to first order |z - z_ref| <= (H/32 + 5) u sum_h |x_h w_h|
    with u = 2^-24 (one rounding per addition)."""
    H = xb.shape[1]
    mag = np.abs(O.bf16_to_f64(xb)) @ np.abs(O.bf16_to_f64(wr)).T
    return (H / 32 + 5) * 2.0 ** -24 * mag * 1.01 + 1e-30


def oracle_routing(z_ref, z_gpu, tol, k, gate):
    """Routing of the oracle on its own float64 logits, for the calls that take hidden states.

    z_ref: float64 logits of the oracle; z_gpu: the kernel's FP32 logits, already checked
    to lie within `tol` (per element) of z_ref.  A token whose float64 k-th and (k+1)-th
    logits lie more than 2 * max(tol) apart has one correct choice, and it is the oracle's.
    A token inside that band is a near tie: either side is a correct choice, so the choice
    the kernel's logits make is taken after checking that it lies inside the band (every
    expert clearly above the band chosen, none clearly below it).
    Returns sel, gates (oracle's gates on float64 logits for decided tokens), the relative
    gate tolerance per token, and the number of near-tie tokens."""
    sel_r, g_r = O.route(z_ref, k, gate)
    sel_g, g_g = O.route(z_gpu, k, gate)
    B, E = z_ref.shape
    sel, gates = sel_r.copy(), g_r.copy()
    rtol = np.full(B, GATE_RTOL)
    near = 0
    for t in range(B):
        zs = np.sort(z_ref[t])[::-1]
        band = 2.0 * float(tol[t].max())
        if k >= E or zs[k - 1] - zs[k] > band:
            assert np.array_equal(sel_g[t], sel_r[t]), f"token {t}: the kernel's logits choose other experts"
            # |d log g| <= 2 max|dz| for each gate function, plus FP32 rounding of the gate
            rtol[t] = 2.02 * float(tol[t].max()) + GATE_RTOL
            continue
        near += 1
        chosen = set(int(e) for e in sel_g[t])
        above = {e for e in range(E) if z_ref[t, e] > zs[k] + band}
        assert above <= chosen, f"token {t}: a clearly larger logit was not chosen"
        assert all(z_ref[t, e] >= zs[k - 1] - band for e in chosen), f"token {t}: a clearly smaller logit was chosen"
        sel[t], gates[t] = sel_g[t], g_g[t]
    return sel, gates, rtol, near


def _F():
    from serving_router_top_dedupe_gb300 import ftmoe

    return ftmoe


class Run:
    """One library handle plus its oracle twin."""

    def __init__(self, w: synth.Workload, banks=None, shared=None, fill_mode=None, max_batch=None,
                 max_prefill_tokens=0, cache_slots=None, gate=0, router=None):
        F = _F()
        self.F = F
        self.w = w
        if banks is None:
            pool = synth.ExpertPool(w)
            banks = pool.routed_banks()
            shared = pool.shared_banks()
        self.banks, self.shared = banks, shared
        self.fp8 = int(w.wtype)  # weight type for the oracle: 0 BF16, 1 FP8, 2 NVFP4
        self.S = w.cache_slots if cache_slots is None else cache_slots
        self.B = w.batch if max_batch is None else max_batch
        cfg = F.make_config(w.n_layers, w.hidden, w.inter, w.n_experts, w.top_k, w.has_shared, w.wtype, self.B,
                            self.S, w.bp_gbps, w.bh_gbps, max_prefill_tokens=max_prefill_tokens,
                            fill_mode=F.FT_FILL_KERNEL if fill_mode is None else fill_mode)
        self.h = F.ft_moe_init(cfg, banks, shared)
        self.sim = O.SlotCache(self.S, w.n_logical)
        self.bp, self.bh = O.mbps(w.bp_gbps), O.mbps(w.bh_gbps)
        self.kcap = min(self.B * w.top_k, w.n_experts)
        self.dev = torch.device("cuda:0")
        self.max_err = 0.0
        self.gate, self.router = gate, router
        self.near_ties = 0          # hidden-state steps: tokens routed inside the float64 tie band
        if router is not None or gate != 0:
            F.ft_moe_set_router(self.h, router, gate)

    def close(self):
        if self.h:
            self.F.ft_moe_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # ----------------------------------------------------------- oracle side
    def expert(self, u):
        return {k: v[u] for k, v in self.banks.items()}

    def shared_expert(self, layer):
        return None if self.shared is None else {k: v[layer] for k, v in self.shared.items()}

    def oracle_rows(self, layer, sel, gates, xb, pairs):
        """float32 [B, k, H]: oracle rows for the listed (t, r) pairs, zeros elsewhere."""
        B, k = sel.shape
        cp = np.zeros((B, k, self.w.hidden), dtype=np.float32)
        for t, r in pairs:
            cp[t, r] = O.pair_row(self.expert(layer * self.w.n_experts + int(sel[t, r])), O.bf16_to_f64(xb[t]),
                                  gates[t, r], self.fp8).astype(np.float32)
        return cp

    def gpu_logits(self, layer, xb):
        """Router logits of the GPU (ft_moe_router_logits), checked against the oracle's
        float64 logits within router_tol."""
        T = xb.shape[0]
        x_d = torch.from_numpy(xb.view(np.int16)).to(self.dev)
        z_d = torch.empty((T, self.w.n_experts), dtype=torch.float32, device=self.dev)
        torch.cuda.synchronize()  # the library runs on its own stream
        self.F.ft_moe_router_logits(self.h, layer, T, x_d, z_d)
        self.F.ft_moe_synchronize(self.h)
        z = z_d.cpu().numpy()
        ref = O.router_logits(xb, self.router[layer])
        err = np.abs(z.astype(np.float64) - ref)
        tol = router_tol(xb, self.router[layer])
        assert np.all(err <= tol), f"layer {layer}: router logit error {err.max():.3e} above its bound"
        return z

    def hidden_routing(self, layer, xb):
        """Decisions for a hidden-state step or chunk: the oracle routes on its own float64
        logits (oracle_routing); returns the kernel's logits too, for the bitwise check of
        the logits the step computes."""
        z = self.gpu_logits(layer, xb)
        z_ref = O.router_logits(xb, self.router[layer])
        sel, gates, rtol, near = oracle_routing(z_ref, z, router_tol(xb, self.router[layer]), self.w.top_k,
                                                self.gate)
        self.near_ties += near
        return z, sel, gates, rtol

    # ------------------------------------------------------------- one step
    def inputs(self, step, layer, trace=None, batch=None):
        w = self.w if batch is None else self.w.with_(batch=batch)
        xb = synth.decode_x(w, step, layer)
        tr = trace if w.logits == "trace" else None
        z = synth.decode_logits(w, step, layer, tr)
        return xb, z

    def step(self, step, layer, trace=None, check_out=False, cpart=None, rows_out=False, batch=None,
             xz=None, hidden=False):
        """Run one decode layer-step on both sides and compare.  Returns (rec, gpu_trace, out, rows).
        hidden: the step takes hidden states (ft_moe_decode_step_hidden); the oracle routes on
        its own float64 logits (hidden_routing)."""
        F = self.F
        xb, z = self.inputs(step, layer, trace, batch) if xz is None else xz
        B = xb.shape[0]
        gate_rtol = GATE_RTOL
        if hidden:
            z, sel, gates, gate_rtol = self.hidden_routing(layer, xb)
        else:
            sel, gates = O.route(z, self.w.top_k, self.gate)
        rec = self.sim.decode_step(layer, self.w.n_experts, sel, self.bp, self.bh)
        if cpart is None:
            cpairs = [(t, r) for t in range(B) for r in range(self.w.top_k) if rec.slot_of_pair[t, r] < 0]
            cpart = self.oracle_rows(layer, sel, gates, xb, cpairs if check_out else [])
        x_d = torch.from_numpy(xb.view(np.int16)).to(self.dev)
        z_d = torch.from_numpy(z).to(self.dev)
        c_d = torch.from_numpy(np.ascontiguousarray(cpart, dtype=np.float32)).to(self.dev)
        out_d = torch.empty((B, self.w.hidden), dtype=torch.float32, device=self.dev)
        rows_d = torch.zeros((B, self.w.top_k, self.w.hidden), dtype=torch.float32, device=self.dev) \
            if rows_out else None
        if hidden:
            lg_d = torch.empty((B, self.w.n_experts), dtype=torch.float32, device=self.dev)
            F.ft_moe_decode_step_hidden(self.h, layer, B, x_d, c_d, out_d, rows_d, lg_d)
            assert np.array_equal(lg_d.cpu().numpy(), z), "router logits inside the step differ"
        else:
            F.ft_moe_decode_step(self.h, layer, B, x_d, z_d, c_d, out_d, rows_d)
        gt = F.ft_moe_get_step_trace(self.h, self.B, self.w.top_k, self.kcap)
        self.compare(rec, sel, gates, gt, gate_rtol)
        out = out_d.cpu().numpy()
        if check_out:
            ref = O.decode_layer_outputs(rec, sel, gates, xb, cpart, self.expert, shared=self.shared_expert(layer),
                                         fp8=self.fp8, n_experts=self.w.n_experts)
            err = O.rel_err_rows(out, ref)
            self.max_err = max(self.max_err, err)
            assert err <= OUT_TOL, f"step {step} layer {layer}: relative error {err:.3e} > {OUT_TOL}"
        return rec, gt, out, (rows_d.cpu().numpy() if rows_out else None)

    def compare(self, rec, sel, gates, gt, gate_rtol=GATE_RTOL):
        ctx = f"layer {rec.layer} clock {rec.clock}"
        assert gt["layer"] == rec.layer and gt["clock"] == rec.clock, ctx
        assert np.array_equal(gt["sel"], sel), f"{ctx}: routing ids"
        rt = np.broadcast_to(np.asarray(gate_rtol, dtype=np.float64).reshape(-1, 1), gates.shape)
        g_gpu = np.asarray(gt["gates"], dtype=np.float64).reshape(gates.shape)
        bad = np.abs(g_gpu - gates) > rt * np.abs(gates.astype(np.float64))
        assert not bad.any(), f"{ctx}: gates {g_gpu[bad]} vs {gates[bad]}"
        assert gt["active"] == rec.A, f"{ctx}: active set"
        assert gt["hit"] == rec.H and gt["miss"] == rec.M, f"{ctx}: hit/miss"
        assert gt["q"] == rec.q, f"{ctx}: q {gt['q']} vs {rec.q}"
        assert gt["victims"] == rec.victims, f"{ctx}: victims"
        assert np.array_equal(gt["slot_of_pair"], rec.slot_of_pair), f"{ctx}: slot rewrite"

    def compare_state(self):
        st = self.F.ft_moe_get_state(self.h, self.w.n_logical, self.sim.S)
        assert st["clock"] == self.sim.clock
        assert np.array_equal(st["res"], self.sim.res), "residency table"
        assert np.array_equal(st["owner"], self.sim.owner), "slot owners"
        assert np.array_equal(st["stamp"].astype(np.int64), self.sim.stamp), "slot stamps"
        s = self.F.ft_moe_get_stats(self.h)
        c = self.sim.cnt
        assert (s.hits, s.misses, s.fills, s.cpu_execs, s.evictions) == \
            (c.hits, c.misses, c.fills, c.cpu_execs, c.evictions)
        assert s.error_word == 0
        return s


def prefill_step(r: Run, chunk: int, layer: int, T: int, check_tokens=None, hidden=False, z=None):
    """One prefill layer on both sides; compares residency state, and outputs of
    `check_tokens` (all when None) against the float64 oracle.  hidden: the call takes
    hidden states (ft_moe_prefill_chunk_hidden) and the oracle routes on its own float64
    logits (Run.hidden_routing).  z: logits to use instead of the workload's."""
    F, w = r.F, r.w
    xb = synth.prefill_x(w, chunk, layer, T)
    if hidden:
        z, sel, gates, _ = r.hidden_routing(layer, xb)
    else:
        if z is None:
            z = synth.prefill_logits(w, chunk, layer, T)
        sel, gates = O.route(z, w.top_k, r.gate)
    if r.S >= 2 * w.n_experts:
        r.sim.prefill_layer(layer, w.n_experts, w.n_layers)
    else:  # the pool cannot hold two full layers: experts on demand
        r.sim.prefill_layer_on_demand(layer, w.n_experts, np.unique(sel))
    x_d = torch.from_numpy(xb.view(np.int16)).to(r.dev)
    z_d = torch.from_numpy(z).to(r.dev)
    out_d = torch.empty((T, w.hidden), dtype=torch.float32, device=r.dev)
    if hidden:
        F.ft_moe_prefill_chunk_hidden(r.h, layer, T, x_d, out_d)
    else:
        F.ft_moe_prefill_chunk(r.h, layer, T, x_d, z_d, out_d)
    st = F.ft_moe_get_state(r.h, w.n_logical, r.sim.S)
    assert st["clock"] == r.sim.clock
    assert np.array_equal(st["res"], r.sim.res), f"prefill layer {layer}: residency table"
    assert np.array_equal(st["owner"], r.sim.owner), f"prefill layer {layer}: slot owners"
    assert np.array_equal(st["stamp"].astype(np.int64), r.sim.stamp), f"prefill layer {layer}: stamps"
    out = out_d.cpu().numpy()
    tokens = range(T) if check_tokens is None else check_tokens
    ref = O.prefill_outputs(layer, sel, gates, xb, r.expert, w.n_experts, tokens=list(tokens),
                            shared=r.shared_expert(layer), fp8=r.fp8)
    err = O.rel_err_rows(out[list(tokens)], ref)
    r.max_err = max(r.max_err, err)
    assert err <= OUT_TOL, f"prefill layer {layer}: relative error {err:.3e}"
    return out
