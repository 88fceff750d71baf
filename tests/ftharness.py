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
        float64 logits within router_tol; the decisions are then taken on these values on
        both sides."""
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
        the GPU router's logits, which gpu_logits has checked against its own."""
        F = self.F
        xb, z = self.inputs(step, layer, trace, batch) if xz is None else xz
        B = xb.shape[0]
        if hidden:
            z = self.gpu_logits(layer, xb)
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
        self.compare(rec, sel, gates, gt)
        out = out_d.cpu().numpy()
        if check_out:
            ref = O.decode_layer_outputs(rec, sel, gates, xb, cpart, self.expert, shared=self.shared_expert(layer),
                                         fp8=self.fp8, n_experts=self.w.n_experts)
            err = O.rel_err_rows(out, ref)
            self.max_err = max(self.max_err, err)
            assert err <= OUT_TOL, f"step {step} layer {layer}: relative error {err:.3e} > {OUT_TOL}"
        return rec, gt, out, (rows_d.cpu().numpy() if rows_out else None)

    def compare(self, rec, sel, gates, gt):
        ctx = f"layer {rec.layer} clock {rec.clock}"
        assert gt["layer"] == rec.layer and gt["clock"] == rec.clock, ctx
        assert np.array_equal(gt["sel"], sel), f"{ctx}: routing ids"
        np.testing.assert_allclose(gt["gates"], gates, rtol=GATE_RTOL, atol=0, err_msg=f"{ctx}: gates")
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


def prefill_step(r: Run, chunk: int, layer: int, T: int, check_tokens=None, hidden=False):
    """One prefill layer on both sides; compares residency state, and outputs of
    `check_tokens` (all when None) against the float64 oracle.  hidden: the call takes
    hidden states (ft_moe_prefill_chunk_hidden) and both sides route on the GPU router's
    logits, checked first against the oracle's."""
    F, w = r.F, r.w
    xb = synth.prefill_x(w, chunk, layer, T)
    z = r.gpu_logits(layer, xb) if hidden else synth.prefill_logits(w, chunk, layer, T)
    if r.S >= 2 * w.n_experts:
        r.sim.prefill_layer(layer, w.n_experts, w.n_layers)
    else:  # the pool cannot hold two full layers: experts on demand
        sel_z, _ = O.route(z, w.top_k, r.gate)
        r.sim.prefill_layer_on_demand(layer, w.n_experts, np.unique(sel_z))
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
    sel, gates = O.route(z, w.top_k, r.gate)
    ref = O.prefill_outputs(layer, sel, gates, xb, r.expert, w.n_experts, tokens=list(tokens),
                            shared=r.shared_expert(layer))
    err = O.rel_err_rows(out[list(tokens)], ref)
    r.max_err = max(r.max_err, err)
    assert err <= OUT_TOL, f"prefill layer {layer}: relative error {err:.3e}"
    return out
