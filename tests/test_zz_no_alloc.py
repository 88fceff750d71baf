"""Allocation-free layer evaluation (ft_moe_decode_resident_noalloc).

The no-alloc call is for callers that cannot call cudaMalloc: an engine that keeps all
device memory in its own pool, or a plug-in host that forbids allocation.  It keeps every
intermediate in the library's fixed device scratch array.  Here the test allocates the
experts and the I/O buffers itself, as such a caller's engine would.

Each case makes one call on other inputs first, so that the scratch holds another call's
lists, then two calls in a row.  Both are checked against the float64 oracle within the
layer-output tolerance, and bitwise against ft_moe_decode_step on a handle whose cache
holds the whole layer.  Batch 1 runs the persistent one-launch kernel, batch > 1 the
batched kernels; both weight types run.  The file is collected last, so a failure here
cannot hide another test's result.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from ftharness import OUT_TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g

    g.build()
    from serving_router_top_dedupe_gb300 import ftmoe

    return ftmoe


def _slot_stride(w):
    esz = 2 if w.wtype == synth.W_BF16 else 1
    used = 3 * w.hidden * w.inter * esz
    if w.wtype == synth.W_FP8_E4M3_B128:
        used += 4 * (2 * w.inter * (w.hidden // 128) + w.hidden * (w.inter // 128))
    return (used + 255) // 256 * 256


def _pack_slots(banks, rows, stride, dev):
    """Experts `rows` of the host banks in the library's slot layout, on the device."""
    order = ["gate", "up", "down", "gate_scale", "up_scale", "down_scale"]
    buf = np.zeros((len(rows), stride), dtype=np.uint8)
    for i, r in enumerate(rows):
        off = 0
        for kname in order:
            if kname in banks:
                b = np.ascontiguousarray(banks[kname][r]).view(np.uint8).reshape(-1)
                buf[i, off:off + b.size] = b
                off += b.size
    return torch.from_numpy(buf).to(dev)


def _workload(kind, batch):
    if kind == "bf16":
        w = synth.decode_bf16(batch=batch).with_(n_layers=1)
    else:
        w = synth.decode_fp8(batch=batch).with_(n_layers=1, n_experts=16)
    return w.with_(cache_slots=w.n_logical, bp_gbps=80.0, bh_gbps=50.0)   # whole layer cached, every miss filled


class _Case:
    def __init__(self, F, w):
        self.F, self.w = F, w
        self.dev = torch.device("cuda:0")
        pool = synth.ExpertPool(w)
        self.pool = pool
        self.banks, self.shared = pool.routed_banks(), pool.shared_banks()
        stride = _slot_stride(w)
        self.experts_d = _pack_slots(self.banks, range(w.n_experts), stride, self.dev)
        self.shared_d = _pack_slots(self.shared, [0], stride, self.dev) if self.shared is not None else None
        self.err_d = torch.full((1,), 0x7777, dtype=torch.int32, device=self.dev)

    def noalloc(self, xb, z):
        F, w = self.F, self.w
        B, H, k = xb.shape[0], w.hidden, w.top_k
        x_d = torch.from_numpy(xb.view(np.int16)).to(self.dev)
        z_d = torch.from_numpy(z).to(self.dev)
        out = torch.full((B, H), float("nan"), dtype=torch.float32, device=self.dev)
        rows = torch.zeros((B, k, H), dtype=torch.float32, device=self.dev)
        F.ft_moe_decode_resident_noalloc(w.n_experts, k, H, w.inter, w.wtype, self.experts_d, self.shared_d, B,
                                         x_d, z_d, out, rows, self.err_d)
        torch.cuda.synchronize()
        return out.cpu().numpy(), rows.cpu().numpy(), int(self.err_d.item())

    def oracle(self, xb, z):
        w = self.w
        sel, gates = O.route(z, w.top_k)
        sh = {kk: v[0] for kk, v in self.shared.items()} if self.shared is not None else None
        return O.prefill_outputs(0, sel, gates, xb, self.pool.expert, w.n_experts, tokens=range(xb.shape[0]),
                                 shared=sh, fp8=int(w.wtype))


@pytest.mark.parametrize("kind,batch", [("bf16", 1), ("bf16", 4), ("fp8", 1), ("fp8", 2)])
def test_noalloc_matches_oracle_and_decode_step(F, kind, batch):
    w = _workload(kind, batch)
    c = _Case(F, w)
    cfg = F.make_config(1, w.hidden, w.inter, w.n_experts, w.top_k, w.has_shared, w.wtype, w.batch, w.cache_slots,
                        w.bp_gbps, w.bh_gbps)
    h = F.ft_moe_init(cfg, c.banks, c.shared)
    try:
        B, H, k = w.batch, w.hidden, w.top_k
        # a call on other inputs first: its lists stay in the scratch, so a read of stale
        # routing in the calls below would give other experts' rows
        c.noalloc(synth.decode_x(w, 7, 0), synth.decode_logits(w, 7, 0))
        for step in range(2):                                  # two calls in a row
            xb = synth.decode_x(w, step, 0)
            z = synth.decode_logits(w, step, 0)
            a, rows, err = c.noalloc(xb, z)
            assert err == 0, f"device error word {err:#x}"
            assert np.isfinite(a).all()
            ref = c.oracle(xb, z)
            e = O.rel_err_rows(a, ref)
            assert e <= OUT_TOL, f"step {step}: relative error {e:.3e} against the oracle"
            # the same layer through the regular entry point: same kernels, same reduction order
            x_d = torch.from_numpy(xb.view(np.int16)).to(c.dev)
            z_d = torch.from_numpy(z).to(c.dev)
            out_ref = torch.empty((B, H), dtype=torch.float32, device=c.dev)
            rows_ref = torch.zeros((B, k, H), dtype=torch.float32, device=c.dev)
            F.ft_moe_decode_step(h, 0, B, x_d, z_d, None, out_ref, rows_ref)
            F.ft_moe_synchronize(h)
            np.testing.assert_array_equal(a, out_ref.cpu().numpy())
            np.testing.assert_array_equal(rows, rows_ref.cpu().numpy())
        assert F.ft_moe_get_stats(h).error_word == 0
    finally:
        F.ft_moe_destroy(h)


def test_noalloc_reports_nan_logits_through_its_error_word(F):
    w = _workload("bf16", 2)
    c = _Case(F, w)
    xb = synth.decode_x(w, 3, 0)
    z = synth.decode_logits(w, 3, 0).copy()
    top = int(np.argmax(z[0]))
    z[0, top] = np.nan                                         # ranks as -inf
    z[1, 5] = np.nan
    a, _, err = c.noalloc(xb, z)
    assert err & F.FT_DEVERR_NAN_LOGIT
    zr = np.where(np.isnan(z), -np.inf, z).astype(np.float32)
    assert O.rel_err_rows(a, c.oracle(xb, zr)) <= OUT_TOL
    # the next call starts with a clear word
    a2, _, err2 = c.noalloc(synth.decode_x(w, 4, 0), synth.decode_logits(w, 4, 0))
    assert err2 == 0


def test_noalloc_rejects_requests_beyond_the_scratch(F):
    # 64 tokens x 16 pairs x 7168 x 4 B of pair rows alone exceed the fixed 8 MiB array
    with pytest.raises(F.FtError) as e:
        F.ft_moe_decode_resident_noalloc(256, 16, 7168, 2048, F.FT_W_FP8_E4M3_B128, 1, None, 64, 1, 1, 1)
    assert e.value.status == F.FT_ERR_CAPACITY
    with pytest.raises(F.FtError) as e:
        F.ft_moe_decode_resident_noalloc(256, 8, 100, 512, F.FT_W_BF16, 1, None, 1, 1, 1, 1)
    assert e.value.status == F.FT_ERR_INVALID
