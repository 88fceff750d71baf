"""Allocation-free layer evaluation (ft_moe_decode_resident_noalloc) against the regular
decode entry point.

The no-alloc call exists for callers that cannot call cudaMalloc (an engine that keeps
all device memory in its own pool, or a plug-in host that forbids allocation): it keeps
every intermediate in the library's fixed device scratch array.  Here the test itself
allocates the experts and the I/O buffers, as such a caller's engine would, and checks
that two calls in a row give the same layer outputs as ft_moe_decode_step on a handle
whose cache holds the whole layer.  Collected last so a failure here cannot hide others.
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


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
def test_noalloc_matches_decode_step_two_calls(F, kind):
    if kind == "bf16":
        w = synth.decode_bf16(batch=4).with_(n_layers=1)
    else:
        w = synth.decode_fp8(batch=2).with_(n_layers=1, n_experts=16)
    w = w.with_(cache_slots=w.n_logical, bp_gbps=80.0, bh_gbps=50.0)   # whole layer cached, every miss filled
    dev = torch.device("cuda:0")
    pool = synth.ExpertPool(w)
    banks, shared = pool.routed_banks(), pool.shared_banks()
    stride = _slot_stride(w)
    experts_d = _pack_slots(banks, range(w.n_experts), stride, dev)
    shared_d = _pack_slots(shared, [0], stride, dev) if shared is not None else None
    cfg = F.make_config(1, w.hidden, w.inter, w.n_experts, w.top_k, w.has_shared, w.wtype, w.batch, w.cache_slots,
                        w.bp_gbps, w.bh_gbps)
    h = F.ft_moe_init(cfg, banks, shared)
    try:
        B, H, k = w.batch, w.hidden, w.top_k
        for step in range(2):                                  # two calls in a row
            xb = synth.decode_x(w, step, 0)
            z = synth.decode_logits(w, step, 0)
            x_d = torch.from_numpy(xb.view(np.int16)).to(dev)
            z_d = torch.from_numpy(z).to(dev)
            out_ref = torch.empty((B, H), dtype=torch.float32, device=dev)
            rows_ref = torch.zeros((B, k, H), dtype=torch.float32, device=dev)
            F.ft_moe_decode_step(h, 0, B, x_d, z_d, None, out_ref, rows_ref)
            F.ft_moe_synchronize(h)
            out = torch.full((B, H), float("nan"), dtype=torch.float32, device=dev)
            rows = torch.zeros((B, k, H), dtype=torch.float32, device=dev)
            F.ft_moe_decode_resident_noalloc(w.n_experts, k, H, w.inter, w.wtype, experts_d, shared_d, B, x_d, z_d,
                                             out, rows)
            torch.cuda.synchronize()
            a, r = out.cpu().numpy(), out_ref.cpu().numpy()
            assert np.isfinite(a).all()
            assert O.rel_err_rows(a, r) <= OUT_TOL
            assert O.rel_err_rows(rows.cpu().numpy().reshape(B * k, H), rows_ref.cpu().numpy().reshape(B * k, H)) \
                <= OUT_TOL
            # same kernels, same reduction order: the results are in fact identical
            np.testing.assert_array_equal(a, r)
        assert F.ft_moe_get_stats(h).error_word == 0
    finally:
        F.ft_moe_destroy(h)


def test_noalloc_rejects_requests_beyond_the_scratch(F):
    # 64 tokens x 16 pairs x 7168 x 4 B of pair rows alone exceed the fixed 8 MiB array
    with pytest.raises(F.FtError) as e:
        F.ft_moe_decode_resident_noalloc(256, 16, 7168, 2048, F.FT_W_FP8_E4M3_B128, 1, None, 64, 1, 1, 1)
    assert e.value.status == F.FT_ERR_CAPACITY
    with pytest.raises(F.FtError) as e:
        F.ft_moe_decode_resident_noalloc(256, 8, 100, 512, F.FT_W_BF16, 1, None, 1, 1, 1, 1)
    assert e.value.status == F.FT_ERR_INVALID
