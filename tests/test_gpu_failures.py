"""Failure detection without faulting the GPU.

- Host-side injection: ft_test_inject_failure makes the n-th device allocation or host-bank
  registration of ft_moe_init / ft_cache_resize fail as if the runtime refused it.  The call
  returns FT_ERR_NOMEM / FT_ERR_PIN, releases what it had taken (device memory back to where
  it was, banks unregistered), and a resize that fails leaves the handle as it was.
- A bounded device wait that runs out: a test control makes the batch-1 persistent GEMV wait
  for one more h row than its CTAs publish, with a 1 ms limit.  The step returns with
  FT_DEVERR_TIMEOUT in the error word (routing and cache decisions still valid), and after
  ft_moe_reset_error the same handle runs correct steps again.
"""
import numpy as np
import pytest
import torch

import synth
from ftharness import Run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g

    g.build()


@pytest.fixture()
def inject():
    from serving_router_top_dedupe_gb300 import ftmoe as F

    def set_(v):
        kind, _, n = v.partition(":")
        if not v:
            F.ft_test_inject_failure(F.FT_INJECT_MALLOC, 0)
            return
        F.ft_test_inject_failure(F.FT_INJECT_MALLOC if kind == "malloc" else F.FT_INJECT_REGISTER, int(n))

    yield set_
    set_("")


def _cfg(F, w, max_batch=1):
    return F.make_config(w.n_layers, w.hidden, w.inter, w.n_experts, w.top_k, w.has_shared, w.wtype, max_batch,
                         w.cache_slots, w.bp_gbps, w.bh_gbps)


def _free_mem():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def _is_registered(arr) -> bool:
    """True when the driver reports the array's memory as page-locked host memory (the driver
    API keeps no error state, so asking changes nothing)."""
    import ctypes

    cu = ctypes.CDLL("libcuda.so.1")
    cu.cuPointerGetAttribute.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong]
    v = ctypes.c_uint(0)
    rc = cu.cuPointerGetAttribute(ctypes.byref(v), 2, arr.ctypes.data)   # CU_POINTER_ATTRIBUTE_MEMORY_TYPE
    return rc == 0 and v.value == 1                                       # CU_MEMORYTYPE_HOST


def _registration_is_observable(banks) -> bool:
    """Whether the query above tells registered from unregistered memory on this system."""
    from serving_router_top_dedupe_gb300 import ftmoe as F

    a = F.host_array((4096,), np.uint8)
    try:
        return _is_registered(a) and not _is_registered(np.zeros(1 << 20, np.uint8))
    finally:
        F.free_host_array(a)


@pytest.mark.parametrize("nth", [1, 2, 5, 12])
def test_injected_device_allocation_failure_releases_everything(inject, nth):
    from serving_router_top_dedupe_gb300 import ftmoe as F

    w = synth.tiny()
    pool = synth.ExpertPool(w)
    banks = pool.routed_banks()
    torch.zeros(1, device="cuda")
    free0 = _free_mem()
    inject(f"malloc:{nth}")
    with pytest.raises(F.FtError) as e:
        F.ft_moe_init(_cfg(F, w), banks)
    assert e.value.status == F.FT_ERR_NOMEM
    inject("")
    assert abs(_free_mem() - free0) < (4 << 20), "device memory not released"
    if _registration_is_observable(banks):
        for k in ("gate", "up", "down"):
            assert not _is_registered(banks[k]), f"bank {k} still registered"
    # the same banks work afterwards
    h = F.ft_moe_init(_cfg(F, w), banks)
    F.ft_moe_destroy(h)


@pytest.mark.parametrize("nth", [1, 3])
def test_injected_registration_failure_is_a_pin_error(inject, nth):
    from serving_router_top_dedupe_gb300 import ftmoe as F

    w = synth.tiny()
    banks = synth.ExpertPool(w).routed_banks()
    torch.zeros(1, device="cuda")
    free0 = _free_mem()
    inject(f"register:{nth}")
    with pytest.raises(F.FtError) as e:
        F.ft_moe_init(_cfg(F, w), banks)
    assert e.value.status == F.FT_ERR_PIN
    assert "no fallback" in F.ft_last_error()
    inject("")
    assert abs(_free_mem() - free0) < (4 << 20)
    if _registration_is_observable(banks):
        for k in ("gate", "up", "down"):
            assert not _is_registered(banks[k]), f"bank {k} still registered"


def test_pinned_banks_from_the_library_allocator_are_used_as_they_are():
    from serving_router_top_dedupe_gb300 import ftmoe as F

    w = synth.tiny()
    pool = synth.ExpertPool(w)
    banks = pool.alloc_banks(w.n_logical, F.host_array)
    pool.fill_banks(banks)
    try:
        with Run(w, banks=banks) as r:
            for s in range(3):
                for l in range(w.n_layers):
                    r.step(s, l, check_out=True)
            r.compare_state()
    finally:
        for a in banks.values():
            F.free_host_array(a)


@pytest.mark.parametrize("nth", [1, 2, 3])
def test_injected_failure_in_resize_leaves_the_handle_as_it_was(inject, nth):
    w = synth.decode_bf16(batch=2).with_(n_layers=3, n_experts=32, hidden=512, inter=256, steps=12, cache_slots=40)
    tr = synth.routing_trace(w)
    with Run(w) as r:
        F = r.F
        for s in range(6):
            for l in range(w.n_layers):
                r.step(s, l, tr)
        for new in (60, 17):                      # grow (pool + state), shrink (state only)
            inject(f"malloc:{nth}")
            if new == 17 and nth == 3:            # a shrink takes two allocations
                inject("malloc:2")
            with pytest.raises(F.FtError) as e:
                F.ft_cache_resize(r.h, new)
            assert e.value.status == F.FT_ERR_NOMEM
            inject("")
            r.compare_state()                     # nothing changed
            for s in range(6, 8):
                for l in range(w.n_layers):
                    r.step(s, l, tr, check_out=True)
        F.ft_cache_resize(r.h, 17)                # and it still resizes
        r.sim.resize(17)
        r.compare_state()


def test_handoff_wait_runs_out_then_the_handle_recovers():
    """Batch 1, 35B expert shape on 2 layers: the persistent GEMV runs.  With the test control
    its hand-off target is never reached; the wait gives up after 1 ms and the error word says
    so.  Decisions of that step still match the oracle; after the reset, steps are correct."""
    w = synth.decode_bf16().with_(n_layers=2, steps=6, cache_slots=synth.capacity_slots(0.5, 2, 256))
    tr = synth.routing_trace(w)
    with Run(w) as r:
        F = r.F
        assert F.ft_moe_get_stats(r.h).batch1_fused == 1
        r.step(0, 0, tr, check_out=True)
        F.ft_moe_test_control(r.h, F.FT_TEST_HANDOFF_TIMEOUT_NS, 1_000_000)
        r.step(0, 1, tr)                          # decisions compared; outputs undefined
        st = F.ft_moe_get_stats(r.h)
        assert st.error_word & F.FT_DEVERR_TIMEOUT
        F.ft_moe_test_control(r.h, F.FT_TEST_HANDOFF_TIMEOUT_NS, 0)
        F.ft_moe_reset_error(r.h)
        assert F.ft_moe_get_stats(r.h).error_word == 0
        for s in range(1, 4):
            for l in range(w.n_layers):
                r.step(s, l, tr, check_out=True)
        r.compare_state()


def test_test_control_rejects_unknown_keys():
    w = synth.tiny()
    with Run(w) as r:
        with pytest.raises(r.F.FtError) as e:
            r.F.ft_moe_test_control(r.h, 99, 1)
        assert e.value.status == r.F.FT_ERR_INVALID
        with pytest.raises(r.F.FtError) as e:
            r.F.ft_moe_test_control(r.h, r.F.FT_TEST_HANDOFF_TIMEOUT_NS, -5)
        assert e.value.status == r.F.FT_ERR_INVALID
