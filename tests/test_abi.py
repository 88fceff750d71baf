"""C-ABI checks that need no GPU: the library loads, exports every entry point the
header declares, the host split mirror agrees with the oracle, and argument
errors come back as status codes."""
import os
import random
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g

    g.build()
    from serving_router_top_dedupe_gb300 import ftmoe

    return ftmoe


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", fn)).read()
        names |= set(re.findall(r"^\s*(?:ft_status|const char\*)\s+(ft_\w+)\s*\(", text, re.M))
    return names


def test_library_exports_every_declared_symbol(F):
    declared = _declared()
    assert len(declared) >= 20
    import ctypes

    lib = ctypes.CDLL(F.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(F.EXPORTED)


def test_binding_argument_counts_match_the_header(F):
    """Every declared entry point takes as many arguments in the binding's ctypes
    signature as in the C declaration."""
    arity = {}
    for fn in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", fn)).read()
        for m in re.finditer(r"^\s*(?:ft_status|const char\*)\s+(ft_\w+)\s*\(([^)]*)\)\s*;", text, re.M):
            args = m.group(2).strip()
            arity[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    assert len(arity) >= 20
    for name, n in arity.items():
        if name in F._SIGS:
            assert len(F._SIGS[name]) == n, name


def test_split_host_mirror_matches_oracle(F):
    rng = random.Random(3)
    for _ in range(2000):
        m = rng.randint(0, 300)
        bp = round(rng.uniform(0.5, 400), 3)
        bh = round(rng.uniform(0.5, 400), 3)
        ev = rng.randint(0, 400)
        assert F.ft_split_misses(m, bp, bh, ev) == O.split_misses(m, O.mbps(bp), O.mbps(bh), ev)
    assert F.ft_split_misses(4, 11.8, 47.5, 99) == 1
    assert F.ft_split_misses(4, 52.7, 77.3, 99) == 3


def test_split_rejects_bad_arguments(F):
    for args in [(-1, 1.0, 1.0, 1), (1, 0.0, 1.0, 1), (1, 1.0, -2.0, 1), (1, 1.0, 1.0, -1)]:
        with pytest.raises(F.FtError) as e:
            F.ft_split_misses(*args)
        assert e.value.status == F.FT_ERR_INVALID


def test_init_rejects_bad_config_without_touching_the_gpu(F):
    banks = {"gate": np.zeros(16, np.uint16), "up": np.zeros(16, np.uint16), "down": np.zeros(16, np.uint16)}
    bad = [
        dict(hidden=100),           # not a multiple of 256
        dict(top_k=0), dict(top_k=17), dict(n_experts=2000), dict(max_batch=65), dict(cache_slots=0),
        dict(inter=100), dict(bh_gbps=0.0), dict(wtype=7),
    ]
    base = dict(n_layers=2, hidden=256, inter=128, n_experts=16, top_k=2, has_shared=False, wtype=F.FT_W_BF16,
                max_batch=1, cache_slots=8, bp_gbps=11.8, bh_gbps=47.5)
    for b in bad:
        with pytest.raises(F.FtError) as e:
            F.ft_moe_init(F.make_config(**{**base, **b}), banks)
        assert e.value.status == F.FT_ERR_INVALID
    with pytest.raises(F.FtError) as e:  # FP8 without scale banks
        F.ft_moe_init(F.make_config(**{**base, "wtype": F.FT_W_FP8_E4M3_B128, "hidden": 512}), banks)
    assert e.value.status == F.FT_ERR_INVALID
    u8 = np.zeros(16, np.uint8)
    for wt in (F.FT_W_NVFP4, F.FT_W_MXFP4):  # block-FP4 without their scale banks
        with pytest.raises(F.FtError) as e:
            F.ft_moe_init(F.make_config(**{**base, "wtype": wt}), {"gate": u8, "up": u8, "down": u8})
        assert e.value.status == F.FT_ERR_INVALID
    with pytest.raises(F.FtError) as e:  # NVFP4 needs the tensor scales too
        F.ft_moe_init(F.make_config(**{**base, "wtype": F.FT_W_NVFP4}),
                      {"gate": u8, "up": u8, "down": u8, "gate_bscale": u8, "up_bscale": u8, "down_bscale": u8})
    assert e.value.status == F.FT_ERR_INVALID


def test_router_and_prefill_calls_reject_a_null_handle(F):
    for call in (lambda: F.ft_moe_set_router(None, None, 0), lambda: F.ft_moe_router_logits(None, 0, 1, 1, 1),
                 lambda: F.ft_moe_decode_step_hidden(None, 0, 1, 1, 1, 1),
                 lambda: F.ft_moe_prefill_chunk_hidden(None, 0, 1, 1, 1),
                 lambda: F.ft_moe_prefill_chunk(None, 0, 1, 1, 1, 1),
                 lambda: F.ft_moe_set_host_hook(None, None), lambda: F.ft_moe_set_prefill_overlap(None, True)):
        with pytest.raises(F.FtError) as e:
            call()
        assert e.value.status == F.FT_ERR_INVALID


def test_null_handle_calls_fail_cleanly(F):
    with pytest.raises(F.FtError):
        F.ft_moe_decode_step(None, 0, 1, 1, 1, 1, 1)
    with pytest.raises(F.FtError):
        F.ft_cache_resize(None, 4)
    with pytest.raises(F.FtError):
        F.ft_moe_get_stats(None)
    F.ft_moe_destroy(None)


def test_binding_without_the_library_fails_loudly(tmp_path):
    """The binding has no fallback: a copy of the package without the built library
    raises at import."""
    import shutil
    import subprocess
    import sys

    pkg = tmp_path / "serving_router_top_dedupe_gb300"
    pkg.mkdir()
    for fn in ("__init__.py", "ftmoe.py"):
        shutil.copy(os.path.join(ROOT, "serving_router_top_dedupe_gb300", fn), pkg / fn)
    r = subprocess.run([sys.executable, "-c", "import serving_router_top_dedupe_gb300.ftmoe"], cwd=tmp_path,
                       capture_output=True, text=True, timeout=120,
                       env={**os.environ, "PYTHONPATH": str(tmp_path)})
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libftmoe.so is missing" in r.stderr
