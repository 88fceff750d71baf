"""Thin Python binding of libftmoe (include/ft_moe.h).

Argument marshalling only: every entry point forwards plain pointers and sizes
to the C ABI; every step of the MoE path runs in the library's CUDA kernels.
Tensors may be torch tensors (their data_ptr() is passed), numpy arrays (their
buffer address) or raw integer addresses.  If the shared library has not been
built, importing this module raises: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libftmoe.so")

FT_OK, FT_ERR_INVALID, FT_ERR_CUDA, FT_ERR_NOMEM, FT_ERR_PIN = 0, 1, 2, 3, 4
FT_ERR_CAPACITY, FT_ERR_STATE, FT_ERR_TIMEOUT, FT_ERR_DEVICE = 5, 6, 7, 8
FT_W_BF16, FT_W_FP8_E4M3_B128, FT_W_NVFP4, FT_W_MXFP4 = 0, 1, 2, 3
FT_FILL_KERNEL, FT_FILL_MEMCPY = 0, 1
FT_GATE_SOFTMAX_TOPK, FT_GATE_SOFTMAX_ALL, FT_GATE_SIGMOID_TOPK = 0, 1, 2
FT_CPU = -1
FT_DEVERR_NAN_LOGIT, FT_DEVERR_BAD_STATE, FT_DEVERR_TIMEOUT, FT_DEVERR_CAPACITY = 1, 2, 4, 8
FT_TEST_HANDOFF_TIMEOUT_NS = 1
FT_INJECT_MALLOC, FT_INJECT_REGISTER = 1, 2
FT_HOST_PINNED, FT_HOST_HUGE_PAGES = 0, 1

PROFILE_KINDS = ("control", "fill", "gate_up", "down_combine", "prefill_route", "prefill_gemm_gate_up",
                 "prefill_combine", "prefill_copy", "prefill_gemm_down", "router")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
_lib = C.CDLL(LIB_PATH)


class FtError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"ft status {status}: {msg}")
        self.status = status


class ft_moe_config(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("hidden", C.c_int), ("inter", C.c_int), ("n_experts", C.c_int),
                ("top_k", C.c_int), ("has_shared", C.c_int), ("wtype", C.c_int), ("max_batch", C.c_int),
                ("max_prefill_tokens", C.c_int), ("cache_slots", C.c_int), ("bp_gbps", C.c_double),
                ("bh_gbps", C.c_double), ("fill_mode", C.c_int), ("device", C.c_int),
                ("compute_stream", C.c_void_p), ("transfer_stream", C.c_void_p)]


_BANK_KEYS = ("gate", "up", "down", "gate_scale", "up_scale", "down_scale", "gate_bscale", "up_bscale",
              "down_bscale", "tensor_scale")


class ft_banks(C.Structure):
    _fields_ = [(k, C.c_void_p) for k in _BANK_KEYS]


class ft_stats(C.Structure):
    _fields_ = [("hits", C.c_uint64), ("misses", C.c_uint64), ("fills", C.c_uint64),
                ("cpu_execs", C.c_uint64), ("evictions", C.c_uint64), ("decode_steps", C.c_uint64),
                ("prefill_layers", C.c_uint64), ("eval_entries", C.c_uint64), ("eval_pairs", C.c_uint64),
                ("error_word", C.c_uint32), ("clock", C.c_uint32),
                ("bp_gbps", C.c_double), ("bh_gbps", C.c_double), ("cache_slots", C.c_int),
                ("batch1_fused", C.c_int32)]


class ft_step_trace(C.Structure):
    _fields_ = [("layer", C.c_int), ("batch", C.c_int), ("q", C.c_int), ("n_active", C.c_int),
                ("n_hit", C.c_int), ("n_miss", C.c_int), ("n_victims", C.c_int), ("n_cpu", C.c_int),
                ("clock", C.c_uint32),
                ("sel", C.c_void_p), ("gates", C.c_void_p), ("slot_of_pair", C.c_void_p),
                ("active", C.c_void_p), ("hit", C.c_void_p), ("miss", C.c_void_p), ("victims", C.c_void_p)]


class ft_profile(C.Structure):
    _fields_ = [("launches", C.c_uint64 * 10), ("total_ms", C.c_double * 10)]


_P = C.c_void_p
_SIGS = {
    "ft_moe_init": [C.POINTER(ft_moe_config), C.POINTER(ft_banks), C.POINTER(ft_banks), C.POINTER(C.c_void_p)],
    "ft_moe_decode_step": [_P, C.c_int, C.c_int, _P, _P, _P, _P, _P],
    "ft_moe_decode_layers": [_P, C.c_int, C.c_int, C.c_int, _P, _P, _P, _P, _P],
    "ft_moe_decode_layers_host": [_P, C.c_int, C.c_int, C.c_int, _P, _P, _P, _P, C.c_int],
    "ft_moe_graph_capture_decode": [_P, C.c_int, C.c_int, C.c_int, _P, _P, _P, _P, _P, C.POINTER(C.c_void_p)],
    "ft_graph_launch": [_P],
    "ft_graph_destroy": [_P],
    "ft_moe_prefill_chunk": [_P, C.c_int, C.c_int, _P, _P, _P],
    "ft_moe_set_prefill_overlap": [_P, C.c_int],
    "ft_moe_set_host_hook": [_P, _P, _P],
    "ft_moe_set_router": [_P, _P, C.c_int],
    "ft_moe_router_logits": [_P, C.c_int, C.c_int, _P, _P],
    "ft_moe_decode_step_hidden": [_P, C.c_int, C.c_int, _P, _P, _P, _P, _P],
    "ft_moe_prefill_chunk_hidden": [_P, C.c_int, C.c_int, _P, _P],
    "ft_cache_resize": [_P, C.c_int],
    "ft_split_misses": [C.c_int, C.c_double, C.c_double, C.c_int, C.POINTER(C.c_int)],
    "ft_bench_bw": [C.c_size_t, C.c_int, C.POINTER(C.c_double)],
    "ft_moe_get_stats": [_P, C.POINTER(ft_stats)],
    "ft_moe_get_step_trace": [_P, C.POINTER(ft_step_trace)],
    "ft_moe_get_state": [_P, _P, _P, _P, _P],
    "ft_moe_set_profiling": [_P, C.c_int],
    "ft_moe_get_profile": [_P, C.POINTER(ft_profile), C.c_int],
    "ft_moe_set_stream": [_P, _P],
    "ft_moe_synchronize": [_P],
    "ft_moe_destroy": [_P],
    "ft_moe_reset_error": [_P],
    "ft_test_inject_failure": [C.c_int, C.c_int],
    "ft_moe_test_control": [_P, C.c_int, C.c_longlong],
    "ft_host_alloc": [C.c_size_t, C.c_int, C.POINTER(C.c_void_p)],
    "ft_host_free": [_P],
    "ft_moe_decode_resident_noalloc": [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, _P, _P, C.c_int, _P, _P, _P, _P,
                                       _P, _P],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = C.c_int
_lib.ft_last_error.argtypes = []
_lib.ft_last_error.restype = C.c_char_p

EXPORTED = tuple(_SIGS) + ("ft_last_error",)


def ft_last_error() -> str:
    return _lib.ft_last_error().decode()


def _check(status: int) -> None:
    if status != FT_OK:
        raise FtError(status, ft_last_error())


def _ptr(t) -> int | None:
    """Address of a torch tensor / numpy array / int (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _banks(d: dict | None) -> ft_banks | None:
    if d is None:
        return None
    return ft_banks(*[_ptr(d.get(k)) for k in _BANK_KEYS])


# ----------------------------------------------------------- same-named calls
def ft_moe_init(cfg: ft_moe_config, host_pool: dict, shared: dict | None = None) -> int:
    h = C.c_void_p()
    hp, sh = _banks(host_pool), _banks(shared)
    _check(_lib.ft_moe_init(C.byref(cfg), C.byref(hp), C.byref(sh) if sh is not None else None, C.byref(h)))
    _hook_k[h.value], _hook_h[h.value] = cfg.top_k, cfg.hidden
    return h.value


def ft_moe_decode_step(h, layer, batch, x_bf16, logits, c_partial, out, rows_out=None) -> None:
    _check(_lib.ft_moe_decode_step(h, layer, batch, _ptr(x_bf16), _ptr(logits), _ptr(c_partial), _ptr(out),
                                   _ptr(rows_out)))


def ft_moe_decode_layers(h, first_layer, n_layers, batch, x_bf16, logits, c_partial, out, rows_out=None) -> None:
    _check(_lib.ft_moe_decode_layers(h, first_layer, n_layers, batch, _ptr(x_bf16), _ptr(logits), _ptr(c_partial),
                                     _ptr(out), _ptr(rows_out)))


def ft_moe_decode_layers_host(h, first_layer, n_layers, batch, x_host, logits_host, c_partial_host, out_host,
                              use_graph=True) -> None:
    _check(_lib.ft_moe_decode_layers_host(h, first_layer, n_layers, batch, _ptr(x_host), _ptr(logits_host),
                                          _ptr(c_partial_host), _ptr(out_host), int(bool(use_graph))))


def ft_moe_graph_capture_decode(h, first_layer, n_layers, batch, x_bf16, logits, c_partial, out,
                                rows_out=None) -> int:
    g = C.c_void_p()
    _check(_lib.ft_moe_graph_capture_decode(h, first_layer, n_layers, batch, _ptr(x_bf16), _ptr(logits),
                                            _ptr(c_partial), _ptr(out), _ptr(rows_out), C.byref(g)))
    return g.value


def ft_graph_launch(g) -> None:
    _check(_lib.ft_graph_launch(g))


def ft_graph_destroy(g) -> None:
    _check(_lib.ft_graph_destroy(g))


def ft_moe_prefill_chunk(h, layer, n_tokens, x_bf16, logits, out) -> None:
    _check(_lib.ft_moe_prefill_chunk(h, layer, n_tokens, _ptr(x_bf16), _ptr(logits), _ptr(out)))


def ft_moe_set_router(h, w_router_bf16, gate=FT_GATE_SOFTMAX_TOPK) -> None:
    """w_router_bf16: host uint16 array [L][E][H] (BF16 bits), or None to keep the weights."""
    if w_router_bf16 is not None:
        w_router_bf16 = np.ascontiguousarray(w_router_bf16, dtype=np.uint16)
    _check(_lib.ft_moe_set_router(h, _ptr(w_router_bf16), int(gate)))


def ft_moe_router_logits(h, layer, n_tokens, x_bf16, logits_out) -> None:
    _check(_lib.ft_moe_router_logits(h, layer, n_tokens, _ptr(x_bf16), _ptr(logits_out)))


def ft_moe_decode_step_hidden(h, layer, batch, x_bf16, c_partial, out, rows_out=None, logits_out=None) -> None:
    _check(_lib.ft_moe_decode_step_hidden(h, layer, batch, _ptr(x_bf16), _ptr(c_partial), _ptr(out),
                                          _ptr(rows_out), _ptr(logits_out)))


def ft_moe_prefill_chunk_hidden(h, layer, n_tokens, x_bf16, out) -> None:
    _check(_lib.ft_moe_prefill_chunk_hidden(h, layer, n_tokens, _ptr(x_bf16), _ptr(out)))


HOST_HOOK = C.CFUNCTYPE(None, C.c_void_p, C.c_int, C.c_int, C.POINTER(C.c_int32), C.POINTER(C.c_float),
                        C.POINTER(C.c_int32), C.POINTER(C.c_float))
_hooks = {}  # handle -> callback object, kept alive while registered


def ft_moe_set_host_hook(h, fn) -> None:
    """fn(layer, batch, sel[B*k], gates[B*k], slot_of_pair[B*k], rows[B*k*H]) with numpy views;
    it must fill the rows of the pairs whose slot is FT_CPU.  None removes the hook.  The
    hook runs on a CUDA driver thread: callers that wait for the stream must release the
    interpreter lock while they wait (ft_moe_synchronize and the other calls here do)."""
    if fn is None:
        _check(_lib.ft_moe_set_host_hook(h, None, None))
        _hooks.pop(h, None)
        return

    def tramp(_user, layer, batch, sel, gates, slot, rows):
        n = batch * _hook_k[h]
        fn(layer, batch, np.ctypeslib.as_array(sel, (n,)), np.ctypeslib.as_array(gates, (n,)),
           np.ctypeslib.as_array(slot, (n,)), np.ctypeslib.as_array(rows, (n, _hook_h[h])))

    cb = HOST_HOOK(tramp)
    _check(_lib.ft_moe_set_host_hook(h, C.cast(cb, C.c_void_p), None))
    _hooks[h] = cb


_hook_k, _hook_h = {}, {}


def ft_moe_set_prefill_overlap(h, on: bool) -> None:
    _check(_lib.ft_moe_set_prefill_overlap(h, 1 if on else 0))


def ft_cache_resize(h, new_slots) -> None:
    _check(_lib.ft_cache_resize(h, new_slots))


def ft_split_misses(m, bp_gbps, bh_gbps, evictable) -> int:
    q = C.c_int()
    _check(_lib.ft_split_misses(m, bp_gbps, bh_gbps, evictable, C.byref(q)))
    return q.value


def ft_bench_bw(nbytes, iters) -> float:
    v = C.c_double()
    _check(_lib.ft_bench_bw(nbytes, iters, C.byref(v)))
    return v.value


def ft_moe_get_stats(h) -> ft_stats:
    s = ft_stats()
    _check(_lib.ft_moe_get_stats(h, C.byref(s)))
    return s


def ft_moe_get_step_trace(h, max_batch, top_k, kcap) -> dict:
    """Decisions of the last decode layer-step as numpy arrays."""
    a = {"sel": np.zeros(max_batch * top_k, np.int32), "gates": np.zeros(max_batch * top_k, np.float32),
         "slot_of_pair": np.zeros(max_batch * top_k, np.int32), "active": np.zeros(kcap, np.int32),
         "hit": np.zeros(kcap, np.int32), "miss": np.zeros(kcap, np.int32), "victims": np.zeros(kcap, np.int32)}
    t = ft_step_trace()
    for k, v in a.items():
        setattr(t, k, v.ctypes.data)
    _check(_lib.ft_moe_get_step_trace(h, C.byref(t)))
    B = t.batch
    return {"layer": t.layer, "batch": B, "q": t.q, "clock": t.clock, "n_cpu": t.n_cpu,
            "sel": a["sel"][:B * top_k].reshape(B, top_k), "gates": a["gates"][:B * top_k].reshape(B, top_k),
            "slot_of_pair": a["slot_of_pair"][:B * top_k].reshape(B, top_k),
            "active": a["active"][:t.n_active].tolist(), "hit": a["hit"][:t.n_hit].tolist(),
            "miss": a["miss"][:t.n_miss].tolist(), "victims": a["victims"][:t.n_victims].tolist()}


def ft_moe_get_state(h, n_logical, n_slots) -> dict:
    res = np.zeros(n_logical, np.int32)
    owner = np.zeros(n_slots, np.int32)
    stamp = np.zeros(n_slots, np.uint32)
    clock = C.c_uint32()
    _check(_lib.ft_moe_get_state(h, res.ctypes.data, owner.ctypes.data, stamp.ctypes.data, C.byref(clock)))
    return {"res": res, "owner": owner, "stamp": stamp, "clock": clock.value}


def ft_moe_set_profiling(h, enable) -> None:
    _check(_lib.ft_moe_set_profiling(h, int(bool(enable))))


def ft_moe_get_profile(h, reset=True) -> dict:
    p = ft_profile()
    _check(_lib.ft_moe_get_profile(h, C.byref(p), int(bool(reset))))
    return {k: (int(p.launches[i]), float(p.total_ms[i])) for i, k in enumerate(PROFILE_KINDS)}


def ft_moe_set_stream(h, stream) -> None:
    _check(_lib.ft_moe_set_stream(h, stream))


def ft_moe_synchronize(h) -> None:
    _check(_lib.ft_moe_synchronize(h))


def ft_moe_destroy(h) -> None:
    _check(_lib.ft_moe_destroy(h))


def ft_moe_decode_resident_noalloc(n_experts, top_k, hidden, inter, wtype, experts_dev, shared_dev, batch, x_bf16,
                                   logits, out, rows_out=None, error_word_out=None, stream=None) -> None:
    """Allocation-free layer evaluation (see include/ft_moe.h): every intermediate lives in
    the library's fixed 8 MiB device scratch array; nothing is allocated by the call.
    error_word_out: optional device uint32 that receives the call's device error bits."""
    st = _lib.ft_moe_decode_resident_noalloc(n_experts, top_k, hidden, inter, wtype, _ptr(experts_dev),
                                             _ptr(shared_dev), batch, _ptr(x_bf16), _ptr(logits), _ptr(out),
                                             _ptr(rows_out), _ptr(error_word_out), stream)
    if st != FT_OK:
        raise FtError(st, "ft_moe_decode_resident_noalloc failed")


def ft_test_inject_failure(kind, nth) -> None:
    _check(_lib.ft_test_inject_failure(kind, nth))


def ft_moe_reset_error(h) -> None:
    _check(_lib.ft_moe_reset_error(h))


def ft_moe_test_control(h, what, value) -> None:
    _check(_lib.ft_moe_test_control(h, what, value))


def ft_host_alloc(nbytes, flags=FT_HOST_PINNED) -> int:
    """Page-locked, mapped host memory for expert banks; returns its address."""
    p = C.c_void_p()
    _check(_lib.ft_host_alloc(nbytes, flags, C.byref(p)))
    return p.value


def ft_host_free(addr) -> None:
    _check(_lib.ft_host_free(addr))


def host_array(shape, dtype, flags=FT_HOST_PINNED):
    """A numpy array over fresh ft_host_alloc memory; release it with free_host_array."""
    dtype = np.dtype(dtype)
    n = int(np.prod(shape)) * dtype.itemsize
    addr = ft_host_alloc(max(n, 16), flags)
    buf = (C.c_uint8 * max(n, 16)).from_address(addr)
    return np.frombuffer(buf, dtype=np.uint8, count=n).view(dtype).reshape(shape)


def free_host_array(a) -> None:
    """Release an array that host_array returned (not a slice of it)."""
    ft_host_free(a.__array_interface__["data"][0])


def make_config(n_layers, hidden, inter, n_experts, top_k, has_shared, wtype, max_batch, cache_slots,
                bp_gbps, bh_gbps, max_prefill_tokens=0, fill_mode=FT_FILL_KERNEL, device=0,
                compute_stream=None, transfer_stream=None) -> ft_moe_config:
    return ft_moe_config(n_layers, hidden, inter, n_experts, top_k, int(has_shared), wtype, max_batch,
                         max_prefill_tokens, cache_slots, bp_gbps, bh_gbps, fill_mode, device,
                         compute_stream, transfer_stream)
