"""Seeded synthetic inputs for the MoE-layer expert-cache path.

This module only *makes inputs*: expert weight banks, activations, router
logits and routing traces.  It holds none of the method's arithmetic (no
routing, no cache policy, no expert math), so the CPU oracle and the CUDA
library can both be fed from it without sharing any computation.

Every random value comes from SplitMix64 (Steele, Lea & Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014) used as a
counter-based generator: value i of a stream is ``splitmix64(key + i)``,
where the key is derived from (base seed, tag, indices) by chaining the same
mixing function.  Any element can therefore be regenerated on its own.

Weight banks are large (64 GB for the 40-layer decode shape), so they are
made from a per-tensor-kind base stream of length P (a prime): the tensor of
logical expert u is the window of P-periodic stream values starting at
offset ``(a*u + b) mod P``.  Because P is prime and a != 0, every expert gets a
distinct window, and materialising a bank is a sequence of contiguous copies.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

MASK64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15

# Stream tags (arbitrary distinct integers).
TAG_GATE, TAG_UP, TAG_DOWN = 1, 2, 3
TAG_GATE_SCALE, TAG_UP_SCALE, TAG_DOWN_SCALE = 4, 5, 6
TAG_TENSOR_SCALE = 8
TAG_OFFSET = 7
TAG_X, TAG_LOGIT = 10, 11
TAG_PERM, TAG_TRACE = 12, 13
TAG_PREFILL_X, TAG_PREFILL_Z = 30, 31
TAG_ROUTER = 40

W_BF16 = 0
W_FP8_E4M3_B128 = 1
W_NVFP4 = 2
W_MXFP4 = 3

FP8_BLOCK = 128


# --------------------------------------------------------------------------- RNG
def _sm64_int(x: int) -> int:
    z = (x + _GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = x.astype(np.uint64, copy=True) + np.uint64(_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def derive_key(*parts: int) -> int:
    """Chain SplitMix64 over integer parts -> a 64-bit stream key."""
    k = 0
    for p in parts:
        k = _sm64_int(k ^ (int(p) & MASK64))
    return k


def raw_u64(key: int, n: int, start: int = 0) -> np.ndarray:
    with np.errstate(over="ignore"):
        idx = np.arange(start, start + n, dtype=np.uint64) + np.uint64(key)
    return splitmix64(idx)


def uniform(key: int, n: int, start: int = 0) -> np.ndarray:
    """n doubles in [0, 1): top 53 bits of each stream value."""
    return (raw_u64(key, n, start) >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))


def normal(key: int, n: int) -> np.ndarray:
    """n standard normals by Box-Muller over consecutive uniform pairs."""
    m = (n + 1) // 2
    u = uniform(key, 2 * m)
    u1 = 1.0 - u[0::2]  # (0, 1]
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n]


# ----------------------------------------------------------------- input rounding
def f32_to_bf16_bits(f) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even), return uint16 bits."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def f32_to_e4m3_codes(f) -> np.ndarray:
    """Saturating round-to-nearest-even E4M3FN encoding (via torch's cast after a clip)."""
    import torch

    t = torch.from_numpy(np.clip(np.asarray(f, dtype=np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


# ------------------------------------------------------------------------ configs
@dataclass(frozen=True)
class Workload:
    """One synthetic workload: model shape, cache size, split bandwidths, input recipe."""

    name: str
    cfg_id: int
    n_layers: int
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    has_shared: bool
    wtype: int
    batch: int
    steps: int
    cache_slots: int
    bp_gbps: float
    bh_gbps: float
    logits: str = "trace"          # "trace" | "normal" | "uniform"
    prefill_tokens: int = 0
    keep_prob: float = 0.7
    zipf_s: float = 1.1
    weight_std: float = 0.02

    @property
    def seed(self) -> int:
        return 20261202 + self.cfg_id

    @property
    def n_logical(self) -> int:
        return self.n_layers * self.n_experts

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def capacity_slots(frac: float, n_layers: int, n_experts: int) -> int:
    """Cache capacity as a fraction of the routed-expert pool -> whole slots."""
    return int(math.floor(frac * n_layers * n_experts + 1e-9))


def tiny() -> Workload:
    return Workload("tiny", 1, 2, 256, 128, 16, 2, False, W_BF16, 1, 8, 8, 11.8, 47.5, logits="normal")


def decode_bf16(batch: int = 1, capacity: float = 0.37, ratio=(52.7, 77.3), cfg_id: int = 2) -> Workload:
    return Workload("decode_bf16", cfg_id, 40, 2048, 512, 256, 8, True, W_BF16, batch, 512,
                    capacity_slots(capacity, 40, 256), ratio[0], ratio[1])


def decode_fp8(batch: int = 1) -> Workload:
    return Workload("decode_fp8", 3, 8, 7168, 2048, 256, 8, False, W_FP8_E4M3_B128, batch, 512,
                    capacity_slots(0.11, 8, 256), 52.7, 77.3)


def prefill() -> Workload:
    return Workload("prefill", 4, 40, 2048, 512, 256, 8, False, W_BF16, 1, 1,
                    capacity_slots(0.37, 40, 256), 52.7, 77.3, logits="uniform", prefill_tokens=8192)


SWEEP_BATCHES = (1, 4, 16, 64)
SWEEP_CAPACITIES = (0.10, 0.25, 0.37, 0.50, 1.00)
SWEEP_RATIOS = ((11.8, 47.5), (25.0, 50.0), (52.7, 77.3))


def sweep_point(batch: int, capacity: float, ratio) -> Workload:
    return decode_bf16(batch=batch, capacity=capacity, ratio=ratio, cfg_id=5).with_(name="sweep")


# ------------------------------------------------------------------ weight banks
def _is_prime(n: int) -> bool:
    if n < 2:
        return False
    if n % 2 == 0:
        return n == 2
    r = int(math.isqrt(n))
    f = 3
    while f <= r:
        if n % f == 0:
            return False
        f += 2
    return True


def _prime_at_least(n: int) -> int:
    n = max(n, 3) | 1
    while not _is_prime(n):
        n += 2
    return n


@dataclass
class _Stream:
    period: int
    ext: np.ndarray      # stream values, extended so any window is contiguous
    a: int
    b: int
    n: int               # elements per expert tensor

    def window(self, u: int) -> np.ndarray:
        off = (self.a * u + self.b) % self.period
        return self.ext[off:off + self.n]


def bank_shapes(w: Workload) -> dict:
    """Per-expert tensor shapes of each bank (row-major, first dim of a bank = logical id)."""
    H, I = w.hidden, w.inter
    s = {"gate": (I, H), "up": (I, H), "down": (H, I)}
    if w.wtype == W_FP8_E4M3_B128:
        s.update({"gate_scale": (I, H // FP8_BLOCK), "up_scale": (I, H // FP8_BLOCK),
                  "down_scale": (H, I // FP8_BLOCK)})
    if w.wtype == W_NVFP4:  # packed E2M1 (two per byte), E4M3 scales per 16, FP32 tensor scales
        s = {"gate": (I, H // 2), "up": (I, H // 2), "down": (H, I // 2),
             "gate_bscale": (I, H // 16), "up_bscale": (I, H // 16), "down_bscale": (H, I // 16),
             "tensor_scale": (4,)}
    if w.wtype == W_MXFP4:  # packed E2M1, E8M0 scales per 32
        s = {"gate": (I, H // 2), "up": (I, H // 2), "down": (H, I // 2),
             "gate_bscale": (I, H // 32), "up_bscale": (I, H // 32), "down_bscale": (H, I // 32)}
    return s


def bank_dtypes(w: Workload) -> dict:
    wd = np.uint16 if w.wtype == W_BF16 else np.uint8
    d = {"gate": wd, "up": wd, "down": wd}
    if w.wtype == W_FP8_E4M3_B128:
        d.update({"gate_scale": np.float32, "up_scale": np.float32, "down_scale": np.float32})
    if w.wtype == W_NVFP4:
        d.update({"gate_bscale": np.uint8, "up_bscale": np.uint8, "down_bscale": np.uint8,
                  "tensor_scale": np.float32})
    if w.wtype == W_MXFP4:
        d.update({"gate_bscale": np.uint8, "up_bscale": np.uint8, "down_bscale": np.uint8})
    return d


_TAGS = {"gate": TAG_GATE, "up": TAG_UP, "down": TAG_DOWN,
         "gate_scale": TAG_GATE_SCALE, "up_scale": TAG_UP_SCALE, "down_scale": TAG_DOWN_SCALE,
         "gate_bscale": TAG_GATE_SCALE, "up_bscale": TAG_UP_SCALE, "down_bscale": TAG_DOWN_SCALE,
         "tensor_scale": TAG_TENSOR_SCALE}


class ExpertPool:
    """Deterministic per-(layer, expert) weights.

    Routed expert (l, e) has logical id u = l*E + e.  The always-on shared
    expert of layer l (when the workload has one) uses id L*E + l, so it never
    coincides with a routed expert.

    BF16 banks: N(0, weight_std) rounded to bfloat16.  FP8 banks: E4M3 codes
    from N(0, weight_std * 448) (saturating RNE), with one FP32 scale per
    128-element block along the reduction dimension drawn from U(0.5, 2)/448,
    so that dequantised weights have roughly the BF16 banks' spread.  NVFP4
    banks: uniform E2M1 codes, E4M3 block scales in [0.5, 2) per 16 elements
    and per-expert FP32 tensor scales in U(0.004, 0.008) (dequantised weights
    of about 0.02 rms).  MXFP4 banks: uniform E2M1 codes and E8M0 block scales
    2^-8 .. 2^-6 per 32 elements.
    """

    def __init__(self, w: Workload):
        self.w = w
        self.shapes = bank_shapes(w)
        self.dtypes = bank_dtypes(w)
        self._streams: dict[str, _Stream] = {}
        for kind, shp in self.shapes.items():
            n = int(np.prod(shp))
            period = _prime_at_least(max(1 << 22, 2 * n + 1))
            key = derive_key(w.seed, _TAGS[kind])
            if kind == "tensor_scale":
                vals = (0.004 + 0.004 * uniform(key, period)).astype(np.float32)
            elif kind.endswith("_bscale") and w.wtype == W_MXFP4:  # E8M0 codes 119..121: 2^-8 .. 2^-6
                vals = (119 + (raw_u64(key, period) % np.uint64(3))).astype(np.uint8)
            elif kind.endswith("_bscale"):  # E4M3 codes 0x30..0x3F: 0.5 .. 1.875
                vals = (0x30 + (raw_u64(key, period) & np.uint64(0xF))).astype(np.uint8)
            elif kind.endswith("_scale"):
                vals = ((0.5 + 1.5 * uniform(key, period)) / 448.0).astype(np.float32)
            elif w.wtype in (W_NVFP4, W_MXFP4):  # two uniform E2M1 codes per byte
                vals = (raw_u64(key, period) & np.uint64(0xFF)).astype(np.uint8)
            elif w.wtype == W_BF16:
                vals = f32_to_bf16_bits((normal(key, period) * w.weight_std).astype(np.float32))
            else:
                vals = f32_to_e4m3_codes((normal(key, period) * (w.weight_std * 448.0)).astype(np.float32))
            reps = (period + n + period - 1) // period
            ext = np.tile(vals, reps)[:period + n]
            ko = derive_key(w.seed, TAG_OFFSET, _TAGS[kind])
            a = 1 + ko % (period - 1)
            b = _sm64_int(ko) % period
            self._streams[kind] = _Stream(period, ext, a, b, n)

    def tensor(self, kind: str, u: int) -> np.ndarray:
        """Read-only view of bank `kind` for logical id u, shaped per `bank_shapes`."""
        return self._streams[kind].window(u).reshape(self.shapes[kind])

    def expert(self, u: int) -> dict:
        return {k: self.tensor(k, u) for k in self.shapes}

    def shared(self, layer: int) -> dict:
        return self.expert(self.w.n_logical + layer)

    def alloc_banks(self, n_rows: int, empty=np.empty) -> dict:
        """Uninitialised banks of n_rows experts; `empty(shape, dtype)` allocates each (e.g. in
        page-locked or huge-page memory)."""
        return {k: empty((n_rows,) + self.shapes[k], self.dtypes[k]) for k in self.shapes}

    def fill_banks(self, banks: dict, first_id: int = 0, threads: int | None = None) -> None:
        """Write experts first_id .. first_id+rows-1 into preallocated banks (rows = first dim)."""
        n_rows = next(iter(banks.values())).shape[0]
        threads = threads or min(16, os.cpu_count() or 1)

        def work(lo, hi):
            for r in range(lo, hi):
                for k, arr in banks.items():
                    arr[r] = self.tensor(k, first_id + r)

        step = max(1, (n_rows + threads - 1) // threads)
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda lo: work(lo, min(n_rows, lo + step)), range(0, n_rows, step)))

    def routed_banks(self, threads: int | None = None, empty=np.empty) -> dict:
        b = self.alloc_banks(self.w.n_logical, empty)
        self.fill_banks(b, 0, threads)
        return b

    def shared_banks(self) -> dict | None:
        if not self.w.has_shared:
            return None
        b = self.alloc_banks(self.w.n_layers)
        self.fill_banks(b, self.w.n_logical, threads=1)
        return b


# ------------------------------------------------------------ activations/logits
def decode_x(w: Workload, step: int, layer: int) -> np.ndarray:
    """Activations of one decode layer-step: bf16 bits [B, H], x ~ N(0, 1)."""
    z = normal(derive_key(w.seed, TAG_X, step, layer), w.batch * w.hidden)
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(w.batch, w.hidden)


def decode_logits(w: Workload, step: int, layer: int, trace: np.ndarray | None = None) -> np.ndarray:
    """Router logits [B, E] float32: N(0, 1), plus 8 on the trace's experts when a trace is given."""
    z = normal(derive_key(w.seed, TAG_LOGIT, step, layer), w.batch * w.n_experts)
    z = z.astype(np.float32).reshape(w.batch, w.n_experts)
    if trace is not None:
        ids = trace[step, layer]  # [B, k]
        for b in range(w.batch):
            z[b, ids[b]] += np.float32(8.0)
    return z


def prefill_x(w: Workload, chunk: int, layer: int, n_tokens: int) -> np.ndarray:
    z = normal(derive_key(w.seed, TAG_PREFILL_X, chunk, layer), n_tokens * w.hidden)
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(n_tokens, w.hidden)


def prefill_logits(w: Workload, chunk: int, layer: int, n_tokens: int) -> np.ndarray:
    """Prefill router logits ~ U(-1, 1): nearly every expert is active in a chunk."""
    u = uniform(derive_key(w.seed, TAG_PREFILL_Z, chunk, layer), n_tokens * w.n_experts)
    return (2.0 * u - 1.0).astype(np.float32).reshape(n_tokens, w.n_experts)


def router_weights(w: Workload) -> np.ndarray:
    """Router projection of every layer: bf16 bits [L, E, H], N(0, (2/sqrt(H))^2), so that
    the logits of x ~ N(0, 1) have a spread of about 2."""
    z = normal(derive_key(w.seed, TAG_ROUTER), w.n_layers * w.n_experts * w.hidden)
    z = z * (2.0 / np.sqrt(w.hidden))
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(w.n_layers, w.n_experts, w.hidden)


# ------------------------------------------------------------------ routing trace
def _zipf_cdf(n: int, s: float) -> np.ndarray:
    p = np.arange(1, n + 1, dtype=np.float64) ** (-s)
    c = np.cumsum(p)
    return c / c[-1]


def routing_trace(w: Workload, steps: int | None = None, batch: int | None = None) -> np.ndarray:
    """Temporal-locality routing trace, int32 [steps, L, B, k] of expert ids.

    Each (layer, sequence) chain is independent.  Step 0 draws k distinct
    experts from Zipf(s) over ranks, mapped to ids by a seeded per-layer
    permutation.  At every later step each of the previous step's experts is
    kept with probability keep_prob; the remaining places are refilled by
    Zipf draws, redrawing duplicates.
    """
    steps = w.steps if steps is None else steps
    B = w.batch if batch is None else batch
    L, E, k = w.n_layers, w.n_experts, w.top_k
    cdf = _zipf_cdf(E, w.zipf_s)
    perms = np.stack([np.argsort(uniform(derive_key(w.seed, TAG_PERM, l), E), kind="stable")
                      for l in range(L)])                                  # rank -> id, [L, E]
    C = L * B
    chain_layer = np.repeat(np.arange(L), B)
    chain_keys = np.array([derive_key(w.seed, TAG_TRACE, c) for c in range(C)], dtype=np.uint64)
    out = np.empty((steps, L, B, k), dtype=np.int32)
    prev = None
    for s in range(steps):
        with np.errstate(over="ignore"):
            skeys = splitmix64(chain_keys ^ np.uint64(s))                  # per (chain, step) key
        chosen = np.full((C, k), -1, dtype=np.int64)
        count = np.zeros(C, dtype=np.int64)
        draw = 0
        if prev is not None:
            keep = _u01(skeys, np.arange(k, dtype=np.uint64)[None, :]) < w.keep_prob   # [C, k]
            for j in range(k):
                m = keep[:, j]
                chosen[m, count[m]] = prev[m, j]
                count[m] += 1
            draw = k
        guard = 0
        while (count < k).any():
            need = np.nonzero(count < k)[0]
            u = _u01(skeys[need], np.uint64(draw))
            rank = np.minimum(np.searchsorted(cdf, u, side="right"), E - 1)
            cand = perms[chain_layer[need], rank]
            dup = (chosen[need] == cand[:, None]).any(axis=1)
            ok = need[~dup]
            chosen[ok, count[ok]] = cand[~dup]
            count[ok] += 1
            draw += 1
            guard += 1
            if guard > 100000:
                raise RuntimeError("routing trace did not converge")
        out[s] = chosen.reshape(L, B, k)
        prev = chosen
    return out


def _u01(keys: np.ndarray, idx) -> np.ndarray:
    """Uniform [0,1) draw number `idx` of each per-chain key (idx scalar or a [1, n] row)."""
    idx = np.asarray(idx, dtype=np.uint64)
    k = keys[:, None] if idx.ndim == 2 else keys
    with np.errstate(over="ignore"):
        v = splitmix64(k + idx)
    return (v >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))
