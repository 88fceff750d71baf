"""Plain CPU oracle for the FreeToken MoE-layer hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code,
tables or constants with the CUDA library, and the library never calls it.

It is written for a reader checking it against the pages, not for speed:
every decision is a total order written out directly, expert maths runs in
float64 on decoded weights, and numpy matmul/sort are the only library steps.

Sources (cited by page title and section):
  [FT]  "FreeToken 完全拆解：带宽自适应执行，让 8GB 笔记本跑 35B、单卡工作站跑 753B 的边缘 MoE 服务系统"
  [FT2] "개인 장치에서 MoE 모델을 서빙하는 FreeToken" (no section headings; cited by paragraph topic)
  [P3]  "OSDI'26 | 双路 CPU + 两张 5090，本地跑满血 671B DeepSeek：云端 SLO 是怎么在消费级硬件上达成的"

Readings taken where the pages are silent or garbled (each is listed in the
design notes with its reason):
  * q* is rounded half-up, computed in integers over bandwidths in MB/s.
  * F is the first q misses in ascending logical id; C is the rest.
  * Hit slots are never victims, so q <= S - |H|.
  * One global clock ticks once per layer-step; LRU ties break by slot index.
  * The C set leaves residency and recency untouched.
  * Router gates are a softmax over the k selected logits; ties pick the lower id.
    Two other gate functions (softmax over all E, normalised sigmoid) are
    written out for routers that use them.
  * FP8 blocks are 1x128 along the reduction dimension of each output row.
  * The output sums, per token, the shared expert first and then the k pair
    rows in ascending expert id.

Parity unpinned: none of the functions here; the pins live in tests/.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

FT_CPU = -1          # rewritten pair id meaning "evaluated on the host (C set)"
FP8_BLOCK = 128


# ============================================================== q* miss split
def mbps(gbps: float) -> int:
    """Bandwidth in GB/s -> integer MB/s, nearest, halves away from zero."""
    v = gbps * 1000.0
    return int(math.floor(v + 0.5)) if v >= 0 else -int(math.floor(-v + 0.5))


def split_misses(m: int, bp_mbs: int, bh_mbs: int, evictable: int) -> int:
    """Number q of the m misses to fill over the host link.

    [FT, "q* 策略"]: fills stream at B_P while the host executes the other
    m-q misses on the residual bandwidth B_H-B_P; equal branch times give
    q* = m*B_P/B_H.  [FT2, paragraph on the miss split]: the residual is
    max(B_H-B_P, 0), so with B_H <= B_P every miss is filled.  q* is rounded
    and at least one fill is kept whenever there is a miss.  The fill count
    cannot exceed the slots that are not hits of this step (evictable).

    Rounding: half up, i.e. floor(m*bp/bh + 1/2) = (2*m*bp + bh) // (2*bh).
    """
    if m <= 0:
        return 0
    if bh_mbs <= bp_mbs:
        q = m
    else:
        q = (2 * m * bp_mbs + bh_mbs) // (2 * bh_mbs)
        q = max(q, 1)
    return max(0, min(q, m, evictable))


# ===================================================================== router
GATE_SOFTMAX_TOPK = 0   # softmax over the k chosen logits
GATE_SOFTMAX_ALL = 1    # softmax over all E logits; the k chosen probabilities as they are
GATE_SIGMOID_TOPK = 2   # sigmoid of each chosen logit, normalised to sum 1 over the k


def route(logits: np.ndarray, k: int, gate_mode: int = GATE_SOFTMAX_TOPK):
    """Top-k router.

    For each token the k experts with the largest logits are chosen (equal
    logits: the lower expert id first), listed in ascending expert id.
    [FT, "Device-side 缓存控制"] (routing precedes dedupe).  The gate function
    is the router's own, which the pages do not print for the models they name
    (Qwen3.6-35B-A3B, DeepSeek-V4-Flash [FT2, opening paragraph]); three
    textbook forms are written out, each in float64 and stored as float32:

      GATE_SOFTMAX_TOPK:  g_r = exp(z_r) / sum_{j chosen} exp(z_j)
      GATE_SOFTMAX_ALL:   g_r = exp(z_r) / sum_{j < E} exp(z_j)
      GATE_SIGMOID_TOPK:  g_r = s(z_r) / sum_{j chosen} s(z_j),  s(z) = 1 / (1 + exp(-z))

    The softmax exponentials are shifted by the largest logit (an exact identity).
    All three gate functions are increasing in z, so the choice is the same.
    A NaN logit ranks as -inf (it then ties with any -inf logit, lower id first);
    -0 and +0 are equal logits.
    """
    B, E = logits.shape
    sel = np.empty((B, k), dtype=np.int64)
    gates = np.empty((B, k), dtype=np.float32)
    ids = np.arange(E)
    for t in range(B):
        z = logits[t].astype(np.float64)
        z = np.where(np.isnan(z), -np.inf, z)
        order = np.lexsort((ids, -z))          # primary: logit desc; secondary: id asc
        chosen = np.sort(order[:k])
        zs = z[chosen]
        if gate_mode == GATE_SOFTMAX_TOPK:
            w = np.exp(zs - zs.max())
            g = w / w.sum()
        elif gate_mode == GATE_SOFTMAX_ALL:
            w = np.exp(z - z.max())
            g = w[chosen] / w.sum()
        elif gate_mode == GATE_SIGMOID_TOPK:
            s = 1.0 / (1.0 + np.exp(-zs))
            g = s / s.sum()
        else:
            raise ValueError(f"unknown gate mode {gate_mode}")
        sel[t] = chosen
        gates[t] = g.astype(np.float32)
    return sel, gates


def router_logits(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """Router logits z[t, e] = sum_h x[t, h] * W_router[e, h], float64 over the
    decoded BF16 values.  x_bits: uint16 [B, H]; w_bits: uint16 [E, H].  The
    router is the layer's gate projection, run on the GPU with the rest of the
    control path ([FT2], decode paragraph: the GPU router dedupes the active
    experts; [P3] §3.3: gate and sort run locally on each GPU)."""
    return bf16_to_f64(x_bits) @ bf16_to_f64(w_bits).T


def dedupe(sel: np.ndarray, layer: int, n_experts: int) -> list[int]:
    """Sorted unique logical ids u = layer*E + e over the whole batch.

    [FT, "Device-side 缓存控制"]; logical id form from [FT, "FTW 权重格式与平台适配"].
    """
    return sorted({layer * n_experts + int(e) for e in sel.reshape(-1)})


# ========================================================== slot-pool cache
@dataclass
class StepRecord:
    layer: int
    clock: int
    A: list
    H: list
    M: list
    q: int
    victims: list
    F: list
    C: list
    slot_of_pair: np.ndarray     # [B, k]: slot id, or FT_CPU


@dataclass
class Counters:
    hits: int = 0
    misses: int = 0
    fills: int = 0
    cpu_execs: int = 0
    evictions: int = 0


class SlotCache:
    """Global slot-pool LRU shared by every MoE layer.

    [FT, "语义感知专家缓存"]: one LRU residency space for all layers; a hit
    refreshes recency, a fill admits the newly chosen expert, an eviction
    removes the expert unused for longest.  [FT2, paragraph on the two-tier
    memory]: a slot holds every tensor of one (layer, expert).

    State: res[u] = slot holding logical expert u or -1; owner[s] = logical
    id in slot s or -1; stamp[s] = clock of the last step that used slot s
    (0 for a slot never used).  One clock for all layers, starting at 0.
    """

    def __init__(self, n_slots: int, n_logical: int):
        self.S = int(n_slots)
        self.res = np.full(n_logical, -1, dtype=np.int64)
        self.owner = np.full(self.S, -1, dtype=np.int64)
        self.stamp = np.zeros(self.S, dtype=np.int64)
        self.clock = 0
        self.cnt = Counters()
        self.buffers: list | None = None
        self.prefill_next_layer: int | None = None

    # -------------------------------------------------------------- decode
    def lru_candidates(self, K: int) -> list[int]:
        """One scan for the K least recently used slots that are not hits of
        this step (stamp < clock), ascending by (stamp, slot).

        [FT, "Device-side 缓存控制"]: a single pass yields K candidates and the
        miss path consumes the first q <= K of them.
        """
        cand = np.nonzero(self.stamp < self.clock)[0]
        order = np.lexsort((cand, self.stamp[cand]))
        return [int(s) for s in cand[order[:K]]]

    def decode_step(self, layer: int, n_experts: int, sel: np.ndarray,
                    bp_mbs: int, bh_mbs: int) -> StepRecord:
        """Cache decisions of one decode layer-step.

        [FT, "Device-side 缓存控制"]: dedupe -> classify against the residency
        table -> fill count q -> victims -> rewrite ids to slots or FT_CPU.
        [FT, "q* 策略"]: F is admitted to the cache; C is executed on the host
        and leaves residency unchanged.
        """
        B, k = sel.shape
        A = dedupe(sel, layer, n_experts)
        self.clock += 1
        H = [u for u in A if self.res[u] >= 0]
        M = [u for u in A if self.res[u] < 0]
        for u in H:
            self.stamp[self.res[u]] = self.clock
        self.cnt.hits += len(H)
        self.cnt.misses += len(M)
        q = split_misses(len(M), bp_mbs, bh_mbs, self.S - len(H))
        K = min(B * k, n_experts)
        victims = self.lru_candidates(K) if q > 0 else []
        for i in range(q):
            v = victims[i]
            old = self.owner[v]
            if old >= 0:
                self.res[old] = -1
                self.cnt.evictions += 1
            self.owner[v] = M[i]
            self.res[M[i]] = v
            self.stamp[v] = self.clock
            self.cnt.fills += 1
        F, C = M[:q], M[q:]
        self.cnt.cpu_execs += len(C)
        slot_of_pair = np.empty((B, k), dtype=np.int64)
        for t in range(B):
            for r in range(k):
                s = self.res[layer * n_experts + int(sel[t, r])]
                slot_of_pair[t, r] = s if s >= 0 else FT_CPU
        self.prefill_next_layer = None
        return StepRecord(layer, self.clock, A, H, M, q, victims, F, C, slot_of_pair)

    # ------------------------------------------------------------- prefill
    def prefill_layer(self, layer: int, n_experts: int, n_layers: int) -> list[int]:
        """Residency effect of one prefill layer with full-layer double buffering.

        [FT, "全层双缓冲"] and [FT2, paragraph on the double buffer]: two
        full-layer buffers are taken from the shared slot pool; layer l is
        computed from one while layer l+1 streams, whole, into the other.
        Reading used here: a chunk starts at a call that does not continue the
        previous prefill layer; it takes the 2E least recently used slots
        (ascending (stamp, slot)); the first E are buffer 0, the next E buffer
        1, and their occupants leave the cache.  Layer l goes to buffer
        (l - first layer) mod 2, expert e of it into the buffer's e-th slot;
        the slot's previous occupant leaves, an older resident copy of the
        same expert is invalidated (slot emptied, stamp 0), and every expert of
        the layer is stamped with this step's clock.  What the last two layers
        leave behind seeds decode.  Prefill is not counted as hits or misses.
        Returns the buffer's slot list (slot of expert e).
        """
        E = n_experts
        if self.S < 2 * E:
            raise ValueError("prefill double buffering needs at least 2E slots")
        if self.prefill_next_layer != layer or self.buffers is None:
            order = np.lexsort((np.arange(self.S), self.stamp))
            bufs = [int(s) for s in order[:2 * E]]
            for v in bufs:
                if self.owner[v] >= 0:
                    self.res[self.owner[v]] = -1
                    self.owner[v] = -1
                    self.stamp[v] = 0
            self.buffers = [bufs[:E], bufs[E:]]
            self.prefill_first = layer
        self.clock += 1
        buf = self.buffers[(layer - self.prefill_first) % 2]
        for e in range(E):
            u = layer * E + e
            v = buf[e]
            if self.owner[v] >= 0 and self.owner[v] != u:
                self.res[self.owner[v]] = -1
            old = self.res[u]
            if old >= 0 and old != v:
                self.owner[old] = -1
                self.stamp[old] = 0
            self.owner[v] = u
            self.res[u] = v
            self.stamp[v] = self.clock
        self.prefill_next_layer = layer + 1 if layer + 1 < n_layers else None
        return list(buf)

    def prefill_layer_on_demand(self, layer: int, n_experts: int, active) -> list[list[int]]:
        """Residency effect of one prefill layer when the pool cannot hold two
        full layers (S < 2E).

        [FT, "全层双缓冲"] and [FT2, paragraph on the double buffer]: without
        room for the two full-layer buffers, prefill loads experts on demand
        instead of oversubscribing memory.  Reading used here: the layer's
        routing is known first; its active experts (sorted unique ids routed by
        the chunk) that are resident are hits and are stamped with this step's
        clock; the others are loaded into the least recently used slots that do
        not hold a hit, ascending (stamp, slot), and stamped too.  When there
        are fewer such slots (W) than misses, the misses are taken in ascending
        id, W at a time, each wave into the same W slots, so the layer ends
        with its hits and its last wave resident.  Prefill is not counted as
        hits, misses or fills.  Returns the waves (lists of logical ids).
        """
        E = n_experts
        self.buffers = None
        self.prefill_next_layer = None
        A = [layer * E + int(e) for e in sorted(set(int(e) for e in active))]
        hits = [u for u in A if self.res[u] >= 0]
        misses = [u for u in A if self.res[u] < 0]
        free = self.S - len(hits)  # slots that hold no hit of this layer
        if misses and free == 0:
            raise ValueError("no slot outside this layer's hits")  # nothing changed
        self.clock += 1
        for u in hits:
            self.stamp[self.res[u]] = self.clock
        victims = self.lru_candidates(min(free, len(misses)))
        waves = [misses[i:i + len(victims)] for i in range(0, len(misses), max(1, len(victims)))]
        for wave in waves:
            for u, v in zip(wave, victims):
                if self.owner[v] >= 0:
                    self.res[self.owner[v]] = -1
                self.owner[v] = u
                self.res[u] = v
                self.stamp[v] = self.clock
        return waves

    # -------------------------------------------------------------- resize
    def resize(self, new_slots: int) -> list[tuple[int, int]]:
        """Safe-point resize of the expert cache.

        [FT, "挑战三"] and [FT2, paragraph on the memory budget]: the cache
        can shrink or grow at run time and the outputs do not change, because
        the host pool stays the source of truth.  Reading used here: growing
        appends empty slots; shrinking keeps the new_slots most recent entries
        by (stamp desc, slot asc), drops the rest, and moves each kept entry
        that sits at a slot >= new_slots into the free slots below new_slots,
        both taken in ascending slot order.  Returns the (from, to) moves.
        """
        n = int(new_slots)
        if n < 0:
            raise ValueError("negative size")
        if n >= self.S:
            self.owner = np.concatenate([self.owner, np.full(n - self.S, -1, dtype=np.int64)])
            self.stamp = np.concatenate([self.stamp, np.zeros(n - self.S, dtype=np.int64)])
            self.S = n
            return []
        occ = np.nonzero(self.owner >= 0)[0]
        order = np.lexsort((occ, -self.stamp[occ]))
        keep = set(int(s) for s in occ[order[:n]])
        for s in occ:
            if int(s) not in keep:
                self.res[self.owner[s]] = -1
                self.owner[s] = -1
                self.stamp[s] = 0
        movers = sorted(s for s in keep if s >= n)
        free = [s for s in range(n) if s not in keep]
        moves = list(zip(movers, free))
        for src, dst in moves:
            u = self.owner[src]
            self.owner[dst] = u
            self.stamp[dst] = self.stamp[src]
            self.res[u] = dst
        self.owner = self.owner[:n].copy()
        self.stamp = self.stamp[:n].copy()
        self.S = n
        self.buffers = None
        self.prefill_next_layer = None
        return moves


# ================================================================ expert maths
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64: the upper half of a float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _e4m3_value(code: int) -> float:
    """One E4M3FN code: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0
    is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity.
    [P3, §4.1] names the format; the definition is the OCP 8-bit float one."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


NVFP4_BLOCK = 16   # elements per block scale along the reduction dimension


def _e2m1_value(code: int) -> float:
    """One E2M1 (FP4) code: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is
    subnormal (m/2).  The block-scaled 4-bit formats that [FT, 主结果] names for its models
    (MXFP4, NVFP4) use these elements."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5
    return s * 2.0 ** (e - 1) * (1.0 + m / 2.0)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def e2m1_unpack_to_f64(packed: np.ndarray) -> np.ndarray:
    """Packed FP4 rows [R][K/2] (byte j: element 2j in the low nibble, 2j+1 in the high
    nibble) -> float64 [R][K]."""
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.float64)
    out[..., 0::2] = E2M1_TABLE[b & 0xF]
    out[..., 1::2] = E2M1_TABLE[b >> 4]
    return out


def matvec_nvfp4(packed: np.ndarray, block_scales: np.ndarray, tensor_scale: float, x: np.ndarray) -> np.ndarray:
    """NVFP4 rows times x: E2M1 elements, one E4M3 scale per 1x16 block along the
    reduction dimension applied after the block's dot product, then the bank's FP32
    tensor scale.  (The post-scaling order of [P3, §4.2], with NVFP4's block size.)"""
    w = e2m1_unpack_to_f64(packed)
    R, K = w.shape
    nb = K // NVFP4_BLOCK
    block_dots = np.einsum("rbk,bk->rb", w.reshape(R, nb, NVFP4_BLOCK),
                           np.asarray(x, dtype=np.float64).reshape(nb, NVFP4_BLOCK))
    return float(tensor_scale) * (block_dots * e4m3_to_f64(block_scales)).sum(axis=1)


MXFP4_BLOCK = 32   # elements per E8M0 block scale along the reduction dimension


def e8m0_to_f64(codes: np.ndarray) -> np.ndarray:
    """E8M0 scale codes (OCP MX): 2^(code - 127); code 255 is NaN."""
    c = np.asarray(codes, dtype=np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, c - 127))


def matvec_mxfp4(packed: np.ndarray, scale_codes: np.ndarray, x: np.ndarray) -> np.ndarray:
    """MXFP4 rows times x: E2M1 elements (packed as for NVFP4), one E8M0 scale per 1x32
    block along the reduction dimension applied after the block's dot product (the
    post-scaling order of [P3, §4.2], with MXFP4's block)."""
    w = e2m1_unpack_to_f64(packed)
    R, K = w.shape
    nb = K // MXFP4_BLOCK
    block_dots = np.einsum("rbk,bk->rb", w.reshape(R, nb, MXFP4_BLOCK),
                           np.asarray(x, dtype=np.float64).reshape(nb, MXFP4_BLOCK))
    return (block_dots * e8m0_to_f64(scale_codes)).sum(axis=1)


def silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def matvec_post_scaled(codes: np.ndarray, scales: np.ndarray, x: np.ndarray) -> np.ndarray:
    """FP8 rows times x, one scale per 1x128 block of each row applied after the block's dot.

    [P3, §4.2]: the block's dot product is formed first and multiplied by the
    block scale once (scale*sum(w*x) = sum(scale*w*x)).
    """
    R, K = codes.shape
    nb = K // FP8_BLOCK
    w = e4m3_to_f64(codes).reshape(R, nb, FP8_BLOCK)
    xb = np.asarray(x, dtype=np.float64).reshape(nb, FP8_BLOCK)
    block_dots = np.einsum("rbk,bk->rb", w, xb)
    return (block_dots * scales.astype(np.float64)).sum(axis=1)


def swiglu_expert(expert: dict, x: np.ndarray, fp8: bool) -> np.ndarray:
    """One SwiGLU expert on one token, float64: y = W_d (silu(W_g x) * (W_u x)).

    Bank layout (per expert, row-major): gate [I][H], up [I][H], down [H][I];
    FP8 scales gate_scale/up_scale [I][H/128], down_scale [H][I/128].
    `fp8` is the weight type: 0/False BF16, 1/True FP8 E4M3, 2 NVFP4 (packed E2M1
    [rows][K/2], E4M3 block scales [rows][K/16], tensor_scale [4] FP32: gate, up,
    down, unused), 3 MXFP4 (packed E2M1, E8M0 block scales [rows][K/32]).
    [FT2, paragraph on the double buffer] / [P3, §4.3] (gate, up, down projections).
    """
    if fp8 == 3:  # MXFP4
        a = matvec_mxfp4(expert["gate"], expert["gate_bscale"], x)
        b = matvec_mxfp4(expert["up"], expert["up_bscale"], x)
        h = silu(a) * b
        return matvec_mxfp4(expert["down"], expert["down_bscale"], h)
    if fp8 == 2:  # NVFP4: tensor_scale holds the gate, up and down banks' scales
        ts = expert["tensor_scale"].astype(np.float64)
        a = matvec_nvfp4(expert["gate"], expert["gate_bscale"], ts[0], x)
        b = matvec_nvfp4(expert["up"], expert["up_bscale"], ts[1], x)
        h = silu(a) * b
        return matvec_nvfp4(expert["down"], expert["down_bscale"], ts[2], h)
    if fp8:
        a = matvec_post_scaled(expert["gate"], expert["gate_scale"], x)
        b = matvec_post_scaled(expert["up"], expert["up_scale"], x)
        h = silu(a) * b
        return matvec_post_scaled(expert["down"], expert["down_scale"], h)
    a = bf16_to_f64(expert["gate"]) @ x
    b = bf16_to_f64(expert["up"]) @ x
    h = silu(a) * b
    return bf16_to_f64(expert["down"]) @ h


def pair_row(expert: dict, x: np.ndarray, gate: float, fp8: bool) -> np.ndarray:
    """Gate-weighted output row of one (token, expert) pair, float64."""
    return np.float64(np.float32(gate)) * swiglu_expert(expert, x, fp8)


def combine(shared_row, rows: list) -> np.ndarray:
    """Fixed-order merge: shared expert first, then the k pair rows in rank
    (= ascending expert id) order.  [FT, "q* 策略"] (exact merge of the GPU
    and host partial sums)."""
    out = np.zeros_like(np.asarray(rows[0], dtype=np.float64)) if shared_row is None \
        else np.asarray(shared_row, dtype=np.float64).copy()
    for r in rows:
        out = out + np.asarray(r, dtype=np.float64)
    return out


def decode_layer_outputs(rec: StepRecord, sel, gates, x_bits, c_partial, expert_of, shared=None,
                         fp8=False, tokens=None, n_experts=None):
    """Layer output rows [len(tokens), H] for a decode step.

    Pair (t, r) in G = H u F (slot_of_pair >= 0) is evaluated here from the
    expert weights; a C pair takes its row from c_partial[t][r].
    [FT, "执行顺序与工程细节"]: grouped evaluation of G, host partials for C,
    then the merge.
    """
    B, k = sel.shape
    tokens = range(B) if tokens is None else tokens
    outs = []
    for t in tokens:
        x = bf16_to_f64(x_bits[t])
        rows = []
        for r in range(k):
            if rec.slot_of_pair[t, r] >= 0:
                u = rec.layer * n_experts + int(sel[t, r])
                rows.append(pair_row(expert_of(u), x, gates[t, r], fp8))
            else:
                rows.append(np.asarray(c_partial[t, r], dtype=np.float64))
        srow = swiglu_expert(shared, x, fp8) if shared is not None else None
        outs.append(combine(srow, rows))
    return np.stack(outs)


def all_pair_rows(layer, sel, gates, x_bits, expert_of, n_experts, fp8=False) -> np.ndarray:
    """Every pair's gate-weighted row, float64 [B, k, H]: what a host executor
    would return for any C pair."""
    B, k = sel.shape
    rows = []
    for t in range(B):
        x = bf16_to_f64(x_bits[t])
        rows.append([pair_row(expert_of(layer * n_experts + int(sel[t, r])), x, gates[t, r], fp8)
                     for r in range(k)])
    return np.asarray(rows)


def prefill_outputs(layer, sel, gates, x_bits, expert_of, n_experts, tokens, shared=None, fp8=False):
    """Prefill output rows for the given tokens: every pair runs on the GPU side."""
    outs = []
    for t in tokens:
        x = bf16_to_f64(x_bits[t])
        rows = [pair_row(expert_of(layer * n_experts + int(sel[t, r])), x, gates[t, r], fp8)
                for r in range(sel.shape[1])]
        srow = swiglu_expert(shared, x, fp8) if shared is not None else None
        outs.append(combine(srow, rows))
    return np.stack(outs)


def rel_err_rows(y: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of max_j |y - ref| / max_j |ref|."""
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    ref = np.atleast_2d(np.asarray(ref, dtype=np.float64))
    num = np.abs(y - ref).max(axis=1)
    den = np.maximum(np.abs(ref).max(axis=1), 1e-30)
    return float((num / den).max())
