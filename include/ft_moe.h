/*
 * ft_moe.h -- C ABI of libftmoe: the MoE-layer hot path of a FreeToken-style
 * edge-serving system, on one GB300 (sm_103a).
 *
 * What the library computes (sources cited by page title and section):
 *   [FT]  "FreeToken 完全拆解：带宽自适应执行，让 8GB 笔记本跑 35B、单卡工作站跑 753B 的边缘 MoE 服务系统"
 *   [FT2] "개인 장치에서 MoE 모델을 서빙하는 FreeToken" (paragraph topics, no headings)
 *   [P3]  "OSDI'26 | 双路 CPU + 两张 5090，本地跑满血 671B DeepSeek：云端 SLO 是怎么在消费级硬件上达成的"
 *
 *  - A slot pool in HBM holds whole experts; one global LRU over all MoE layers,
 *    addressed by the logical id u = layer*E + expert ([FT] "语义感知专家缓存",
 *    [FT] "FTW 权重格式与平台适配").
 *  - Per decode layer-step, one control kernel routes (top-k and gates), dedupes the
 *    batch's experts, classifies hits/misses against the residency table, computes
 *    the fill count q, finds the K least recently used victims in one pass and
 *    rewrites routed ids to slots or FT_CPU ([FT] "Device-side 缓存控制").
 *  - q = round(m * B_P / B_H), at least one fill when m > 0 ([FT] "q* 策略").
 *    The F set is copied host->slots by a copy kernel (or, in FT_FILL_MEMCPY mode, by
 *    copies on the transfer stream); the C set's gate-weighted rows are an INPUT
 *    (c_partial): no host executor lives here.
 *  - G = H u F is evaluated by SwiGLU GEMV kernels (BF16; FP8 E4M3 with one FP32
 *    scale per 1x128 block applied after the block's dot product, [P3] §4.2; NVFP4
 *    and MXFP4),
 *    then a combine sums, per token, the shared expert and the k pair rows in
 *    ascending expert id (fixed order), so outputs do not depend on cache size or
 *    on the F/C split ([FT] "q* 策略").
 *  - Prefill chunks stream whole layers into two pool buffers while the previous
 *    layer runs a tcgen05 grouped GEMM ([FT] "全层双缓冲").
 *
 * Conventions for every entry point:
 *  - Return FT_OK or an ft_status; ft_last_error() gives a thread-local message.
 *  - Argument errors are returned synchronously and change no state.
 *  - Decode/prefill calls only enqueue work on the library's compute stream (no
 *    host synchronisation), except where a function says it synchronises.
 *    Errors found by kernels (bad ids in inputs, NaN logits, a wait that timed
 *    out) set bits in a device error word, read by ft_moe_get_stats().
 *  - "dev" pointers are device (HBM) addresses owned by the caller; "host"
 *    pointers are host addresses owned by the caller.
 *  - BF16 values are passed as raw 16-bit patterns (uint16_t storage).
 */
#ifndef FT_MOE_H
#define FT_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FT_OK = 0,
  FT_ERR_INVALID = 1,   /* bad argument or configuration */
  FT_ERR_CUDA = 2,      /* a CUDA runtime/driver call failed */
  FT_ERR_NOMEM = 3,     /* device or host allocation failed */
  FT_ERR_PIN = 4,       /* the host pool could not be pinned/registered; no fallback */
  FT_ERR_CAPACITY = 5,  /* the slot pool is too small for the request */
  FT_ERR_STATE = 6,     /* call not allowed in the current state (e.g. during capture) */
  FT_ERR_TIMEOUT = 7,   /* a bounded device-side wait gave up */
  FT_ERR_DEVICE = 8     /* the device error word is non-zero */
} ft_status;

/* Expert weight formats.
 *   FT_W_BF16           BF16 weights.
 *   FT_W_FP8_E4M3_B128  E4M3 weights, one FP32 scale per 1x128 block along the reduction
 *                       dimension, applied after the block's dot product ([P3] §4.2).
 *   FT_W_NVFP4          E2M1 (FP4) weights packed two per byte (element 2j in the low
 *                       nibble), one E4M3 scale per 1x16 block along the reduction
 *                       dimension applied after the block's dot product, then one FP32
 *                       tensor scale per bank of each expert ([FT] 主结果 names NVFP4
 *                       experts).
 *   FT_W_MXFP4          E2M1 weights packed as for NVFP4, one E8M0 scale (2^(code-127))
 *                       per 1x32 block along the reduction dimension, applied after the
 *                       block's dot product; no tensor scale ([FT] 主结果: MXFP4 checkpoints).
 * Prefill decodes FP8 and FP4 weights to BF16 in shared memory (each weight times its block
 * scale in FP32, rounded once) before the tensor-core product: the block-scaled tensor-core
 * forms take FP8 / FP4 activations, and the activations here are BF16. */
typedef enum { FT_W_BF16 = 0, FT_W_FP8_E4M3_B128 = 1, FT_W_NVFP4 = 2, FT_W_MXFP4 = 3 } ft_wtype;

/* How a decode step moves F-set experts from the host pool into their slots.
 * FT_FILL_KERNEL: one fixed-shape copy kernel on the compute stream, between the
 *   control kernel and the evaluation, reads the device-resident copy list and pulls
 *   bytes from the mapped host pool (16 CTAs of SM loads); the whole step can be
 *   captured into a CUDA graph.  In a multi-layer call the copy can start while the
 *   previous layer's evaluation still runs, when none of its victim slots belongs to
 *   the previous layer-step.
 * FT_FILL_MEMCPY: the host waits for the control kernel, reads the copy list and
 *   issues one cudaMemcpyAsync per bank per filled expert on the transfer stream.
 *   One host synchronisation per layer; not capturable. */
typedef enum { FT_FILL_KERNEL = 0, FT_FILL_MEMCPY = 1 } ft_fill_mode;

/* Rewritten pair id of a C-set pair (executed on the host; row taken from c_partial). */
#define FT_CPU (-1)

/* Bits of the device error word. */
#define FT_DEVERR_NAN_LOGIT 0x1u   /* a NaN router logit (treated as -inf) */
#define FT_DEVERR_BAD_STATE 0x2u   /* residency table inconsistent (should never happen) */
#define FT_DEVERR_TIMEOUT 0x4u     /* a bounded wait gave up */
#define FT_DEVERR_CAPACITY 0x8u    /* a work list overflowed its fixed shape */

typedef struct {
  int n_layers;           /* L: MoE layers */
  int hidden;             /* H: model width (multiple of 256; FP8: of 512) */
  int inter;              /* I: expert intermediate width (multiple of 128) */
  int n_experts;          /* E: routed experts per layer (<= 1024) */
  int top_k;              /* k (<= 16, <= E) */
  int has_shared;         /* 1: one always-on shared expert per layer (weight 1) */
  int wtype;              /* ft_wtype */
  int max_batch;          /* largest decode batch B (<= 64) */
  int max_prefill_tokens; /* largest prefill chunk T (0: no prefill) */
  int cache_slots;        /* S: slots in the HBM pool */
  double bp_gbps;         /* B_P, pinned host -> HBM GB/s; <= 0: measured at init */
  double bh_gbps;         /* B_H, host-side expert processing GB/s (supplied) */
  int fill_mode;          /* ft_fill_mode */
  int device;             /* CUDA device ordinal */
  void* compute_stream;   /* cudaStream_t, or NULL for a library-created stream */
  void* transfer_stream;  /* cudaStream_t, or NULL for a library-created stream */
} ft_moe_config;

/* Host expert banks ([FT] "FTW 权重格式与平台适配": first dimension of every bank is
 * the logical id; rows with the same id form one expert).  Row-major:
 *   gate, up   [L*E][I][H]        BF16 bits (uint16), E4M3 codes (uint8), or NVFP4:
 *                                 [L*E][I][H/2] packed E2M1 codes
 *   down       [L*E][H][I]        (NVFP4: [L*E][H][I/2])
 *   gate_scale, up_scale [L*E][I][H/128] FP32 (FP8 only; NULL otherwise)
 *   down_scale [L*E][H][I/128]           FP32 (FP8 only)
 *   gate_bscale, up_bscale [L*E][I][H/16] E4M3 codes (NVFP4), [L*E][I][H/32] E8M0 codes
 *                                          (MXFP4); NULL otherwise
 *   down_bscale [L*E][H][I/16] (NVFP4) or [L*E][H][I/32] (MXFP4)
 *   tensor_scale [L*E][4] FP32: gate, up, down, unused (NVFP4 only)
 * For the shared-expert banks the first dimension is L (one per layer). */
typedef struct {
  const void* gate;
  const void* up;
  const void* down;
  const float* gate_scale;
  const float* up_scale;
  const float* down_scale;
  const uint8_t* gate_bscale;
  const uint8_t* up_bscale;
  const uint8_t* down_bscale;
  const float* tensor_scale;
} ft_banks;

typedef struct ft_moe ft_moe;
typedef struct ft_graph ft_graph;

typedef struct {
  uint64_t hits, misses, fills, cpu_execs, evictions;
  uint64_t decode_steps, prefill_layers;
  uint64_t eval_entries;  /* decode: experts evaluated on the GPU (G entries + shared), summed over steps */
  uint64_t eval_pairs;    /* decode: (expert, token) pairs evaluated on the GPU, summed over steps */
  uint32_t error_word;  /* FT_DEVERR_* bits */
  uint32_t clock;       /* global LRU clock (one tick per layer-step) */
  double bp_gbps, bh_gbps;
  int cache_slots;
  int32_t batch1_fused; /* 1: batch-1 steps run the persistent one-launch GEMV (its grid fits on
                           the device, checked at init); 0: they run the batched kernels */
} ft_stats;

/* Last decode layer-step's decisions, for parity checks.  The caller provides
 * host arrays of the stated sizes (K = min(max_batch*top_k, n_experts)); any
 * pointer may be NULL to skip that array. */
typedef struct {
  int layer, batch, q, n_active, n_hit, n_miss, n_victims, n_cpu;
  uint32_t clock;
  int32_t* sel;          /* [batch*top_k] expert ids, ascending per token */
  float* gates;          /* [batch*top_k] gates (ft_gate of ft_moe_set_router) */
  int32_t* slot_of_pair; /* [batch*top_k] slot id, or FT_CPU */
  int32_t* active;       /* [K] A: sorted unique logical ids */
  int32_t* hit;          /* [K] H, ascending */
  int32_t* miss;         /* [K] M, ascending; F = first q, C = the rest */
  int32_t* victims;      /* [K] LRU candidates, ascending (stamp, slot); first q used */
} ft_step_trace;

/* Per-kernel CUDA-event timing collected while profiling is on. */
typedef struct {
  uint64_t launches[10]; /* 0 control, 1 fill, 2 gemv phase 1 (gate/up), 3 gemv phase 2 (down)
                            + combine, 4 prefill routing (route, scan, place), 5 prefill grouped
                            GEMM gate/up + SwiGLU, 6 prefill combine, 7 prefill layer copy,
                            8 prefill grouped GEMM down + gate weighting, 9 router logits */
  double total_ms[10];
} ft_profile;

/* Create the library state: allocates the slot pool (S * slot bytes) and the work
 * buffers in HBM, copies the shared experts to HBM, and registers (pins + maps)
 * each host bank with cudaHostRegister unless it is already pinned.
 * On any error everything allocated or registered so far is released (ft_test_inject_failure
 * makes these paths testable).
 *   cfg      configuration (copied)
 *   host_pool routed-expert banks, caller-owned, must outlive the handle
 *   shared   shared-expert banks (first dim L) or NULL when cfg->has_shared == 0
 *   out      receives the handle
 * Errors: FT_ERR_INVALID (shape limits above), FT_ERR_NOMEM, FT_ERR_PIN (no
 * fallback path), FT_ERR_CUDA.  Synchronises. */
ft_status ft_moe_init(const ft_moe_config* cfg, const ft_banks* host_pool, const ft_banks* shared,
                      ft_moe** out);

/* In-step host evaluation of the C set ([FT] "Device-side 缓存控制": the host branch of a
 * layer-step runs inside the step, and only its result joins the GPU's).  When a hook is
 * set, every decode layer-step enqueues after its control kernel: a copy of the step's
 * routing (sel, gates and slot_of_pair, where FT_CPU marks the C pairs) into pinned host
 * memory, a call of the hook in stream order (cudaLaunchHostFunc, on a driver thread;
 * graph-capturable as a host node), and a copy of the rows the hook wrote back to the
 * device, which then serve as the step's c_partial (the c_partial argument is ignored and
 * may be NULL).  The hook must write rows[(t*top_k + r)*H .. +H) = gate-weighted expert
 * output for every pair with slot_of_pair[t*top_k + r] == FT_CPU, may leave other rows
 * unwritten, and must not call CUDA.  Arrays are [batch*top_k] and [batch*top_k*H],
 * row-major; they stay valid only during the call.  The library itself executes no expert
 * arithmetic on the host.  fn = NULL removes the hook.  Errors: FT_ERR_INVALID (null
 * handle), FT_ERR_STATE (called while a graph of this handle is being captured). */
typedef void (*ft_host_hook)(void* user, int layer, int batch, const int32_t* sel, const float* gates,
                             const int32_t* slot_of_pair, float* rows);
ft_status ft_moe_set_host_hook(ft_moe* h, ft_host_hook fn, void* user);

/* One decode layer-step ([FT] "执行顺序与工程细节", "Device-side 缓存控制").
 *   layer     0 <= layer < L
 *   batch     1 <= batch <= max_batch tokens
 *   x_bf16    dev [batch][H] BF16 activations
 *   logits    dev [batch][E] FP32 router logits
 *   c_partial dev [batch][top_k][H] FP32 gate-weighted rows of host-executed pairs;
 *             row (t, r) is read only if that pair lands in the C set.  May be NULL
 *             only when B_H <= B_P (every miss is filled).
 *   out       dev [batch][H] FP32 layer output
 *   rows_out  optional dev [batch][top_k][H] FP32: GPU pair rows (g_r * expert(x_t));
 *             rows of C pairs are left untouched.
 * Enqueues on the compute stream; graph-capturable with FT_FILL_KERNEL. */
ft_status ft_moe_decode_step(ft_moe* h, int layer, int batch, const void* x_bf16, const float* logits,
                             const float* c_partial, float* out, float* rows_out);

/* n_layers consecutive decode layer-steps (layers first_layer .. first_layer+n-1,
 * one token batch), with per-layer inputs packed layer-major:
 * x [n][batch][H], logits [n][batch][E], c_partial [n][batch][k][H], out [n][batch][H],
 * rows_out [n][batch][k][H] or NULL.  Same results as n calls of ft_moe_decode_step.
 * Every layer's logits are an input of the call, complete in stream order before it (a
 * kernel enqueued earlier on the compute stream may write them): the control kernel of a
 * layer after the first takes its routing and cache decisions from them before its
 * dependency wait, while the previous layer is still evaluated. */
ft_status ft_moe_decode_layers(ft_moe* h, int first_layer, int n_layers, int batch, const void* x_bf16,
                               const float* logits, const float* c_partial, float* out, float* rows_out);

/* Same as ft_moe_decode_layers with HOST buffers: copies the inputs into library
 * staging buffers (H2D), runs the layers (through a cached CUDA graph when
 * use_graph != 0 and fill_mode == FT_FILL_KERNEL), copies out back (D2H) and
 * synchronises.  out_host may be NULL (no D2H). */
ft_status ft_moe_decode_layers_host(ft_moe* h, int first_layer, int n_layers, int batch,
                                    const void* x_host, const float* logits_host,
                                    const float* c_partial_host, float* out_host, int use_graph);

/* Capture ft_moe_decode_layers(...) with these exact device buffers into a CUDA
 * graph (requires FT_FILL_KERNEL).  Replays re-read the buffers' current contents. */
ft_status ft_moe_graph_capture_decode(ft_moe* h, int first_layer, int n_layers, int batch,
                                      const void* x_bf16, const float* logits, const float* c_partial,
                                      float* out, float* rows_out, ft_graph** g);
/* Enqueue one replay on the handle's compute stream (no host synchronisation).  A prefill
 * chunk in progress on the handle is ended first (the next prefill call starts a new
 * chunk).  Errors: FT_ERR_INVALID (null graph),
 * FT_ERR_STATE (the handle was destroyed, or resized after the capture: capture again),
 * FT_ERR_CUDA (the launch failed). */
ft_status ft_graph_launch(ft_graph* g);
/* Free a captured graph (NULL is a no-op).  Replays already enqueued are not waited for:
 * CUDA keeps an executing graph alive until it completes.  Always returns FT_OK. */
ft_status ft_graph_destroy(ft_graph* g);

/* One prefill layer of a chunk ([FT] "全层双缓冲"): a call that does not continue
 * the previous prefill layer starts a chunk and takes the 2E least recently used
 * slots as two full-layer buffers (chosen on the device; the transfer stream waits for
 * the choice).  Layer l's experts are in buffer (l - first) mod 2; the whole of layer
 * l+1 is copied into the other buffer while layer l's routing and grouped GEMMs run on
 * the compute stream: a copy kernel on the transfer stream (16 SMs) reads the mapped
 * pinned banks over the host link, and the GEMMs take the other SMs meanwhile.  All
 * pairs run on the GPU.
 * When the pool cannot hold two full layers (S < 2E), experts are loaded on demand
 * instead, after the layer's routing: the chunk's resident experts are hits, the
 * others go (ascending id) into the least recently used slots outside the hits, in
 * waves when they outnumber those slots; this path synchronises with the host.
 *   n_tokens  1 <= T <= max_prefill_tokens
 *   x_bf16    dev [T][H] BF16;  logits dev [T][E] FP32;  out dev [T][H] FP32
 * Errors: FT_ERR_CAPACITY when every slot holds an expert of the layer that the chunk
 * uses and a miss remains (on-demand path only). */
ft_status ft_moe_prefill_chunk(ft_moe* h, int layer, int n_tokens, const void* x_bf16, const float* logits,
                               float* out);

/* Ablation switch for the prefill double buffer ([FT] "全层双缓冲" measures the loss
 * when the second buffer is off).  on = 1 (default): layer l+1 streams into the other
 * buffer while layer l computes.  on = 0: each layer's weights are copied at the start
 * of its own call, after all compute enqueued before it (as into a single buffer), and
 * the computation waits for them; residency decisions and outputs are identical either
 * way.  Takes effect at the next prefill call.
 * Errors: FT_ERR_INVALID (null handle). */
ft_status ft_moe_set_prefill_overlap(ft_moe* h, int on);

/* Gate functions of the router: how the k chosen logits of a token become its gates.
 * The choice itself is always the k largest logits (equal logits: lower expert id).
 *   FT_GATE_SOFTMAX_TOPK  g_r = exp(z_r) / sum over the k chosen of exp(z_j)  (default)
 *   FT_GATE_SOFTMAX_ALL   g_r = exp(z_r) / sum over all E experts of exp(z_j)  (not renormalised)
 *   FT_GATE_SIGMOID_TOPK  g_r = s(z_r) / sum over the k chosen of s(z_j),  s = logistic sigmoid */
typedef enum { FT_GATE_SOFTMAX_TOPK = 0, FT_GATE_SOFTMAX_ALL = 1, FT_GATE_SIGMOID_TOPK = 2 } ft_gate;

/* Router of the layers, for the calls that take hidden states instead of logits ([FT2]
 * decode paragraph: the GPU router dedupes the layer's active experts; [P3] §3.3: gate and
 * sort run on the GPU).
 *   w_router_bf16  host [L][E][H] BF16: row e of layer l gives logit e (z = x . row); copied
 *                  into device memory owned by the library.  NULL keeps the weights
 *                  already set (none at init).
 *   gate           ft_gate; applies to every later decode and prefill call, with logits
 *                  given or computed.
 * Synchronises.  Errors: FT_ERR_INVALID (null handle, unknown gate), FT_ERR_STATE (called
 * during a graph capture), FT_ERR_NOMEM, FT_ERR_CUDA. */
ft_status ft_moe_set_router(ft_moe* h, const void* w_router_bf16, int gate);

/* Router logits z[t][e] = sum_h x[t][h] * W_router[layer][e][h]: BF16 products accumulated
 * in FP32 in a fixed order, so the same inputs give the same bits in every call, inside a
 * decode step or not.
 *   n_tokens    1 <= n <= max(max_batch, max_prefill_tokens)
 *   x_bf16      dev [n][H] BF16, 16-byte aligned
 *   logits_out  dev [n][E] FP32
 * Enqueues on the compute stream.  Errors: FT_ERR_INVALID (arguments), FT_ERR_STATE (no
 * router weights set). */
ft_status ft_moe_router_logits(ft_moe* h, int layer, int n_tokens, const void* x_bf16, float* logits_out);

/* ft_moe_decode_step with the router inside the step: a router kernel computes the
 * logits from x (as ft_moe_router_logits) and the step continues on them, in the same
 * chain of kernels and graph-capturable in the same way.
 *   logits_out  optional dev [batch][E] FP32: receives the step's logits; NULL uses a
 *               library buffer.
 * Other arguments and errors as ft_moe_decode_step, plus FT_ERR_STATE (no router weights). */
ft_status ft_moe_decode_step_hidden(ft_moe* h, int layer, int batch, const void* x_bf16, const float* c_partial,
                                    float* out, float* rows_out, float* logits_out);

/* ft_moe_prefill_chunk with the router inside the call: the chunk's logits are computed
 * from x into a library buffer, then the layer proceeds as ft_moe_prefill_chunk.
 * Errors as ft_moe_prefill_chunk, plus FT_ERR_STATE (no router weights). */
ft_status ft_moe_prefill_chunk_hidden(ft_moe* h, int layer, int n_tokens, const void* x_bf16, float* out);

/* Safe-point resize of the slot pool ([FT] "挑战三"; [FT2] paragraph on the memory
 * budget).  Growing adds empty slots.  Shrinking keeps the new_slots most recently
 * used experts (stamp desc, slot asc), drops the rest and moves kept experts from
 * slots >= new_slots into the free slots below, in ascending order.  Outputs of
 * later steps do not change (the host pool stays authoritative).  Synchronises;
 * reallocates the pool when growing.  Errors: FT_ERR_INVALID (new_slots < 1),
 * FT_ERR_NOMEM, FT_ERR_STATE (called while a graph of this handle is being captured). */
ft_status ft_cache_resize(ft_moe* h, int new_slots);

/* Host mirror of the device split rule ([FT] "q* 策略"; [FT2] paragraph on the miss
 * split): q = clamp(round_half_up(m * bp / bh), 1, m) for m > 0, with bp, bh rounded
 * to integer MB/s; q = m when bh <= bp; then q <= evictable.  No GPU needed.
 * Errors: FT_ERR_INVALID (m < 0, evictable < 0, bandwidths <= 0, q_out NULL). */
ft_status ft_split_misses(int m, double bp_gbps, double bh_gbps, int evictable, int* q_out);

/* Pinned host -> HBM copy bandwidth with cudaMemcpyAsync on the current device,
 * timed with CUDA events over `iters` copies of `bytes` (the calibration step,
 * [FT] "q* 策略", "ft bench bw").  Allocates and frees its own buffers; synchronises. */
ft_status ft_bench_bw(size_t bytes, int iters, double* bp_gbps);

/* Counters, error word, clock.  Synchronises the library's streams.  Errors: FT_ERR_INVALID
 * (null handle or out), FT_ERR_CUDA (a CUDA call failed, e.g. after a device fault). */
ft_status ft_moe_get_stats(ft_moe* h, ft_stats* out);

/* Clear the device error word (after a reported FT_DEVERR_* condition has been handled);
 * counters, state and cache contents are kept.  Synchronises.  Errors: FT_ERR_INVALID (null
 * handle), FT_ERR_STATE (called during a capture). */
ft_status ft_moe_reset_error(ft_moe* h);

/* Test controls: they change no result of a correct run and exist so that the error paths
 * can be exercised without faulting a GPU.
 *   FT_TEST_HANDOFF_TIMEOUT_NS  value > 0: the batch-1 persistent GEMV waits for one more h
 *                               row than its CTAs publish, giving up after `value` ns; the
 *                               step then returns with FT_DEVERR_TIMEOUT set and its outputs
 *                               undefined, while routing and cache decisions stay valid.
 *                               0 (default): off.
 * Takes effect for steps enqueued afterwards (graphs capture the value in force).  Errors:
 * FT_ERR_INVALID (null handle, unknown control, negative value). */
typedef enum { FT_TEST_HANDOFF_TIMEOUT_NS = 1 } ft_test_control;
ft_status ft_moe_test_control(ft_moe* h, int what, long long value);

/* Failure injection for tests of the error paths, process-wide: after this call the nth
 * request of the given kind (counted from this call) fails once as if the CUDA runtime had
 * refused it.  FT_INJECT_MALLOC: device allocations of ft_moe_init, ft_cache_resize and
 * ft_moe_set_router (the call returns FT_ERR_NOMEM); FT_INJECT_REGISTER: cudaHostRegister of
 * a host bank in ft_moe_init (FT_ERR_PIN).  nth = 0 disarms.  Errors: FT_ERR_INVALID. */
typedef enum { FT_INJECT_MALLOC = 1, FT_INJECT_REGISTER = 2 } ft_inject_kind;
ft_status ft_test_inject_failure(int kind, int nth);

/* Decisions of the last decode layer-step (see ft_step_trace).  Synchronises. */
ft_status ft_moe_get_step_trace(ft_moe* h, ft_step_trace* out);

/* Copy of the residency state: res [L*E], owner [S], stamp [S] (host arrays, any may
 * be NULL), clock.  Synchronises. */
ft_status ft_moe_get_state(ft_moe* h, int32_t* res, int32_t* owner, uint32_t* stamp, uint32_t* clock);

/* Turn per-kernel CUDA-event timing on (1) or off (0); ft_moe_get_profile reads and
 * (reset != 0) clears the totals.  Timing events are recorded on the stream each
 * kernel is launched on.  A graph captured while profiling is on carries its timing
 * events as graph nodes: reading the profile after a replay adds that replay's kernel
 * times (read after every replay; earlier replays are overwritten).  Synchronises. */
ft_status ft_moe_set_profiling(ft_moe* h, int enable);
ft_status ft_moe_get_profile(ft_moe* h, ft_profile* out, int reset);

/* Replace the compute stream (e.g. to follow a framework's current stream): waits for the
 * handle's work, then uses compute_stream (caller-owned, must outlive its use) or, for
 * NULL, a new library-owned stream.  Graphs captured before are replayed on the new
 * stream.  Errors: FT_ERR_INVALID (null handle), FT_ERR_CUDA. */
ft_status ft_moe_set_stream(ft_moe* h, void* compute_stream);

/* Wait for all work the handle has enqueued (transfer stream, then compute stream).
 * Errors: FT_ERR_INVALID (null handle), FT_ERR_CUDA (an enqueued kernel or copy failed). */
ft_status ft_moe_synchronize(ft_moe* h);

/* Release device memory, streams and host registrations (NULL is a no-op).  Synchronises.
 * Graphs captured on the handle stay valid objects but can no longer be launched
 * (FT_ERR_STATE); free them with ft_graph_destroy.  Always returns FT_OK. */
ft_status ft_moe_destroy(ft_moe* h);

/* Allocation-free layer evaluation.  The pages have no counterpart: this entry point is
 * for callers that cannot call cudaMalloc, such as an engine that reserved all device
 * memory for its own pool at start-up and forbids further allocation, or a plug-in host
 * that only lets a library use memory it was handed.  It evaluates one decode MoE layer
 * whose E routed experts all sit in device memory owned by the caller: top-k softmax
 * routing, grouped SwiGLU evaluation of every routed pair, and the fixed-order combine
 * (shared expert first, then the k rows in ascending expert id).  The result equals what
 * ft_moe_decode_step returns for a cache that holds the whole layer.
 *   experts_dev  dev, E slots of stride S_b = round_up(used, 256) bytes, each laid out
 *                gate [I][H] | up [I][H] | down [H][I] (BF16, 2 B/elem; or E4M3 codes,
 *                1 B/elem, followed by gate_scale [I][H/128] | up_scale [I][H/128] |
 *                down_scale [H][I/128] FP32), used = the sum of those sizes
 *   shared_dev   dev, one slot in the same layout, or NULL (no shared expert)
 *   x_bf16 [batch][H] BF16, logits [batch][E] FP32, out [batch][H] FP32 (dev);
 *   rows_out     optional dev [batch][top_k][H] FP32 gate-weighted pair rows
 *   error_word_out optional dev uint32: receives this call's FT_DEVERR_* bits (for example
 *                FT_DEVERR_NAN_LOGIT for a NaN logit, ranked as -inf), written in stream
 *                order after the output; NULL skips it
 *   stream       cudaStream_t to enqueue on (NULL: legacy default stream)
 * It calls no cudaMalloc, cudaFree or other allocating routine.  All intermediates live
 * in one file-scope device array of 8 MiB that every GPU loading the library holds until
 * the process exits; a request whose intermediates do not fit returns FT_ERR_CAPACITY
 * (e.g. batch * top_k * H * 4 bytes of pair rows alone must stay well below 8 MiB).
 * The first call on a device, with that device current, looks up the array's device
 * address and sets kernel launch limits; make that first call before any stream capture.
 * Every call shares the array and the array keeps the last call's contents (the call
 * resets what must start fresh), so calls that overlap on the GPU -- on different streams,
 * or from several threads -- race with each other: serialise them.
 * Other errors: FT_ERR_INVALID (the ft_moe_init shape limits; batch <= 64), FT_ERR_CUDA.
 * Returns after enqueueing; no error message is stored for ft_last_error. */
ft_status ft_moe_decode_resident_noalloc(int n_experts, int top_k, int hidden, int inter, int wtype,
                                         const void* experts_dev, const void* shared_dev, int batch,
                                         const void* x_bf16, const float* logits, float* out,
                                         float* rows_out, uint32_t* error_word_out, void* stream);

/* Page-locked, device-mapped host memory for expert banks ([FT] "FTW 权重格式与平台适配":
 * banks are exact-size pinned host arrays).  ft_moe_init uses such memory as it is (no
 * registration of its own).
 *   FT_HOST_PINNED      cudaHostAlloc (mapped, portable).  The fill kernel reads it fastest:
 *                       on a GB300 host whose memory a long test run had fragmented, 112 GB/s
 *                       against 48 GB/s (FT_HOST_HUGE_PAGES) and 40 GB/s (malloc'd banks
 *                       registered by ft_moe_init).
 *   FT_HOST_HUGE_PAGES  anonymous memory advised for transparent huge pages, then registered
 *                       (cudaHostRegister, mapped, portable): the copy engine reads it at the
 *                       link rate however fragmented host memory is (211 GB/s, against 62 GB/s
 *                       for registered base pages on the same host).
 * `bytes` > 0; *out receives the host address, which kernels can also use on every device.
 * Errors: FT_ERR_INVALID, FT_ERR_NOMEM (no address space), FT_ERR_PIN (the runtime refused to
 * pin; nothing is kept).  ft_host_free releases memory from ft_host_alloc (NULL: no-op); the
 * caller must first destroy every handle using it.  Errors: FT_ERR_INVALID (not an
 * ft_host_alloc address). */
typedef enum { FT_HOST_PINNED = 0, FT_HOST_HUGE_PAGES = 1 } ft_host_alloc_flags;
ft_status ft_host_alloc(size_t bytes, int flags, void** out);
ft_status ft_host_free(void* p);

/* Thread-local message describing the last error of this thread ("" if none). */
const char* ft_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* FT_MOE_H */
