// Internal definitions of libftmoe (device structs, limits, kernel entry points).
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <utility>

#include "ft_moe.h"

namespace ft {

constexpr int kMaxE = 1024;           // routed experts per layer
constexpr int kMaxK = 16;             // top-k
constexpr int kMaxBatch = 64;         // decode tokens per step
constexpr int kMaxPairs = kMaxBatch * kMaxK;
constexpr int kCtrlThreads = 512;     // decode control kernel (one CTA)
constexpr int kEvalThreads = 256;     // GEMV CTAs: 8 warps
constexpr int kRowsPerItem2 = 32;     // down-projection rows per work item (= combine block)
constexpr uint32_t kSpinLimit = 1u << 22;

// Device-resident counters and clock of one handle.
struct DevState {
  uint32_t clock;
  uint32_t error_word;
  unsigned long long hits, misses, fills, cpu_execs, evictions;
  unsigned long long decode_steps, prefill_layers;
  unsigned long long eval_entries, eval_pairs;  // G entries (+shared) and (entry, token) pairs evaluated
};

// Indices into DecodeWork::counts (written by the control kernel, read by the
// fill / evaluation kernels and by the host for traces).
enum CountIdx {
  C_NACTIVE = 0, C_NHIT, C_NMISS, C_Q, C_NVICT, C_NG, C_NENTRIES, C_NGPAIRS,
  C_LAYER, C_BATCH, C_CLOCK, C_EVICT, C_NCOUNTS = 16
};

// Fixed-shape work lists of a decode layer-step.  One set per handle; every
// layer-step overwrites it, and the valid counts tell kernels how much is live.
struct DecodeWork {
  int32_t* sel;            // [maxB*k] expert ids, ascending per token
  float* gates;            // [maxB*k]
  int32_t* slot_of_pair;   // [maxB*k] slot, or FT_CPU
  int32_t* active;         // [Kmax] A (logical ids)
  int32_t* hit;            // [Kmax]
  int32_t* miss;           // [Kmax]
  int32_t* victims;        // [Kmax]
  int32_t* copy_u;         // [Kmax] F: logical id to fill
  int32_t* copy_slot;      // [Kmax] F: destination slot
  int32_t* counts;         // [C_NCOUNTS]
  // Evaluation entries: 0..n_g-1 are G = H u F in ascending logical id; entry
  // n_g is the shared expert when the model has one.
  const uint8_t** g_w;     // [Kmax+1] base address of the entry's weights
  int32_t* g_fill;         // [Kmax+1] 1 if the entry's slot is being filled in this step
  uint32_t* ready;         // [Kmax+1] batch-1 fused kernel: h rows published per entry (zeroed by control)
  int32_t* g_off;          // [Kmax+2] prefix offsets into g_pair
  int32_t* g_pair;         // [maxB*k + maxB] routed: pair id t*k+r; shared: token t
  float* h;                // [(maxB*k + maxB) * I] intermediate, indexed like g_pair
  float* rows;             // [maxB*k*H] GPU pair rows when the caller gives no rows_out
  float* shared_rows;      // [maxB*H]
  uint32_t* blk_count;     // [H / kRowsPerItem2] combine arrival counters (self-resetting)
  // Copy list taken before the control kernel's dependency wait, two buffers by the parity of
  // the step's clock: {clock (written last, release), q, ids[kmax], slots[kmax]}
  int32_t* ecopy;
  int kmax;                // capacity of the per-expert lists
};

// Byte layout of one slot: gate | up | down [| gate_scale | up_scale | down_scale].
struct SlotLayout {
  size_t gate, up, down, gs, us, ds;  // byte offsets
  size_t gate_b, down_b, gs_b, ds_b;  // byte sizes (up == gate, us == gs)
  size_t ts, ts_b;                    // NVFP4 tensor scales (4 FP32), else ts_b == 0
  size_t used, stride;                // bytes used, slot stride (256-aligned)
};

SlotLayout make_layout(int wtype, int H, int I);

struct CtrlParams {
  const float* logits;
  int B, E, k, layer, S, kcap, has_shared;
  int gate;  // FT_GATE_*
  long long bp_mbs, bh_mbs;
  int32_t* res;
  int32_t* owner;
  uint32_t* stamp;
  DevState* st;
  DecodeWork w;
  const uint8_t* pool;
  size_t slot_stride;
  const uint8_t* shared_w;  // shared expert of this layer, or nullptr
  bool pdl;                 // launched as a programmatic dependent
  // the logits were complete before the kernel right before this one started (a later layer
  // of one multi-layer call): they may be read before the dependency wait
  bool logits_early;
};

struct FillParams {
  const int32_t* counts;
  const int32_t* copy_u;
  const int32_t* copy_slot;
  uint8_t* pool;
  SlotLayout lay;
  const uint8_t* src[7];    // device-visible addresses of the host banks
  size_t src_row[7];        // bytes per logical id in each bank
  int n_banks;
  bool pdl;
  const int32_t* ecopy;     // DecodeWork::ecopy (nullptr: no early start)
  const DevState* st;       // the step clock: st->clock + 1 while the step's control kernel runs
  int kmax;
};

struct EvalParams {
  const int32_t* counts;
  const uint8_t* const* g_w;
  const int32_t* g_fill;
  uint32_t* ready;          // [entries] h rows published per entry (batch-1 fused kernel)
  const int32_t* g_off;
  const int32_t* g_pair;
  const float* gates;
  const int32_t* slot_of_pair;
  const uint16_t* x;        // [B][H] bf16
  float* h;
  float* rows;              // [B*k][H]
  float* shared_rows;       // [B][H]
  const float* c_partial;   // [B*k][H] or nullptr
  float* out;               // [B][H]
  uint32_t* blk_count;
  uint32_t* error_word;
  SlotLayout lay;
  int H, I, k, B, has_shared;
  int n_sm;                 // CTAs of the batch-1 GEMV (one per SM it may use)
  int max_entries;          // capacity of the entry lists (kcap + 1)
  bool pdl;                 // launched as programmatic dependents
  bool allow_fused;         // batch 1 may run the persistent one-launch kernel (its grid fits)
  uint32_t wait_extra;      // added to the batch-1 hand-off target: 0, or 1 in the timeout test
  unsigned long long wait_ns;  // limit of the batch-1 hand-off wait
};

// Limit of the batch-1 kernel's wait for the h rows of other CTAs: a lost signal sets
// FT_DEVERR_TIMEOUT and the kernel returns instead of hanging.
constexpr unsigned long long kHandoffWaitNs = 2000000000ull;  // 2 s

// Programmatic dependent launch.  Kernels of the decode chain (control -> fill -> gate/up
// -> down+combine -> next control) are launched with programmatic stream serialization.
// Each kernel triggers its dependents only after its own wait, so when kernel n+1 starts,
// kernel n-1 has completed: a prologue may read what kernels two or more back wrote, and
// must wait before reading what the previous kernel wrote.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` with the programmatic-serialization attribute when `pdl` is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct RouterParams {
  const uint16_t* x;  // [T][H] BF16 hidden states
  const uint16_t* w;  // [E][H] BF16 router projection of the layer
  float* z;           // [T][E] FP32 logits
  int T, E, H;
  int tok_tile;       // token rows staged per CTA
  int e_per_warp;     // router rows per warp
  bool pdl;
};

// Fill kernel shape: CTAs (SMs) that carry the host-link copy, threads per CTA, and the
// shared memory each reserves so that no batch-1 GEMV CTA (~150 KB) shares its SM.
constexpr int kFillSms = 16;
constexpr int kFillThreads = 512;
constexpr size_t kFillSmemReserve = 120 * 1024;

// Kernel launchers (stream-ordered, no synchronisation).
cudaError_t launch_control(const CtrlParams& p, cudaStream_t s);
// Router logits (router.cu): launch shape for T tokens, then the launch.
void router_shape(int T, int E, int H, int* tok_tile, int* e_per_warp);
size_t router_smem_bytes(int tok_tile, int H);
cudaError_t launch_router(const RouterParams& p, cudaStream_t s);
cudaError_t prepare_router();
// Raise the control kernel's shared-memory limit (call once per device, before capture).
cudaError_t prepare_control();
cudaError_t launch_fill(const FillParams& p, int grid, cudaStream_t s);
cudaError_t launch_gate_up(const EvalParams& p, int wtype, int grid, cudaStream_t s);
cudaError_t launch_down_combine(const EvalParams& p, int wtype, int grid, cudaStream_t s);
// Set the dynamic shared-memory limits of every evaluation kernel (call once, before capture).
cudaError_t prepare_kernels(int wtype, int H, int I);
// Batch-1 decode evaluation in one persistent launch (decode_fused.cu).
bool fused_gemv_supported(int wtype, int H, int I, int max_entries, int n_sm);
// True when one CTA of the batch-1 kernel fits on an SM (occupancy >= 1), so that its grid of
// n_sm CTAs can be resident at once on an idle device.
bool fused_gemv_fits(int wtype, int H, int I, int max_entries, int n_sm);
cudaError_t launch_fused_gemv(const EvalParams& p, int wtype, int n_sm, int max_entries, cudaStream_t s);
cudaError_t prepare_fused_gemv();
// Entries of a batch-1 step: at most k routed experts plus the shared expert.
inline int batch1_entries(const EvalParams& p) { return p.max_entries < p.k + 1 ? p.max_entries : p.k + 1; }
// True when launch_gate_up runs the whole layer (launch_down_combine then launches nothing).
bool eval_fused(const EvalParams& p, int wtype);

}  // namespace ft
