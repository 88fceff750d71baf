// Internal interface of the prefill path (full-layer double buffering + grouped GEMM).
#pragma once

#include <string>
#include <utility>
#include <vector>

#include "ft_internal.cuh"

namespace ft {

struct PrefillCtx {
  cudaStream_t cs, ts;
  int L, E, K, H, I, S, has_shared, max_tokens, n_sm;
  SlotLayout lay;
  uint8_t* pool;
  const uint8_t* shared_w;
  int32_t* res;
  int32_t* owner;
  uint32_t* stamp;
  DevState* st;
  const uint8_t* bank_host[7];  // host banks (pinned): gate, up, down, then the scale banks
  const uint8_t* bank_dev[7];   // the same banks as the device addresses them (mapped)
  size_t bank_row[7];           // bytes per logical id in each bank
  int n_banks;
  int wtype;                    // ft_wtype of the experts
  bool prof;
  bool overlap;  // stream layer l+1 while layer l computes (the double buffer)
  int gate;      // FT_GATE_*
};

// Arguments of the grouped GEMM (prefill_gemm.cu).  Entries 0..E-1 are the layer's
// routed experts (weights in pool slots buf_slots[e]); entry E, when present, is the
// shared expert (weights in the shared-expert array, row block `layer`).
struct GemmDesc {
  int n_entries, E, layer, I, H;
  int mt;                    // M tiles per entry: gate/up I/64, down H/128
  int kb;                    // K steps of 64: gate/up H/64, down I/64
  const int32_t* entry_off;  // [n_entries+1] first pair of each entry (pairs sorted by entry, token)
  const int32_t* tile_off;   // [n_entries+1] prefix of N tiles per entry
  const int4* tiles;         // [N tiles] {entry, first pair, valid pairs, N (multiple of 16)}
  const int32_t* buf_slots;  // [E]
  const int32_t* pair_tok;   // [P] token of each pair
  const float* pair_gate;    // [P] gate of each pair (1 for the shared expert)
  uint16_t* h;               // [P][I] BF16 (gate/up output)
  uint16_t* rows;            // [P][H] BF16 (down output)
  uint32_t* error_word;
  // FP8 / FP4 experts: where the dequantising warps find each weight row's block scales
  const uint8_t* pool;       // slot pool (routed experts)
  const uint8_t* shared_w;   // shared experts, one slot-layout row block per layer
  size_t stride;             // slot stride in bytes
  size_t off_gs, off_us, off_ds, off_ts;  // scale-bank offsets within a slot
};

// Tensor maps and launch of the grouped GEMM.  mode 0: gate/up + SwiGLU from the token
// rows in pair order (xp); mode 1: down + gate weighting from h.  wtype picks the weight
// form: BF16 tiles go straight to the tensor cores; FP8 and FP4 tiles are decoded to BF16
// in shared memory first.
struct GemmMaps;
cudaError_t gemm_maps_create(GemmMaps** out, const uint8_t* pool, int S, const uint8_t* shared_w, int L, int H,
                             int I, const uint16_t* h_buf, const uint16_t* xp_buf, int max_pairs, int wtype,
                             const SlotLayout& lay);
void gemm_maps_destroy(GemmMaps* m);
cudaError_t launch_grouped_gemm(int mode, const GemmMaps* m, const uint16_t* x, int T, const GemmDesc& d, int grid,
                                cudaStream_t s);

struct PrefillState;

using ProfEvents = std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>>;

cudaError_t prefill_create(PrefillState** out, const PrefillCtx& c);
void prefill_destroy(PrefillState* p);
// Ends an open chunk.  If the next layer was already streaming into a buffer whose
// residency still names the layer before it, that layer's weights are copied back so
// data and residency agree.  Enqueues on the streams of the last prefill call.
void prefill_interrupt(PrefillState* p);
cudaError_t prefill_layer(PrefillState* p, const PrefillCtx& c, int layer, int T, const uint16_t* x,
                          const float* logits, float* out, ProfEvents* prof, std::string* err);
// One prefill layer with experts loaded on demand, for pools smaller than two full layers
// (S < 2E).  Host-synchronising.  Returns cudaErrorNotSupported with *err naming the
// capacity when a miss has no slot outside the layer's hits.
cudaError_t prefill_layer_on_demand(PrefillState* p, const PrefillCtx& c, int layer, int T, const uint16_t* x,
                                    const float* logits, float* out, ProfEvents* prof, std::string* err);

}  // namespace ft
