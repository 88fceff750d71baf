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
  const uint8_t* bank_host[3];  // gate, up, down host banks (pinned)
  size_t bank_row[3];
  bool prof;
};

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

}  // namespace ft
