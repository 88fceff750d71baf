// Per-token top-k routing, shared by the decode control kernel and the prefill router
// ("FreeToken 完全拆解", section "Device-side 缓存控制": routing precedes dedupe).  One
// warp routes one token: the k largest logits (equal logits: lower expert id first) are
// chosen and listed in ascending expert id.  Their gates follow the router's gate
// function (FT_GATE_*): a softmax over the k chosen logits, a softmax over all E logits
// (not renormalised), or the chosen logits' sigmoids normalised to sum 1.  All three
// increase with the logit, so the choice does not depend on the gate function.  NaN
// logits rank as -inf and raise `err`.
//
// Lane l holds the logits of experts l, l+32, l+64, ... as order-preserving 32-bit
// keys.  Each of the k rounds takes the warp-wide largest key with one redux.sync and
// the lowest expert id holding it with a second one, so a round costs two warp
// reductions instead of a shuffle butterfly over (value, id) pairs.
#pragma once

#include <climits>

#include "ft_internal.cuh"

namespace ft {

// float -> uint32 with the same order; -0 is taken as +0 first, so equal logits give equal
// keys (and then the lower expert id wins, as for any tie)
__device__ __forceinline__ uint32_t route_key(float v) {
  const uint32_t u = v == 0.f ? 0u : __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float route_key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// This lane's logits of one token: experts lane, lane+32, ... (-inf past E).
template <int NPL>
__device__ __forceinline__ void load_logits_warp(const float* z, int E, int lane, float (&raw)[NPL]) {
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = lane + 32 * j;
    raw[j] = e < E ? __ldg(z + e) : -INFINITY;
  }
}

// Calls emit(e, gate, rank) once for each of the token's k choices, from the lane that
// holds expert e; rank is e's position among the k choices in ascending expert id.  The
// logits come as this lane's raw values (load_logits_warp).
template <int NPL, typename F>  // logits held per lane: E <= 32*NPL
__device__ __forceinline__ void route_token_warp_loaded(const float (&raw)[NPL], int E, int k, int gate, int lane,
                                                        uint32_t* err, F&& emit) {
  constexpr uint32_t kFull = 0xffffffffu;
  float v[NPL];
  uint32_t key[NPL];
  uint32_t taken = 0;
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = lane + 32 * j;
    float x = -INFINITY;
    key[j] = 0u;  // not an expert: below every logit, never chosen (k <= E)
    if (e < E) {
      x = raw[j];
      if (x != x) {
        x = -INFINITY;
        atomicOr(err, FT_DEVERR_NAN_LOGIT);
      }
      key[j] = route_key(x);
    }
    v[j] = x;
  }
  uint32_t zmax_key = 0;
  for (int r = 0; r < k; ++r) {
    // this lane's best untaken key; equal keys keep the lower j (= lower expert id)
    uint32_t best = 0;
    int bj = 0;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const bool free = !((taken >> j) & 1u);
      if (free && key[j] > best) {
        best = key[j];
        bj = j;
      }
    }
    const uint32_t kmax = __reduce_max_sync(kFull, best);
    // lowest expert id holding kmax (a lane's best is its lowest untaken j with that key)
    const uint32_t cand = (best == kmax && best != 0u) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu;
    const uint32_t emin = __reduce_min_sync(kFull, cand);
    if ((int)(emin & 31u) == lane) taken |= 1u << (emin >> 5);
    if (r == 0) zmax_key = kmax;
  }
  // ranks in ascending expert id: experts are ordered by (j, lane)
  const float zmax = route_key_value(zmax_key);  // the largest chosen logit
  uint32_t below = 0;  // chosen experts with a smaller j, then this j's lower lanes
  float ex[NPL];
  float sum = 0.f;
  if (gate == FT_GATE_SIGMOID_TOPK) {
    // s(z_j) / s(zmax), an exact rewrite of the sigmoid ratio in which no exponential
    // overflows: (1 + e^-zmax) / (1 + e^-z) above zero, e^(z - zmax) (1 + e^zmax) / (1 + e^z)
    // at or below it
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      float w = 0.f;
      if ((taken >> j) & 1u)
        w = zmax > 0.f ? (1.f + expf(-zmax)) / (1.f + expf(-v[j]))
                       : expf(v[j] - zmax) * (1.f + expf(zmax)) / (1.f + expf(v[j]));
      ex[j] = w;
      sum += w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const bool in = gate == FT_GATE_SOFTMAX_ALL ? lane + 32 * j < E : ((taken >> j) & 1u) != 0u;
      const float e = in ? expf(v[j] - zmax) : 0.f;
      ex[j] = e;
      sum += e;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const uint32_t b = __ballot_sync(kFull, (taken >> j) & 1u);
    if ((taken >> j) & 1u) emit(lane + 32 * j, ex[j] / sum, (int)(below + __popc(b & ((1u << lane) - 1u))));
    below += __popc(b);
  }
}

template <int NPL, typename F>
__device__ __forceinline__ void route_token_warp(const float* z, int E, int k, int gate, int lane, uint32_t* err,
                                                 F&& emit) {
  float raw[NPL];
  load_logits_warp<NPL>(z, E, lane, raw);
  route_token_warp_loaded<NPL>(raw, E, k, gate, lane, err, emit);
}

// Dispatch on E (the number of logits each lane holds).
template <typename F>
__device__ __forceinline__ void route_token_any(const float* z, int E, int k, int gate, int lane, uint32_t* err,
                                                F&& emit) {
  if (E <= 32) route_token_warp<1>(z, E, k, gate, lane, err, emit);
  else if (E <= 64) route_token_warp<2>(z, E, k, gate, lane, err, emit);
  else if (E <= 128) route_token_warp<4>(z, E, k, gate, lane, err, emit);
  else if (E <= 256) route_token_warp<8>(z, E, k, gate, lane, err, emit);
  else if (E <= 512) route_token_warp<16>(z, E, k, gate, lane, err, emit);
  else route_token_warp<32>(z, E, k, gate, lane, err, emit);
}

}  // namespace ft
