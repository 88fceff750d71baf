// Per-token top-k softmax routing, shared by the decode control kernel and the
// prefill router ("FreeToken 完全拆解", section "Device-side 缓存控制": routing
// precedes dedupe).  One warp routes one token: the k largest logits (equal logits:
// lower expert id first) are chosen, listed in ascending expert id, and their gates
// are a softmax over those k logits.  NaN logits rank as -inf and raise `err`.
#pragma once

#include <climits>

#include "ft_internal.cuh"

namespace ft {

__device__ __forceinline__ bool route_better(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}

// On return, lane r < k holds the token's rank-r choice: out_e (expert id, ascending in
// r), out_g (gate), out_rank (= r); lanes >= k hold out_rank = -1.
template <int NPL>  // logits held per lane: E <= 32*NPL
__device__ __forceinline__ void route_token_warp(const float* z, int E, int k, int lane, uint32_t* err, int& out_e,
                                                 float& out_g, int& out_rank) {
  float v[NPL];
  uint32_t taken = 0;
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = lane + 32 * j;
    float x = -INFINITY;
    if (e < E) {
      x = __ldg(z + e);
      if (x != x) {
        x = -INFINITY;
        atomicOr(err, FT_DEVERR_NAN_LOGIT);
      }
    } else {
      taken |= 1u << j;  // not an expert
    }
    v[j] = x;
  }
  int my_e = INT_MAX;
  float my_z = -INFINITY, zmax = -INFINITY;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = lane + 32 * j;
      if (!(taken & (1u << j)) && route_better(v[j], e, bv, be)) {
        bv = v[j];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (route_better(ov, oe, bv, be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == r) {
      my_e = be;
      my_z = bv;
    }
    if (r == 0) zmax = bv;
  }
  int rank = 0;
  for (int j = 0; j < k; ++j) {
    const int oe = __shfl_sync(0xffffffffu, my_e, j);
    if (lane < k && oe < my_e) ++rank;
  }
  const float ex = lane < k ? expf(my_z - zmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  out_e = my_e;
  out_g = ex / sum;
  out_rank = lane < k ? rank : -1;
}

// Dispatch on E (the number of logits each lane holds).
template <typename F>
__device__ __forceinline__ void route_token_any(const float* z, int E, int k, int lane, uint32_t* err, F&& emit) {
  int e, rank;
  float g;
  if (E <= 32) route_token_warp<1>(z, E, k, lane, err, e, g, rank);
  else if (E <= 64) route_token_warp<2>(z, E, k, lane, err, e, g, rank);
  else if (E <= 128) route_token_warp<4>(z, E, k, lane, err, e, g, rank);
  else if (E <= 256) route_token_warp<8>(z, E, k, lane, err, e, g, rank);
  else if (E <= 512) route_token_warp<16>(z, E, k, lane, err, e, g, rank);
  else route_token_warp<32>(z, E, k, lane, err, e, g, rank);
  if (rank >= 0) emit(e, g, rank);
}

}  // namespace ft
