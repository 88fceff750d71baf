// Per-layer decode control kernel: one CTA does every routing-dependent decision of
// a decode layer-step on the device, so the step needs no host synchronisation and
// can replay inside a CUDA graph.
//
// Order of work ("FreeToken 完全拆解", section "Device-side 缓存控制"):
//   route (top-k softmax per token) -> dedupe over the batch -> classify against the
//   residency table -> fill count q -> one scan for the K least recently used slots
//   -> install the first q misses in the first q victims -> rewrite routed ids to
//   slots or FT_CPU -> fixed-shape evaluation lists with device-resident counts.
// Split rule: "FreeToken 完全拆解", section "q* 策略"; residual bandwidth
// max(B_H-B_P, 0): "개인 장치에서 MoE 모델을 서빙하는 FreeToken", paragraph on the miss split.
#include <cfloat>
#include <climits>

#include "ft_internal.cuh"
#include "ft_route.cuh"

namespace ft {
namespace {


// Fill count: q = clamp(floor(m*bp/bh + 1/2), 1, m) for m > 0; all misses when the
// residual bandwidth B_H - B_P is not positive; never more than `evictable`.
__device__ __forceinline__ int split_q(int m, long long bp, long long bh, int evictable) {
  if (m <= 0) return 0;
  long long q;
  if (bh <= bp) {
    q = m;
  } else {
    q = (2LL * m * bp + bh) / (2LL * bh);
    if (q < 1) q = 1;
  }
  if (q > m) q = m;
  if (q > evictable) q = evictable;
  return q < 0 ? 0 : (int)q;
}

constexpr int kRegJ = 16;      // stamps per thread held in registers (S <= 16K)
constexpr int kDigit = 11;     // radix-select digit
constexpr int kBins = 1 << kDigit;

__global__ void __launch_bounds__(kCtrlThreads, 1) control_kernel(CtrlParams p) {
  __shared__ uint32_t s_bitmap[kMaxE / 32];
  __shared__ int s_sel[kMaxPairs];
  __shared__ int s_active[kMaxE];
  __shared__ int s_hit[kMaxE];
  __shared__ int s_miss[kMaxE];
  __shared__ int s_gidx[kMaxE];
  __shared__ int s_victims[kMaxE];
  __shared__ int s_res[kMaxE];                         // res[] of this layer's experts
  __shared__ uint32_t s_hitbits[kRegJ * kCtrlThreads / 32];  // hit slots (register-stamp path)
  __shared__ uint32_t s_wsum[32];
  __shared__ uint8_t s_fflag[kMaxE];                   // expert of this layer filled in this step
  extern __shared__ unsigned long long s_dyn[];
  unsigned long long* s_vkeys = s_dyn;                 // [kMaxE]
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(s_dyn + kMaxE);  // [kBins]
  __shared__ int s_gcount[kMaxE + 1];
  __shared__ uint32_t s_err;
  __shared__ uint32_t s_clock;
  __shared__ int s_nactive, s_nhit, s_nmiss, s_q, s_nv, s_ng, s_evict, s_ncand;
  __shared__ unsigned long long s_prefix;
  __shared__ int s_kk;
  __shared__ uint32_t s_lo, s_hi;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, k = p.k, B = p.B, S = p.S;
  const int base_u = p.layer * E;

  // State loads first, so their latency overlaps the routing: this layer's residency
  // slice to shared memory, slot stamps to registers (S <= 16K slots).
  const bool in_reg = S <= kRegJ * kCtrlThreads;
  uint32_t rs[kRegJ];
#pragma unroll
  for (int j = 0; j < kRegJ; ++j) {
    const int s = tid + j * kCtrlThreads;
    rs[j] = (in_reg && s < S) ? p.stamp[s] : UINT_MAX;
  }
  for (int i = tid; i < E; i += blockDim.x) s_res[i] = p.res[base_u + i];
  for (int i = tid; i < kMaxE / 32; i += blockDim.x) s_bitmap[i] = 0;
  for (int i = tid; i < kRegJ * kCtrlThreads / 32; i += blockDim.x) s_hitbits[i] = 0;
  for (int i = tid; i < E; i += blockDim.x) {
    s_gidx[i] = -1;
    s_fflag[i] = 0;
  }
  // Everything above reads state the previous control kernel wrote (it has completed);
  // logits and the work lists belong to the kernel right before this one: wait for it.
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    s_err = 0;
    s_clock = p.st->clock + 1u;
    s_evict = 0;
    s_nv = 0;
    s_lo = UINT_MAX;
    s_hi = 0;
    s_ncand = 0;
  }
  __syncthreads();
  const uint32_t clock = s_clock;

  // ---- 1. route: one warp per token
  for (int t = warp; t < B; t += blockDim.x / 32) {
    route_token_any(p.logits + (size_t)t * E, E, k, lane, &s_err, [&](int e, float g, int rank) {
      const int idx = t * k + rank;
      p.w.sel[idx] = e;
      p.w.gates[idx] = g;
      s_sel[idx] = e;
      atomicOr(&s_bitmap[e >> 5], 1u << (e & 31));
    });
  }
  __syncthreads();

  // ---- 2. dedupe + classify (warp 0; A is at most min(B*k, E) ids)
  if (warp == 0) {
    const int nwords = (E + 31) / 32;
    uint32_t word = lane < nwords ? s_bitmap[lane] : 0u;
    int cnt = __popc(word), incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int pos = incl - cnt;
    while (word) {
      int b = __ffs(word) - 1;
      word &= word - 1;
      s_active[pos++] = base_u + lane * 32 + b;
    }
    const int nact = __shfl_sync(0xffffffffu, incl, 31);
    int nh = 0, nm = 0;
    for (int c = 0; c < nact; c += 32) {
      int i = c + lane;
      int u = i < nact ? s_active[i] : -1;
      int slot = u >= 0 ? s_res[u - base_u] : -1;
      if (slot >= S) {  // cannot happen with a consistent table
        atomicOr(&s_err, FT_DEVERR_BAD_STATE);
        slot = -1;
      }
      bool valid = i < nact, hit = valid && slot >= 0;
      uint32_t hb = __ballot_sync(0xffffffffu, hit);
      uint32_t mb = __ballot_sync(0xffffffffu, valid && !hit);
      uint32_t lt = (1u << lane) - 1u;
      if (hit) {
        s_hit[nh + __popc(hb & lt)] = u;
        p.stamp[slot] = clock;  // hit refreshes recency
        if (in_reg) atomicOr(&s_hitbits[slot >> 5], 1u << (slot & 31));
      } else if (valid) {
        s_miss[nm + __popc(mb & lt)] = u;
      }
      nh += __popc(hb);
      nm += __popc(mb);
    }
    if (lane == 0) {
      s_nactive = nact;
      s_nhit = nh;
      s_nmiss = nm;
      s_q = split_q(nm, p.bp_mbs, p.bh_mbs, S - nh);
    }
  }
  __syncthreads();

  const int q = s_q;
  const int kcap = p.kcap;

  // ---- 3. one-pass K-LRU victim scan over slots not hit in this step
  if (q > 0) {
    // register stamps were read before this step's hits refreshed them: hits are excluded
    // through s_hitbits instead
#define FOR_CANDIDATES(...)                                          \
  if (in_reg) {                                                      \
    _Pragma("unroll") for (int j = 0; j < kRegJ; ++j) {              \
      const int s = tid + j * kCtrlThreads;                          \
      const uint32_t st = rs[j];                                     \
      if (s < S && st < clock && !((s_hitbits[s >> 5] >> (s & 31)) & 1u)) { __VA_ARGS__ } \
    }                                                                \
  } else {                                                           \
    for (int s = tid; s < S; s += kCtrlThreads) {                    \
      const uint32_t st = p.stamp[s];                                \
      if (st < clock) { __VA_ARGS__ }                                \
    }                                                                \
  }
    // range of candidate stamps and their count
    uint32_t lo = UINT_MAX, hi = 0;
    int nc = 0;
    FOR_CANDIDATES(lo = min(lo, st); hi = max(hi, st); ++nc;)
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      nc += __shfl_xor_sync(0xffffffffu, nc, o);
    }
    if (lane == 0) {
      atomicMin(&s_lo, lo);
      atomicMax(&s_hi, hi);
      atomicAdd(&s_ncand, nc);
    }
    __syncthreads();
    const uint32_t st_lo = s_lo;
    const int ncand = s_ncand;
    const int want = min(kcap, ncand);
    const int sbits = S > 1 ? 32 - __clz((unsigned)(S - 1)) : 1;
    const uint32_t range = s_hi - st_lo;
    const int width = (range ? 32 - __clz(range) : 0) + sbits;  // <= 52 bits
    // key = (stamp - lowest stamp, slot): unique, ordered like (stamp, slot)
#define KEY_OF(s, st) ((((unsigned long long)((st) - st_lo)) << sbits) | (unsigned long long)(s))
    unsigned long long thresh = ~0ull;
    if (want < ncand) {
      // radix select of the want-th smallest key, kDigit bits per pass, most significant first
      const int passes = (width + kDigit - 1) / kDigit;
      if (tid == 0) {
        s_prefix = 0;
        s_kk = want;
      }
      for (int ps = passes - 1; ps >= 0; --ps) {
        const int shift = ps * kDigit;
        for (int i = tid; i < kBins; i += kCtrlThreads) s_hist[i] = 0;
        __syncthreads();
        const unsigned long long pre = s_prefix;
        FOR_CANDIDATES(const unsigned long long key = KEY_OF(s, st);
                       if ((key >> (shift + kDigit)) == pre) atomicAdd(&s_hist[(key >> shift) & (kBins - 1)], 1u);)
        __syncthreads();
        {
          // block-wide exclusive scan: thread t owns bins 2t and 2t+1
          const uint32_t h0 = s_hist[2 * tid], h1 = s_hist[2 * tid + 1], v = h0 + h1;
          uint32_t incl = v;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          if (lane == 31) s_wsum[warp] = incl;
          __syncthreads();
          if (warp == 0) {
            uint32_t ws = s_wsum[lane], wi = ws;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
              if (lane >= o) wi += y;
            }
            s_wsum[lane] = wi - ws;  // exclusive prefix of warp totals
          }
          __syncthreads();
          const uint32_t kk = (uint32_t)s_kk;
          const uint32_t excl = s_wsum[warp] + incl - v;
          if (excl < kk && excl + v >= kk) {  // exactly one thread
            const bool first = excl + h0 >= kk;
            const uint32_t run = first ? excl : excl + h0;
            s_prefix = (pre << kDigit) | (unsigned long long)(2 * tid + (first ? 0 : 1));
            s_kk = (int)(kk - run);
          }
        }
        __syncthreads();
      }
      thresh = s_prefix;
    }
    // collect the `want` smallest keys (keys are unique), then order them
    FOR_CANDIDATES(const unsigned long long key = KEY_OF(s, st); if (key <= thresh) {
      const int i = atomicAdd(&s_nv, 1);
      if (i < kMaxE) s_vkeys[i] = key;
    })
#undef FOR_CANDIDATES
#undef KEY_OF
    __syncthreads();
    const int nv = min(s_nv, want);
    const unsigned long long smask = (1ull << sbits) - 1ull;
    for (int i = tid; i < nv; i += kCtrlThreads) {
      const unsigned long long ki = s_vkeys[i];
      int rank = 0;
      for (int j = 0; j < nv; ++j) rank += s_vkeys[j] < ki;
      s_victims[rank] = (int)(ki & smask);
    }
    if (tid == 0) s_nv = nv;
    __syncthreads();

    // ---- 4. install F = first q misses into the first q victims
    for (int i = tid; i < q; i += blockDim.x) {
      int v = s_victims[i];
      int u = s_miss[i];
      int old = p.owner[v];
      if (old >= 0) {
        p.res[old] = -1;
        atomicAdd(&s_evict, 1);
      }
      p.owner[v] = u;
      p.res[u] = v;
      s_res[u - base_u] = v;
      s_fflag[u - base_u] = 1;
      p.stamp[v] = clock;
      p.w.copy_u[i] = u;
      p.w.copy_slot[i] = v;
    }
  }
  __syncthreads();

  // ---- 5. G = resident part of A (ascending u): evaluation entries
  if (warp == 0) {
    const int nact = s_nactive;
    int ng = 0;
    for (int c = 0; c < nact; c += 32) {
      int i = c + lane;
      int u = i < nact ? s_active[i] : -1;
      int slot = u >= 0 ? s_res[u - base_u] : -1;
      bool in = slot >= 0;
      uint32_t b = __ballot_sync(0xffffffffu, in);
      if (in) {
        int g = ng + __popc(b & ((1u << lane) - 1u));
        s_gidx[u - base_u] = g;
        p.w.g_w[g] = p.pool + (size_t)slot * p.slot_stride;
        p.w.g_fill[g] = s_fflag[u - base_u];
      }
      ng += __popc(b);
    }
    if (lane == 0) s_ng = ng;
  }
  for (int i = tid; i <= kMaxE; i += blockDim.x) s_gcount[i] = 0;
  __syncthreads();
  const int ng = s_ng;

  // rewrite pairs to slots / FT_CPU and count pairs per entry
  const int npairs = B * k;
  for (int pi = tid; pi < npairs; pi += blockDim.x) {
    int e = s_sel[pi];
    int g = s_gidx[e];
    p.w.slot_of_pair[pi] = g >= 0 ? s_res[e] : FT_CPU;
    if (g >= 0) atomicAdd(&s_gcount[g], 1);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of per-entry pair counts -> g_off
    int carry = 0;
    for (int c = 0; c < ng; c += 32) {
      int i = c + lane;
      int v = i < ng ? s_gcount[i] : 0, incl = v;
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (i < ng) {
        p.w.g_off[i] = carry + incl - v;
        s_gcount[i] = carry + incl - v;  // becomes the offset
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      p.w.g_off[ng] = carry;
      s_gcount[ng] = carry;
      int ne = ng;
      if (p.has_shared) {
        p.w.g_w[ng] = p.shared_w;
        p.w.g_fill[ng] = 0;
        p.w.g_off[ng + 1] = carry + B;
        ne = ng + 1;
      }
      int* cnt = p.w.counts;
      cnt[C_NACTIVE] = s_nactive;
      cnt[C_NHIT] = s_nhit;
      cnt[C_NMISS] = s_nmiss;
      cnt[C_Q] = q;
      cnt[C_NVICT] = q > 0 ? s_nv : 0;
      cnt[C_NG] = ng;
      cnt[C_NENTRIES] = ne;
      cnt[C_NGPAIRS] = carry;
      cnt[C_LAYER] = p.layer;
      cnt[C_BATCH] = B;
      cnt[C_CLOCK] = (int)clock;
      cnt[C_EVICT] = s_evict;
    }
  }
  __syncthreads();
  // place pairs: within an entry, ascending pair id
  for (int pi = tid; pi < npairs; pi += blockDim.x) {
    int e = s_sel[pi];
    int g = s_gidx[e];
    if (g < 0) continue;
    int pos = 0;
    for (int j = 0; j < pi; ++j) pos += (s_sel[j] == e);
    p.w.g_pair[s_gcount[g] + pos] = pi;
  }
  if (p.has_shared) {
    const int base = s_gcount[ng];
    for (int t = tid; t < B; t += blockDim.x) p.w.g_pair[base + t] = t;
  }
  // lists for traces
  for (int i = tid; i < s_nactive; i += blockDim.x) p.w.active[i] = s_active[i];
  for (int i = tid; i < s_nhit; i += blockDim.x) p.w.hit[i] = s_hit[i];
  for (int i = tid; i < s_nmiss; i += blockDim.x) p.w.miss[i] = s_miss[i];
  if (q > 0)
    for (int i = tid; i < s_nv; i += blockDim.x) p.w.victims[i] = s_victims[i];
  if (tid == 0) {
    DevState* st = p.st;
    st->clock = clock;
    st->hits += (unsigned long long)s_nhit;
    st->misses += (unsigned long long)s_nmiss;
    st->fills += (unsigned long long)q;
    st->cpu_execs += (unsigned long long)(s_nmiss - q);
    st->evictions += (unsigned long long)s_evict;
    st->decode_steps += 1ull;
    st->eval_entries += (unsigned long long)(s_ng + (p.has_shared ? 1 : 0));
    st->eval_pairs += (unsigned long long)(s_gcount[s_ng] + (p.has_shared ? B : 0));
    if (s_err) atomicOr(&st->error_word, s_err);
  }
}

}  // namespace

constexpr size_t kCtrlDynSmem = kMaxE * sizeof(unsigned long long) + kBins * sizeof(uint32_t);

cudaError_t launch_control(const CtrlParams& p, cudaStream_t s) {
  return launch_k(control_kernel, dim3(1), dim3(kCtrlThreads), kCtrlDynSmem, s, p.pdl, p);
}

cudaError_t prepare_control() {
  return cudaFuncSetAttribute(control_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCtrlDynSmem);
}

}  // namespace ft
