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
//
// The kernel is latency-bound and its code is fetched cold on every launch (the weight
// streams of the evaluation kernels pass through L2 in between), so it is kept compact:
// one router width per instantiation, plain loops, slot stamps staged once in shared
// memory, and a radix select that stops as soon as the selected bin holds exactly the
// keys still wanted.
#include <cfloat>
#include <climits>

#include "ft_internal.cuh"
#include "ft_ptx.cuh"
#include "ft_route.cuh"

namespace ft {
namespace {

constexpr int kThreads = kCtrlThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kDigit = 9;  // radix-select digit: one histogram bin per thread
constexpr int kBins = 1 << kDigit;
static_assert(kBins == kThreads, "one histogram bin per thread");
constexpr int kSmemSlots = 16384;  // slot stamps staged in shared memory up to this many slots
constexpr int kSmemOwners = 8192;  // slot owners staged too up to this many slots
constexpr size_t kDynSmemMax = kMaxE * sizeof(unsigned long long) + kSmemSlots * sizeof(uint32_t);
static_assert(kSmemOwners * 2 <= kSmemSlots, "owners share the stamp area's budget");

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

constexpr int kTour = 16;  // victim lists up to this length take the warp tournament

// Warp-wide minimum of a 64-bit key: high halves first, then the low halves that tie.
__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
  const uint32_t hi = __reduce_min_sync(0xffffffffu, (uint32_t)(v >> 32));
  const uint32_t lo = __reduce_min_sync(0xffffffffu, (uint32_t)(v >> 32) == hi ? (uint32_t)v : 0xffffffffu);
  return ((unsigned long long)hi << 32) | lo;
}

// Exclusive prefix sum of one value per thread over the block; *total gets the sum.
__device__ __noinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* s_wsum, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t ws = lane < kWarps ? s_wsum[lane] : 0u;
    uint32_t wi = ws;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kWarps) s_wsum[lane] = wi - ws;
    if (lane == kWarps - 1) s_wsum[kWarps] = wi;
  }
  __syncthreads();
  *total = s_wsum[kWarps];
  const uint32_t r = s_wsum[warp] + incl - v;
  __syncthreads();  // s_wsum may be reused right after
  return r;
}

template <int NPL>
__global__ void __launch_bounds__(kThreads, 1) control_kernel(CtrlParams p) {
  __shared__ uint32_t s_bitmap[kMaxE / 32];
  __shared__ int s_sel[kMaxPairs];
  __shared__ int s_active[kMaxE];
  __shared__ int s_hit[kMaxE];
  __shared__ int s_miss[kMaxE];
  __shared__ int s_gidx[kMaxE];
  __shared__ int s_victims[kMaxE];
  __shared__ int s_cand[kTour];                // LRU candidates taken before the dependency wait
  __shared__ float s_gate[kMaxPairs];          // gates of the routed pairs
  __shared__ int s_gent[kMaxE];                // expert (index in the layer) of evaluation entry g
  __shared__ int s_res[kMaxE];                 // res[] of this layer's experts
  __shared__ unsigned long long s_tok[kMaxE];  // tokens routed to each expert of this layer
  __shared__ int s_goff[kMaxE + 1];
  __shared__ uint8_t s_fflag[kMaxE];           // expert of this layer filled in this step
  __shared__ uint32_t s_hist[kBins];
  __shared__ uint32_t s_wsum[kWarps + 1];
  __shared__ int s_wcnt[kWarps];
  __shared__ uint32_t s_err, s_clock, s_lo, s_hi;
  __shared__ int s_nactive, s_nhit, s_nmiss, s_q, s_nv, s_ng, s_evict, s_ncand, s_kk, s_done, s_npre;
  __shared__ int s_free;  // no victim was touched by the previous layer-step (its kernels may still run)
  __shared__ unsigned long long s_prefix;
  extern __shared__ unsigned long long s_dyn[];
  unsigned long long* s_vkeys = s_dyn;                              // [kMaxE]
  uint32_t* s_stamp = reinterpret_cast<uint32_t*>(s_dyn + kMaxE);  // [min(S, kSmemSlots)]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, k = p.k, B = p.B, S = p.S;
  const int base_u = p.layer * E;
  const bool in_smem = S <= kSmemSlots;
  uint32_t* stv = in_smem ? s_stamp : p.stamp;  // stamps as the victim scan sees them
  // slot owners, needed only by the install: staged with the stamps for small pools so that
  // the install does not wait on global memory
  const bool own_smem = S <= kSmemOwners;
  int32_t* s_owner = reinterpret_cast<int32_t*>(s_stamp + S);

  // State written by the previous control kernel (complete when this one starts, since
  // every kernel of the chain triggers its dependents only after its own wait): this
  // layer's residency slice and the slot stamps, staged while the previous kernel ends.
  for (int i = tid; i < E; i += kThreads) {
    s_res[i] = p.res[base_u + i];
    s_gidx[i] = -1;
    s_fflag[i] = 0;
    s_tok[i] = 0ull;
  }
  if (in_smem)
    for (int s = tid; s < S; s += kThreads) s_stamp[s] = p.stamp[s];
  if (own_smem)
    for (int s = tid; s < S; s += kThreads) s_owner[s] = p.owner[s];
  for (int i = tid; i < kMaxE / 32; i += kThreads) s_bitmap[i] = 0;
  if (tid == 0) {
    s_err = 0;
    s_clock = p.st->clock + 1u;
    s_evict = 0;
    s_nv = 0;
    s_lo = UINT_MAX;
    s_hi = 0;
    s_ncand = 0;
    s_done = 0;
    s_free = 1;
  }
  const int sbits = S > 1 ? 32 - __clz((unsigned)(S - 1)) : 1;
  // Small K (batch 1-2): the `want` (<= kTour) smallest keys (stamp << sbits | slot) over the
  // slots with stamp < clock, ascending, into out[]; returns how many (fewer when fewer
  // slots qualify), or -1 when the gather overflows its buffer (the radix select then
  // runs).  Each thread's smallest key is found in one scan; the want-th smallest of those
  // per-thread minima bounds the want-th smallest key overall, since they are distinct
  // keys.  A warp tournament over the minima finds that bound T, a second scan gathers every
  // key <= T, and rank counting orders them.  Every thread calls it.
  auto small_k_select = [&](int want, int* out) -> int {
    const uint32_t clk = s_clock;
    const int nit = S > tid ? (S - tid + kThreads - 1) / kThreads : 0;  // slots tid + j*kThreads
    unsigned long long mk = ~0ull;
    for (int j = 0; j < nit; ++j) {
      const int sl = tid + j * kThreads;
      const uint32_t st = s_stamp[sl];
      const unsigned long long key = ((unsigned long long)st << sbits) | (unsigned)sl;
      if (st < clk && key < mk) mk = key;
    }
    int r = 0;
    for (; r < want; ++r) {  // this warp's `want` smallest minima, ascending
      const unsigned long long win = warp_min_u64(mk);
      if (win == ~0ull) break;
      if (mk == win) mk = ~0ull;
      if (lane == 0) s_vkeys[warp * kTour + r] = win;
    }
    if (lane == 0) s_wcnt[warp] = r;
    if (tid == 0) s_nv = 0;
    __syncthreads();
    if (warp == 0) {
      uint32_t taken = 0;
      unsigned long long kth = ~0ull - 1ull;  // fewer than `want` minima: every key qualifies
      for (int n = 0; n < want; ++n) {
        unsigned long long m2 = ~0ull;
        int mj = 0;
        for (int j = 0; j < kWarps * kTour / 32; ++j) {
          const int it = lane + 32 * j, w = it / kTour, rr = it - w * kTour;
          if (rr < s_wcnt[w] && !((taken >> j) & 1u) && s_vkeys[it] < m2) {
            m2 = s_vkeys[it];
            mj = j;
          }
        }
        const unsigned long long win = warp_min_u64(m2);
        if (win == ~0ull) break;
        if (m2 == win) taken |= 1u << mj;
        if (n == want - 1) kth = win;
      }
      if (lane == 0) s_prefix = kth;
    }
    __syncthreads();
    const unsigned long long bound = s_prefix;
    for (int j = 0; j < nit; ++j) {
      const int sl = tid + j * kThreads;
      const uint32_t st = s_stamp[sl];
      const unsigned long long key = ((unsigned long long)st << sbits) | (unsigned)sl;
      if (st < clk && key <= bound) {
        const int i = atomicAdd(&s_nv, 1);
        if (i < kMaxE) s_vkeys[i] = key;
      }
    }
    __syncthreads();
    const int nc = s_nv;
    if (nc > kMaxE) return -1;
    const unsigned long long smask = (1ull << sbits) - 1ull;
    for (int i = tid; i < nc; i += kThreads) {
      const unsigned long long ki = s_vkeys[i];
      int rank = 0;
      for (int j = 0; j < nc; ++j) rank += s_vkeys[j] < ki;
      if (rank < want) out[rank] = (int)(ki & smask);
    }
    return min(nc, want);
  };
  // Victim candidates before the wait (the slot stamps are final: only the previous control
  // kernel writes them, and this kernel's own hits come later).  Hits of this step can
  // remove at most kcap of them, so the 2*kcap least recently used slots always hold the
  // kcap victims; after the wait only the hits are filtered out.  This takes the victim
  // scan off the step's critical path, while the previous layer's evaluation still runs
  // (launched as a programmatic dependent; otherwise nothing runs beside the prologue).
  // When the logits were complete before the previous kernel started (p.logits_early: a
  // later layer of one multi-layer call), every decision of the step is taken before the
  // dependency wait, while the previous layer's evaluation still runs: the residency state
  // is final (only the previous control kernel writes it), and the decisions write only
  // that state and shared memory.  The work lists, which the previous fill and evaluation
  // kernels read, are published after the wait.  Otherwise the logits may be written by
  // the kernel right before this one, so the decisions follow the wait.
  const bool early = p.logits_early && B <= kWarps;
  if (tid == 0) s_npre = -1;
  if (!early && p.pdl && in_smem && 2 * p.kcap <= kTour) {
    __syncthreads();  // stamps staged, s_clock set
    const int n = small_k_select(2 * p.kcap, s_cand);
    if (tid == 0) s_npre = n;
  }
  // an L2 prefetch of the logits is safe before the wait (the L2 is coherent and a prefetch
  // returns no data) and takes the DRAM latency off the routing step
  float zpre[NPL];
  if (early) {
    if (warp < B) load_logits_warp<NPL>(p.logits + (size_t)warp * E, E, lane, zpre);
  } else {
    for (int i = tid * 32; i < B * E; i += kThreads * 32)
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p.logits + i));
  }

  auto decide = [&]() {
    const uint32_t clock = s_clock;
    // ---- 1. route: one warp per token
    for (int t = warp; t < B; t += kWarps) {
      auto emit = [&](int e, float g, int rank) {
        const int idx = t * k + rank;
        s_gate[idx] = g;
        s_sel[idx] = e;
        atomicOr(&s_bitmap[e >> 5], 1u << (e & 31));
        atomicOr(reinterpret_cast<uint32_t*>(&s_tok[e]) + (t >> 5), 1u << (t & 31));  // 32-bit half of the mask
      };
      if (early) route_token_warp_loaded<NPL>(zpre, E, k, p.gate, lane, &s_err, emit);
      else route_token_warp<NPL>(p.logits + (size_t)t * E, E, k, p.gate, lane, &s_err, emit);
    }
    __syncthreads();

    // ---- 2. dedupe + classify (warp 0; A is at most min(B*k, E) ids, ascending)
    if (warp == 0) {
      const int nwords = (E + 31) / 32;
      int nact = 0, nh = 0, nm = 0;
      for (int c = 0; c < nwords; c += 32) {
        uint32_t word = c + lane < nwords ? s_bitmap[c + lane] : 0u;
        const int cnt = __popc(word);
        int incl = cnt;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        int pos = nact + incl - cnt;
        while (word) {
          const int b = __ffs(word) - 1;
          word &= word - 1;
          s_active[pos++] = base_u + (c + lane) * 32 + b;
        }
        nact += __shfl_sync(0xffffffffu, incl, 31);
      }
      __syncwarp();
      for (int c = 0; c < nact; c += 32) {
        const int i = c + lane;
        const bool valid = i < nact;
        const int u = valid ? s_active[i] : -1;
        int slot = valid ? s_res[u - base_u] : -1;
        if (slot >= S) {  // cannot happen with a consistent table
          atomicOr(&s_err, FT_DEVERR_BAD_STATE);
          slot = -1;
        }
        const bool hit = valid && slot >= 0;
        const uint32_t hb = __ballot_sync(0xffffffffu, hit);
        const uint32_t mb = __ballot_sync(0xffffffffu, valid && !hit);
        const uint32_t lt = (1u << lane) - 1u;
        if (hit) {
          s_hit[nh + __popc(hb & lt)] = u;
          p.stamp[slot] = clock;  // a hit refreshes recency
          stv[slot] = clock;
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
    // ---- 3. one-pass K-LRU victim scan over slots not touched in this step
    if (q > 0) {
      bool picked = false;
      if (s_npre >= 0) {
        // candidates taken before the wait, minus this step's hits (now stamped with clock)
        if (warp == 0) {
          const int v = lane < s_npre ? s_cand[lane] : -1;
          const bool ok = v >= 0 && s_stamp[v] < clock;
          const uint32_t okb = __ballot_sync(0xffffffffu, ok);
          const int rank = __popc(okb & ((1u << lane) - 1u));
          if (ok && rank < kcap) s_victims[rank] = v;
          if (lane == 0) s_nv = min(__popc(okb), kcap);
        }
        picked = true;
        __syncthreads();
      } else if (in_smem && kcap <= kTour) {
        const int n = small_k_select(kcap, s_victims);
        __syncthreads();  // every thread has read the gather count before it is overwritten
        if (n >= 0) {
          picked = true;
          if (tid == 0) s_nv = n;
        }
        __syncthreads();
      }
      if (!picked) {
        // range of candidate stamps (stamp < clock: hits of this step are excluded) and count
        uint32_t lo = UINT_MAX, hi = 0;
        int nc = 0;
        for (int s = tid; s < S; s += kThreads) {
          const uint32_t st = stv[s];
          if (st < clock) {
            lo = min(lo, st);
            hi = max(hi, st);
            ++nc;
          }
        }
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
        const uint32_t range = s_hi - st_lo;
        const int width = (range ? 32 - __clz(range) : 0) + sbits;  // <= 52 bits
        // key = (stamp - lowest candidate stamp, slot): unique, ordered like (stamp, slot)
        unsigned long long thresh = ~0ull;
        if (want < ncand) {
          // radix select of the want-th smallest key, most significant digit first.  Digits are
          // taken from the top of the key's actual width, so the first pass spreads the keys
          // over all kBins bins (few shared-memory atomics collide).
          if (tid == 0) {
            s_prefix = 0;
            s_kk = want;
          }
          for (int hi_bit = width; hi_bit > 0;) {
            const int shift = hi_bit > kDigit ? hi_bit - kDigit : 0;
            const int dbits = hi_bit - shift;
            s_hist[tid] = 0;
            __syncthreads();
            const unsigned long long pre = s_prefix;
            for (int s = tid; s < S; s += kThreads) {
              const uint32_t st = stv[s];
              if (st >= clock) continue;
              const unsigned long long key = ((unsigned long long)(st - st_lo) << sbits) | (unsigned)s;
              if ((key >> hi_bit) == pre) atomicAdd(&s_hist[(key >> shift) & ((1u << dbits) - 1u)], 1u);
            }
            __syncthreads();
            const uint32_t h = s_hist[tid];
            const uint32_t kk = (uint32_t)s_kk;
            uint32_t total;
            const uint32_t excl = block_excl_scan(h, s_wsum, &total);
            if (excl < kk && excl + h >= kk) {  // exactly one thread: the bin holding the kk-th key
              s_prefix = (pre << dbits) | (unsigned long long)tid;
              s_kk = (int)(kk - excl);
              s_done = excl + h == kk;  // every key of the bin is wanted: no finer digit needed
            }
            __syncthreads();
            if (s_done || shift == 0) {
              thresh = (s_prefix << shift) | ((1ull << shift) - 1ull);
              break;
            }
            hi_bit = shift;
          }
        }
        // collect the `want` smallest keys (keys are unique), then order them
        for (int s = tid; s < S; s += kThreads) {
          const uint32_t st = stv[s];
          if (st >= clock) continue;
          const unsigned long long key = ((unsigned long long)(st - st_lo) << sbits) | (unsigned)s;
          if (key <= thresh) {
            const int i = atomicAdd(&s_nv, 1);
            if (i < kMaxE) s_vkeys[i] = key;
          }
        }
        __syncthreads();
        const int nv = min(s_nv, want);
        const unsigned long long smask = (1ull << sbits) - 1ull;
        for (int i = tid; i < nv; i += kThreads) {
          const unsigned long long ki = s_vkeys[i];
          int rank = 0;
          for (int j = 0; j < nv; ++j) rank += s_vkeys[j] < ki;
          s_victims[rank] = (int)(ki & smask);
        }
        __syncthreads();
        if (tid == 0) s_nv = nv;
      }

      // ---- 4. install F = first q misses into the first q victims
      for (int i = tid; i < q; i += kThreads) {
        const int v = s_victims[i];
        const int u = s_miss[i];
        // the previous layer-step stamped its entries and victims with clock - 1
        if (stv[v] + 1u >= clock) s_free = 0;
        const int old = own_smem ? s_owner[v] : p.owner[v];
        if (old >= 0) {
          p.res[old] = -1;
          atomicAdd(&s_evict, 1);
        }
        p.owner[v] = u;
        p.res[u] = v;
        s_res[u - base_u] = v;
        s_fflag[u - base_u] = 1;
        p.stamp[v] = clock;
      }
    }
    __syncthreads();

    // ---- 5. G = resident part of A (ascending u): evaluation entries and pair offsets
    if (warp == 0) {
      const int nact = s_nactive;
      int ng = 0, carry = 0;
      for (int c = 0; c < nact; c += 32) {
        const int i = c + lane;
        const int e = i < nact ? s_active[i] - base_u : -1;
        const int slot = e >= 0 ? s_res[e] : -1;
        const bool in = slot >= 0;
        const int cnt = in ? __popcll(s_tok[e]) : 0;
        int incl = cnt;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t b = __ballot_sync(0xffffffffu, in);
        if (in) {
          const int g = ng + __popc(b & ((1u << lane) - 1u));
          s_gidx[e] = g;
          s_gent[g] = e;
          s_goff[g] = carry + incl - cnt;
        }
        ng += __popc(b);
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        s_ng = ng;
        s_goff[ng] = carry;
      }
    }
    __syncthreads();
  };  // decide

  if (early) {
    __syncthreads();  // stamps and residency staged, s_clock set
    decide();
    // The fill may start now when no victim slot belongs to the previous layer-step, whose
    // evaluation (and fill) may still read (and write) its slots: the copy list goes out
    // tagged with the step's clock, released after its entries, and the fill kernel is let
    // launch.  It still waits for this kernel before it lets the evaluation start.
    const int q = s_q;
    if (p.w.ecopy != nullptr && q > 0 && s_free) {
      const uint32_t clock = s_clock;
      int32_t* el = p.w.ecopy + (size_t)(clock & 1u) * (2 + 2 * p.w.kmax);
      for (int i = tid; i < q; i += kThreads) {
        el[2 + i] = s_miss[i];
        el[2 + p.w.kmax + i] = s_victims[i];
      }
      if (tid == 0) el[1] = q;
      __syncthreads();
      if (tid == 0) ptx::st_release_gpu(reinterpret_cast<uint32_t*>(el), clock);
    }
    pdl_trigger();
  }
  // the work lists belong to the kernels right before this one (and the logits, unless early)
  pdl_wait();
  if (!early) pdl_trigger();
  __syncthreads();
  if (!early) decide();

  // ---- publish the step's lists
  const uint32_t clock = s_clock;
  const int q = s_q;
  const int kcap = p.kcap;
  const int ng = s_ng, carry = s_goff[ng];
  const int npairs = B * k;
  for (int i = tid; i < npairs; i += kThreads) {
    p.w.sel[i] = s_sel[i];
    p.w.gates[i] = s_gate[i];
  }
  for (int i = tid; i < q; i += kThreads) {
    p.w.copy_u[i] = s_miss[i];
    p.w.copy_slot[i] = s_victims[i];
  }
  for (int g = tid; g < ng; g += kThreads) {
    const int e = s_gent[g];
    p.w.g_w[g] = p.pool + (size_t)s_res[e] * p.slot_stride;
    p.w.g_fill[g] = s_fflag[e];
    p.w.g_off[g] = s_goff[g];
  }
  if (tid == 0) {
    p.w.g_off[ng] = carry;
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
  // rewrite pairs to slots / FT_CPU and place them: within an entry, ascending pair id
  // (= ascending token, since a token routes to an expert at most once)
  for (int pi = tid; pi < npairs; pi += kThreads) {
    const int e = s_sel[pi];
    const int g = s_gidx[e];
    p.w.slot_of_pair[pi] = g >= 0 ? s_res[e] : FT_CPU;
    if (g >= 0) {
      const int t = pi / k;
      const int pos = __popcll(s_tok[e] & ((1ull << t) - 1ull));
      p.w.g_pair[s_goff[g] + pos] = pi;
    }
  }
  if (p.has_shared)
    for (int t = tid; t < B; t += kThreads) p.w.g_pair[carry + t] = t;
  for (int i = tid; i <= kcap; i += kThreads) p.w.ready[i] = 0u;
  // lists for traces
  for (int i = tid; i < s_nactive; i += kThreads) p.w.active[i] = s_active[i];
  for (int i = tid; i < s_nhit; i += kThreads) p.w.hit[i] = s_hit[i];
  for (int i = tid; i < s_nmiss; i += kThreads) p.w.miss[i] = s_miss[i];
  if (q > 0)
    for (int i = tid; i < s_nv; i += kThreads) p.w.victims[i] = s_victims[i];
  if (tid == 0) {
    DevState* st = p.st;
    st->clock = clock;
    // counter updates without a read back (reductions): nothing on this path waits for them
    atomicAdd(&st->hits, (unsigned long long)s_nhit);
    atomicAdd(&st->misses, (unsigned long long)s_nmiss);
    atomicAdd(&st->fills, (unsigned long long)q);
    atomicAdd(&st->cpu_execs, (unsigned long long)(s_nmiss - q));
    atomicAdd(&st->evictions, (unsigned long long)s_evict);
    atomicAdd(&st->decode_steps, 1ull);
    atomicAdd(&st->eval_entries, (unsigned long long)(ng + (p.has_shared ? 1 : 0)));
    atomicAdd(&st->eval_pairs, (unsigned long long)(carry + (p.has_shared ? B : 0)));
    if (s_err) atomicOr(&st->error_word, s_err);
  }
}

template <int NPL>
cudaError_t launch_npl(const CtrlParams& p, cudaStream_t s) {
  const size_t smem = kMaxE * sizeof(unsigned long long) +
                      (size_t)(p.S <= kSmemSlots ? p.S : 0) * sizeof(uint32_t) +
                      (size_t)(p.S <= kSmemOwners ? p.S : 0) * sizeof(int32_t);
  return launch_k(control_kernel<NPL>, dim3(1), dim3(kThreads), smem, s, p.pdl, p);
}

template <int NPL>
cudaError_t prepare_npl() {
  return cudaFuncSetAttribute(control_kernel<NPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmemMax);
}

}  // namespace

// One router width per instantiation: E <= 32 * NPL logits per lane.
cudaError_t launch_control(const CtrlParams& p, cudaStream_t s) {
  if (p.E <= 32) return launch_npl<1>(p, s);
  if (p.E <= 64) return launch_npl<2>(p, s);
  if (p.E <= 128) return launch_npl<4>(p, s);
  if (p.E <= 256) return launch_npl<8>(p, s);
  if (p.E <= 512) return launch_npl<16>(p, s);
  return launch_npl<32>(p, s);
}

cudaError_t prepare_control() {
  cudaError_t e;
  if ((e = prepare_npl<1>()) != cudaSuccess) return e;
  if ((e = prepare_npl<2>()) != cudaSuccess) return e;
  if ((e = prepare_npl<4>()) != cudaSuccess) return e;
  if ((e = prepare_npl<8>()) != cudaSuccess) return e;
  if ((e = prepare_npl<16>()) != cudaSuccess) return e;
  return prepare_npl<32>();
}

}  // namespace ft
