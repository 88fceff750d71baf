// Prefill path: full-layer double buffering from the shared slot pool, routing of a
// whole chunk, the grouped GEMMs (prefill_gemm.cu) and the fixed-order combine.
//
// "FreeToken 完全拆解", section "全层双缓冲": two full-layer buffers come from the same
// global slot pool as the decode cache; while layer l is computed from one, a transfer
// stream copies every expert of layer l+1 into the other without waiting for routing;
// what the last layers leave behind seeds decode.  Reading used here (the pages fix no
// finer policy): a chunk starts at a prefill call that does not continue the previous
// prefill layer and takes the 2E least recently used slots (ascending (stamp, slot)),
// evicting their occupants; layer l uses buffer (l - first) mod 2, expert e in its e-th
// slot; installing a layer drops the buffer's previous occupants, invalidates any older
// resident copy of the layer's experts and stamps every expert of the layer with that
// step's clock.  Prefill does not count as hits or misses.
#include <algorithm>
#include <cstring>

#include "ft_dot.cuh"
#include "ft_prefill.cuh"
#include "ft_route.cuh"

namespace ft {
namespace {

constexpr int kPickThreads = 1024;
constexpr int kPickMaxSlots = 16384;  // slots sorted in shared memory when a chunk starts
constexpr int kTileN = 256;  // token rows of one grouped-GEMM tile at most

// Layer copy: SM loads of the mapped host banks.  One CTA step moves a 64 KB piece of one
// expert's bank (512 threads x 8 loads of 16 bytes in flight).  16 CTAs already hold the host
// link at its read rate (~200 GB/s for SM loads; the copy engine managed 110-150 GB/s on the
// scattered 2 MB pieces of a layer); each reserves enough shared memory that no grouped-GEMM
// CTA shares its SM, and the GEMMs run on the other SMs meanwhile.
constexpr int kCopySms = 16;
constexpr int kCopyThreads = 512;
constexpr int kCopyUnroll = 8;
constexpr size_t kCopyPiece = (size_t)kCopyThreads * kCopyUnroll * 16;
constexpr size_t kCopySmemReserve = 120 * 1024;

struct LayerCopyArgs {
  const uint8_t* src[7];  // device view of the host banks
  size_t row[7];          // bytes per logical id in bank j (a multiple of 16)
  size_t off[7];          // byte offset of bank j within a slot
  uint32_t pieces[7];     // 64 KB pieces per expert in bank j
  uint32_t per_expert;    // sum of pieces[]
  int n_banks, E, layer;
  const int32_t* slots;   // [E] destination slot of each expert of the layer
  uint8_t* pool;
  size_t stride;
};

__global__ void __launch_bounds__(kCopyThreads) layer_copy_kernel(const LayerCopyArgs a) {
  const size_t total = (size_t)a.E * a.per_expert;
  for (size_t c = blockIdx.x; c < total; c += gridDim.x) {
    const int e = (int)(c / a.per_expert);
    uint32_t r = (uint32_t)(c - (size_t)e * a.per_expert);
    const uint8_t* sb = a.src[0];
    size_t row = a.row[0], off = a.off[0];
    uint32_t np = a.pieces[0];
#pragma unroll
    for (int j = 1; j < 7; ++j)
      if (r >= np && j < a.n_banks) {
        r -= np;
        sb = a.src[j];
        row = a.row[j];
        off = a.off[j];
        np = a.pieces[j];
      }
    const size_t lo = (size_t)r * kCopyPiece;
    const size_t n16 = (row - lo < kCopyPiece ? row - lo : kCopyPiece) / 16;
    const uint4* src = reinterpret_cast<const uint4*>(sb + ((size_t)a.layer * a.E + e) * row + lo);
    uint4* dst = reinterpret_cast<uint4*>(a.pool + (size_t)__ldg(a.slots + e) * a.stride + off + lo);
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const size_t i = threadIdx.x + (size_t)u * kCopyThreads;
      if (i < n16) v[u] = dot::ld_host(src + i);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const size_t i = threadIdx.x + (size_t)u * kCopyThreads;
      if (i < n16) dst[i] = v[u];
    }
  }
}

// Sorts all slots by (stamp, slot) in shared memory (bitonic), writes the 2E least
// recently used to out[] in order and evicts their occupants.
__global__ void __launch_bounds__(kPickThreads) pick_buffers_kernel(int32_t* res, int32_t* owner, uint32_t* stamp,
                                                                   int S, int n_pick, int32_t* out) {
  extern __shared__ unsigned long long keys[];
  int n2 = 1;
  while (n2 < S) n2 <<= 1;
  for (int i = threadIdx.x; i < n2; i += blockDim.x)
    keys[i] = i < S ? (((unsigned long long)stamp[i] << 32) | (unsigned)i) : ~0ull;
  __syncthreads();
  for (int kk = 2; kk <= n2; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & kk) == 0;
          const unsigned long long a = keys[i], b = keys[ixj];
          if ((a > b) == up) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n_pick; i += blockDim.x) {
    const int v = (int)(keys[i] & 0xffffffffu);
    out[i] = v;
    const int o = owner[v];
    if (o >= 0) res[o] = -1;
    owner[v] = -1;
    stamp[v] = 0u;
  }
}

// Residency effect of computing layer `layer` from buffer `buf` (one CTA).
__global__ void __launch_bounds__(1024) install_layer_kernel(int layer, int E, const int32_t* buf, int32_t* res,
                                                            int32_t* owner, uint32_t* stamp, DevState* st) {
  __shared__ uint32_t s_clock;
  if (threadIdx.x == 0) s_clock = st->clock + 1u;
  // phase 1: read previous occupants and older copies
  int prev[4], old[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = threadIdx.x + j * blockDim.x;
    prev[j] = old[j] = -1;
    if (e < E) {
      prev[j] = owner[buf[e]];
      old[j] = res[layer * E + e];
    }
  }
  __syncthreads();
  const uint32_t clock = s_clock;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = threadIdx.x + j * blockDim.x;
    if (e >= E) continue;
    const int u = layer * E + e, v = buf[e];
    if (prev[j] >= 0 && prev[j] != u) res[prev[j]] = -1;
    if (old[j] >= 0 && old[j] != v) {
      owner[old[j]] = -1;
      stamp[old[j]] = 0u;
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = threadIdx.x + j * blockDim.x;
    if (e >= E) continue;
    const int u = layer * E + e, v = buf[e];
    owner[v] = u;
    res[u] = v;
    stamp[v] = clock;
  }
  if (threadIdx.x == 0) {
    st->clock = clock;
    st->prefill_layers += 1ull;
  }
}

// One warp per token: top-k routing and gates, then the token's bit in each chosen
// expert's mask.
__global__ void __launch_bounds__(256) prefill_route_kernel(const float* logits, int T, int E, int k, int gate, int W,
                                                           int32_t* sel, float* gates, uint32_t* masks,
                                                           uint32_t* error_word) {
  __shared__ uint32_t s_err;
  if (threadIdx.x == 0) s_err = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (t < T) {
    route_token_any(logits + (size_t)t * E, E, k, gate, lane, &s_err, [&](int e, float g, int rank) {
      sel[(size_t)t * k + rank] = e;
      gates[(size_t)t * k + rank] = g;
      atomicOr(masks + (size_t)e * W + (t >> 5), 1u << (t & 31));
    });
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_err) atomicOr(error_word, s_err);
}

// Per expert: exclusive prefix of popcounts over its mask words (token order), its
// pair count; then pair offsets and N-tile offsets over entries (one CTA).
__global__ void __launch_bounds__(1024) prefill_scan_kernel(const uint32_t* masks, int W, int E, int T,
                                                           int has_shared, int32_t* wpre, int32_t* entry_off,
                                                           int32_t* tile_off) {
  __shared__ int s_cnt[kMaxE + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int per = (W + 31) / 32;  // contiguous words per lane
  for (int e = warp; e < E; e += nw) {
    const uint32_t* m = masks + (size_t)e * W;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int w = lane * per + i;
      if (w < W) local += __popc(m[w]);
    }
    int incl = local;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int w = lane * per + i;
      if (w < W) {
        wpre[(size_t)e * W + w] = run;
        run += __popc(m[w]);
      }
    }
    if (lane == 31) s_cnt[e] = incl;
  }
  if (threadIdx.x == 0 && has_shared) s_cnt[E] = T;
  __syncthreads();
  if (warp == 0) {
    const int n = E + (has_shared ? 1 : 0);
    int carry_p = 0, carry_t = 0;
    for (int c = 0; c < n; c += 32) {
      const int i = c + lane;
      const int v = i < n ? s_cnt[i] : 0;
      const int nt = (v + kTileN - 1) / kTileN;
      int ip = v, it = nt;
      for (int o = 1; o < 32; o <<= 1) {
        const int yp = __shfl_up_sync(0xffffffffu, ip, o), yt = __shfl_up_sync(0xffffffffu, it, o);
        if (lane >= o) {
          ip += yp;
          it += yt;
        }
      }
      if (i < n) {
        entry_off[i] = carry_p + ip - v;
        tile_off[i] = carry_t + it - nt;
      }
      carry_p += __shfl_sync(0xffffffffu, ip, 31);
      carry_t += __shfl_sync(0xffffffffu, it, 31);
    }
    if (lane == 0) {
      entry_off[n] = carry_p;
      tile_off[n] = carry_t;
    }
  }
}

// Pair (t, r) -> its position in the expert-sorted pair list (tokens ascending within
// an expert); shared-expert pairs follow all routed pairs, one per token.
__global__ void prefill_place_kernel(const int32_t* sel, const float* gates, const uint32_t* masks,
                                     const int32_t* wpre, const int32_t* entry_off, int T, int k, int E, int W,
                                     int has_shared, int32_t* pair_tok, float* pair_gate, int32_t* pos_of) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < T * k) {
    const int t = i / k;
    const int e = sel[i];
    const int w = t >> 5;
    const uint32_t below = masks[(size_t)e * W + w] & ((1u << (t & 31)) - 1u);
    const int pos = entry_off[e] + wpre[(size_t)e * W + w] + __popc(below);
    pair_tok[pos] = t;
    pair_gate[pos] = gates[i];
    pos_of[i] = pos;
  } else if (has_shared && i < T * k + T) {
    const int t = i - T * k;
    const int pos = entry_off[E] + t;
    pair_tok[pos] = t;
    pair_gate[pos] = 1.0f;
  }
}

// Token rows in pair order: xp[p] = x[pair_tok[p]] (BF16, one warp per row, 16-byte
// vectors).  The gate/up GEMM then reads each N tile of tokens as one contiguous TMA box.
__global__ void __launch_bounds__(256) prefill_permute_kernel(const uint16_t* x, const int32_t* pair_tok, int P,
                                                             int H, uint16_t* xp) {
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  for (int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < P; p += nw) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)__ldg(pair_tok + p) * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)p * H);
    for (int i = lane; i < H / 8; i += 32) dst[i] = __ldg(src + i);
  }
}

// N tiles of every entry: an entry with n_e pairs is split into ceil(n_e / kTileN) tiles
// of equal size rounded up to 16.  tiles[q] = {entry, first pair, valid pairs, N}.
__global__ void prefill_tiles_kernel(const int32_t* entry_off, const int32_t* tile_off, int n_entries, int4* tiles) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n_entries) return;
  const int p0 = entry_off[e], ne = entry_off[e + 1] - p0;
  const int t0 = tile_off[e], nt = tile_off[e + 1] - t0;
  if (nt <= 0) return;
  const int tsize = ((ne + nt - 1) / nt + 15) & ~15;
  for (int j = 0; j < nt; ++j) {
    const int n0 = j * tsize;
    const int nvalid = min(tsize, ne - n0);
    tiles[t0 + j] = make_int4(e, p0 + n0, nvalid, (nvalid + 15) & ~15);
  }
}

// out[t] = shared row (if any) + the k pair rows in rank order (ascending expert id).
__global__ void prefill_combine_kernel(const uint16_t* rows, const int32_t* pos_of, const int32_t* entry_off, int T,
                                       int k, int H, int E, int has_shared, float* out) {
  const int per_tok = H / 8;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)T * per_tok) return;
  const int t = (int)(i / per_tok), j0 = (int)(i - (size_t)t * per_tok) * 8;
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  auto add_row = [&](int p) {
    const uint4 v = *reinterpret_cast<const uint4*>(rows + (size_t)p * H + j0);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[2 * q] += __uint_as_float(w[q] << 16);
      acc[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
    }
  };
  if (has_shared) add_row(entry_off[E] + t);
  for (int r = 0; r < k; ++r) add_row(pos_of[(size_t)t * k + r]);
  float4* o = reinterpret_cast<float4*>(out + (size_t)t * H + j0);
  o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

}  // namespace

struct PrefillState {
  int T_max = 0, E = 0, K = 0, H = 0, I = 0, L = 0, S = 0, W = 0, has_shared = 0, n_sm = 0;
  // routing and GEMM buffers
  int32_t *sel = nullptr, *wpre = nullptr, *entry_off = nullptr, *tile_off = nullptr;
  int32_t *pair_tok = nullptr, *pos_of = nullptr, *buf_dev = nullptr, *pick_dev = nullptr;
  float *gates = nullptr, *pair_gate = nullptr;
  uint32_t* masks = nullptr;
  uint16_t *h = nullptr, *rows = nullptr, *xp = nullptr;
  int4* tiles = nullptr;
  GemmMaps* maps = nullptr;
  // chunk state (host)
  bool active = false;
  int first = 0, next_layer = -1, pending = -1;
  cudaEvent_t ev_loaded[2] = {nullptr, nullptr}, ev_free[2] = {nullptr, nullptr}, ev_restore = nullptr;
  cudaEvent_t ev_pick = nullptr;  // the chunk's buffer slots are in buf_dev (the copies read them)
  cudaEvent_t ev_serial = nullptr;  // second buffer off: this layer's copy waits for all prior compute
  bool free_recorded[2] = {false, false};
  cudaStream_t cs = nullptr, ts = nullptr;
  // what a restore copy needs
  uint8_t* pool = nullptr;
  SlotLayout lay{};
  const uint8_t* bank_host[7] = {};
  const uint8_t* bank_dev[7] = {};
  size_t bank_row[7] = {};
  int n_banks = 3;
  int wtype = FT_W_BF16;
};

namespace {

// Byte offset of bank j within a slot: gate, up, down, then the scale banks.
size_t bank_offset(const SlotLayout& l, int j) {
  const size_t off[7] = {l.gate, l.up, l.down, l.gs, l.us, l.ds, l.ts};
  return off[j];
}

}  // namespace

namespace {

// Where the decoding warps of the FP8 / FP4 grouped GEMM find the block scales.
void set_weight_info(GemmDesc& d, const PrefillCtx& c) {
  d.pool = c.pool;
  d.shared_w = c.shared_w;
  d.stride = c.lay.stride;
  d.off_gs = c.lay.gs;
  d.off_us = c.lay.us;
  d.off_ds = c.lay.ds;
  d.off_ts = c.lay.ts;
}

// Copy every expert of `layer` from the host banks into the slots of buffer b (slot ids in
// buf_dev), ordered after the work already on ts and completed in ts's order.
cudaError_t copy_layer(PrefillState* p, int layer, int b, cudaStream_t ts) {
  LayerCopyArgs a{};
  a.per_expert = 0;
  for (int j = 0; j < p->n_banks; ++j) {
    a.src[j] = p->bank_dev[j];
    a.row[j] = p->bank_row[j];
    a.off[j] = bank_offset(p->lay, j);
    a.pieces[j] = (uint32_t)((p->bank_row[j] + kCopyPiece - 1) / kCopyPiece);
    a.per_expert += a.pieces[j];
  }
  a.n_banks = p->n_banks;
  a.E = p->E;
  a.layer = layer;
  a.slots = p->buf_dev + (size_t)b * p->E;
  a.pool = p->pool;
  a.stride = p->lay.stride;
  layer_copy_kernel<<<kCopySms, kCopyThreads, kCopySmemReserve, ts>>>(a);
  return cudaGetLastError();
}

// Enqueue the load of `layer` into buffer b on the transfer stream, after the compute
// that last used buffer b.
cudaError_t load_buffer(PrefillState* p, int layer, int b, ProfEvents* prof) {
  cudaError_t e;
  if (p->free_recorded[b] && (e = cudaStreamWaitEvent(p->ts, p->ev_free[b], 0)) != cudaSuccess) return e;
  cudaEvent_t a = nullptr, z = nullptr;
  if (prof) {
    cudaEventCreate(&a);
    cudaEventCreate(&z);
    cudaEventRecord(a, p->ts);
  }
  if ((e = copy_layer(p, layer, b, p->ts)) != cudaSuccess) return e;
  if (prof) {
    cudaEventRecord(z, p->ts);
    prof->push_back({7, {a, z}});
  }
  return cudaEventRecord(p->ev_loaded[b], p->ts);
}

template <typename T>
cudaError_t dev_alloc(T** ptr, size_t n) {
  return cudaMalloc(reinterpret_cast<void**>(ptr), (n ? n : 1) * sizeof(T));
}

// Route a chunk and sort its pairs by entry: per-expert token masks, pair offsets and N
// tiles per entry, the pair lists, the tile table and the token rows in pair order.
cudaError_t route_chunk(PrefillState* p, const PrefillCtx& c, int T, const uint16_t* x, const float* logits) {
  const int E = p->E, k = p->K;
  cudaError_t r = cudaMemsetAsync(p->masks, 0, sizeof(uint32_t) * (size_t)E * p->W, c.cs);
  if (r != cudaSuccess) return r;
  prefill_route_kernel<<<(T + 7) / 8, 256, 0, c.cs>>>(logits, T, E, k, c.gate, p->W, p->sel, p->gates, p->masks,
                                                      &c.st->error_word);
  prefill_scan_kernel<<<1, 1024, 0, c.cs>>>(p->masks, p->W, E, T, p->has_shared, p->wpre, p->entry_off, p->tile_off);
  const int n_pl = T * k + (p->has_shared ? T : 0);
  prefill_place_kernel<<<(n_pl + 255) / 256, 256, 0, c.cs>>>(p->sel, p->gates, p->masks, p->wpre, p->entry_off, T, k,
                                                             E, p->W, p->has_shared, p->pair_tok, p->pair_gate,
                                                             p->pos_of);
  const int n_ent = E + (p->has_shared ? 1 : 0);
  prefill_tiles_kernel<<<(n_ent + 255) / 256, 256, 0, c.cs>>>(p->entry_off, p->tile_off, n_ent, p->tiles);
  prefill_permute_kernel<<<p->n_sm * 8, 256, 0, c.cs>>>(x, p->pair_tok, n_pl, p->H, p->xp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_create(PrefillState** out, const PrefillCtx& c) {
  if (c.S > kPickMaxSlots) return cudaErrorInvalidValue;
  // BF16 tiles are read through 2-D maps over the whole pool (slot stride = the three banks);
  // FP8 / FP4 tiles through 3-D maps (any stride)
  if ((c.wtype == FT_W_BF16 && c.lay.stride != c.lay.used) || c.H % 128 || c.I % 64) return cudaErrorInvalidValue;
  PrefillState* p = new PrefillState();
  p->T_max = c.max_tokens;
  p->E = c.E;
  p->K = c.K;
  p->H = c.H;
  p->I = c.I;
  p->L = c.L;
  p->S = c.S;
  p->W = (c.max_tokens + 31) / 32;
  p->has_shared = c.has_shared;
  p->n_sm = c.n_sm;
  p->pool = c.pool;
  p->lay = c.lay;
  p->n_banks = c.n_banks;
  p->wtype = c.wtype;
  for (int j = 0; j < c.n_banks; ++j) {
    p->bank_host[j] = c.bank_host[j];
    p->bank_dev[j] = c.bank_dev[j];
    p->bank_row[j] = c.bank_row[j];
  }
  const size_t T = c.max_tokens, k = c.K, P = T * k + (c.has_shared ? T : 0);
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = dev_alloc(&p->sel, T * k);
  if (e == cudaSuccess) e = dev_alloc(&p->gates, T * k);
  if (e == cudaSuccess) e = dev_alloc(&p->masks, (size_t)c.E * p->W);
  if (e == cudaSuccess) e = dev_alloc(&p->wpre, (size_t)c.E * p->W);
  if (e == cudaSuccess) e = dev_alloc(&p->entry_off, (size_t)c.E + 2);
  if (e == cudaSuccess) e = dev_alloc(&p->tile_off, (size_t)c.E + 2);
  if (e == cudaSuccess) e = dev_alloc(&p->pair_tok, P);
  if (e == cudaSuccess) e = dev_alloc(&p->pair_gate, P);
  if (e == cudaSuccess) e = dev_alloc(&p->pos_of, T * k);
  if (e == cudaSuccess) e = dev_alloc(&p->h, P * c.I);
  if (e == cudaSuccess) e = dev_alloc(&p->xp, P * c.H);
  if (e == cudaSuccess) e = dev_alloc(&p->tiles, P / kTileN + (size_t)c.E + 2);
  if (e == cudaSuccess) e = dev_alloc(&p->rows, P * c.H);
  if (e == cudaSuccess) e = dev_alloc(&p->buf_dev, (size_t)2 * c.E);
  if (e == cudaSuccess) e = dev_alloc(&p->pick_dev, (size_t)2 * c.E);
  for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
    e = cudaEventCreateWithFlags(&p->ev_loaded[b], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_free[b], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_restore, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_pick, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_serial, cudaEventDisableTiming);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(layer_copy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCopySmemReserve);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pick_buffers_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPickMaxSlots * (int)sizeof(unsigned long long));
  if (e == cudaSuccess)
    e = gemm_maps_create(&p->maps, c.pool, c.S, c.shared_w, c.L, c.H, c.I, p->h, p->xp, (int)P, c.wtype, c.lay);
  if (e != cudaSuccess) {
    prefill_destroy(p);
    return e;
  }
  *out = p;
  return cudaSuccess;
}

void prefill_destroy(PrefillState* p) {
  if (!p) return;
  prefill_interrupt(p);
  if (p->cs) cudaStreamSynchronize(p->cs);
  if (p->ts) cudaStreamSynchronize(p->ts);
  void* bufs[] = {p->sel, p->gates, p->masks, p->wpre, p->entry_off, p->tile_off, p->pair_tok,
                  p->pair_gate, p->pos_of, p->h, p->rows, p->xp, p->tiles, p->buf_dev, p->pick_dev};
  for (void* b : bufs)
    if (b) cudaFree(b);
  for (int b = 0; b < 2; ++b) {
    if (p->ev_loaded[b]) cudaEventDestroy(p->ev_loaded[b]);
    if (p->ev_free[b]) cudaEventDestroy(p->ev_free[b]);
  }
  if (p->ev_restore) cudaEventDestroy(p->ev_restore);
  if (p->ev_pick) cudaEventDestroy(p->ev_pick);
  if (p->ev_serial) cudaEventDestroy(p->ev_serial);
  gemm_maps_destroy(p->maps);
  delete p;
}

void prefill_interrupt(PrefillState* p) {
  if (!p || !p->active) return;
  if (p->pending >= 0) {
    // buffer of the streaming layer still holds (in the residency table) the layer two
    // before it: copy that layer's weights back so data and table agree again
    const int b = (p->pending - p->first) & 1;
    const int back = p->pending - 2;
    if (back >= p->first) {
      copy_layer(p, back, b, p->ts);
    }
    cudaEventRecord(p->ev_restore, p->ts);
    cudaStreamWaitEvent(p->cs, p->ev_restore, 0);
  }
  p->active = false;
  p->pending = -1;
  p->next_layer = -1;
}

cudaError_t prefill_layer(PrefillState* p, const PrefillCtx& c, int layer, int T, const uint16_t* x,
                          const float* logits, float* out, ProfEvents* prof, std::string* err) {
  cudaError_t e;
  p->cs = c.cs;
  p->ts = c.ts;
  const int E = p->E, k = p->K;
  auto timed = [&](int kind, auto&& body) -> cudaError_t {
    cudaEvent_t a = nullptr, z = nullptr;
    if (prof) {
      cudaEventCreate(&a);
      cudaEventCreate(&z);
      cudaEventRecord(a, c.cs);
    }
    cudaError_t r = body();
    if (prof) {
      cudaEventRecord(z, c.cs);
      prof->push_back({kind, {a, z}});
    }
    return r;
  };

  // ---- chunk start: take the 2E least recently used slots as the two buffers
  if (!p->active || p->next_layer != layer) {
    prefill_interrupt(p);
    pick_buffers_kernel<<<1, kPickThreads, kPickMaxSlots * sizeof(unsigned long long), c.cs>>>(
        c.res, c.owner, c.stamp, c.S, 2 * E, p->pick_dev);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(p->buf_dev, p->pick_dev, sizeof(int32_t) * 2 * E, cudaMemcpyDeviceToDevice, c.cs)) !=
            cudaSuccess ||
        (e = cudaEventRecord(p->ev_pick, c.cs)) != cudaSuccess || (e = cudaStreamWaitEvent(c.ts, p->ev_pick, 0)))
      return e;
    p->active = true;
    p->first = layer;
    p->pending = -1;
    p->free_recorded[0] = p->free_recorded[1] = false;
  }
  const int b = (layer - p->first) & 1;

  // ---- this layer's weights: already streaming (prefetched) or load now.  With the second
  // buffer off the copy also waits for the previous layer's compute, as a single buffer would.
  if (p->pending != layer) {
    if (!c.overlap && ((e = cudaEventRecord(p->ev_serial, c.cs)) != cudaSuccess ||
                       (e = cudaStreamWaitEvent(c.ts, p->ev_serial, 0)) != cudaSuccess))
      return e;
    if ((e = load_buffer(p, layer, b, prof)) != cudaSuccess) return e;
  }
  p->pending = -1;
  if ((e = cudaStreamWaitEvent(c.cs, p->ev_loaded[b], 0)) != cudaSuccess) return e;
  install_layer_kernel<<<1, 1024, 0, c.cs>>>(layer, E, p->buf_dev + (size_t)b * E, c.res, c.owner, c.stamp, c.st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // ---- stream the whole next layer into the other buffer while this one computes
  if (c.overlap && layer + 1 < p->L) {
    if ((e = load_buffer(p, layer + 1, b ^ 1, prof)) != cudaSuccess) return e;
    p->pending = layer + 1;
  }

  // ---- route the chunk and sort its pairs by expert
  e = timed(4, [&]() -> cudaError_t { return route_chunk(p, c, T, x, logits); });
  if (e != cudaSuccess) return e;

  // ---- grouped GEMMs on the tensor cores
  GemmDesc d{};
  d.n_entries = E + (p->has_shared ? 1 : 0);
  d.E = E;
  d.layer = layer;
  d.I = p->I;
  d.H = p->H;
  d.entry_off = p->entry_off;
  d.tile_off = p->tile_off;
  d.tiles = p->tiles;
  d.buf_slots = p->buf_dev + (size_t)b * E;
  d.pair_tok = p->pair_tok;
  d.pair_gate = p->pair_gate;
  d.h = p->h;
  d.rows = p->rows;
  d.error_word = &c.st->error_word;
  set_weight_info(d, c);
  // while the next layer's copy runs, its CTAs hold kCopySms SMs: the GEMMs take the others
  const int grid = p->pending == layer + 1 ? std::max(1, p->n_sm - kCopySms) : p->n_sm;
  e = timed(5, [&]() -> cudaError_t {
    d.mt = p->I / 64;
    d.kb = p->H / 64;
    return launch_grouped_gemm(0, p->maps, x, T, d, grid, c.cs);
  });
  if (e == cudaSuccess)
    e = timed(8, [&]() -> cudaError_t {
      d.mt = p->H / 128;
      d.kb = p->I / 64;
      return launch_grouped_gemm(1, p->maps, x, T, d, grid, c.cs);
    });
  if (e != cudaSuccess) {
    if (err) *err = "grouped GEMM launch";
    return e;
  }
  e = timed(6, [&]() -> cudaError_t {
    const size_t n = (size_t)T * (p->H / 8);
    prefill_combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, c.cs>>>(p->rows, p->pos_of, p->entry_off, T, k,
                                                                          p->H, E, p->has_shared, out);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return e;
  if ((e = cudaEventRecord(p->ev_free[b], c.cs)) != cudaSuccess) return e;
  p->free_recorded[b] = true;
  if (layer + 1 < p->L) {
    p->next_layer = layer + 1;
  } else {
    p->active = false;
    p->next_layer = -1;
  }
  return cudaSuccess;
}

}  // namespace ft

namespace ft {
namespace {

__global__ void count_prefill_layer_kernel(DevState* st) { st->prefill_layers += 1ull; }

}  // namespace

// One prefill layer when the pool cannot hold two full-layer buffers (S < 2E): the
// experts are loaded on demand instead ("FreeToken 完全拆解", section "全层双缓冲": without
// room for the two buffers, prefill falls back to on-demand loading rather than
// oversubscribing memory).  The chunk is routed first.  Its active experts that are
// resident are hits and are stamped with the step's clock; the others go, in ascending
// id, into the least recently used slots that hold no hit, W at a time when there are
// more misses than such slots, each wave into the same W slots.  Every wave copies its
// experts from the host pool and runs the two grouped GEMMs over its entries (the first
// wave also over the hits and the shared expert); one combine follows.  The decisions are
// taken on the host, between host synchronisations: this path serves pools too small for
// the streamed one, where the host link is the bound anyway.
cudaError_t prefill_layer_on_demand(PrefillState* p, const PrefillCtx& c, int layer, int T, const uint16_t* x,
                                    const float* logits, float* out, ProfEvents* prof, std::string* err) {
  cudaError_t e;
  if (p->active) prefill_interrupt(p);  // a streamed chunk cannot continue here
  p->cs = c.cs;
  p->ts = c.ts;
  const int E = p->E, L = p->L, S = c.S;
  const bool sh = p->has_shared != 0;
  const int n_ent = E + (sh ? 1 : 0);
  auto timed = [&](int kind, auto&& body) -> cudaError_t {
    cudaEvent_t a = nullptr, z = nullptr;
    if (prof) {
      cudaEventCreate(&a);
      cudaEventCreate(&z);
      cudaEventRecord(a, c.cs);
    }
    cudaError_t r = body();
    if (prof) {
      cudaEventRecord(z, c.cs);
      prof->push_back({kind, {a, z}});
    }
    return r;
  };

  // ---- route the chunk, then read its per-expert pair offsets and the residency state
  if ((e = timed(4, [&]() -> cudaError_t { return route_chunk(p, c, T, x, logits); })) != cudaSuccess) return e;
  std::vector<int32_t> eoff(n_ent + 1), res((size_t)L * E), owner(S);
  std::vector<uint32_t> stamp(S);
  uint32_t clock = 0;
  if ((e = cudaMemcpyAsync(eoff.data(), p->entry_off, sizeof(int32_t) * (n_ent + 1), cudaMemcpyDeviceToHost, c.cs)) ||
      (e = cudaMemcpyAsync(res.data(), c.res, sizeof(int32_t) * res.size(), cudaMemcpyDeviceToHost, c.cs)) ||
      (e = cudaMemcpyAsync(owner.data(), c.owner, sizeof(int32_t) * S, cudaMemcpyDeviceToHost, c.cs)) ||
      (e = cudaMemcpyAsync(stamp.data(), c.stamp, sizeof(uint32_t) * S, cudaMemcpyDeviceToHost, c.cs)) ||
      (e = cudaMemcpyAsync(&clock, &c.st->clock, sizeof(uint32_t), cudaMemcpyDeviceToHost, c.cs)) ||
      (e = cudaStreamSynchronize(c.cs)))
    return e;

  // ---- decisions: hits, misses (ascending id), LRU slots outside the hits
  const int base = layer * E;
  std::vector<int> hits, misses;
  for (int x_e = 0; x_e < E; ++x_e) {
    if (eoff[x_e + 1] <= eoff[x_e]) continue;
    (res[base + x_e] >= 0 ? hits : misses).push_back(base + x_e);
  }
  std::vector<char> hit_slot(S, 0);
  for (int u : hits) hit_slot[res[u]] = 1;
  std::vector<int> cand;
  for (int v = 0; v < S; ++v)
    if (!hit_slot[v]) cand.push_back(v);
  if (!misses.empty() && cand.empty()) {
    if (err) *err = "capacity: every slot holds an expert of this layer that the chunk uses";
    return cudaErrorNotSupported;
  }
  std::sort(cand.begin(), cand.end(), [&](int a, int b) { return stamp[a] != stamp[b] ? stamp[a] < stamp[b] : a < b; });
  const int width = std::min((int)cand.size(), (int)misses.size());
  const uint32_t now = clock + 1;
  std::vector<int32_t> slot_of(E, 0);  // slot the GEMM reads for each expert of the layer (idle ones: 0)
  for (int u : hits) {
    stamp[res[u]] = now;
    slot_of[u - base] = res[u];
  }

  // ---- waves
  const int n_waves = misses.empty() ? 1 : ((int)misses.size() + width - 1) / width;
  std::vector<int32_t> toff(n_ent + 1);
  for (int w = 0; w < n_waves; ++w) {
    std::vector<char> in_wave(n_ent, 0);
    if (w == 0) {
      for (int u : hits) in_wave[u - base] = 1;
      if (sh) in_wave[E] = 1;
    }
    const int m0 = w * width, m1 = std::min((int)misses.size(), m0 + width);
    for (int i = m0; i < m1; ++i) {
      const int u = misses[i], v = cand[i - m0];
      if (owner[v] >= 0) res[owner[v]] = -1;
      owner[v] = u;
      res[u] = v;
      stamp[v] = now;
      in_wave[u - base] = 1;
      slot_of[u - base] = v;
      // after the previous wave's GEMMs (same stream), which read this slot
      for (int j = 0; j < p->n_banks; ++j)
        if ((e = cudaMemcpyAsync(p->pool + (size_t)v * p->lay.stride + bank_offset(p->lay, j),
                                 p->bank_host[j] + (size_t)u * p->bank_row[j], p->bank_row[j], cudaMemcpyHostToDevice,
                                 c.cs)) != cudaSuccess)
          return e;
    }
    toff[0] = 0;
    for (int i = 0; i < n_ent; ++i)
      toff[i + 1] = toff[i] + (in_wave[i] ? (eoff[i + 1] - eoff[i] + kTileN - 1) / kTileN : 0);
    if ((e = cudaMemcpyAsync(p->tile_off, toff.data(), sizeof(int32_t) * (n_ent + 1), cudaMemcpyHostToDevice, c.cs)) ||
        (e = cudaMemcpyAsync(p->buf_dev, slot_of.data(), sizeof(int32_t) * E, cudaMemcpyHostToDevice, c.cs)))
      return e;
    prefill_tiles_kernel<<<(n_ent + 255) / 256, 256, 0, c.cs>>>(p->entry_off, p->tile_off, n_ent, p->tiles);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    GemmDesc d{};
    d.n_entries = n_ent;
    d.E = E;
    d.layer = layer;
    d.I = p->I;
    d.H = p->H;
    d.entry_off = p->entry_off;
    d.tile_off = p->tile_off;
    d.tiles = p->tiles;
    d.buf_slots = p->buf_dev;
    d.pair_tok = p->pair_tok;
    d.pair_gate = p->pair_gate;
    d.h = p->h;
    d.rows = p->rows;
    d.error_word = &c.st->error_word;
    set_weight_info(d, c);
    e = timed(5, [&]() -> cudaError_t {
      d.mt = p->I / 64;
      d.kb = p->H / 64;
      return launch_grouped_gemm(0, p->maps, x, T, d, p->n_sm, c.cs);
    });
    if (e == cudaSuccess)
      e = timed(8, [&]() -> cudaError_t {
        d.mt = p->H / 128;
        d.kb = p->I / 64;
        return launch_grouped_gemm(1, p->maps, x, T, d, p->n_sm, c.cs);
      });
    if (e != cudaSuccess) {
      if (err) *err = "grouped GEMM launch";
      return e;
    }
    // the host arrays above are rewritten by the next wave: let this wave's copies finish
    if ((e = cudaStreamSynchronize(c.cs)) != cudaSuccess) return e;
  }

  // ---- residency state back, then the fixed-order combine
  if ((e = cudaMemcpyAsync(c.res, res.data(), sizeof(int32_t) * res.size(), cudaMemcpyHostToDevice, c.cs)) ||
      (e = cudaMemcpyAsync(c.owner, owner.data(), sizeof(int32_t) * S, cudaMemcpyHostToDevice, c.cs)) ||
      (e = cudaMemcpyAsync(c.stamp, stamp.data(), sizeof(uint32_t) * S, cudaMemcpyHostToDevice, c.cs)) ||
      (e = cudaMemcpyAsync(&c.st->clock, &now, sizeof(uint32_t), cudaMemcpyHostToDevice, c.cs)))
    return e;
  count_prefill_layer_kernel<<<1, 1, 0, c.cs>>>(c.st);
  e = timed(6, [&]() -> cudaError_t {
    const size_t n = (size_t)T * (p->H / 8);
    prefill_combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, c.cs>>>(p->rows, p->pos_of, p->entry_off, T, p->K,
                                                                          p->H, E, p->has_shared, out);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return e;
  // the host copies of the state are locals: they must be read before returning
  if ((e = cudaStreamSynchronize(c.cs)) != cudaSuccess) return e;
  p->active = false;
  p->next_layer = -1;
  return cudaSuccess;
}

}  // namespace ft
