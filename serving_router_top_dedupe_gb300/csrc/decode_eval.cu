// Decode-side data movement and expert evaluation.
//
//  fill_kernel        F-set fill: copies whole experts (every bank) from the mapped
//                     host pool into their victim slots, driven by the device copy
//                     list and its valid count ("FreeToken 完全拆解", section
//                     "Device-side 缓存控制": one fixed-shape launch across all banks).
//  gate_up_kernel     h = silu(W_g x) * (W_u x) for every (entry, token) of G = H u F
//                     plus the shared expert.
//  down_combine_kernel y = W_d h, pair row = g * y, and per row block the last CTA to
//                     finish sums shared + the k pair rows (GPU row, or the caller's
//                     c_partial row for C pairs) in ascending expert id.
//
// GEMV design for HBM: every weight byte is read once with 16-byte streaming loads,
// one warp per row, all of a row's loads issued before any arithmetic.  The reduction
// order of each (token, expert) dot product is fixed (lane-strided chunks, then an xor
// butterfly), independent of slot, batch composition or split, so outputs are identical
// across cache capacities.  FP8 E4M3 rows are decoded with the hardware e4m3x2->f16x2
// conversion; each 1x128 block's dot product is summed over the 8 lanes holding its chunks
// and then multiplied by its FP32 scale once ("OSDI'26 | 双路 CPU + 两张 5090…", §4.2,
// post-scaling).  FP8 and FP4 activations enter as F16 after an exact per-token
// power-of-two prescale (act_shift), undone on the finished sum.  The block-FP4 formats named in
// "FreeToken 完全拆解" (section 主结果) take the same order: E2M1 pairs are decoded with the
// hardware e2m1x2->f16x2 conversion, each block's partial dot (16 elements for NVFP4, 32 for
// MXFP4) is multiplied by its scale (E4M3, or E8M0 = 2^(code-127)), and NVFP4's per-bank FP32
// tensor scale multiplies the finished row sum.
#include <cuda_fp16.h>

#include <algorithm>

#include "ft_internal.cuh"
#include "ft_dot.cuh"
#include "ft_ptx.cuh"

namespace ft {
namespace {

using namespace dot;

// E8M0 scale code -> float: 2^(code - 127), built from the float's exponent field
// (code 0 is the subnormal 2^-127; code 255, NaN in the format, is never written).
__device__ __forceinline__ float e8m0_to_float(uint32_t code) {
  return __uint_as_float(code ? code << 23 : 0x00400000u);
}

// ------------------------------------------------------------------------- fill
// Work = q experts x n_banks contiguous segments.  CTA b copies a share of segment
// b mod nseg (addresses computed once per segment), issuing FILL_UNROLL 16-byte loads
// from the mapped host pool before storing any, so the grid keeps ~0.5 MB of host reads
// in flight: one 6 MB expert then moves at the host link's rate.
//
// The grid is a few CTAs on SMs of their own.  A streaming CTA that shares an SM with a
// fill CTA stalls behind the fill's host loads until the fill ends (measured on GB300:
// such SMs finished their share of the resident experts ~33 us late, at the fill's end,
// while the other SMs took ~11 us), so each fill CTA reserves enough shared memory that
// no batch-1 GEMV CTA is placed beside it, and the GEMV runs on the remaining SMs.  The
// next layer's control CTA still fits beside a fill CTA.
constexpr int FILL_UNROLL = 4;

__device__ __forceinline__ void copy_segment(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n16,
                                             size_t first, size_t stride) {
  for (size_t base = first; base < n16; base += stride * FILL_UNROLL) {
    uint4 v[FILL_UNROLL];
#pragma unroll
    for (int u = 0; u < FILL_UNROLL; ++u) {
      const size_t c = base + u * stride;
      if (c < n16) v[u] = ld_host(src + c);
    }
#pragma unroll
    for (int u = 0; u < FILL_UNROLL; ++u) {
      const size_t c = base + u * stride;
      if (c < n16) dst[c] = v[u];
    }
  }
}

// The kernel is launched while the control kernel right before still runs.  When that kernel
// took its decisions early and none of its victim slots belongs to the previous layer-step,
// it has released a copy list tagged with this step's clock: the copy starts at once, while
// warp 0 waits for the control kernel to complete and only then lets the evaluation kernel
// launch (whose prologue reads the control kernel's lists).  Otherwise every thread waits and
// the list comes from the published work lists.  Both lists hold the same entries.
__global__ void __launch_bounds__(kFillThreads) fill_kernel(FillParams p) {
  __shared__ int s_early;  // 0, or 1 + the parity of the early list
  if (threadIdx.x == 0) {
    int e = 0;
    if (p.pdl && p.ecopy != nullptr) {
      const uint32_t expect = *reinterpret_cast<const volatile uint32_t*>(&p.st->clock) + 1u;
      const int32_t* l = p.ecopy + (size_t)(expect & 1u) * (2 + 2 * p.kmax);
      if (ptx::ld_acquire_gpu(reinterpret_cast<const uint32_t*>(l)) == expect) e = 1 + (int)(expect & 1u);
    }
    s_early = e;
  }
  __syncthreads();
  // warp 0 lets the evaluation launch once the control kernel is done; the other warps copy.
  // The copy's split over threads is the same on both paths, since CTAs of one launch can
  // take different paths (a CTA that starts after the control kernel published its clock
  // finds no early list).
  if (threadIdx.x < 32) {
    pdl_wait();
    pdl_trigger();
    return;
  }
  const int early = s_early;
  const int ct = threadIdx.x - 32, nct = blockDim.x - 32;  // copying threads
  const int32_t *copy_u = p.copy_u, *copy_slot = p.copy_slot;
  int q;
  if (early) {
    const int32_t* l = p.ecopy + (size_t)(early - 1) * (2 + 2 * p.kmax);
    q = l[1];
    copy_u = l + 2;
    copy_slot = l + 2 + p.kmax;
  } else {
    pdl_wait();  // the copy list comes from the control kernel right before
    q = p.counts[C_Q];
  }
  if (q <= 0) return;
  const int nseg = q * p.n_banks;
  const int G = gridDim.x;
  for (int sgi = nseg >= G ? blockIdx.x : blockIdx.x % nseg; sgi < nseg; sgi += G) {
    const int i = sgi / p.n_banks, j = sgi - i * p.n_banks;
    // CTAs sharing this segment: those with the same residue mod nseg (all of them when nseg < G)
    const int part = nseg >= G ? 0 : blockIdx.x / nseg;
    const int nparts = nseg >= G ? 1 : (G - 1 - sgi) / nseg + 1;
    size_t nbytes, doff;
    const uint8_t* sb;
    switch (j) {
      case 0: nbytes = p.src_row[0]; doff = p.lay.gate; sb = p.src[0]; break;
      case 1: nbytes = p.src_row[1]; doff = p.lay.up; sb = p.src[1]; break;
      case 2: nbytes = p.src_row[2]; doff = p.lay.down; sb = p.src[2]; break;
      case 3: nbytes = p.src_row[3]; doff = p.lay.gs; sb = p.src[3]; break;
      case 4: nbytes = p.src_row[4]; doff = p.lay.us; sb = p.src[4]; break;
      case 5: nbytes = p.src_row[5]; doff = p.lay.ds; sb = p.src[5]; break;
      default: nbytes = p.src_row[6]; doff = p.lay.ts; sb = p.src[6]; break;
    }
    const int uid = copy_u[i];
    const uint4* src = reinterpret_cast<const uint4*>(sb + (size_t)uid * nbytes);
    uint4* dst = reinterpret_cast<uint4*>(p.pool + (size_t)copy_slot[i] * p.lay.stride + doff);
    copy_segment(src, dst, nbytes / 16, (size_t)part * nct + ct, (size_t)nparts * nct);
    if (nseg < G) break;  // one segment share per CTA
  }
}

// ------------------------------------------------------------- work items
// Items of the batched kernels: (entry g, row block rb, chunk ch of TG of the entry's
// tokens), chunks innermost, so that the chunks of one row block run on neighbouring CTAs at
// the same time and share its weight rows through L2.  An entry with many tokens (the shared
// expert takes all B) is thus spread over many CTAs instead of one CTA looping over its
// chunks.  pref[g] = items before entry g (block-wide prefix, by warp 0); returns the total.
template <int TG>
__device__ int item_prefix(const int32_t* g_off, int ne, int rows_blocks, int* pref) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    int carry = 0;
    for (int c0 = 0; c0 < ne; c0 += 32) {
      const int g = c0 + lane;
      const int v = g < ne ? (g_off[g + 1] - g_off[g] + TG - 1) / TG * rows_blocks : 0;
      int incl = v;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (g < ne) pref[g] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pref[ne] = carry;
  }
  __syncthreads();
  return pref[ne];
}

// item -> (entry, row block, chunk): the last entry whose prefix is <= item
__device__ __forceinline__ void item_decode(const int* pref, int ne, const int32_t* g_off, int item, int TG, int& g,
                                            int& rb, int& ch) {
  int lo = 0, hi = ne - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= item) lo = mid;
    else hi = mid - 1;
  }
  g = lo;
  const int nch = (g_off[g + 1] - g_off[g] + TG - 1) / TG;
  const int local = item - pref[g];
  rb = local / nch;
  ch = local - rb * nch;
}

// ---------------------------------------------------------------- gate / up
// Work item = (entry, block of 8 rows of I, chunk of TG tokens): warp w computes row
// 8*rb + w for the chunk's tokens, staged in shared memory.
template <int WT, int SEG, int TG>
__global__ void __launch_bounds__(kEvalThreads) gate_up_kernel(EvalParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_wait();  // filled slots are written by the kernel right before
  const uint64_t pol = ptx::l2_evict_first();
  pdl_trigger();
  const int ne = p.counts[C_NENTRIES];
  const int I = p.I, H = p.H;
  const int rbs = I / 8;
  __shared__ int s_pref[kMaxE + 3];
  const int n_items = item_prefix<TG>(p.g_off, ne, rbs, s_pref);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int EPC = WT == FT_W_BF16 ? 8 : (WT == FT_W_FP8_E4M3_B128 ? 16 : 32);  // elements per 16-byte chunk
  const int row_chunks = H / EPC;
  // x tile: BF16 path keeps raw bf16 (2 B); FP8 and FP4 paths keep f16 (2 B) -> H*2 bytes per token
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  __shared__ int s_shift[TG];  // FP8 / FP4: per-token power-of-two prescale of x (act_shift)

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    int g, rb, ch;
    item_decode(s_pref, ne, p.g_off, item, TG, g, rb, ch);
    const int i = rb * 8 + warp;
    const uint8_t* W = p.g_w[g];
    const uint8_t* wg = W + p.lay.gate + (size_t)i * row_chunks * 16;
    const uint8_t* wu = W + p.lay.up + (size_t)i * row_chunks * 16;
    const float* sg = reinterpret_cast<const float*>(W + p.lay.gs) + (size_t)i * (H / 128);
    const float* su = reinterpret_cast<const float*>(W + p.lay.us) + (size_t)i * (H / 128);
    // NVFP4: two E4M3 block scales per 16-byte chunk, read as one 16-bit word;
    // MXFP4: one E8M0 block scale per 16-byte chunk
    const uint16_t* bg = reinterpret_cast<const uint16_t*>(W + p.lay.gs) + (size_t)i * (H / 32);
    const uint16_t* bu = reinterpret_cast<const uint16_t*>(W + p.lay.us) + (size_t)i * (H / 32);
    const uint8_t* mg = W + p.lay.gs + (size_t)i * (H / 32);
    const uint8_t* mu = W + p.lay.us + (size_t)i * (H / 32);
    const int p0 = p.g_off[g], np = p.g_off[g + 1] - p0;
    const bool shared_entry = p.has_shared && g == ne - 1;
    {
      const int t0 = ch * TG;
      const int nt = min(TG, np - t0);
      __syncthreads();
      if (WT != FT_W_BF16) {  // one warp per token: the exponent of its largest |x|
        for (int tt = warp; tt < nt; tt += kEvalThreads / 32) {
          const int pr = p.g_pair[p0 + t0 + tt];
          const uint16_t* xr = p.x + (size_t)(shared_entry ? pr : pr / p.k) * H;
          uint32_t m = 0;
          for (int c8 = lane; c8 < H / 8; c8 += 32) m = bf16x8_maxbits(*reinterpret_cast<const uint4*>(xr + c8 * 8), m);
          m = __reduce_max_sync(0xffffffffu, m);
          if (lane == 0) s_shift[tt] = act_shift(m);
        }
        __syncthreads();
      }
      for (int idx = threadIdx.x; idx < nt * (H / 8); idx += blockDim.x) {
        const int tt = idx / (H / 8), c8 = idx - tt * (H / 8);
        const int pr = p.g_pair[p0 + t0 + tt];
        const int tok = shared_entry ? pr : pr / p.k;
        uint4 v = *reinterpret_cast<const uint4*>(p.x + (size_t)tok * H + c8 * 8);
        if (WT != FT_W_BF16) v = bf16x8_to_f16x8_scaled(v, pow2i(-s_shift[tt]));  // exact
        *reinterpret_cast<uint4*>(xs + (size_t)tt * H + c8 * 8) = v;
      }
      __syncthreads();
      float acc_a[TG], acc_b[TG];
#pragma unroll
      for (int tt = 0; tt < TG; ++tt) acc_a[tt] = acc_b[tt] = 0.f;
      for (int c0 = 0; c0 < row_chunks; c0 += 32 * SEG) {
        uint4 wa[SEG], wb[SEG];
#pragma unroll
        for (int s = 0; s < SEG; ++s) {
          const int c = c0 + s * 32 + lane;
          if (c < row_chunks) {
            wa[s] = ld_stream(wg + (size_t)c * 16, pol);
            wb[s] = ld_stream(wu + (size_t)c * 16, pol);
          }
        }
#pragma unroll
        for (int s = 0; s < SEG; ++s) {
          const int c = c0 + s * 32 + lane;
          if (c < row_chunks) {
            if (WT == FT_W_BF16) {
#pragma unroll
              for (int tt = 0; tt < TG; ++tt) {
                if (tt < nt) {
                  const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)tt * H + c * 8);
                  acc_a[tt] = dot_bf16_bf16(wa[s], xv, acc_a[tt]);
                  acc_b[tt] = dot_bf16_bf16(wb[s], xv, acc_b[tt]);
                }
              }
            } else if (WT == FT_W_FP8_E4M3_B128) {
              const float scg = __ldg(sg + c / 8), scu = __ldg(su + c / 8);
#pragma unroll
              for (int tt = 0; tt < TG; ++tt) {
                if (tt < nt) {
                  const uint4* xp = reinterpret_cast<const uint4*>(xs + (size_t)tt * H + c * 16);
                  const uint4 xa = xp[0], xb = xp[1];
                  // the 1x128 block's dot product over its 8 lanes, then its scale once
                  acc_a[tt] = fmaf(group8_sum(dot_e4m3_f16(wa[s], xa, xb)), scg, acc_a[tt]);
                  acc_b[tt] = fmaf(group8_sum(dot_e4m3_f16(wb[s], xa, xb)), scu, acc_b[tt]);
                }
              }
            } else if (WT == FT_W_MXFP4) {
              const float scg = e8m0_to_float(__ldg(mg + c)), scu = e8m0_to_float(__ldg(mu + c));
#pragma unroll
              for (int tt = 0; tt < TG; ++tt) {
                if (tt < nt) {
                  const uint4* xp = reinterpret_cast<const uint4*>(xs + (size_t)tt * H + c * 32);
                  const uint4 x0 = xp[0], x1 = xp[1], x2 = xp[2], x3 = xp[3];
                  const float da = dot16_e2m1_f16(wa[s].x, wa[s].y, x0, x1) + dot16_e2m1_f16(wa[s].z, wa[s].w, x2, x3);
                  const float db = dot16_e2m1_f16(wb[s].x, wb[s].y, x0, x1) + dot16_e2m1_f16(wb[s].z, wb[s].w, x2, x3);
                  acc_a[tt] = fmaf(da, scg, acc_a[tt]);
                  acc_b[tt] = fmaf(db, scu, acc_b[tt]);
                }
              }
            } else {
              const float2 sg2 = e4m3x2_to_float2(__ldg(bg + c)), su2 = e4m3x2_to_float2(__ldg(bu + c));
#pragma unroll
              for (int tt = 0; tt < TG; ++tt) {
                if (tt < nt) {
                  const uint4* xp = reinterpret_cast<const uint4*>(xs + (size_t)tt * H + c * 32);
                  const uint4 x0 = xp[0], x1 = xp[1], x2 = xp[2], x3 = xp[3];
                  acc_a[tt] = fmaf(dot16_e2m1_f16(wa[s].x, wa[s].y, x0, x1), sg2.x, acc_a[tt]);
                  acc_a[tt] = fmaf(dot16_e2m1_f16(wa[s].z, wa[s].w, x2, x3), sg2.y, acc_a[tt]);
                  acc_b[tt] = fmaf(dot16_e2m1_f16(wb[s].x, wb[s].y, x0, x1), su2.x, acc_b[tt]);
                  acc_b[tt] = fmaf(dot16_e2m1_f16(wb[s].z, wb[s].w, x2, x3), su2.y, acc_b[tt]);
                }
              }
            }
          }
        }
      }
      // NVFP4: the banks' tensor scales multiply the finished sums
      const float tsa = WT == FT_W_NVFP4 ? __ldg(reinterpret_cast<const float*>(W + p.lay.ts)) : 1.f;
      const float tsb = WT == FT_W_NVFP4 ? __ldg(reinterpret_cast<const float*>(W + p.lay.ts) + 1) : 1.f;
#pragma unroll
      for (int tt = 0; tt < TG; ++tt) {
        // FP8: every lane of a block group holds the group's sum; FP8 / FP4: undo the prescale
        const float xsc = WT == FT_W_BF16 ? 1.f : pow2i(tt < nt ? s_shift[tt] : 0);
        const float a = (WT == FT_W_FP8_E4M3_B128 ? groups_sum(acc_a[tt]) : warp_sum(acc_a[tt])) * xsc;
        const float b = (WT == FT_W_FP8_E4M3_B128 ? groups_sum(acc_b[tt]) : warp_sum(acc_b[tt])) * xsc;
        if (lane == 0 && tt < nt)
          p.h[(size_t)(p0 + t0 + tt) * I + i] = WT == FT_W_NVFP4 ? silu_mul(a * tsa, b * tsb) : silu_mul(a, b);
      }
    }
  }
}

// ------------------------------------------------------------ down + combine
// Work item = (entry, block of 32 output rows): warp w computes rows 32*rb + 4w .. +3.
// (Spreading an entry's token chunks over CTAs, as the gate/up kernel does, measured slower
// here: 514 against 416 us at batch 64, 136 against 129 at batch 16, with one combine arrival
// per chunk.)
template <int WT, int RPW, int TG>
// BF16: registers capped for three CTAs per SM (80, no spill; the uncapped build took 116 and
// two CTAs: batch 16 down 122 -> 117 us); the FP8 / FP4 forms keep two CTAs per SM
__global__ void __launch_bounds__(kEvalThreads, WT == FT_W_BF16 ? 3 : 2) down_combine_kernel(EvalParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_wait();
  const uint64_t pol = ptx::l2_evict_first();
  pdl_trigger();
  __shared__ int s_last;
  __shared__ uint8_t s_gpu_pair[kMaxPairs];  // combine: pair evaluated on the GPU (else host row)
  const int ne = p.counts[C_NENTRIES];
  const int I = p.I, H = p.H, k = p.k, B = p.B;
  constexpr int R2 = 8 * RPW;
  static_assert(R2 == kRowsPerItem2, "row block");
  const int nrb = H / R2;
  const int n_items = ne * nrb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int EPC = WT == FT_W_BF16 ? 8 : (WT == FT_W_FP8_E4M3_B128 ? 16 : 32);  // elements per 16-byte chunk
  const int row_chunks = I / EPC;
  float* hs = reinterpret_cast<float*>(smem);  // [TG][I]

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    // entries in the order ne-1, 0, 1, ..: the shared expert, which takes all B tokens and so
    // the longest items, goes first instead of forming the tail
    const int gi = item / nrb, rb = item - gi * nrb;
    const int g = gi == 0 ? ne - 1 : gi - 1;
    const uint8_t* W = p.g_w[g];
    const int p0 = p.g_off[g], np = p.g_off[g + 1] - p0;
    const bool shared_entry = p.has_shared && g == ne - 1;
    const int j0 = rb * R2 + warp * RPW;
    constexpr int SEG = WT == FT_W_BF16 ? 2 : 4;
    // BF16 rows of one K segment (I <= 512) are loaded once per item, before h is staged:
    // their HBM latency then overlaps the staging, and every token chunk reuses them
    const bool early_w = WT == FT_W_BF16 && row_chunks <= 32 * SEG;
    uint4 wv[RPW][SEG];
    if (early_w) {
#pragma unroll
      for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int s = 0; s < SEG; ++s) {
          const int c = s * 32 + lane;
          if (c < row_chunks)
            wv[r][s] = ld_stream(W + p.lay.down + (size_t)(j0 + r) * row_chunks * 16 + (size_t)c * 16, pol);
        }
    }
    for (int t0 = 0; t0 < np; t0 += TG) {
      const int nt = min(TG, np - t0);
      // lane tt holds the chunk's pair tt and its gate, loaded while h is staged
      int my_pr = 0;
      if (lane < nt) my_pr = p.g_pair[p0 + t0 + lane];
      __syncthreads();
      for (int idx = threadIdx.x; idx < nt * (I / 4); idx += blockDim.x) {
        const int tt = idx / (I / 4), c4 = idx - tt * (I / 4);
        *reinterpret_cast<float4*>(hs + (size_t)tt * I + c4 * 4) =
            *reinterpret_cast<const float4*>(p.h + (size_t)(p0 + t0 + tt) * I + c4 * 4);
      }
      const float my_gate = lane < nt && !shared_entry ? p.gates[my_pr] : 0.f;
      __syncthreads();
      float acc[RPW][TG];
#pragma unroll
      for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int tt = 0; tt < TG; ++tt) acc[r][tt] = 0.f;
      for (int c0 = 0; c0 < row_chunks; c0 += 32 * SEG) {
        if (!early_w) {
#pragma unroll
          for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int s = 0; s < SEG; ++s) {
              const int c = c0 + s * 32 + lane;
              if (c < row_chunks)
                wv[r][s] = ld_stream(W + p.lay.down + (size_t)(j0 + r) * row_chunks * 16 + (size_t)c * 16, pol);
            }
        }
#pragma unroll
        for (int s = 0; s < SEG; ++s) {
          const int c = c0 + s * 32 + lane;
          if (WT == FT_W_FP8_E4M3_B128) {
            // row_chunks is a multiple of 8, so a block's 8 lanes are all live or all idle;
            // the shuffles of the block sum run on every lane of the warp
            if (c0 + s * 32 >= row_chunks) break;
            const bool cv = c < row_chunks;
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
              const float sc = cv ? __ldg(reinterpret_cast<const float*>(W + p.lay.ds) + (size_t)(j0 + r) * (I / 128) +
                                          c / 8)
                                  : 0.f;
#pragma unroll
              for (int tt = 0; tt < TG; ++tt)
                if (tt < nt) {
                  const float d = group8_sum(cv ? dot_e4m3_f32(wv[r][s], hs + (size_t)tt * I + c * 16) : 0.f);
                  acc[r][tt] = fmaf(d, sc, acc[r][tt]);
                }
            }
            continue;
          }
          if (c < row_chunks) {
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
              if (WT == FT_W_BF16) {
#pragma unroll
                for (int tt = 0; tt < TG; ++tt)
                  if (tt < nt) acc[r][tt] = dot_bf16_f32(wv[r][s], hs + (size_t)tt * I + c * 8, acc[r][tt]);
              } else if (WT == FT_W_MXFP4) {
                const float sd = e8m0_to_float(__ldg(W + p.lay.ds + (size_t)(j0 + r) * (I / 32) + c));
#pragma unroll
                for (int tt = 0; tt < TG; ++tt)
                  if (tt < nt) {
                    const float* hv = hs + (size_t)tt * I + c * 32;
                    const float d = dot16_e2m1_f32(wv[r][s].x, wv[r][s].y, hv) + dot16_e2m1_f32(wv[r][s].z, wv[r][s].w, hv + 16);
                    acc[r][tt] = fmaf(d, sd, acc[r][tt]);
                  }
              } else {
                const float2 sd = e4m3x2_to_float2(
                    __ldg(reinterpret_cast<const uint16_t*>(W + p.lay.ds) + (size_t)(j0 + r) * (I / 32) + c));
#pragma unroll
                for (int tt = 0; tt < TG; ++tt)
                  if (tt < nt) {
                    const float* hv = hs + (size_t)tt * I + c * 32;
                    acc[r][tt] = fmaf(dot16_e2m1_f32(wv[r][s].x, wv[r][s].y, hv), sd.x, acc[r][tt]);
                    acc[r][tt] = fmaf(dot16_e2m1_f32(wv[r][s].z, wv[r][s].w, hv + 16), sd.y, acc[r][tt]);
                  }
              }
            }
          }
        }
      }
      const float tsd = WT == FT_W_NVFP4 ? __ldg(reinterpret_cast<const float*>(W + p.lay.ts) + 2) : 1.f;
#pragma unroll
      for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int tt = 0; tt < TG; ++tt) {
          const float y = WT == FT_W_NVFP4 ? warp_sum(acc[r][tt]) * tsd
                                           : (WT == FT_W_FP8_E4M3_B128 ? groups_sum(acc[r][tt]) : warp_sum(acc[r][tt]));
          const int pr = __shfl_sync(0xffffffffu, my_pr, tt);
          const float gate = __shfl_sync(0xffffffffu, my_gate, tt);
          if (lane == 0 && tt < nt) {
            if (shared_entry) p.shared_rows[(size_t)pr * H + j0 + r] = y;
            else p.rows[(size_t)pr * H + j0 + r] = gate * y;
          }
        }
    }
    // arrival at this row block; the last entry to arrive combines it
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const uint32_t prev = atomicAdd(p.blk_count + rb, 1u);
      s_last = prev == (uint32_t)(ne - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      // which pairs run on the GPU, read once; then per output the k rows' loads are issued
      // together (L2 loads of the other CTAs' rows) and summed in the fixed order: the shared
      // row, then r ascending
      for (int i = threadIdx.x; i < B * k; i += blockDim.x) s_gpu_pair[i] = p.slot_of_pair[i] >= 0;
      __syncthreads();
      for (int idx = threadIdx.x; idx < B * R2; idx += blockDim.x) {
        const int t = idx / R2, j = rb * R2 + (idx - t * R2);
        float o = p.has_shared ? __ldcg(p.shared_rows + (size_t)t * H + j) : 0.f;
#pragma unroll 4
        for (int r = 0; r < k; ++r) {
          const int pr = t * k + r;
          float v = 0.f;
          if (s_gpu_pair[pr]) {
            v = __ldcg(p.rows + (size_t)pr * H + j);
          } else if (p.c_partial) {
            v = p.c_partial[(size_t)pr * H + j];
          } else if (j == 0) {
            atomicOr(p.error_word, FT_DEVERR_CAPACITY);
          }
          o += v;
        }
        p.out[(size_t)t * H + j] = o;
      }
      if (threadIdx.x == 0) p.blk_count[rb] = 0u;
    }
  }
}

template <int WT, int SEG, int TG>
cudaError_t gate_up_launch(const EvalParams& p, int grid, cudaStream_t s) {
  return launch_k(gate_up_kernel<WT, SEG, TG>, dim3(grid), dim3(kEvalThreads), (size_t)TG * p.H * 2, s, p.pdl, p);
}

template <int WT, int TG>
cudaError_t down_launch(const EvalParams& p, int grid, cudaStream_t s) {
  return launch_k(down_combine_kernel<WT, 4, TG>, dim3(grid), dim3(kEvalThreads), (size_t)TG * p.I * 4, s, p.pdl,
                  p);
}

template <typename F>
cudaError_t set_smem(F f, size_t bytes) {
  return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_fill(const FillParams& p, int grid, cudaStream_t s) {
  return launch_k(fill_kernel, dim3(grid), dim3(kFillThreads), kFillSmemReserve, s, p.pdl, p);
}

bool eval_fused(const EvalParams& p, int wtype) {
  return p.B == 1 && p.allow_fused &&
         fused_gemv_supported(wtype, p.H, p.I, batch1_entries(p), p.n_sm);
}

cudaError_t launch_gate_up(const EvalParams& p, int wtype, int grid, cudaStream_t s) {
  if (eval_fused(p, wtype)) return launch_fused_gemv(p, wtype, p.n_sm, batch1_entries(p), s);
  const bool one = p.B == 1;
  if (wtype == FT_W_BF16) {
    return one ? gate_up_launch<FT_W_BF16, 8, 1>(p, grid, s) : gate_up_launch<FT_W_BF16, 8, 4>(p, grid, s);
  }
  if (wtype == FT_W_NVFP4)
    return one ? gate_up_launch<FT_W_NVFP4, 4, 1>(p, grid, s) : gate_up_launch<FT_W_NVFP4, 4, 4>(p, grid, s);
  if (wtype == FT_W_MXFP4)
    return one ? gate_up_launch<FT_W_MXFP4, 4, 1>(p, grid, s) : gate_up_launch<FT_W_MXFP4, 4, 4>(p, grid, s);
  return one ? gate_up_launch<FT_W_FP8_E4M3_B128, 7, 1>(p, grid, s)
             : gate_up_launch<FT_W_FP8_E4M3_B128, 7, 4>(p, grid, s);
}

cudaError_t prepare_kernels(int wtype, int H, int I) {
  cudaError_t e = cudaSuccess;
  if ((e = prepare_fused_gemv()) != cudaSuccess) return e;
  if ((e = set_smem(fill_kernel, kFillSmemReserve)) != cudaSuccess) return e;
  const size_t gu1 = (size_t)H * 2, gu4 = 4 * gu1, dn1 = (size_t)I * 4, dn4 = 4 * dn1;
  if (wtype == FT_W_BF16) {
    if ((e = set_smem(gate_up_kernel<FT_W_BF16, 8, 1>, gu1)) != cudaSuccess) return e;
    if ((e = set_smem(gate_up_kernel<FT_W_BF16, 8, 4>, gu4)) != cudaSuccess) return e;
    if ((e = set_smem(down_combine_kernel<FT_W_BF16, 4, 1>, dn1)) != cudaSuccess) return e;
    e = set_smem(down_combine_kernel<FT_W_BF16, 4, 4>, dn4);
  } else if (wtype == FT_W_NVFP4) {
    if ((e = set_smem(gate_up_kernel<FT_W_NVFP4, 4, 1>, gu1)) != cudaSuccess) return e;
    if ((e = set_smem(gate_up_kernel<FT_W_NVFP4, 4, 4>, gu4)) != cudaSuccess) return e;
    if ((e = set_smem(down_combine_kernel<FT_W_NVFP4, 4, 1>, dn1)) != cudaSuccess) return e;
    e = set_smem(down_combine_kernel<FT_W_NVFP4, 4, 4>, dn4);
  } else if (wtype == FT_W_MXFP4) {
    if ((e = set_smem(gate_up_kernel<FT_W_MXFP4, 4, 1>, gu1)) != cudaSuccess) return e;
    if ((e = set_smem(gate_up_kernel<FT_W_MXFP4, 4, 4>, gu4)) != cudaSuccess) return e;
    if ((e = set_smem(down_combine_kernel<FT_W_MXFP4, 4, 1>, dn1)) != cudaSuccess) return e;
    e = set_smem(down_combine_kernel<FT_W_MXFP4, 4, 4>, dn4);
  } else {
    if ((e = set_smem(gate_up_kernel<FT_W_FP8_E4M3_B128, 7, 1>, gu1)) != cudaSuccess) return e;
    if ((e = set_smem(gate_up_kernel<FT_W_FP8_E4M3_B128, 7, 4>, gu4)) != cudaSuccess) return e;
    if ((e = set_smem(down_combine_kernel<FT_W_FP8_E4M3_B128, 4, 1>, dn1)) != cudaSuccess) return e;
    e = set_smem(down_combine_kernel<FT_W_FP8_E4M3_B128, 4, 4>, dn4);
  }
  return e;
}

cudaError_t launch_down_combine(const EvalParams& p, int wtype, int grid, cudaStream_t s) {
  if (eval_fused(p, wtype)) return cudaSuccess;  // the fused batch-1 kernel did the whole layer
  const bool one = p.B == 1;
  if (wtype == FT_W_BF16) return one ? down_launch<FT_W_BF16, 1>(p, grid, s) : down_launch<FT_W_BF16, 4>(p, grid, s);
  if (wtype == FT_W_NVFP4) return one ? down_launch<FT_W_NVFP4, 1>(p, grid, s) : down_launch<FT_W_NVFP4, 4>(p, grid, s);
  if (wtype == FT_W_MXFP4) return one ? down_launch<FT_W_MXFP4, 1>(p, grid, s) : down_launch<FT_W_MXFP4, 4>(p, grid, s);
  return one ? down_launch<FT_W_FP8_E4M3_B128, 1>(p, grid, s) : down_launch<FT_W_FP8_E4M3_B128, 4>(p, grid, s);
}

}  // namespace ft
