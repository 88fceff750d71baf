// Decode expert evaluation at batch 1 in one persistent launch: gate/up GEMV + SwiGLU,
// down GEMV and the fixed-order combine, for BF16, FP8 (E4M3, 1x128 FP32 block scales) and the
// block-FP4 formats (NVFP4, MXFP4).
//
// A decode layer reads every byte of its G-set experts once (about 1 FLOP per byte), so
// it is bound by HBM, and at batch 1 a layer is only ~10 us of traffic: what costs is
// every point where the weight stream stops.  One CTA per SM keeps up to ~190 KB of weight
// rows in flight in a ring of shared-memory stages filled by cp.async.bulk, and the same
// ring carries both halves of the layer:
//
//  phase 0 (gate/up): units (entry, row i), split evenly over the CTAs; a stage holds gate
//                     rows i0.. and the same up rows of one entry; a consumer warp forms
//                     a = W_g[i].x, b = W_u[i].x and writes h[g][i] = silu(a)*b.
//  phase 1 (down):    each CTA owns output rows j0..j0+nj-1 and streams W_down[g][j] of
//                     every entry g for them.  These rows do not depend on h, so the
//                     producer streams them right behind its phase-0 rows; only the
//                     consumers wait, until every CTA has published its h rows.
//  combine:           out[j] = shared + the k pair rows in ascending expert id (GPU row
//                     gate_r * y, or the caller's c_partial row for a host-evaluated pair).
//
// Both phases run twice: first for the experts resident before the step, then, once the
// fill kernel of the step has completed, for the experts it filled.  While a fill crosses
// the host link, the resident experts' whole layer (both phases) is evaluated; after it,
// only the filled experts' rows remain, spread over every CTA.
//
// The hand-off between the phases is a per-entry counter that each CTA raises by the h rows
// it wrote (release), and that consumers wait on (acquire, bounded).  It needs every CTA to
// be resident: the grid is one CTA per SM and a CTA takes more than half of an SM's shared
// memory, and no kernel this grid could wait behind depends on it.
//
// Per (entry, row) the lane-strided 16-byte chunk order and the xor butterfly are those of
// the batched decode kernels, so results are bit-identical to them.
//
// FP8 E4M3 weights: each 1x128 block's dot product is formed first (its 8 chunks sit in 8
// lanes and are summed across them) and then multiplied by the block's FP32 scale once
// ("OSDI'26 | 双路 CPU + 两张 5090 …", §4.2).  The token enters the FP8 products as F16 after
// an exact per-token power-of-two prescale, undone on the finished sums.
#include "ft_dot.cuh"
#include "ft_internal.cuh"
#include "ft_ptx.cuh"

namespace ft {
namespace {

using namespace dot;
using namespace ptx;

// E8M0 scale code -> 2^(code - 127) (code 0: the subnormal 2^-127; 255 is never written)
__device__ __forceinline__ float e8m0_float(uint32_t code) { return __uint_as_float(code ? code << 23 : 0x00400000u); }

constexpr int kConsumers = 8;
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kMaxStages = 8;
// Ring stage size: 48 KB for BF16 rows (four stages; measured 22.7 against 23.2 us per
// 35B-shape layer with 32 KB stages), 32 KB for the FP8 / FP4 rows, whose h and activation
// planes leave less room for the ring.
constexpr size_t kStageTargetBF16 = 48 * 1024;
constexpr size_t kStageTarget = 32 * 1024;
constexpr size_t kSmemBudget = 220 * 1024;  // largest ring
constexpr int kRowsILP = 4;                 // phase-1 rows a consumer warp forms at once

__host__ __device__ inline size_t round128(size_t b) { return (b + 127) / 128 * 128; }

struct FusedPlan {
  int pairs;     // phase-0 (gate, up) row pairs per stage
  int drows;     // phase-1 down rows per stage
  int nst;       // ring stages
  int sbh, sbi;  // block-scale bytes of an H row / an I row carried in the ring (0: read from HBM)
  size_t stage;  // bytes per stage
  size_t xs, hs, ybuf, cb;
};

// Block-scale bytes per row of H (or I) elements: FP32 per 128 (FP8), E4M3 per 16 (NVFP4),
// E8M0 per 32 (MXFP4).
__host__ __device__ inline int scale_row_bytes(int wtype, int n) {
  return wtype == FT_W_FP8_E4M3_B128 ? n / 128 * 4 : (wtype == FT_W_NVFP4 ? n / 16 : (wtype == FT_W_MXFP4 ? n / 32 : 0));
}

__host__ __device__ inline FusedPlan make_fused_plan(int wtype, int H, int I, int max_entries, int n_cta) {
  // stored bytes per row: 2 per element (BF16), 1 (FP8), 1/2 (NVFP4, MXFP4)
  const size_t epc = wtype == FT_W_BF16 ? 8 : (wtype == FT_W_FP8_E4M3_B128 ? 16 : 32);  // elements per 16 B
  const size_t rh = (size_t)H / epc * 16, ri = (size_t)I / epc * 16;
  FusedPlan pl;
  // The block scales of a stage's rows travel in the same stage (one bulk copy per run of
  // rows), so the consumers read them from shared memory instead of waiting on HBM for them;
  // that needs 16-byte multiples per row (bulk copies move 16-byte units).
  const int sh = scale_row_bytes(wtype, H), si = scale_row_bytes(wtype, I);
  const bool carry = sh > 0 && sh % 16 == 0 && si % 16 == 0;
  pl.sbh = carry ? sh : 0;
  pl.sbi = carry ? si : 0;
  const size_t ph = rh + pl.sbh, pi = ri + pl.sbi;  // ring bytes per H row / per I row
  pl.stage = wtype == FT_W_BF16 ? kStageTargetBF16 : kStageTarget;
  if (pl.stage < 2 * ph) pl.stage = 2 * ph;
  if (pl.stage < pi) pl.stage = pi;
  pl.pairs = (int)(pl.stage / (2 * ph));
  pl.drows = (int)(pl.stage / pi);
  pl.xs = round128((size_t)H * 2);
  pl.hs = round128((size_t)max_entries * I * 4);
  const int jpc = (H + n_cta - 1) / n_cta;
  pl.ybuf = round128((size_t)jpc * max_entries * 4);
  pl.cb = round128((size_t)jpc * kMaxK * 4);
  const size_t fixed = pl.xs + pl.hs + pl.ybuf + pl.cb + 1024;
  // The deepest ring that fits: bytes in flight per SM set the streaming rate.  (No CTA of
  // another kernel shares the SM: the next layer's control kernel runs beside a fill CTA.)
  const int nst = fixed >= kSmemBudget ? 0 : (int)((kSmemBudget - fixed) / pl.stage);
  pl.nst = nst > kMaxStages ? kMaxStages : nst;
  return pl;
}

inline size_t fused_smem_bytes(const FusedPlan& pl) {
  return (size_t)pl.nst * pl.stage + pl.xs + pl.hs + pl.ybuf + pl.cb + 2 * kMaxStages * 8 + kMaxStages * 16 + 16 +
         128;
}

// HC, IC: 16-byte chunks per lane of an H row and of an I row when the shape is known at
// compile time (0: taken from the parameters).  With them the dot loops are straight-line
// code; with runtime bounds the guarded loops measured ~2.7x slower per row on GB300.
template <int WT, int HC, int IC>
__global__ void __launch_bounds__(kThreads, 1) fused_gemv_kernel(EvalParams p, FusedPlan pl) {
  extern __shared__ uint8_t smem_raw[];
  // rounded up by pointer arithmetic on the shared array, so that the compiler still knows
  // every derived pointer is in shared memory (shared loads, not generic ones)
  uint8_t* smem = smem_raw + ((128u - (ptx::smem_u32(smem_raw) & 127u)) & 127u);
  uint8_t* stages = smem;
  uint16_t* xs = reinterpret_cast<uint16_t*>(stages + (size_t)pl.nst * pl.stage);
  float* hs = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xs) + pl.xs);
  float* ybuf = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(hs) + pl.hs);
  float* cb = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ybuf) + pl.ybuf);  // [jl][r] host rows
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(cb) + pl.cb);
  uint64_t* empty = full + kMaxStages;
  int4* meta = reinterpret_cast<int4*>(empty + kMaxStages);  // per stage: phase, first row, rows
  volatile int* abort_flag = reinterpret_cast<volatile int*>(meta + kMaxStages);

  constexpr int EPC = WT == FT_W_BF16 ? 8 : (WT == FT_W_FP8_E4M3_B128 ? 16 : 32);  // weights per 16-byte chunk
  constexpr bool kFP4 = WT == FT_W_NVFP4 || WT == FT_W_MXFP4;
  const int ne = p.counts[C_NENTRIES];
  // compile-time shapes make the unit and row index arithmetic constant as well
  const int H = HC > 0 ? HC * 32 * EPC : p.H, I = IC > 0 ? IC * 32 * EPC : p.I, k = p.k;
  const size_t rh = (size_t)H / EPC * 16, ri = (size_t)I / EPC * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Entries split into two passes: those resident before this step (pass 0) and those the
  // fill kernel right before writes (pass 1).  Within a pass, phase-0 units v (entry
  // pe[v / I], row v % I) are split evenly over the CTAs; phase-1 rows t (entry pe[t / nj],
  // output row j0 + t % nj) are this CTA's output rows of every entry of the pass.
  __shared__ int s_pe[2][kMaxK + 2];
  __shared__ int s_np[2];
  // the entries' weight bases, read once: the producer would otherwise wait on a global load
  // before every copy it issues
  __shared__ const uint8_t* s_gw[kMaxK + 2];
  const int j0 = (int)((long long)H * blockIdx.x / gridDim.x);
  const int nj = (int)((long long)H * (blockIdx.x + 1) / gridDim.x) - j0;

  __shared__ int s_fill[kMaxK + 2];
  if (threadIdx.x < ne && threadIdx.x < kMaxK + 2) {  // one thread per entry: the loads overlap
    s_fill[threadIdx.x] = p.g_fill[threadIdx.x];
    s_gw[threadIdx.x] = p.g_w[threadIdx.x];
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < pl.nst; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kConsumers);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n[2] = {0, 0};
    for (int g = 0; g < ne && g < kMaxK + 2; ++g) {
      const int ps = s_fill[g] != 0 ? 1 : 0;
      s_pe[ps][n[ps]++] = g;
    }
    s_np[0] = n[0];
    s_np[1] = n[1];
  }
  __syncthreads();

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();
      int c = 0;
      // Pass 0 streams the experts that were resident before this step (the fill kernel
      // right before does not write their slots): their gate/up rows, then their down rows.
      // Pass 1 joins the dependency chain and streams the filled experts the same way.
      for (int pass = 0; pass < 2 && !*abort_flag; ++pass) {
        if (pass == 1) pdl_wait();
        const int npe = s_np[pass];
        const int* pe = s_pe[pass];
        const long long R0 = (long long)npe * I;
        const int v1 = (int)(R0 * (blockIdx.x + 1) / gridDim.x);
        for (int v = (int)(R0 * blockIdx.x / gridDim.x); v < v1 && !*abort_flag;) {
          const int gi = v / I, i = v - gi * I, g = pe[gi];
          const int nr = min(pl.pairs, min(v1, (gi + 1) * I) - v);
          const int s = c % pl.nst, use = c / pl.nst;
          if (!mbar_wait(smem_u32(empty + s), (uint32_t)(use & 1) ^ 1u, abort_flag, p.error_word)) break;
          meta[s] = make_int4(0, v, nr, pass);
          const uint32_t fb = smem_u32(full + s), dst = smem_u32(stages + (size_t)s * pl.stage);
          const uint8_t* src = s_gw[g] + p.lay.gate + (size_t)i * rh;
          mbar_arrive_expect_tx(fb, (uint32_t)(2 * nr * (rh + pl.sbh)));
          bulk_g2s_hint(dst, src, (uint32_t)(nr * rh), fb, pol);
          bulk_g2s_hint(dst + (uint32_t)(nr * rh), src + (size_t)I * rh, (uint32_t)(nr * rh), fb, pol);
          if (pl.sbh) {  // gate scales, then up scales, behind the rows
            const uint32_t sdst = dst + (uint32_t)(2 * nr * rh);
            bulk_g2s_hint(sdst, s_gw[g] + p.lay.gs + (size_t)i * pl.sbh, (uint32_t)(nr * pl.sbh), fb, pol);
            bulk_g2s_hint(sdst + (uint32_t)(nr * pl.sbh), s_gw[g] + p.lay.us + (size_t)i * pl.sbh,
                          (uint32_t)(nr * pl.sbh), fb, pol);
          }
          v += nr;
          ++c;
        }
        // The next layer's control kernel may start once the pre-fill gate/up rows are on
        // their way: its prologue reads only state that earlier control kernels wrote, and
        // it waits for this grid to complete before anything else.
        if (pass == 0) pdl_trigger();
        const int n1 = npe * nj;
        // phase-1 stages hold whole entries when an entry's rows fit in a stage
        const int p1_rows = nj > 0 && nj <= pl.drows ? pl.drows / nj * nj : pl.drows;
        for (int t = 0; t < n1 && !*abort_flag;) {
          const int s = c % pl.nst, use = c / pl.nst;
          if (!mbar_wait(smem_u32(empty + s), (uint32_t)(use & 1) ^ 1u, abort_flag, p.error_word)) break;
          const int nr = min(p1_rows, n1 - t);
          meta[s] = make_int4(1, t, nr, pass);
          const uint32_t fb = smem_u32(full + s), dst = smem_u32(stages + (size_t)s * pl.stage);
          mbar_arrive_expect_tx(fb, (uint32_t)(nr * (ri + pl.sbi)));
          // a stage may span entries: one bulk copy per entry segment (its rows are contiguous),
          // and one for the segment's block scales behind all the stage's rows
          uint32_t off = 0;
          for (int tt = t; tt < t + nr;) {
            const int gi = tt / nj, jl = tt - gi * nj;
            const int seg = min(t + nr, (gi + 1) * nj) - tt;
            bulk_g2s_hint(dst + off, s_gw[pe[gi]] + p.lay.down + (size_t)(j0 + jl) * ri, (uint32_t)(seg * ri), fb,
                          pol);
            if (pl.sbi)
              bulk_g2s_hint(dst + (uint32_t)(nr * ri) + (uint32_t)((tt - t) * pl.sbi),
                            s_gw[pe[gi]] + p.lay.ds + (size_t)(j0 + jl) * pl.sbi, (uint32_t)(seg * pl.sbi), fb, pol);
            off += (uint32_t)(seg * ri);
            tt += seg;
          }
          t += nr;
          ++c;
        }
      }
      if (*abort_flag)  // let copies already issued land before the CTA exits
        for (int cc = (c > pl.nst ? c - pl.nst : 0); cc < c; ++cc)
          for (uint32_t i = 0;
               i < kWaitLimit && !mbar_try_wait(smem_u32(full + cc % pl.nst), (uint32_t)((cc / pl.nst) & 1)); ++i) {
          }
    }
  } else {
    // ------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int ct = threadIdx.x - 32;  // 0..255
    // the token as bf16 (BF16 weights) or f16 after an exact power-of-two prescale (FP8, FP4)
    int xshift = 0;
    if (WT != FT_W_BF16) {
      __shared__ uint32_t s_xmax[kConsumers];
      uint32_t m = 0;
      for (int idx = ct; idx < H / 8; idx += 32 * kConsumers)
        m = bf16x8_maxbits(*reinterpret_cast<const uint4*>(p.x + (size_t)idx * 8), m);
      m = __reduce_max_sync(0xffffffffu, m);
      if (lane == 0) s_xmax[cw] = m;
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumers) : "memory");
      m = 0;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) m = max(m, s_xmax[w]);
      xshift = act_shift(m);
    }
    for (int idx = ct; idx < H / 8; idx += 32 * kConsumers) {
      uint4 v = *reinterpret_cast<const uint4*>(p.x + (size_t)idx * 8);
      if (WT != FT_W_BF16) v = bf16x8_to_f16x8_scaled(v, pow2i(-xshift));
      // plane layout: piece q (8 elements) of chunk c at plane q, so that each lane's 16-byte
      // pieces of consecutive chunks lie side by side (no bank conflicts)
      constexpr int kXP = EPC / 8;  // x pieces (planes) per chunk
      const int c = idx / kXP, q = idx - c * kXP;
      *reinterpret_cast<uint4*>(xs + (size_t)q * (H / kXP) + (size_t)c * 8) = v;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumers) : "memory");

    // combine inputs that do not depend on h: lane r < k holds pair r
    const bool res_r = lane < k && p.slot_of_pair[lane] >= 0;
    const uint32_t res_mask = __ballot_sync(0xffffffffu, res_r);
    const int gi_r = __popc(res_mask & ((1u << lane) - 1u));
    const float gate_r = lane < k ? p.gates[lane] : 0.f;

    // the caller's rows of host-evaluated pairs, [jl][r]
    auto fetch_cb = [&]() {
      for (int idx = ct; idx < nj * k; idx += 32 * kConsumers) {
        const int jl = idx / k, r = idx - jl * k;
        float val = 0.f;
        if (p.slot_of_pair[r] < 0) {
          if (p.c_partial) val = p.c_partial[(size_t)r * H + j0 + jl];
          else atomicOr(p.error_word, FT_DEVERR_CAPACITY);
        }
        cb[idx] = val;
      }
    };
    bool cb_done = false;

    int c = 0;
    for (int pass = 0; pass < 2; ++pass) {
      const int npe = s_np[pass];
      if (npe == 0) continue;
      const int* pe = s_pe[pass];
      if (WT != FT_W_BF16 && pass == 1) pdl_wait();  // block scales of filled slots are read directly
      const long long R0 = (long long)npe * I;
      const int v0 = (int)(R0 * blockIdx.x / gridDim.x);
      const int n0 = (int)(R0 * (blockIdx.x + 1) / gridDim.x) - v0;

      // ---- phase 0: h = silu(W_g x) * (W_u x)
      for (int done = 0; done < n0;) {
        const int s = c % pl.nst, use = c / pl.nst;
        if (!mbar_wait(smem_u32(full + s), (uint32_t)(use & 1), abort_flag, p.error_word)) break;
        const int4 m = meta[s];
        const uint8_t* st = stages + (size_t)s * pl.stage;
        // items rotate over the warps from stage to stage, so small stages keep all warps busy
        for (int q = ((cw - done) % kConsumers + kConsumers) % kConsumers; q < m.z; q += kConsumers) {
          const int v = m.y + q, gi = v / I, i = v - gi * I, g = pe[gi];
          const uint8_t* rg = st + (size_t)q * rh;          // gate row
          const uint8_t* ru = st + ((size_t)m.z + q) * rh;  // the same up row
          float a = 0.f, b = 0.f;                           // two independent chains
          if (WT == FT_W_BF16 && HC > 0) {
#pragma unroll
            for (int cc = 0; cc < HC; ++cc) {
              const int c16 = lane + 32 * cc;
              const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)c16 * 8);
              a = dot_bf16_bf16(*reinterpret_cast<const uint4*>(rg + (size_t)c16 * 16), xv, a);
              b = dot_bf16_bf16(*reinterpret_cast<const uint4*>(ru + (size_t)c16 * 16), xv, b);
            }
          } else if (WT == FT_W_BF16) {
            for (int c16 = lane; c16 < H / EPC; c16 += 32) {
              const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)c16 * 8);
              a = dot_bf16_bf16(*reinterpret_cast<const uint4*>(rg + (size_t)c16 * 16), xv, a);
              b = dot_bf16_bf16(*reinterpret_cast<const uint4*>(ru + (size_t)c16 * 16), xv, b);
            }
          } else if (kFP4) {
            // a chunk holds 32 elements: two NVFP4 blocks or one MXFP4 block, each block's dot
            // product taken first and multiplied by its scale (as in the batched kernels)
            const int sb = WT == FT_W_NVFP4 ? H / 16 : H / 32;  // scale bytes per row
            // the stage's copy of the scales when the ring carries them (generic loads serve both)
            const uint8_t* bg = pl.sbh ? st + (size_t)2 * m.z * rh + (size_t)q * sb : s_gw[g] + p.lay.gs + (size_t)i * sb;
            const uint8_t* bu = pl.sbh ? st + (size_t)2 * m.z * rh + (size_t)(m.z + q) * sb
                                       : s_gw[g] + p.lay.us + (size_t)i * sb;
            for (int c16 = lane; c16 < H / EPC; c16 += 32) {
              const uint4 x0 = *reinterpret_cast<const uint4*>(xs + (size_t)c16 * 8);
              const uint4 x1 = *reinterpret_cast<const uint4*>(xs + (size_t)H / 4 + (size_t)c16 * 8);
              const uint4 x2 = *reinterpret_cast<const uint4*>(xs + (size_t)H / 2 + (size_t)c16 * 8);
              const uint4 x3 = *reinterpret_cast<const uint4*>(xs + (size_t)3 * H / 4 + (size_t)c16 * 8);
              const uint4 wa = *reinterpret_cast<const uint4*>(rg + (size_t)c16 * 16);
              const uint4 wb = *reinterpret_cast<const uint4*>(ru + (size_t)c16 * 16);
              if (WT == FT_W_NVFP4) {
                const float2 ga = e4m3x2_to_float2(reinterpret_cast<const uint16_t*>(bg)[c16]);
                const float2 gb = e4m3x2_to_float2(reinterpret_cast<const uint16_t*>(bu)[c16]);
                a = fmaf(dot16_e2m1_f16(wa.x, wa.y, x0, x1), ga.x, a);
                a = fmaf(dot16_e2m1_f16(wa.z, wa.w, x2, x3), ga.y, a);
                b = fmaf(dot16_e2m1_f16(wb.x, wb.y, x0, x1), gb.x, b);
                b = fmaf(dot16_e2m1_f16(wb.z, wb.w, x2, x3), gb.y, b);
              } else {
                const float da = dot16_e2m1_f16(wa.x, wa.y, x0, x1) + dot16_e2m1_f16(wa.z, wa.w, x2, x3);
                const float db = dot16_e2m1_f16(wb.x, wb.y, x0, x1) + dot16_e2m1_f16(wb.z, wb.w, x2, x3);
                a = fmaf(da, e8m0_float(bg[c16]), a);
                b = fmaf(db, e8m0_float(bu[c16]), b);
              }
            }
          } else {
            const float* sg = pl.sbh ? reinterpret_cast<const float*>(st + (size_t)2 * m.z * rh) + (size_t)q * (H / 128)
                                     : reinterpret_cast<const float*>(s_gw[g] + p.lay.gs) + (size_t)i * (H / 128);
            const float* su = pl.sbh
                                  ? reinterpret_cast<const float*>(st + (size_t)2 * m.z * rh) + (size_t)(m.z + q) * (H / 128)
                                  : reinterpret_cast<const float*>(s_gw[g] + p.lay.us) + (size_t)i * (H / 128);
            // H / 16 is a multiple of 32: every lane runs every step.  Each 1x128 block's dot
            // product is summed over its 8 lanes, then multiplied by the block's scale once.
#pragma unroll 4
            for (int c16 = lane; c16 < H / EPC; c16 += 32) {
              const uint4 x0 = *reinterpret_cast<const uint4*>(xs + (size_t)c16 * 8);
              const uint4 x1 = *reinterpret_cast<const uint4*>(xs + (size_t)H / 2 + (size_t)c16 * 8);
              const float da = group8_sum(dot_e4m3_f16(*reinterpret_cast<const uint4*>(rg + (size_t)c16 * 16), x0, x1));
              const float db = group8_sum(dot_e4m3_f16(*reinterpret_cast<const uint4*>(ru + (size_t)c16 * 16), x0, x1));
              a = fmaf(da, sg[c16 / 8], a);
              b = fmaf(db, su[c16 / 8], b);
            }
          }
          const float xsc = WT == FT_W_BF16 ? 1.f : pow2i(xshift);
          // NVFP4: the banks' FP32 tensor scales multiply the finished sums
          const float tsa = WT == FT_W_NVFP4 ? __ldg(reinterpret_cast<const float*>(s_gw[g] + p.lay.ts)) : 1.f;
          const float tsb = WT == FT_W_NVFP4 ? __ldg(reinterpret_cast<const float*>(s_gw[g] + p.lay.ts) + 1) : 1.f;
          const float ab2[2] = {(WT == FT_W_FP8_E4M3_B128 ? groups_sum(a) : warp_sum(a)) * xsc * tsa,
                                (WT == FT_W_FP8_E4M3_B128 ? groups_sum(b) : warp_sum(b)) * xsc * tsb};
          if (lane == 0) p.h[(size_t)g * I + i] = silu_mul(ab2[0], ab2[1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + s));
        done += m.z;
        ++c;
      }

      if (!cb_done) {
        fetch_cb();  // while the other CTAs finish phase 0
        cb_done = true;
      }

      // ---- hand-off: publish this CTA's h rows of the pass, wait for the pass's entries,
      // stage their h
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumers) : "memory");
      if (ct == 0) {
        __threadfence();
        for (int v = v0; v < v0 + n0;) {
          const int gi = v / I;
          const int end = min(v0 + n0, (gi + 1) * I);
          atomicAdd(p.ready + pe[gi], (uint32_t)(end - v));
          v = end;
        }
      }
      // every warp waits on its own entries' counters, so the polls run side by side
      if (lane == 0)
        for (int gi = cw; gi < npe; gi += kConsumers)
          if (!wait_counter(p.ready + pe[gi], (uint32_t)I + p.wait_extra, abort_flag, p.error_word, p.wait_ns)) break;
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumers) : "memory");
      // one flat loop, so that every thread's loads of all the pass's entries are in flight
      // together
      for (int idx = ct; idx < npe * (I / 4); idx += 32 * kConsumers) {
        const int gi = idx / (I / 4), i4 = idx - gi * (I / 4);
        const size_t off = (size_t)pe[gi] * (I / 4) + i4;
        // per entry, float4 piece q of chunk c at plane q (planes of I / EPC float4)
        constexpr int kHP = EPC / 4;  // h pieces per chunk
        const int c = i4 / kHP, q = i4 - c * kHP;
        reinterpret_cast<float4*>(hs)[(size_t)pe[gi] * (I / 4) + (size_t)q * (I / EPC) + c] =
            __ldcg(reinterpret_cast<const float4*>(p.h) + off);
      }
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumers) : "memory");

      // ---- phase 1: y[g][j] = W_d[g][j] . h[g]
      const int n1 = npe * nj;
      for (int done = 0; done < n1;) {
        const int s = c % pl.nst, use = c / pl.nst;
        if (!mbar_wait(smem_u32(full + s), (uint32_t)(use & 1), abort_flag, p.error_word)) break;
        const int4 m = meta[s];
        const uint8_t* st = stages + (size_t)s * pl.stage;
        const int rot = ((cw - done) % kConsumers + kConsumers) % kConsumers;
        if (WT == FT_W_BF16 && IC > 0) {
          // Work items are blocks of kRowsILP consecutive rows of one entry, so a warp loads
          // that entry's h chunks once into registers for all the rows of the block.
          // Products and their order per row are those of the per-row form below.
          // items: entry-runs of the stage split into blocks of kRowsILP rows; a block past a
          // run's end computes clamped duplicate rows and stores only its own
          const int gfirst = m.y / nj, glast = (m.y + m.z - 1) / nj;
          const int nb = (nj + kRowsILP - 1) / kRowsILP;  // blocks per run, at most
          for (int item = rot; item < (glast - gfirst + 1) * nb; item += kConsumers) {
            const int gi = gfirst + item / nb;
            const int ra = max(m.y, gi * nj), rb = min(m.y + m.z, (gi + 1) * nj);
            const int r0 = ra + (item % nb) * kRowsILP;
            if (r0 >= rb) continue;
            const int g = pe[gi];
            const float* hv = hs + (size_t)g * I;
            float4 h0[IC > 0 ? IC : 1], h1[IC > 0 ? IC : 1];
#pragma unroll
            for (int cc = 0; cc < IC; ++cc) {
              const int c16 = lane + 32 * cc;
              h0[cc] = reinterpret_cast<const float4*>(hv)[c16];
              h1[cc] = reinterpret_cast<const float4*>(hv)[I / EPC + c16];
            }
            const uint8_t* wrow[kRowsILP];
#pragma unroll
            for (int r = 0; r < kRowsILP; ++r) wrow[r] = st + (size_t)(min(r0 + r, rb - 1) - m.y) * ri;
            float acc[kRowsILP];
#pragma unroll
            for (int r = 0; r < kRowsILP; ++r) acc[r] = 0.f;
#pragma unroll
            for (int cc = 0; cc < IC; ++cc) {
              const int c16 = lane + 32 * cc;
#pragma unroll
              for (int r = 0; r < kRowsILP; ++r)
                acc[r] = dot_bf16_f32v(*reinterpret_cast<const uint4*>(wrow[r] + (size_t)c16 * 16), h0[cc], h1[cc],
                                       acc[r]);
            }
#pragma unroll
            for (int r = 0; r < kRowsILP; ++r) {
              const float v = warp_sum(acc[r]);
              if (r0 + r < rb && lane == 0) ybuf[(size_t)g * nj + (r0 + r - gi * nj)] = v;  // [entry][jl]
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(empty + s));
          done += m.z;
          ++c;
          continue;
        }
        // up to kRowsILP rows per warp at once: independent chains, each row in the usual order
        for (int q = rot; q < m.z; q += kRowsILP * kConsumers) {
          float acc[kRowsILP];
          const float* hv[kRowsILP];
          const float* sc[kRowsILP];
          const uint8_t* sb4[kRowsILP];
          float ts4[kRowsILP];
          int yi[kRowsILP];
          bool ok[kRowsILP];
#pragma unroll
          for (int r = 0; r < kRowsILP; ++r) {
            const int qq = q + r * kConsumers;
            ok[r] = qq < m.z;
            const int t = m.y + (ok[r] ? qq : q), gi = t / nj, jl = t - gi * nj, g = pe[gi];
            yi[r] = g * nj + jl;
            hv[r] = hs + (size_t)g * I;
            // block scales: the stage's copy when the ring carries them, else the slot's
            const uint8_t* sbase = pl.sbi ? st + (size_t)m.z * ri + (size_t)(ok[r] ? qq : q) * pl.sbi
                                          : s_gw[g] + p.lay.ds + (size_t)(j0 + jl) * scale_row_bytes(WT, I);
            sc[r] = WT == FT_W_FP8_E4M3_B128 ? reinterpret_cast<const float*>(sbase) : nullptr;
            sb4[r] = kFP4 ? sbase : nullptr;
            ts4[r] = WT == FT_W_NVFP4 ? __ldg(reinterpret_cast<const float*>(s_gw[g] + p.lay.ts) + 2) : 1.f;
            acc[r] = 0.f;
          }
          if (WT == FT_W_BF16) {
#pragma unroll 4
            for (int c16 = lane; c16 < I / EPC; c16 += 32) {
#pragma unroll
              for (int r = 0; r < kRowsILP; ++r) {
                if (!ok[r]) continue;
                const uint4 wv =
                    *reinterpret_cast<const uint4*>(st + (size_t)(q + r * kConsumers) * ri + (size_t)c16 * 16);
                const float4* h4 = reinterpret_cast<const float4*>(hv[r]);
                acc[r] = dot_bf16_f32v(wv, h4[c16], h4[I / EPC + c16], acc[r]);
              }
            }
          } else if (kFP4) {
            for (int c16 = lane; c16 < I / EPC; c16 += 32) {
#pragma unroll
              for (int r = 0; r < kRowsILP; ++r) {
                if (!ok[r]) continue;
                const uint4 wv =
                    *reinterpret_cast<const uint4*>(st + (size_t)(q + r * kConsumers) * ri + (size_t)c16 * 16);
                const float4* h4 = reinterpret_cast<const float4*>(hv[r]);
                float hv32[32];
#pragma unroll
                for (int q = 0; q < 8; ++q) *reinterpret_cast<float4*>(hv32 + 4 * q) = h4[(size_t)q * (I / EPC) + c16];
                if (WT == FT_W_NVFP4) {
                  const float2 sd = e4m3x2_to_float2(reinterpret_cast<const uint16_t*>(sb4[r])[c16]);
                  acc[r] = fmaf(dot16_e2m1_f32(wv.x, wv.y, hv32), sd.x, acc[r]);
                  acc[r] = fmaf(dot16_e2m1_f32(wv.z, wv.w, hv32 + 16), sd.y, acc[r]);
                } else {
                  const float d = dot16_e2m1_f32(wv.x, wv.y, hv32) + dot16_e2m1_f32(wv.z, wv.w, hv32 + 16);
                  acc[r] = fmaf(d, e8m0_float(sb4[r][c16]), acc[r]);
                }
              }
            }
          } else {
            // I / 16 is a multiple of 8: a block's 8 lanes are all live or all idle, and the
            // block-sum shuffles run on every lane
            for (int cb = 0; cb < I / EPC; cb += 32) {
              const int c16 = cb + lane;
              const bool cv = c16 < I / EPC;
#pragma unroll
              for (int r = 0; r < kRowsILP; ++r) {
                if (!ok[r]) continue;  // the same for every lane
                float d = 0.f;
                if (cv) {
                  const float4* h4 = reinterpret_cast<const float4*>(hv[r]);
                  const float4 hq[4] = {h4[c16], h4[I / EPC + c16], h4[2 * (I / EPC) + c16], h4[3 * (I / EPC) + c16]};
                  d = dot_e4m3_f32v(
                      *reinterpret_cast<const uint4*>(st + (size_t)(q + r * kConsumers) * ri + (size_t)c16 * 16), hq);
                }
                d = group8_sum(d);
                if (cv) acc[r] = fmaf(d, sc[r][c16 / 8], acc[r]);
              }
            }
          }
#pragma unroll
          for (int r = 0; r < kRowsILP; ++r) {
            const float v = (WT == FT_W_FP8_E4M3_B128 ? groups_sum(acc[r]) : warp_sum(acc[r])) * ts4[r];
            if (ok[r] && lane == 0) ybuf[yi[r]] = v;  // [entry][jl]
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + s));
        done += m.z;
        ++c;
      }
    }
    if (!cb_done) fetch_cb();  // no GPU entry at all: every pair is host-evaluated
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumers) : "memory");

    // ---- combine: one warp per output row; lane r < k holds pair r (ascending expert id)
    for (int jl = cw; jl < nj; jl += kConsumers) {
      const int j = j0 + jl;
      float val = 0.f;
      if (lane < k) {
        if (res_r) {
          val = gate_r * ybuf[(size_t)gi_r * nj + jl];
          p.rows[(size_t)lane * H + j] = val;
        } else {
          val = cb[jl * k + lane];
        }
      }
      float o = p.has_shared ? ybuf[(size_t)(ne - 1) * nj + jl] : 0.f;
      for (int r = 0; r < k; ++r) o += __shfl_sync(0xffffffffu, val, r);
      if (lane == 0) p.out[j] = o;
    }
  }
  __syncthreads();
}

template <int WT, int HC, int IC>
cudaError_t launch_fused_t(const EvalParams& p, int n_sm, int max_entries, cudaStream_t s) {
  const FusedPlan pl = make_fused_plan(WT, p.H, p.I, max_entries, n_sm);
  return launch_k(fused_gemv_kernel<WT, HC, IC>, dim3(n_sm), dim3(kThreads), fused_smem_bytes(pl), s, p.pdl, p, pl);
}

// Shapes compiled with fixed chunk counts: the 35B-A3B expert shape (H 2048, I 512, BF16)
// and the large FP8 expert shape (H 7168, I 2048, E4M3).
template <int WT, int HC, int IC>
constexpr bool fixed_shape_matches(int H, int I) {
  return H == HC * 32 * (WT == FT_W_BF16 ? 8 : 16) && I == IC * 32 * (WT == FT_W_BF16 ? 8 : 16);
}

}  // namespace

bool fused_gemv_supported(int wtype, int H, int I, int max_entries, int n_sm) {
  const FusedPlan pl = make_fused_plan(wtype, H, I, max_entries, n_sm);
  return pl.nst >= 2 && fused_smem_bytes(pl) <= kSmemBudget + 4096;
}

bool fused_gemv_fits(int wtype, int H, int I, int max_entries, int n_sm) {
  if (!fused_gemv_supported(wtype, H, I, max_entries, n_sm)) return false;
  const FusedPlan pl = make_fused_plan(wtype, H, I, max_entries, n_sm);
  int nb = 0;
  const size_t smem = fused_smem_bytes(pl);
  cudaError_t e;
  switch (wtype) {
    case FT_W_BF16:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fused_gemv_kernel<FT_W_BF16, 0, 0>, kThreads, smem);
      break;
    case FT_W_FP8_E4M3_B128:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fused_gemv_kernel<FT_W_FP8_E4M3_B128, 0, 0>, kThreads,
                                                        smem);
      break;
    case FT_W_NVFP4:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fused_gemv_kernel<FT_W_NVFP4, 0, 0>, kThreads, smem);
      break;
    default:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fused_gemv_kernel<FT_W_MXFP4, 0, 0>, kThreads, smem);
      break;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return nb >= 1;
}

cudaError_t launch_fused_gemv(const EvalParams& p, int wtype, int n_sm, int max_entries, cudaStream_t s) {
  if (wtype == FT_W_BF16 && fixed_shape_matches<FT_W_BF16, 8, 2>(p.H, p.I))
    return launch_fused_t<FT_W_BF16, 8, 2>(p, n_sm, max_entries, s);
  if (wtype == FT_W_FP8_E4M3_B128 && fixed_shape_matches<FT_W_FP8_E4M3_B128, 14, 4>(p.H, p.I))
    return launch_fused_t<FT_W_FP8_E4M3_B128, 14, 4>(p, n_sm, max_entries, s);
  switch (wtype) {
    case FT_W_BF16: return launch_fused_t<FT_W_BF16, 0, 0>(p, n_sm, max_entries, s);
    case FT_W_FP8_E4M3_B128: return launch_fused_t<FT_W_FP8_E4M3_B128, 0, 0>(p, n_sm, max_entries, s);
    case FT_W_NVFP4: return launch_fused_t<FT_W_NVFP4, 0, 0>(p, n_sm, max_entries, s);
    default: return launch_fused_t<FT_W_MXFP4, 0, 0>(p, n_sm, max_entries, s);
  }
}

cudaError_t prepare_fused_gemv() {
  const int lim = (int)(kSmemBudget + 4096);
  const void* k[] = {(const void*)fused_gemv_kernel<FT_W_BF16, 8, 2>,
                     (const void*)fused_gemv_kernel<FT_W_FP8_E4M3_B128, 14, 4>,
                     (const void*)fused_gemv_kernel<FT_W_BF16, 0, 0>,
                     (const void*)fused_gemv_kernel<FT_W_FP8_E4M3_B128, 0, 0>,
                     (const void*)fused_gemv_kernel<FT_W_NVFP4, 0, 0>,
                     (const void*)fused_gemv_kernel<FT_W_MXFP4, 0, 0>};
  for (const void* f : k) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ft
