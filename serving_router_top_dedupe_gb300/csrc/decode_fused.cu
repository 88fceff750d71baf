// Decode expert evaluation at batch 1 in one persistent launch: gate/up GEMV + SwiGLU,
// down GEMV and the fixed-order combine.
//
// A decode layer reads every byte of its G-set experts once (about 1 FLOP per byte), so
// it is bound by HBM, and at batch 1 a layer is only ~10 us of traffic: what costs is
// every point where the weight stream stops.  One CTA per SM streams its share of the
// layer's weight rows through a ring of shared-memory stages filled by cp.async.bulk
// (one elected producer thread, eight consumer warps).  Every CTA takes a slice of every
// entry g (the layer's G-set experts and the shared expert):
//
//  phase 0 of g: h rows i0..i0+ni-1: a stage holds gate rows and the same up rows; a
//                consumer warp forms a = W_g[i].x, b = W_u[i].x, writes h[g][i] =
//                silu(a)*b and adds its rows to the entry's counter ready[g].
//  phase 1 of g: output rows j0..j0+nj-1 of W_down[g]; the rows need every CTA's h[g], so
//                consumers wait (bounded) until ready[g] = I, then form y[g][j] = W_d[g][j].h[g].
//
// The ring carries the entries in the order phase0(g0), phase0(g1), phase0(g2),
// phase1(g0), phase0(g3), phase1(g1), ...: the down rows of an entry stream right behind
// the gate/up rows of later entries, so the h hand-off between CTAs overlaps the stream
// instead of stopping it.  Experts resident before this step come first; experts filled in
// this step come last, after the producer has waited for the fill kernel.
//
//  combine: out[j] = shared + the k pair rows in ascending expert id (GPU row gate_r * y,
//           or the caller's c_partial row for a host-evaluated pair).
//
// The counters need every CTA of the grid to be resident: the grid is one CTA per SM and
// a CTA takes more than half of an SM's shared memory; no kernel this grid could wait
// behind depends on it.  Every wait is bounded (FT_DEVERR_TIMEOUT on expiry).
//
// Per (entry, row) the lane-strided 16-byte chunk order and the xor butterfly are those of
// the batched decode kernels, so results are bit-identical to them.
//
// FP8 E4M3 weights: each 128-element block's dot product is formed first and then
// multiplied by the block's FP32 scale ("OSDI'26 | 双路 CPU + 两张 5090 …", §4.2).
#include "ft_dot.cuh"
#include "ft_internal.cuh"
#include "ft_ptx.cuh"

namespace ft {
namespace {

using namespace dot;
using namespace ptx;

constexpr int kConsumers = 8;
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kMaxStages = 8;
constexpr int kLag = 2;                     // entries between an entry's phase 0 and its phase 1
constexpr size_t kStageTarget = 32 * 1024;
constexpr size_t kSmemBudget = 220 * 1024;  // largest ring
constexpr size_t kSmemShared = 150 * 1024;  // ring that still lets a control-kernel CTA share the SM
constexpr int kRowsILP = 4;                 // phase-1 rows a consumer warp forms at once
constexpr int kMaxEntries = kMaxK + 1;      // batch 1: k routed experts + the shared expert

__host__ __device__ inline size_t round128(size_t b) { return (b + 127) / 128 * 128; }

struct FusedPlan {
  int pairs;     // phase-0 (gate, up) row pairs per stage
  int drows;     // phase-1 down rows per stage
  int nst;       // ring stages
  size_t stage;  // bytes per stage
  size_t xs, ybuf, cb;
};

__host__ __device__ inline FusedPlan make_fused_plan(int wtype, int H, int I, int n_cta) {
  const size_t esz = wtype == FT_W_BF16 ? 2 : 1;
  const size_t rh = (size_t)H * esz, ri = (size_t)I * esz;
  FusedPlan pl;
  pl.stage = kStageTarget;
  if (pl.stage < 2 * rh) pl.stage = 2 * rh;
  if (pl.stage < ri) pl.stage = ri;
  pl.pairs = (int)(pl.stage / (2 * rh));
  pl.drows = (int)(pl.stage / ri);
  pl.xs = round128((size_t)H * 2);
  const int jpc = (H + n_cta - 1) / n_cta;
  pl.ybuf = round128((size_t)jpc * kMaxEntries * 4);
  pl.cb = round128((size_t)jpc * kMaxK * 4);
  const size_t fixed = pl.xs + pl.ybuf + pl.cb + 1024;
  // Prefer a ring that leaves room on the SM for the next layer's control kernel, so that
  // its prologue overlaps this kernel's tail; take the large ring when that would leave
  // fewer than three stages.
  int nst = fixed >= kSmemShared ? 0 : (int)((kSmemShared - fixed) / pl.stage);
  if (nst < 3) nst = fixed >= kSmemBudget ? 0 : (int)((kSmemBudget - fixed) / pl.stage);
  pl.nst = nst > kMaxStages ? kMaxStages : nst;
  return pl;
}

inline size_t fused_smem_bytes(const FusedPlan& pl) {
  return (size_t)pl.nst * pl.stage + pl.xs + pl.ybuf + pl.cb + 2 * kMaxStages * 8 + kMaxStages * 16 + 16 + 128;
}

template <int WT>
__global__ void __launch_bounds__(kThreads, 1) fused_gemv_kernel(EvalParams p, FusedPlan pl) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_order[kMaxEntries];
  __shared__ int s_nres;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
  uint8_t* stages = smem;
  uint16_t* xs = reinterpret_cast<uint16_t*>(stages + (size_t)pl.nst * pl.stage);
  float* ybuf = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xs) + pl.xs);   // [entry][jl]
  float* cb = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ybuf) + pl.ybuf);  // [jl][r] host rows
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(cb) + pl.cb);
  uint64_t* empty = full + kMaxStages;
  int4* meta = reinterpret_cast<int4*>(empty + kMaxStages);  // per stage: phase, entry, first row, rows
  volatile int* abort_flag = reinterpret_cast<volatile int*>(meta + kMaxStages);

  constexpr int ESZ = WT == FT_W_BF16 ? 2 : 1;
  constexpr int EPC = 16 / ESZ;  // weights per 16-byte chunk
  const int ne = min(p.counts[C_NENTRIES], kMaxEntries);
  const int H = p.H, I = p.I, k = p.k;
  const size_t rh = (size_t)H * ESZ, ri = (size_t)I * ESZ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // this CTA's slice of every entry: h rows [i0, i0+ni), output rows [j0, j0+nj)
  const int i0 = (int)((long long)I * blockIdx.x / gridDim.x);
  const int ni = (int)((long long)I * (blockIdx.x + 1) / gridDim.x) - i0;
  const int j0 = (int)((long long)H * blockIdx.x / gridDim.x);
  const int nj = (int)((long long)H * (blockIdx.x + 1) / gridDim.x) - j0;
  const int st0 = (ni + pl.pairs - 1) / pl.pairs, st1 = (nj + pl.drows - 1) / pl.drows;  // stages per entry

  if (threadIdx.x == 0) {
    for (int s = 0; s < pl.nst; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kConsumers);
    }
    *abort_flag = 0;
    mbar_fence_init();
    // entry order: resident before this step first, then filled in this step
    int n = 0;
    for (int g = 0; g < ne; ++g)
      if (!p.g_fill[g]) s_order[n++] = g;
    s_nres = n;
    for (int g = 0; g < ne; ++g)
      if (p.g_fill[g]) s_order[n++] = g;
  }
  __syncthreads();

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();
      const int nres = s_nres;
      // join the dependency chain (the fill kernel right before) before the first filled
      // entry; with none, after the first two entries' gate/up rows are on their way
      const int wait_at = nres < ne ? nres : min(2, ne);
      bool waited = false;
      int c = 0;
      auto acquire = [&](int& s) -> bool {
        s = c % pl.nst;
        return mbar_wait(smem_u32(empty + s), (uint32_t)((c / pl.nst) & 1) ^ 1u, abort_flag, p.error_word);
      };
      for (int idx = 0; idx < ne + kLag && !*abort_flag; ++idx) {
        if (idx == wait_at && !waited) {
          pdl_wait();
          pdl_trigger();
          waited = true;
        }
        if (idx < ne) {  // gate/up rows of entry order[idx]
          const int g = s_order[idx];
          for (int t = 0; t < ni; t += pl.pairs) {
            int s;
            if (!acquire(s)) break;
            const int nr = min(pl.pairs, ni - t);
            meta[s] = make_int4(0, g, i0 + t, nr);
            const uint32_t fb = smem_u32(full + s), dst = smem_u32(stages + (size_t)s * pl.stage);
            const uint8_t* src = p.g_w[g] + p.lay.gate + (size_t)(i0 + t) * rh;
            mbar_arrive_expect_tx(fb, (uint32_t)(2 * nr * rh));
            bulk_g2s_hint(dst, src, (uint32_t)(nr * rh), fb, pol);
            bulk_g2s_hint(dst + (uint32_t)(nr * rh), src + (size_t)I * rh, (uint32_t)(nr * rh), fb, pol);
            ++c;
          }
        }
        if (idx >= kLag) {  // down rows of entry order[idx - kLag]
          const int g = s_order[idx - kLag];
          for (int t = 0; t < nj; t += pl.drows) {
            int s;
            if (!acquire(s)) break;
            const int nr = min(pl.drows, nj - t);
            meta[s] = make_int4(1, g, t, nr);
            const uint32_t fb = smem_u32(full + s), dst = smem_u32(stages + (size_t)s * pl.stage);
            mbar_arrive_expect_tx(fb, (uint32_t)(nr * ri));
            bulk_g2s_hint(dst, p.g_w[g] + p.lay.down + (size_t)(j0 + t) * ri, (uint32_t)(nr * ri), fb, pol);
            ++c;
          }
        }
      }
      if (!waited) {
        pdl_wait();
        pdl_trigger();
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
    // the token as bf16 (BF16 weights) or f16 (FP8 weights)
    for (int idx = ct; idx < H / 8; idx += 32 * kConsumers) {
      uint4 v = *reinterpret_cast<const uint4*>(p.x + (size_t)idx * 8);
      if (WT == FT_W_FP8_E4M3_B128) {
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          __half2 hh = __floats2half2_rn(__uint_as_float(in[q] << 16), __uint_as_float(in[q] & 0xffff0000u));
          o[q] = *reinterpret_cast<uint32_t*>(&hh);
        }
        v = make_uint4(o[0], o[1], o[2], o[3]);
      }
      *reinterpret_cast<uint4*>(xs + (size_t)idx * 8) = v;
    }
    // combine inputs that depend on neither phase: lane r < k holds pair r; the caller's
    // rows of host-evaluated pairs go to shared memory
    const bool res_r = lane < k && p.slot_of_pair[lane] >= 0;
    const uint32_t res_mask = __ballot_sync(0xffffffffu, res_r);
    const int gi_r = __popc(res_mask & ((1u << lane) - 1u));
    const float gate_r = lane < k ? p.gates[lane] : 0.f;
    for (int idx = ct; idx < nj * k; idx += 32 * kConsumers) {
      const int jl = idx / k, r = idx - jl * k;
      float v = 0.f;
      if (p.slot_of_pair[r] < 0) {
        if (p.c_partial) v = p.c_partial[(size_t)r * H + j0 + jl];
        else atomicOr(p.error_word, FT_DEVERR_CAPACITY);
      }
      cb[idx] = v;
    }
    if (WT == FT_W_FP8_E4M3_B128) pdl_wait();  // block scales of filled slots are read directly
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumers) : "memory");

    const int total = ne * (st0 + st1);
    int rot = 0;  // rows handed out so far: items rotate over the warps from stage to stage
    for (int c = 0; c < total; ++c) {
      const int s = c % pl.nst;
      if (!mbar_wait(smem_u32(full + s), (uint32_t)((c / pl.nst) & 1), abort_flag, p.error_word)) break;
      const int4 m = meta[s];
      const int g = m.y;
      const uint8_t* st = stages + (size_t)s * pl.stage;
      const int q0 = ((cw - rot) % kConsumers + kConsumers) % kConsumers;
      if (m.x == 0) {
        // ---- phase 0: h[g][i] = silu(W_g[i].x) * (W_u[i].x)
        int done = 0;
        for (int q = q0; q < m.w; q += kConsumers) {
          const int i = m.z + q;
          const uint8_t* rg = st + (size_t)q * rh;          // gate row
          const uint8_t* ru = st + ((size_t)m.w + q) * rh;  // the same up row
          float a = 0.f, b = 0.f;                           // two independent chains
          if (WT == FT_W_BF16) {
            for (int c16 = lane; c16 < H / EPC; c16 += 32) {
              const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)c16 * 8);
              a = dot_bf16_bf16(*reinterpret_cast<const uint4*>(rg + (size_t)c16 * 16), xv, a);
              b = dot_bf16_bf16(*reinterpret_cast<const uint4*>(ru + (size_t)c16 * 16), xv, b);
            }
          } else {
            const float* sg = reinterpret_cast<const float*>(p.g_w[g] + p.lay.gs) + (size_t)i * (H / 128);
            const float* su = reinterpret_cast<const float*>(p.g_w[g] + p.lay.us) + (size_t)i * (H / 128);
            for (int c16 = lane; c16 < H / EPC; c16 += 32) {
              const uint4* xp = reinterpret_cast<const uint4*>(xs + (size_t)c16 * 16);
              const uint4 x0 = xp[0], x1 = xp[1];
              a = fmaf(dot_e4m3_f16(*reinterpret_cast<const uint4*>(rg + (size_t)c16 * 16), x0, x1),
                       __ldg(sg + c16 / 8), a);
              b = fmaf(dot_e4m3_f16(*reinterpret_cast<const uint4*>(ru + (size_t)c16 * 16), x0, x1),
                       __ldg(su + c16 / 8), b);
            }
          }
          const float ha = warp_sum(a), hb = warp_sum(b);
          if (lane == 0) p.h[(size_t)g * I + i] = silu_mul(ha, hb);
          ++done;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(empty + s));
          if (done) {  // publish this warp's h rows (release)
            __threadfence();
            atomicAdd(p.ready + g, (uint32_t)done);
          }
        }
      } else if (q0 < m.w) {
        // ---- phase 1: y[g][j] = W_d[g][j] . h[g], once every CTA has published h[g]
        if (lane == 0) wait_counter(p.ready + g, (uint32_t)I, abort_flag, p.error_word);
        __syncwarp();
        const float* hg = p.h + (size_t)g * I;
        for (int q = q0; q < m.w; q += kRowsILP * kConsumers) {
          float acc[kRowsILP];
          const float* sc[kRowsILP];
          bool ok[kRowsILP];
#pragma unroll
          for (int r = 0; r < kRowsILP; ++r) {
            const int qq = q + r * kConsumers;
            ok[r] = qq < m.w;
            sc[r] = WT == FT_W_BF16 ? nullptr
                                    : reinterpret_cast<const float*>(p.g_w[g] + p.lay.ds) +
                                          (size_t)(j0 + m.z + (ok[r] ? qq : q)) * (I / 128);
            acc[r] = 0.f;
          }
          for (int c16 = lane; c16 < I / EPC; c16 += 32) {
            // h written by other CTAs in this launch: read through L2
            if (WT == FT_W_BF16) {
              const float4 ha = __ldcg(reinterpret_cast<const float4*>(hg + c16 * EPC));
              const float4 hb = __ldcg(reinterpret_cast<const float4*>(hg + c16 * EPC + 4));
#pragma unroll
              for (int r = 0; r < kRowsILP; ++r)
                if (ok[r])
                  acc[r] = dot_bf16_f32v(
                      *reinterpret_cast<const uint4*>(st + (size_t)(q + r * kConsumers) * ri + (size_t)c16 * 16), ha,
                      hb, acc[r]);
            } else {
              float4 hv[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) hv[u] = __ldcg(reinterpret_cast<const float4*>(hg + c16 * EPC + 4 * u));
#pragma unroll
              for (int r = 0; r < kRowsILP; ++r)
                if (ok[r])
                  acc[r] = fmaf(
                      dot_e4m3_f32v(
                          *reinterpret_cast<const uint4*>(st + (size_t)(q + r * kConsumers) * ri + (size_t)c16 * 16),
                          hv),
                      __ldg(sc[r] + c16 / 8), acc[r]);
            }
          }
#pragma unroll
          for (int r = 0; r < kRowsILP; ++r) {
            const float v = warp_sum(acc[r]);
            if (ok[r] && lane == 0) ybuf[g * nj + m.z + q + r * kConsumers] = v;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + s));
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + s));
      }
      rot += m.w;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumers) : "memory");

    // ---- combine: one warp per output row; lane r < k holds pair r (ascending expert id)
    for (int jl = cw; jl < nj; jl += kConsumers) {
      const int j = j0 + jl;
      float val = 0.f;
      if (lane < k) {
        if (res_r) {
          val = gate_r * ybuf[gi_r * nj + jl];
          p.rows[(size_t)lane * H + j] = val;
        } else {
          val = cb[jl * k + lane];
        }
      }
      float o = p.has_shared ? ybuf[(ne - 1) * nj + jl] : 0.f;
      for (int r = 0; r < k; ++r) o += __shfl_sync(0xffffffffu, val, r);
      if (lane == 0) p.out[j] = o;
    }
  }
  __syncthreads();
}

template <int WT>
cudaError_t launch_fused_t(const EvalParams& p, int n_sm, cudaStream_t s) {
  const FusedPlan pl = make_fused_plan(WT, p.H, p.I, n_sm);
  return launch_k(fused_gemv_kernel<WT>, dim3(n_sm), dim3(kThreads), fused_smem_bytes(pl), s, p.pdl, p, pl);
}

}  // namespace

bool fused_gemv_supported(int wtype, int H, int I, int max_entries, int n_sm) {
  const FusedPlan pl = make_fused_plan(wtype, H, I, n_sm);
  return max_entries <= kMaxEntries && pl.nst >= 2 && fused_smem_bytes(pl) <= kSmemBudget + 4096;
}

cudaError_t launch_fused_gemv(const EvalParams& p, int wtype, int n_sm, int max_entries, cudaStream_t s) {
  (void)max_entries;
  return wtype == FT_W_BF16 ? launch_fused_t<FT_W_BF16>(p, n_sm, s) : launch_fused_t<FT_W_FP8_E4M3_B128>(p, n_sm, s);
}

cudaError_t prepare_fused_gemv() {
  const int lim = (int)(kSmemBudget + 4096);
  cudaError_t e = cudaFuncSetAttribute(fused_gemv_kernel<FT_W_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_gemv_kernel<FT_W_FP8_E4M3_B128>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  return e;
}

}  // namespace ft
