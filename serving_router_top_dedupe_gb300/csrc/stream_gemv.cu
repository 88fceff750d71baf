// Decode expert GEMV at batch 1, streamed through shared memory with bulk async copies.
//
// A decode layer reads every byte of its G-set experts once (~1 FLOP per byte), so the
// kernel is bound by HBM; the question is only how many bytes each SM keeps in flight.
// Register-staged loads cap that at a few tens of KB per SM, so each SM's share (hundreds
// of KB) takes several dependent round trips.  Here one CTA per SM keeps up to ~190 KB of
// weight rows in flight in a ring of shared-memory stages filled by cp.async.bulk (no
// registers spent), and eight consumer warps form the dot products from shared memory.
//
//  phase 0 (gate/up): units = entries x I; a stage holds gate rows i0..i0+n-1 and the
//                     same up rows (two bulk copies); a warp forms a = W_g[i].x and
//                     b = W_u[i].x and writes h[entry][i] = silu(a)*b.
//  phase 1 (down):    each CTA owns a range of output rows j, and streams W_down[g][j] of
//                     every entry g for them; vector = h_g (staged in shared memory);
//                     then out[j] = shared + the k pair rows in ascending
//                     expert id (GPU row g_r*y, or the caller's c_partial row).
//
// Per (entry, row) the lane-strided 16-byte chunk order and the xor butterfly match the
// other decode kernels, so results are bit-identical to them.  Warp 0 lane 0 is the
// producer; every mbarrier wait is bounded (FT_DEVERR_TIMEOUT on expiry).
#include "ft_dot.cuh"
#include "ft_internal.cuh"
#include "ft_ptx.cuh"

namespace ft {
namespace {

using namespace dot;
using namespace ptx;

constexpr int kConsumers = 8;
constexpr int kStreamThreads = 32 * (kConsumers + 1);
constexpr int kMaxStages = 8;
constexpr size_t kStageTarget = 32 * 1024;   // bytes per stage: one contiguous bulk copy
constexpr size_t kSmemBudget = 220 * 1024;

struct StreamPlan {
  int rps;          // rows per stage (at most; a stage never spans two experts)
  int nst;          // stages
  size_t stage;     // bytes per stage
  size_t vec;       // bytes of the vector area (x, or h of every entry)
  size_t ybuf;      // bytes of per-(entry, j) results (phase 1)
};

__host__ __device__ inline StreamPlan make_plan(int phase, int wtype, int H, int I, int max_entries, int n_cta) {
  const size_t esz = wtype == FT_W_BF16 ? 2 : 1;
  const size_t row = phase == 0 ? (size_t)H * esz : (size_t)I * esz;
  StreamPlan pl;
  pl.rps = (int)(kStageTarget / row) > 0 ? (int)(kStageTarget / row) : 1;
  if (phase == 0) pl.rps = pl.rps >= 2 ? pl.rps / 2 * 2 : 2;  // pairs of (gate, up) rows
  pl.stage = (size_t)pl.rps * row;
  pl.vec = phase == 0 ? (size_t)H * 2 : (size_t)max_entries * I * 4;
  const int jpc = (H + n_cta - 1) / n_cta;
  pl.ybuf = phase == 0 ? 0 : ((size_t)jpc * max_entries * 4 + 127) / 128 * 128;  // keeps the mbarriers 8-aligned
  const size_t fixed = pl.vec + pl.ybuf + 1024;
  int nst = fixed >= kSmemBudget ? 0 : (int)((kSmemBudget - fixed) / pl.stage);
  pl.nst = nst > kMaxStages ? kMaxStages : nst;
  return pl;
}

template <int WT, int PHASE>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_gemv_kernel(EvalParams p, StreamPlan pl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
  uint8_t* stages = smem;
  uint8_t* vec = stages + (size_t)pl.nst * pl.stage;
  float* ybuf = reinterpret_cast<float*>(vec + pl.vec);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ybuf) + pl.ybuf);
  uint64_t* empty = full + kMaxStages;
  int2* meta = reinterpret_cast<int2*>(empty + kMaxStages);  // per stage: first local row, row count
  volatile int* abort_flag = reinterpret_cast<volatile int*>(meta + kMaxStages);

  constexpr int ESZ = WT == FT_W_BF16 ? 2 : 1;
  constexpr int EPC = 16 / ESZ;
  const int ne = p.counts[C_NENTRIES];
  const int H = p.H, I = p.I, k = p.k;
  const int row_elems = PHASE == 0 ? H : I;
  const size_t row_bytes = (size_t)row_elems * ESZ;
  const int row_chunks = row_elems / EPC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // This CTA's rows, in an order where each expert's rows are contiguous in memory.
  //  phase 0: local row t = global row r_begin + t, r = g*2I + rr (gate rows, then up rows)
  //  phase 1: local row t = g*nj + jl for output row j0 + jl of entry g
  //  phase 0: local unit t = global unit r_begin + t = g*I + i (gate row i and up row i)
  int r_begin = 0, n_rows, j0 = 0, nj = 0;
  if (PHASE == 0) {
    const long long R = (long long)ne * I;
    r_begin = (int)(R * blockIdx.x / gridDim.x);
    n_rows = (int)(R * (blockIdx.x + 1) / gridDim.x) - r_begin;
  } else {
    j0 = (int)((long long)H * blockIdx.x / gridDim.x);
    nj = (int)((long long)H * (blockIdx.x + 1) / gridDim.x) - j0;
    n_rows = nj * ne;
  }
  auto entry_of = [&](int t) { return PHASE == 0 ? (r_begin + t) / I : t / max(nj, 1); };
  auto row_src = [&](int t) -> const uint8_t* {
    if (PHASE == 0) {
      const int r = r_begin + t, g = r / I, i = r - g * I;
      return p.g_w[g] + p.lay.gate + (size_t)i * row_bytes;
    }
    const int g = t / nj, jl = t - g * nj;
    return p.g_w[g] + p.lay.down + (size_t)(j0 + jl) * row_bytes;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < pl.nst; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kConsumers);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      // Phase 0 streams the rows of experts that were resident before this step first
      // (their slots are not written by the fill kernel running right before), then waits
      // for the fill and streams the filled experts.  Phase 1 only needs data of kernels
      // two or more back, so it streams everything and waits before its consumers read h.
      int c = 0;
      bool waited = false;
      for (int pass = 0; pass < (PHASE == 0 ? 2 : 1) && !*abort_flag; ++pass) {
        if (PHASE == 0 && pass == 1) {
          pdl_wait();
          pdl_trigger();
          waited = true;
        }
        int t = 0;
        while (t < n_rows) {
          const int g = entry_of(t);
          const int last = PHASE == 0 ? (g + 1) * I - r_begin : (g + 1) * nj;
          if (PHASE == 0 && (p.g_fill[g] != 0) != (pass == 1)) {  // not this pass: skip the entry
            t = last;
            continue;
          }
          const int s = c % pl.nst, use = c / pl.nst;
          if (PHASE == 1 && !waited && use > 0) {  // ring is full: join the dependency chain now
            pdl_wait();
            pdl_trigger();
            waited = true;
          }
          if (!mbar_wait(smem_u32(empty + s), (uint32_t)(use & 1) ^ 1u, abort_flag, p.error_word)) break;
          const int cap = PHASE == 0 ? pl.rps / 2 : pl.rps;
          const int nr = min(min(cap, n_rows - t), last - t);
          meta[s] = make_int2(t, nr);
          const uint32_t fb = smem_u32(full + s);
          const uint32_t dst = smem_u32(stages + (size_t)s * pl.stage);
          if (PHASE == 0) {  // gate rows, then the same up rows (I rows further on in the slot)
            mbar_arrive_expect_tx(fb, (uint32_t)(2 * nr * row_bytes));
            bulk_g2s(dst, row_src(t), (uint32_t)(nr * row_bytes), fb);
            bulk_g2s(dst + (uint32_t)(nr * row_bytes), row_src(t) + (size_t)I * row_bytes, (uint32_t)(nr * row_bytes),
                     fb);
          } else {
            mbar_arrive_expect_tx(fb, (uint32_t)(nr * row_bytes));
            bulk_g2s(dst, row_src(t), (uint32_t)(nr * row_bytes), fb);
          }
          t += nr;
          ++c;
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
    if (PHASE == 0) {
      uint16_t* xs = reinterpret_cast<uint16_t*>(vec);  // the token: bf16 (BF16 weights) or f16 (FP8)
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
    } else {
      pdl_wait();  // h is written by the kernel right before
      // h of every entry (written by phase 0): independent 16-byte loads
      float4* hs = reinterpret_cast<float4*>(vec);
      const float4* hg = reinterpret_cast<const float4*>(p.h);
      const int n4 = ne * I / 4;
      for (int i0 = ct; i0 < n4; i0 += 4 * 32 * kConsumers) {
        float4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (i0 + q * 32 * kConsumers < n4) v[q] = __ldcg(hg + i0 + q * 32 * kConsumers);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (i0 + q * 32 * kConsumers < n4) hs[i0 + q * 32 * kConsumers] = v[q];
      }
    }
    if (PHASE == 0 && WT == FT_W_FP8_E4M3_B128) pdl_wait();  // block scales of filled slots
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumers) : "memory");
    int t_done = 0, c = 0;
    while (t_done < n_rows) {
      const int s = c % pl.nst, use = c / pl.nst;
      if (!mbar_wait(smem_u32(full + s), (uint32_t)(use & 1), abort_flag, p.error_word)) break;
      const int2 m = meta[s];
      const uint8_t* st = stages + (size_t)s * pl.stage;
      for (int q = cw; q < m.y; q += kConsumers) {  // rows of the stage split over the warps
        const int t = m.x + q;
        const uint8_t* rowp = st + (size_t)q * row_bytes;
        float acc = 0.f;
        (void)rowp;
        (void)acc;
        if (PHASE == 0) {
          const int r = r_begin + t, g = r / I, i = r - g * I;
          const uint16_t* xs = reinterpret_cast<const uint16_t*>(vec);
          float ab2[2];
#pragma unroll
          for (int half = 0; half < 2; ++half) {  // gate row, then up row
            const uint8_t* rp = st + ((size_t)half * m.y + q) * row_bytes;
            const float* sc = WT == FT_W_BF16
                                  ? nullptr
                                  : reinterpret_cast<const float*>(p.g_w[g] + (half ? p.lay.us : p.lay.gs)) +
                                        (size_t)i * (H / 128);
            float a = 0.f;
            for (int c16 = lane; c16 < row_chunks; c16 += 32) {
              const uint4 wv = *reinterpret_cast<const uint4*>(rp + (size_t)c16 * 16);
              if (WT == FT_W_BF16) {
                a = dot_bf16_bf16(wv, *reinterpret_cast<const uint4*>(xs + (size_t)c16 * 8), a);
              } else {
                const uint4* xp = reinterpret_cast<const uint4*>(xs + (size_t)c16 * 16);
                a = fmaf(dot_e4m3_f16(wv, xp[0], xp[1]), __ldg(sc + c16 / 8), a);
              }
            }
            ab2[half] = warp_sum(a);
          }
          if (lane == 0) p.h[(size_t)g * I + i] = silu_mul(ab2[0], ab2[1]);
        } else {
          const int g = t / nj, jl = t - g * nj;
          const float* hg = reinterpret_cast<const float*>(vec) + (size_t)g * I;
          const float* sc = WT == FT_W_BF16 ? nullptr
                                             : reinterpret_cast<const float*>(p.g_w[g] + p.lay.ds) +
                                                   (size_t)(j0 + jl) * (I / 128);
          for (int c16 = lane; c16 < row_chunks; c16 += 32) {
            const uint4 wv = *reinterpret_cast<const uint4*>(rowp + (size_t)c16 * 16);
            if (WT == FT_W_BF16) acc = dot_bf16_f32(wv, hg + c16 * EPC, acc);
            else acc = fmaf(dot_e4m3_f32(wv, hg + c16 * EPC), __ldg(sc + c16 / 8), acc);
          }
          const float v = warp_sum(acc);
          if (lane == 0) ybuf[t] = v;  // [entry][jl]
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(empty + s));
      t_done += m.y;
      ++c;
    }
    if (PHASE == 1) {
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumers) : "memory");
      // combine: one warp per output row; lane r < k holds pair r
      const bool res_r = lane < k && p.slot_of_pair[lane] >= 0;
      const uint32_t res_mask = __ballot_sync(0xffffffffu, res_r);
      const int gi_r = __popc(res_mask & ((1u << lane) - 1u));
      const float gate_r = lane < k ? p.gates[lane] : 0.f;
      for (int jl = cw; jl < nj; jl += kConsumers) {
        const int j = j0 + jl;
        float val = 0.f;
        if (lane < k) {
          if (res_r) {
            val = gate_r * ybuf[(size_t)gi_r * nj + jl];
            p.rows[(size_t)lane * H + j] = val;
          } else if (p.c_partial) {
            val = p.c_partial[(size_t)lane * H + j];
          } else {
            atomicOr(p.error_word, FT_DEVERR_CAPACITY);
          }
        }
        float o = p.has_shared ? ybuf[(size_t)(ne - 1) * nj + jl] : 0.f;
        for (int r = 0; r < k; ++r) o += __shfl_sync(0xffffffffu, val, r);
        if (lane == 0) p.out[j] = o;
      }
    }
  }
  __syncthreads();
}

template <int WT, int PHASE>
cudaError_t launch_stream(const EvalParams& p, int n_sm, int max_entries, cudaStream_t s) {
  const StreamPlan pl = make_plan(PHASE, WT, p.H, p.I, max_entries, n_sm);
  const size_t smem = (size_t)pl.nst * pl.stage + pl.vec + pl.ybuf + 2 * kMaxStages * 8 + kMaxStages * 8 + 16 + 128;
  return launch_k(stream_gemv_kernel<WT, PHASE>, dim3(n_sm), dim3(kStreamThreads), smem, s, p.pdl, p, pl);
}

}  // namespace

cudaError_t prepare_stream_gemv() {
  const int lim = (int)(kSmemBudget + 4096);
  cudaError_t e = cudaFuncSetAttribute(stream_gemv_kernel<FT_W_BF16, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_gemv_kernel<FT_W_BF16, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_gemv_kernel<FT_W_FP8_E4M3_B128, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             lim);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_gemv_kernel<FT_W_FP8_E4M3_B128, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             lim);
  return e;
}

bool stream_gemv_supported(int wtype, int H, int I, int max_entries, int n_sm) {
  for (int phase = 0; phase < 2; ++phase) {
    const StreamPlan pl = make_plan(phase, wtype, H, I, max_entries, n_sm);
    if (pl.nst < 2) return false;
  }
  return true;
}

cudaError_t launch_stream_gemv(int phase, const EvalParams& p, int wtype, int n_sm, int max_entries,
                               cudaStream_t s) {
  if (wtype == FT_W_BF16)
    return phase == 0 ? launch_stream<FT_W_BF16, 0>(p, n_sm, max_entries, s)
                      : launch_stream<FT_W_BF16, 1>(p, n_sm, max_entries, s);
  return phase == 0 ? launch_stream<FT_W_FP8_E4M3_B128, 0>(p, n_sm, max_entries, s)
                    : launch_stream<FT_W_FP8_E4M3_B128, 1>(p, n_sm, max_entries, s);
}

}  // namespace ft
