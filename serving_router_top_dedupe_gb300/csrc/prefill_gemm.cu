// Prefill grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMA + TMEM).
//
// A prefill chunk routes thousands of tokens, so nearly every expert of a layer gets
// ~T*k/E tokens ("FreeToken 完全拆解", section "挑战一"): the expert evaluation is a real
// dense contraction per expert.  Both projections use the weight-stationary ("swap-AB")
// form D[m, n] = sum_k W[m, k] * X[n, k]: the M side is 128 weight rows, the N side is up
// to 256 of the expert's tokens (a multiple of 16), so ragged token counts pad only to 16.
//
//  mode 0 (gate/up + SwiGLU): one 128-row M tile holds 64 gate rows and the same 64 up
//    rows of the expert (two TMA boxes), K = H.  The N operand is the expert's token rows,
//    copied into pair order beforehand so that a tile is one TMA box.  Epilogue:
//    h[p][i] = silu(g) * u as BF16.
//  mode 1 (down + gate weighting): M tile = 128 rows of W_down, K = I, the N operand is
//    the expert's contiguous rows of h.  Epilogue: rows[p][j] = BF16(gate_p * y).
//
// One CTA per SM, persistent over tiles.  Warp 0 issues TMA into a 4-stage shared-memory
// ring, warp 1 issues tcgen05.mma (one thread) into one of two TMEM accumulators, warps
// 2-9 drain the other accumulator (tcgen05.ld; two warps per TMEM lane quarter, taking
// alternate 16-column steps) while the next tile accumulates.  Every
// mbarrier wait is bounded: on timeout the kernel records FT_DEVERR_TIMEOUT, stops
// issuing work, drains its outstanding copies (bounded) and frees TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "ft_dot.cuh"
#include "ft_prefill.cuh"

namespace ft {
namespace {

constexpr int BM = 128, BK = 64, BN_MAX = 256, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int B_BYTES = BN_MAX * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
// FP8 / FP4 weights: each stage also holds the raw tile (BM rows x BK elements as stored),
// which four dequantising warps turn into the BF16 A tile; three stages fit.
constexpr int STAGES_Q = 3;
constexpr int RAW_BYTES = BM * BK;         // FP8: 8 KB (FP4: half of it used)
constexpr int STAGE_BYTES_Q = A_BYTES + B_BYTES + RAW_BYTES;
constexpr int DQ_WARPS = 4;
constexpr int EPI_COLS = 16;               // TMEM columns drained per step
constexpr int STG_PITCH = EPI_COLS + 1;    // staging row pitch (floats), bank-conflict free
constexpr int SB_BYTES = EPI_COLS * BM * 2;  // BF16 output tile of one epilogue step
constexpr int EPI_HALF_BYTES = BM * STG_PITCH * 4 + SB_BYTES;
constexpr int EPI_WARPS = 8;              // two epilogue warps per TMEM lane quarter
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int GEMM_THREADS_Q = GEMM_THREADS + 32 * DQ_WARPS;

template <int WT>
struct WCfg {
  static constexpr bool q = WT != FT_W_BF16;                                  // decoded in shared memory
  static constexpr int stages = q ? STAGES_Q : STAGES;
  static constexpr int stage_bytes = q ? STAGE_BYTES_Q : STAGE_BYTES;
  static constexpr int threads = q ? GEMM_THREADS_Q : GEMM_THREADS;
  static constexpr int raw_row = WT == FT_W_FP8_E4M3_B128 ? BK : BK / 2;    // stored bytes of BK elements
};
constexpr uint32_t kWaitLimit = 1u << 24;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with parity `parity` to complete.  On timeout sets the
// error word and the CTA's abort flag and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* error_word) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  atomicOr(error_word, FT_DEVERR_TIMEOUT);
  return false;
}

// 2-D TMA tile load completing on `bar`, with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}

// 3-D TMA tile load (x innermost) completing on `bar`, with an L2 cache policy.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}

// L2 policies: weight tiles are read by the one or two N tiles of their expert at about the
// same time, then never again in this layer (evict first); token tiles are re-read by every
// M tile of the expert (evict last).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Shared-memory matrix descriptor: K-major tile, rows of 128 bytes with the 128-byte
// swizzle, 8-row atoms 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: BF16 A and B, FP32 accumulator, both K-major.
__device__ __forceinline__ uint32_t bf16_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t b = __float_as_uint(f);
  b += 0x7FFFu + ((b >> 16) & 1u);  // round to nearest even (inputs are finite)
  return (uint16_t)(b >> 16);
}

// Two decoded weights (as floats) times the scale, as a BF16 pair (element 0 low): one
// rounding of the scaled product.
__device__ __forceinline__ uint32_t scaled_bf16x2(float2 f, float sc) {
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x * sc, f.y * sc);
  return *reinterpret_cast<uint32_t*>(&b);
}

// 16 stored E4M3 codes (element 0 in the low byte) times sc -> 16 BF16 (two 16-byte pieces)
__device__ __forceinline__ void e4m3x16_to_bf16(uint4 w, float sc, uint4& lo, uint4& hi) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t o[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    o[2 * q] = scaled_bf16x2(dot::e4m3x2_to_float2((uint16_t)(in[q] & 0xffffu)), sc);
    o[2 * q + 1] = scaled_bf16x2(dot::e4m3x2_to_float2((uint16_t)(in[q] >> 16)), sc);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// 8 stored bytes of E2M1 codes (16 elements, element 2j in the low nibble of byte j) times sc
// -> 16 BF16 (two 16-byte pieces)
__device__ __forceinline__ void e2m1x16_to_bf16(uint32_t w0, uint32_t w1, float sc, uint4& lo, uint4& hi) {
  const uint32_t in[2] = {w0, w1};
  uint32_t o[8];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t h2 = dot::e2m1x2_to_f16x2((in[q] >> (8 * b)) & 0xffu);
      o[4 * q + b] = scaled_bf16x2(__half22float2(*reinterpret_cast<const __half2*>(&h2)), sc);
    }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ float e8m0_value(uint32_t code) {
  return __uint_as_float(code ? code << 23 : 0x00400000u);
}

struct TileInfo {
  int e, m, nvalid, N, pbase;
};

// Global tile g -> (entry, M tile, N range).  M tiles are innermost, so the M tiles of one
// N tile run on neighbouring CTAs at the same time and share its token rows through L2.
__device__ __forceinline__ TileInfo decode_tile(const GemmDesc& d, int g) {
  TileInfo t;
  t.m = g % d.mt;
  const int4 q = __ldg(d.tiles + g / d.mt);
  t.e = q.x;
  t.pbase = q.y;
  t.nvalid = q.z;
  t.N = q.w;
  return t;
}

template <int MODE, int WT>
__global__ void __launch_bounds__(WCfg<WT>::threads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAs,
                        const __grid_constant__ CUtensorMap tmB, const GemmDesc d) {
  using C = WCfg<WT>;
  constexpr int NST = C::stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  // per stage: A tile (BF16, SW128) | B tile | raw weight tile (FP8 / FP4 only); then per
  // epilogue half: FP32 staging [BM][STG_PITCH] and a BF16 output tile [EPI_COLS][BM]
  uint8_t* epi = smem + NST * C::stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + 2 * EPI_HALF_BYTES);
  uint64_t* full = bars;                 // TMA bytes landed (raw or A, and B)
  uint64_t* empty = bars + NST;          // MMAs of the stage done
  uint64_t* afull = bars + 2 * NST;      // A tile decoded (FP8 / FP4)
  uint64_t* tfull = bars + 3 * NST;
  uint64_t* tempty = bars + 3 * NST + 2;
  uint64_t* done = bars + 3 * NST + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * NST + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
      mbar_init(smem_u32(afull + s), DQ_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(tfull + b), 1);
      mbar_init(smem_u32(tempty + b), 32 * EPI_WARPS);
    }
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {  // 512 TMEM columns: two 256-column FP32 accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = d.mt * __ldg(d.tile_off + d.n_entries);
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int last_par[NST];
#pragma unroll
    for (int s = 0; s < NST; ++s) last_par[s] = -1;
    for (int g = blockIdx.x; g < total; g += gridDim.x) {
      const TileInfo t = decode_tile(d, g);
      if (t.nvalid <= 0) continue;
      const bool sh = t.e >= d.E;
      const CUtensorMap* mA = sh ? &tmAs : &tmA;
      const int wbase = sh ? d.layer : __ldg(d.buf_slots + t.e);
      int arow0, arow1 = 0;
      if (C::q) {  // 3-D maps: (byte within the row, row within the slot's bank, slot)
        arow0 = MODE == 0 ? t.m * 64 : t.m * BM;
        arow1 = arow0 + d.I;                // up rows follow the gate rows
      } else if (MODE == 0) {
        arow0 = wbase * 3 * d.I + t.m * 64;  // gate rows
        arow1 = arow0 + d.I;                 // up rows
      } else {
        arow0 = wbase * 3 * d.H + 2 * d.H + t.m * BM;  // down rows
      }
      bool ok = true;
      for (int kb = 0; kb < d.kb; ++kb) {
        int w_ok = lane == 0 ? (int)mbar_wait(smem_u32(empty + stage), phase ^ 1u, abort_flag, d.error_word) : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        const uint32_t a_dst = smem_base + stage * C::stage_bytes, b_dst = a_dst + A_BYTES;
        const uint32_t raw_dst = b_dst + B_BYTES;
        const uint32_t fb = smem_u32(full + stage);
        if (lane == 0) {
          // the token box is always BN_MAX rows (rows past the tile belong to the next entry
          // or lie beyond the buffer and are zero-filled; the epilogue ignores them)
          if (C::q) {
            mbar_arrive_expect_tx(fb, BM * C::raw_row + B_BYTES);
            if (MODE == 0) {
              tma_load_3d_hint(raw_dst, mA, kb * C::raw_row, arow0, wbase, fb, pol_w);
              tma_load_3d_hint(raw_dst + 64 * C::raw_row, mA, kb * C::raw_row, arow1, wbase, fb, pol_w);
            } else {
              tma_load_3d_hint(raw_dst, mA, kb * C::raw_row, arow0, wbase, fb, pol_w);
            }
          } else {
            mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
            if (MODE == 0) {
              tma_load_2d_hint(a_dst, mA, kb * BK, arow0, fb, pol_w);
              tma_load_2d_hint(a_dst + A_BYTES / 2, mA, kb * BK, arow1, fb, pol_w);
            } else {
              tma_load_2d_hint(a_dst, mA, kb * BK, arow0, fb, pol_w);
            }
          }
          tma_load_2d_hint(b_dst, &tmB, kb * BK, t.pbase, fb, pol_x);
        }
        __syncwarp();
        last_par[stage] = (int)phase;
        if (++stage == NST) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    if (*abort_flag && lane == 0) {  // drain copies still in flight before the CTA exits
      for (int s = 0; s < NST; ++s)
        if (last_par[s] >= 0)
          for (uint32_t i = 0; i < kWaitLimit && !mbar_try_wait(smem_u32(full + s), (uint32_t)last_par[s]); ++i) {
          }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int g = blockIdx.x; g < total && ok; g += gridDim.x) {
        const TileInfo t = decode_tile(d, g);
        if (t.nvalid <= 0) continue;
        if (!mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1u, abort_flag, d.error_word)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN_MAX);
        const uint32_t idesc = bf16_idesc(BM, t.N);
        for (int kb = 0; kb < d.kb; ++kb) {
          // FP8 / FP4: the decoded tile (its warps waited for the TMA bytes, so B has landed too)
          if (!mbar_wait(smem_u32((C::q ? afull : full) + stage), phase, abort_flag, d.error_word)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_base + stage * C::stage_bytes, b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d_tmem, sw128_desc(a_addr + 32 * k), sw128_desc(b_addr + 32 * k), idesc, (kb | k) != 0);
          umma_commit(smem_u32(empty + stage));
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(tfull + acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA issued above has completed once `done` flips
      umma_commit(smem_u32(done));
      for (uint32_t i = 0; i < kWaitLimit && !mbar_try_wait(smem_u32(done), 0u); ++i) {
      }
    }
    __syncwarp();
  } else if (warp < 2 + EPI_WARPS) {
    // --------------------------------------------------------------- epilogue
    const int half = (threadIdx.x - 64) >> 7;  // the two halves take alternate column steps
    const int et = (threadIdx.x - 64) & 127;   // 0..127 within the half
    const int q4 = warp & 3;                   // TMEM lane quarter this warp may access
    float* stg = reinterpret_cast<float*>(epi + half * EPI_HALF_BYTES);
    uint16_t* sb = reinterpret_cast<uint16_t*>(stg + BM * STG_PITCH);
    const uint32_t bar_id = 1 + half;
    const int m = 32 * q4 + lane;          // accumulator row (TMEM lane)
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int g = blockIdx.x; g < total; g += gridDim.x) {
      const TileInfo t = decode_tile(d, g);
      if (t.nvalid <= 0) continue;
      if (!mbar_wait(smem_u32(tfull + acc), acc_phase, abort_flag, d.error_word)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * q4) << 16) + (uint32_t)(acc * BN_MAX);
      for (int c0 = half * EPI_COLS; c0 < t.N; c0 += 2 * EPI_COLS) {
        float v[EPI_COLS];
        tmem_ld16(tbase + c0, v);
        // results go out as 16-byte row pieces through a BF16 tile in shared memory
        if (MODE == 0) {
#pragma unroll
          for (int c = 0; c < EPI_COLS; ++c) stg[m * STG_PITCH + c] = v[c];
          asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
          const int i = et & 63, cb = (et >> 6) * (EPI_COLS / 2);
#pragma unroll
          for (int c = 0; c < EPI_COLS / 2; ++c) {  // h[n][i] for this thread's 8 tokens
            const float gv = stg[i * STG_PITCH + cb + c], uv = stg[(64 + i) * STG_PITCH + cb + c];
            sb[(cb + c) * 64 + i] = f2bf(gv / (1.0f + expf(-gv)) * uv);
          }
          asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
          {  // 16 tokens x 64 h values: one 16-byte piece per thread
            const int n = et >> 3, ch = et & 7;
            if (c0 + n < t.nvalid)
              *reinterpret_cast<uint4*>(d.h + (size_t)(t.pbase + c0 + n) * d.I + t.m * 64 + ch * 8) =
                  *reinterpret_cast<const uint4*>(sb + n * 64 + ch * 8);
          }
          asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
        } else {
#pragma unroll
          for (int c = 0; c < EPI_COLS; ++c) {
            const int n = c0 + c;
            const float gate = n < t.nvalid ? __ldg(d.pair_gate + t.pbase + n) : 0.f;
            sb[c * BM + m] = f2bf(gate * v[c]);
          }
          asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
#pragma unroll
          for (int q = 0; q < EPI_COLS * BM / 8 / 128; ++q) {  // 16 tokens x 128 outputs
            const int idx = et + 128 * q, n = idx >> 4, ch = idx & 15;
            if (c0 + n < t.nvalid)
              *reinterpret_cast<uint4*>(d.rows + (size_t)(t.pbase + c0 + n) * d.H + t.m * BM + ch * 8) =
                  *reinterpret_cast<const uint4*>(sb + n * BM + ch * 8);
          }
          asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(tempty + acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if (C::q) {
    // ---------------------------------------------------------- weight decoding
    // Thread r decodes row r of the A tile: each of its BK stored weights times the scale of
    // its block (FP8: one FP32 scale per 1x128 block; NVFP4: E4M3 scale per 16 elements times
    // the bank's FP32 tensor scale; MXFP4: E8M0 scale per 32 elements), rounded once to BF16
    // and written in the 128-byte-swizzled K-major layout the MMA reads.
    const int r = threadIdx.x - GEMM_THREADS;  // 0..127
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int g = blockIdx.x; g < total && ok; g += gridDim.x) {
      const TileInfo t = decode_tile(d, g);
      if (t.nvalid <= 0) continue;
      const bool sh = t.e >= d.E;
      const uint8_t* slot = sh ? d.shared_w + (size_t)d.layer * d.stride
                               : d.pool + (size_t)__ldg(d.buf_slots + t.e) * d.stride;
      const int K = MODE == 0 ? d.H : d.I;                      // reduction length of the row
      const int row = MODE == 0 ? t.m * 64 + (r & 63) : t.m * BM + r;
      const size_t soff = MODE == 0 ? (r < 64 ? d.off_gs : d.off_us) : d.off_ds;
      const int bank = MODE == 0 ? (r < 64 ? 0 : 1) : 2;
      const float tsc = WT == FT_W_NVFP4 ? __ldg(reinterpret_cast<const float*>(slot + d.off_ts) + bank) : 1.f;
      for (int kb = 0; kb < d.kb; ++kb) {
        if (!mbar_wait(smem_u32(full + stage), phase, abort_flag, d.error_word)) {
          ok = false;
          break;
        }
        const uint8_t* st = smem + stage * C::stage_bytes;
        const uint4* src = reinterpret_cast<const uint4*>(st + A_BYTES + B_BYTES + r * C::raw_row);
        uint8_t* arow = const_cast<uint8_t*>(st) + r * 128;
        auto put = [&](int ch, uint4 v) { *reinterpret_cast<uint4*>(arow + ((ch ^ (r & 7)) << 4)) = v; };
        if (WT == FT_W_FP8_E4M3_B128) {
          const float sc = __ldg(reinterpret_cast<const float*>(slot + soff) + (size_t)row * (K / 128) + kb / 2);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 lo, hi;
            e4m3x16_to_bf16(src[q], sc, lo, hi);
            put(2 * q, lo);
            put(2 * q + 1, hi);
          }
        } else if (WT == FT_W_NVFP4) {
          // four E4M3 block scales for the BK = 64 elements of this step
          const uint32_t sc4 = __ldg(reinterpret_cast<const uint32_t*>(slot + soff + (size_t)row * (K / 16)) + kb);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint4 w = src[q];
            const float2 s01 = dot::e4m3x2_to_float2((uint16_t)(q == 0 ? (sc4 & 0xffffu) : (sc4 >> 16)));
            uint4 lo, hi;
            e2m1x16_to_bf16(w.x, w.y, s01.x * tsc, lo, hi);
            put(4 * q, lo);
            put(4 * q + 1, hi);
            e2m1x16_to_bf16(w.z, w.w, s01.y * tsc, lo, hi);
            put(4 * q + 2, lo);
            put(4 * q + 3, hi);
          }
        } else {
          // two E8M0 block scales for the BK = 64 elements of this step
          const uint32_t sc2 =
              __ldg(reinterpret_cast<const uint16_t*>(slot + soff + (size_t)row * (K / 32)) + kb);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint4 w = src[q];
            const float sc = e8m0_value(q == 0 ? (sc2 & 0xffu) : (sc2 >> 8));
            uint4 lo, hi;
            e2m1x16_to_bf16(w.x, w.y, sc, lo, hi);
            put(4 * q, lo);
            put(4 * q + 1, hi);
            e2m1x16_to_bf16(w.z, w.w, sc, lo, hi);
            put(4 * q + 2, lo);
            put(4 * q + 3, hi);
          }
        }
        // the MMA reads the tile through the async proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(afull + stage));
        if (++stage == NST) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base) : "memory");
  }
}

}  // namespace

// ------------------------------------------------------------------------ host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder() {
  if (g_encode) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e != cudaSuccess ? e : cudaErrorNotSupported;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

// 2-D BF16 tensor [outer][inner] with row pitch row_bytes, 128-byte swizzled boxes.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                     uint32_t box_inner, uint32_t box_outer) {
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D byte tensor (stored weights of one bank per slot): dims {row bytes, rows, slots},
// unswizzled boxes {box_bytes, box_rows, 1}.
cudaError_t make_map_raw3d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
                           uint64_t slot_stride, uint32_t box_bytes, uint32_t box_rows) {
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[3] = {row_bytes, rows, slots};
  const cuuint64_t strides[2] = {row_bytes, slot_stride};
  const cuuint32_t box[3] = {box_bytes, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int WT>
size_t gemm_smem_bytes() {
  return 1024 + WCfg<WT>::stages * WCfg<WT>::stage_bytes + 2 * EPI_HALF_BYTES + (3 * WCfg<WT>::stages + 5) * 8 + 16;
}

template <int WT>
cudaError_t set_gemm_attrs() {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<0, WT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)gemm_smem_bytes<WT>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<1, WT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gemm_smem_bytes<WT>());
  return e;
}

template <int WT>
void launch_t(int mode, const CUtensorMap& a, const CUtensorMap& as, const CUtensorMap& b, const GemmDesc& d, int grid,
              cudaStream_t s) {
  if (mode == 0) grouped_gemm_kernel<0, WT><<<grid, WCfg<WT>::threads, gemm_smem_bytes<WT>(), s>>>(a, as, b, d);
  else grouped_gemm_kernel<1, WT><<<grid, WCfg<WT>::threads, gemm_smem_bytes<WT>(), s>>>(a, as, b, d);
}

}  // namespace

struct GemmMaps {
  CUtensorMap a_gu, a_gu_sh;    // weight rows of width H (gate, up): pool / shared experts
  CUtensorMap a_dn, a_dn_sh;    // weight rows of width I (down)
  CUtensorMap h_map;            // h [P][I]
  CUtensorMap x_map;            // token rows in pair order [P][H]
  int H, I, wtype;
};

cudaError_t gemm_maps_create(GemmMaps** out, const uint8_t* pool, int S, const uint8_t* shared_w, int L, int H,
                             int I, const uint16_t* h_buf, const uint16_t* xp_buf, int max_pairs, int wtype,
                             const SlotLayout& lay) {
  GemmMaps* m = new GemmMaps();
  m->H = H;
  m->I = I;
  m->wtype = wtype;
  const void* sh = shared_w ? (const void*)shared_w : (const void*)pool;
  const uint64_t sh_rows = shared_w ? (uint64_t)L : (uint64_t)S;
  cudaError_t e = cudaSuccess;
  if (wtype == FT_W_BF16) {
    // a slot is gate [I][H] | up [I][H] | down [H][I]: 3I rows of width H, or 3H rows of width I
    e = make_map(&m->a_gu, pool, H, (uint64_t)S * 3 * I, (uint64_t)H * 2, BK, 64);
    if (e == cudaSuccess) e = make_map(&m->a_dn, pool, I, (uint64_t)S * 3 * H, (uint64_t)I * 2, BK, BM);
    if (e == cudaSuccess) e = make_map(&m->a_gu_sh, sh, H, sh_rows * 3 * I, (uint64_t)H * 2, BK, 64);
    if (e == cudaSuccess) e = make_map(&m->a_dn_sh, sh, I, sh_rows * 3 * H, (uint64_t)I * 2, BK, BM);
  } else {
    // stored weights, one 3-D map per bank kind: (byte in row, row, slot); gate and up rows
    // are contiguous, so one map covers both (rows 0..2I-1)
    const uint64_t div = wtype == FT_W_FP8_E4M3_B128 ? 1 : 2;  // elements per stored byte
    const uint32_t raw = (uint32_t)(BK / div);
    const uint8_t* shb = static_cast<const uint8_t*>(sh);
    e = make_map_raw3d(&m->a_gu, pool + lay.gate, (uint64_t)H / div, 2 * (uint64_t)I, (uint64_t)S, lay.stride, raw,
                       64);
    if (e == cudaSuccess)
      e = make_map_raw3d(&m->a_dn, pool + lay.down, (uint64_t)I / div, (uint64_t)H, (uint64_t)S, lay.stride, raw, BM);
    if (e == cudaSuccess)
      e = make_map_raw3d(&m->a_gu_sh, shb + lay.gate, (uint64_t)H / div, 2 * (uint64_t)I, sh_rows, lay.stride, raw,
                         64);
    if (e == cudaSuccess)
      e = make_map_raw3d(&m->a_dn_sh, shb + lay.down, (uint64_t)I / div, (uint64_t)H, sh_rows, lay.stride, raw, BM);
  }
  if (e == cudaSuccess) e = make_map(&m->h_map, h_buf, I, (uint64_t)max_pairs, (uint64_t)I * 2, BK, BN_MAX);
  if (e == cudaSuccess) e = make_map(&m->x_map, xp_buf, H, (uint64_t)max_pairs, (uint64_t)H * 2, BK, BN_MAX);
  if (e == cudaSuccess) {
    switch (wtype) {
      case FT_W_BF16: e = set_gemm_attrs<FT_W_BF16>(); break;
      case FT_W_FP8_E4M3_B128: e = set_gemm_attrs<FT_W_FP8_E4M3_B128>(); break;
      case FT_W_NVFP4: e = set_gemm_attrs<FT_W_NVFP4>(); break;
      default: e = set_gemm_attrs<FT_W_MXFP4>(); break;
    }
  }
  if (e != cudaSuccess) {
    delete m;
    return e;
  }
  *out = m;
  return cudaSuccess;
}

void gemm_maps_destroy(GemmMaps* m) { delete m; }

cudaError_t launch_grouped_gemm(int mode, const GemmMaps* m, const uint16_t* x, int T, const GemmDesc& d, int grid,
                                cudaStream_t s) {
  (void)x;
  (void)T;
  const CUtensorMap& a = mode == 0 ? m->a_gu : m->a_dn;
  const CUtensorMap& as = mode == 0 ? m->a_gu_sh : m->a_dn_sh;
  const CUtensorMap& b = mode == 0 ? m->x_map : m->h_map;
  switch (m->wtype) {
    case FT_W_BF16: launch_t<FT_W_BF16>(mode, a, as, b, d, grid, s); break;
    case FT_W_FP8_E4M3_B128: launch_t<FT_W_FP8_E4M3_B128>(mode, a, as, b, d, grid, s); break;
    case FT_W_NVFP4: launch_t<FT_W_NVFP4>(mode, a, as, b, d, grid, s); break;
    default: launch_t<FT_W_MXFP4>(mode, a, as, b, d, grid, s); break;
  }
  return cudaGetLastError();
}

}  // namespace ft
