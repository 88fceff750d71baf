// Router logits from hidden states: z[t][e] = sum_h x[t][h] * W_router[e][h], BF16
// operands, FP32 accumulation.  The router runs on the GPU with the rest of the
// routing-dependent control ("개인 장치에서 MoE 모델을 서빙하는 FreeToken", decode
// paragraph: the GPU router dedupes the active experts; "OSDI'26 | 双路 CPU + 两张
// 5090…", §3.3: gate and sort run on the GPU), so a decode layer can take hidden states
// instead of precomputed logits.
//
// The router projection of one layer is E x H BF16 (1 MB at E = 256, H = 2048): a GEMV
// at decode batch sizes.  One warp owns one router row at a time and keeps its first
// 2048 elements in registers, loaded before the programmatic-dependency wait, because
// the weights do not depend on the previous kernel; a CTA stages a tile of token rows
// in shared memory after the wait and every warp of the CTA reuses it.  Each logit is
// one lane-strided FP32 dot product followed by an xor butterfly, so its bits do not
// depend on the launch shape.
#include <algorithm>

#include "ft_internal.cuh"
#include "ft_dot.cuh"

namespace ft {
namespace {

constexpr int kRouterWarps = 8;
constexpr int kRouterRegVecs = 8;  // 16-byte vectors of a router row held per lane

__device__ __forceinline__ void load_row_regs(const uint4* wrow, int nvec, int lane, uint4 (&wr)[kRouterRegVecs]) {
#pragma unroll
  for (int i = 0; i < kRouterRegVecs; ++i) {
    const int idx = lane + 32 * i;
    wr[i] = idx < nvec ? __ldg(wrow + idx) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// grid (ceil(E / (kRouterWarps * e_per_warp)), ceil(T / tok_tile)); dynamic shared memory
// tok_tile * H * 2 bytes.  Warp w of CTA x handles experts (x * e_per_warp + j) * 8 + w.
__global__ void __launch_bounds__(kRouterWarps * 32) router_logits_kernel(RouterParams p) {
  extern __shared__ uint4 s_x[];  // [tok_tile][H / 8]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = p.H >> 3;
  const int t0 = blockIdx.y * p.tok_tile;
  const int nt = min(p.tok_tile, p.T - t0);
  const uint4* wbase = reinterpret_cast<const uint4*>(p.w);
  const int e_first = blockIdx.x * p.e_per_warp * kRouterWarps + warp;

  uint4 wr[kRouterRegVecs];
  load_row_regs(wbase + (size_t)min(e_first, p.E - 1) * nvec, nvec, lane, wr);
  if (p.pdl) pdl_wait();
  const uint4* xg = reinterpret_cast<const uint4*>(p.x) + (size_t)t0 * nvec;
  for (int i = threadIdx.x; i < nt * nvec; i += blockDim.x) s_x[i] = xg[i];
  __syncthreads();
  if (p.pdl) pdl_trigger();

  for (int j = 0; j < p.e_per_warp; ++j) {
    const int e = e_first + j * kRouterWarps;
    if (e >= p.E) break;
    const uint4* wrow = wbase + (size_t)e * nvec;
    if (j > 0) load_row_regs(wrow, nvec, lane, wr);
    for (int t = 0; t < nt; ++t) {
      const uint4* xs = s_x + (size_t)t * nvec;
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kRouterRegVecs; ++i) {
        const int idx = lane + 32 * i;
        if (idx < nvec) acc = dot::dot_bf16_bf16(wr[i], xs[idx], acc);
      }
      for (int idx = lane + 32 * kRouterRegVecs; idx < nvec; idx += 32)
        acc = dot::dot_bf16_bf16(__ldg(wrow + idx), xs[idx], acc);
      acc = dot::warp_sum(acc);
      if (lane == 0) p.z[(size_t)(t0 + t) * p.E + e] = acc;
    }
  }
}

}  // namespace

size_t router_smem_bytes(int tok_tile, int H) { return (size_t)tok_tile * H * 2; }

void router_shape(int T, int E, int H, int* tok_tile, int* e_per_warp) {
  // decode batches: one router row per warp, the tokens in tiles of 8 (x tiles stay
  // small and every SM holds several CTAs); prefill chunks: 4 rows per warp over tiles
  // of 16 tokens, so each staged token tile serves 32 experts
  int tt = T <= 64 ? 8 : 16;
  while (tt > 1 && router_smem_bytes(tt, H) > 96 * 1024) tt >>= 1;
  *tok_tile = tt;
  *e_per_warp = T <= 64 ? 1 : std::max(1, std::min(4, (E + kRouterWarps - 1) / kRouterWarps));
}

cudaError_t prepare_router() {
  return cudaFuncSetAttribute(router_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
}

cudaError_t launch_router(const RouterParams& p, cudaStream_t s) {
  const int rows_per_cta = kRouterWarps * p.e_per_warp;
  const dim3 grid((p.E + rows_per_cta - 1) / rows_per_cta, (p.T + p.tok_tile - 1) / p.tok_tile);
  return launch_k(router_logits_kernel, grid, dim3(kRouterWarps * 32), router_smem_bytes(p.tok_tile, p.H), s,
                  p.pdl, p);
}

}  // namespace ft
