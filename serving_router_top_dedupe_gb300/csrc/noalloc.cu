// Allocation-free evaluation of one fully resident MoE layer.
//
// Some callers cannot call cudaMalloc: an engine that reserved all device memory at
// start-up for its own pool (for example a KV-cache allocator that was handed the rest
// of HBM) and forbids further allocation, or a plug-in host that only allows memory
// it hands out.  This entry point lets such a caller run the routed-expert layer with
// no allocation at all: the caller passes inputs and outputs, and every intermediate
// (routing lists, cache bookkeeping, SwiGLU intermediates, pair rows, combine counters)
// lives in one file-scope device array of fixed size, kFtScratchBytes.  That array is
// held by every GPU that loads the library until the process exits.
//
// The layer uses the same kernels as ft_moe_decode_step, run with a bookkeeping table
// that marks every expert resident, so every routed pair is evaluated on the GPU and
// the output is what ft_moe_decode_step returns for a cache that holds the whole layer.
#include <mutex>

#include "ft_internal.cuh"

namespace {

constexpr size_t kFtScratchBytes = (size_t)8 << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

// The scratch.  In host code `ft_noalloc_scratch` is only a host-side stand-in for the
// symbol: its device address must be looked up with cudaGetSymbolAddress per device.
static __device__ __align__(256) unsigned char ft_noalloc_scratch[kFtScratchBytes];

struct DevSetup {
  bool done = false;
  unsigned char* scratch = nullptr;  // device address of ft_noalloc_scratch on this device
  int n_sm = 0;
  int prepared_wtype[2] = {0, 0};
  int prepared_h[2] = {0, 0}, prepared_i[2] = {0, 0};
};
DevSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

// Resets the per-call bookkeeping: every expert resident in its own slot, clock 0,
// combine counters 0.
__global__ void noalloc_reset(int32_t* res, int32_t* owner, uint32_t* stamp, ft::DevState* st,
                              uint32_t* blk_count, int E, int n_blk) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < E; i += gridDim.x * blockDim.x) {
    res[i] = i;
    owner[i] = i;
    stamp[i] = 0u;
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_blk; i += gridDim.x * blockDim.x) blk_count[i] = 0u;
  if (blockIdx.x == 0 && threadIdx.x == 0) *st = ft::DevState{};
}

// Copies this call's device error word (cleared by noalloc_reset at the start of the call)
// to the caller's word.
__global__ void noalloc_export_error(const ft::DevState* st, uint32_t* out) {
  if (threadIdx.x == 0) *out = *reinterpret_cast<const volatile uint32_t*>(&st->error_word);
}

// Bump allocator over the scratch array (offsets only; nothing is allocated).
struct Carve {
  unsigned char* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t n) {
    off = (off + 255) & ~(size_t)255;
    T* p = reinterpret_cast<T*>(base + off);
    off += n * sizeof(T);
    return p;
  }
};

}  // namespace

extern "C" ft_status ft_moe_decode_resident_noalloc(int n_experts, int top_k, int hidden, int inter, int wtype,
                                                    const void* experts_dev, const void* shared_dev, int batch,
                                                    const void* x_bf16, const float* logits, float* out,
                                                    float* rows_out, uint32_t* error_word_out, void* stream) {
  if (n_experts < 1 || n_experts > ft::kMaxE || top_k < 1 || top_k > ft::kMaxK || top_k > n_experts)
    return FT_ERR_INVALID;
  if (wtype != FT_W_BF16 && wtype != FT_W_FP8_E4M3_B128) return FT_ERR_INVALID;
  const int hmul = wtype == FT_W_BF16 ? 256 : 512;
  if (hidden < hmul || hidden % hmul || inter < 128 || inter % 128) return FT_ERR_INVALID;
  if (batch < 1 || batch > ft::kMaxBatch) return FT_ERR_INVALID;
  if (!experts_dev || !x_bf16 || !logits || !out) return FT_ERR_INVALID;
  const int E = n_experts, k = top_k, B = batch, H = hidden, I = inter;
  const int kcap = B * k < E ? B * k : E;
  const int has_shared = shared_dev != nullptr;
  const size_t npair = (size_t)B * k, ngp = npair + B;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FT_ERR_CUDA;
  DevSetup* su = &g_setup[dev];
  {
    // First call on this device (with it current): look up the scratch address.
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!su->done) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, ft_noalloc_scratch) != cudaSuccess || !p) return FT_ERR_CUDA;
      if (cudaDeviceGetAttribute(&su->n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FT_ERR_CUDA;
      su->scratch = static_cast<unsigned char*>(p);
      if (ft::prepare_control() != cudaSuccess) return FT_ERR_CUDA;
      su->done = true;
    }
    const int wi = wtype == FT_W_BF16 ? 0 : 1;
    if (su->prepared_h[wi] < H || su->prepared_i[wi] < I) {
      const int ph = su->prepared_h[wi] > H ? su->prepared_h[wi] : H;
      const int pi = su->prepared_i[wi] > I ? su->prepared_i[wi] : I;
      if (ft::prepare_kernels(wtype, ph, pi) != cudaSuccess) return FT_ERR_CUDA;
      su->prepared_h[wi] = ph;
      su->prepared_i[wi] = pi;
    }
  }

  // Lay out every intermediate inside the scratch array; refuse sizes beyond it.
  Carve cv{su->scratch};
  int32_t* res = cv.take<int32_t>(E);
  int32_t* owner = cv.take<int32_t>(E);
  uint32_t* stamp = cv.take<uint32_t>(E);
  ft::DevState* st = cv.take<ft::DevState>(1);
  ft::DecodeWork w{};
  w.sel = cv.take<int32_t>(npair);
  w.gates = cv.take<float>(npair);
  w.slot_of_pair = cv.take<int32_t>(npair);
  w.active = cv.take<int32_t>(kcap);
  w.hit = cv.take<int32_t>(kcap);
  w.miss = cv.take<int32_t>(kcap);
  w.victims = cv.take<int32_t>(kcap);
  w.copy_u = cv.take<int32_t>(kcap);
  w.copy_slot = cv.take<int32_t>(kcap);
  w.counts = cv.take<int32_t>(ft::C_NCOUNTS);
  w.g_w = cv.take<const uint8_t*>((size_t)kcap + 1);
  w.g_fill = cv.take<int32_t>((size_t)kcap + 1);
  w.g_off = cv.take<int32_t>((size_t)kcap + 2);
  w.g_pair = cv.take<int32_t>(ngp);
  w.h = cv.take<float>(ngp * I);
  w.ready = cv.take<uint32_t>((size_t)kcap + 1);
  w.rows = cv.take<float>(npair * H);
  w.shared_rows = cv.take<float>((size_t)B * H);
  w.blk_count = cv.take<uint32_t>((size_t)H / ft::kRowsPerItem2);
  w.kmax = kcap;
  if (cv.off > kFtScratchBytes) return FT_ERR_CAPACITY;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const ft::SlotLayout lay = ft::make_layout(wtype, H, I);
  noalloc_reset<<<4, 256, 0, s>>>(res, owner, stamp, st, w.blk_count, E, H / ft::kRowsPerItem2);
  if (cudaGetLastError() != cudaSuccess) return FT_ERR_CUDA;

  ft::CtrlParams cp{};
  cp.logits = logits;
  cp.B = B;
  cp.E = E;
  cp.k = k;
  cp.layer = 0;
  cp.S = E;
  cp.kcap = kcap;
  cp.has_shared = has_shared;
  cp.bp_mbs = 1;  // every expert is resident: there are never misses to split
  cp.bh_mbs = 1;
  cp.res = res;
  cp.owner = owner;
  cp.stamp = stamp;
  cp.st = st;
  cp.w = w;
  cp.pool = static_cast<const uint8_t*>(experts_dev);
  cp.slot_stride = lay.stride;
  cp.shared_w = static_cast<const uint8_t*>(shared_dev);
  // Plain stream order, no programmatic dependent launch: the control kernel's prologue
  // reads the table that noalloc_reset writes, and at batch 1 the evaluation kernel's
  // prologue reads the lists the control kernel writes (in ft_moe_decode_step a fill
  // kernel sits between the two; here nothing does).
  cp.pdl = false;
  if (ft::launch_control(cp, s) != cudaSuccess) return FT_ERR_CUDA;

  ft::EvalParams ep{};
  ep.counts = w.counts;
  ep.g_w = w.g_w;
  ep.g_fill = w.g_fill;
  ep.g_off = w.g_off;
  ep.g_pair = w.g_pair;
  ep.gates = w.gates;
  ep.slot_of_pair = w.slot_of_pair;
  ep.x = static_cast<const uint16_t*>(x_bf16);
  ep.h = w.h;
  ep.ready = w.ready;
  ep.rows = rows_out ? rows_out : w.rows;
  ep.shared_rows = w.shared_rows;
  ep.c_partial = nullptr;
  ep.out = out;
  ep.blk_count = w.blk_count;
  ep.error_word = &st->error_word;
  ep.lay = lay;
  ep.H = H;
  ep.I = I;
  ep.k = k;
  ep.B = B;
  ep.has_shared = has_shared;
  ep.n_sm = su->n_sm;
  ep.max_entries = kcap + 1;
  ep.pdl = false;
  ep.allow_fused = true;
  ep.wait_extra = 0;
  ep.wait_ns = ft::kHandoffWaitNs;
  if (ft::launch_gate_up(ep, wtype, su->n_sm * 4, s) != cudaSuccess) return FT_ERR_CUDA;
  if (ft::launch_down_combine(ep, wtype, su->n_sm * 4, s) != cudaSuccess) return FT_ERR_CUDA;
  if (error_word_out) {
    noalloc_export_error<<<1, 32, 0, s>>>(st, error_word_out);
    if (cudaGetLastError() != cudaSuccess) return FT_ERR_CUDA;
  }
  return FT_OK;
}
