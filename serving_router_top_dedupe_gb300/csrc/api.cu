// Host runtime of libftmoe: the C ABI declared in include/ft_moe.h.
//
// Owns the HBM slot pool, the residency state, the fixed-shape work lists, the
// compute and transfer streams, cached CUDA graphs and the host-pool registrations.
// Every routing-dependent decision runs in kernels (control.cu); this file only
// validates arguments, enqueues work and moves bytes.
#include <cuda.h>
#include <cuda_runtime.h>
#include <sys/mman.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <memory>
#include <string>
#include <tuple>
#include <vector>

#include "ft_internal.cuh"
#include "ft_prefill.cuh"

namespace {

thread_local std::string g_last_error;

ft_status fail(ft_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

// Memory of ft_host_alloc: the registered address -> its mapping (base NULL: cudaHostAlloc).
struct HostMap {
  void* base;
  size_t len;
};
std::mutex g_host_mu;
std::map<void*, HostMap> g_host_maps;

// Transparent huge page size of this host (the PMD size: 2 MB with 4 KB base pages, 512 MB
// with 64 KB ones); 2 MB when the kernel does not say.
size_t huge_page_bytes() {
  size_t v = 0;
  if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
    unsigned long long x = 0;
    if (std::fscanf(f, "%llu", &x) == 1) v = (size_t)x;
    std::fclose(f);
  }
  return v >= 4096 && (v & (v - 1)) == 0 ? v : ((size_t)2 << 20);
}

// Test hook for the failure paths (ft_test_inject_failure): the armed kind's nth request
// from the moment of arming fails as if the CUDA runtime had refused it, once.
std::mutex g_inject_mu;
int g_inject_kind = 0, g_inject_left = 0;

bool injected_failure(int kind) {
  std::lock_guard<std::mutex> lock(g_inject_mu);
  if (g_inject_kind != kind || g_inject_left <= 0) return false;
  if (--g_inject_left > 0) return false;
  g_inject_kind = 0;
  return true;
}

cudaError_t dev_malloc(void** p, size_t bytes) {
  if (injected_failure(FT_INJECT_MALLOC)) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(p, bytes);
}

#define FT_CUDA(call)                                                                        \
  do {                                                                                       \
    cudaError_t e_ = (call);                                                                 \
    if (e_ != cudaSuccess)                                                                   \
      return fail(e_ == cudaErrorMemoryAllocation ? FT_ERR_NOMEM : FT_ERR_CUDA, "%s: %s (%s:%d)", \
                  #call, cudaGetErrorString(e_), __FILE__, __LINE__);                        \
  } while (0)

long long to_mbps(double gbps) { return (long long)std::floor(gbps * 1000.0 + 0.5); }

struct HostBank {
  const uint8_t* host = nullptr;  // caller's pointer
  const uint8_t* dev = nullptr;   // device-visible alias
  size_t row = 0;                 // bytes per logical id
  size_t bytes = 0;
  bool registered = false;        // registered by us (unregister at destroy)
};

struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};

}  // namespace

struct ft_graph {
  ft_moe* owner = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  std::vector<ProfRec> prof;  // timing events captured as graph nodes (profiling on at capture)
  uint64_t pending = 0;       // replays since the profile was last read
};

struct ft_moe {
  ft_moe_config cfg{};
  int dev = 0, n_sm = 0;
  cudaStream_t cs = nullptr, ts = nullptr;
  bool own_cs = false, own_ts = false;
  bool pf_overlap = true;  // prefill double buffer on
  // router (hidden-state entry points): device weights [L][E][H], logits buffer
  int gate = FT_GATE_SOFTMAX_TOPK;
  uint16_t* router_w = nullptr;
  float* router_z = nullptr;  // [max(max_batch, max_prefill_tokens)][E]
  // in-step host hook for the C set: pinned staging of routing and rows, device rows
  ft_host_hook hook = nullptr;
  void* hook_user = nullptr;
  int32_t *hk_sel = nullptr, *hk_slot = nullptr;
  float *hk_gates = nullptr, *hk_rows = nullptr, *hk_rows_dev = nullptr;
  std::vector<std::pair<ft_moe*, std::pair<int, int>>> hook_ctx;  // (handle, (layer, batch)), stable
  ft::SlotLayout lay{};
  int S = 0, L = 0, E = 0, K = 0, H = 0, I = 0, kcap = 0;
  bool logits_early_next = false;  // the next control kernel may read its logits before its wait
  long long bp_mbs = 0, bh_mbs = 0;
  double bp_gbps = 0, bh_gbps = 0;
  HostBank bank[7];
  int n_banks = 3;
  uint8_t* pool = nullptr;
  uint8_t* shared_w = nullptr;
  int32_t* res = nullptr;
  int32_t* owner = nullptr;
  uint32_t* stamp = nullptr;
  ft::DevState* st = nullptr;
  ft::DecodeWork w{};
  std::vector<void*> allocs;  // work-list allocations
  int32_t* counts_host = nullptr;  // pinned mirror (memcpy fill mode)
  int32_t* copy_host = nullptr;    // pinned [2*kcap]
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_ctrl = nullptr;
  int grid_eval = 0, grid_fill = 0;
  bool fused_ok = true;              // the batch-1 persistent GEMV's grid fits (checked at init)
  uint64_t test_handoff_ns = 0;      // test control: unreachable hand-off target, wait limit (ns)
  // host-buffer staging (lazy)
  uint16_t* stg_x = nullptr;
  float *stg_logits = nullptr, *stg_cp = nullptr, *stg_out = nullptr;
  std::map<std::tuple<int, int, int>, ft_graph*> host_graphs;
  // profiling
  bool prof = false;
  std::vector<ProfRec> prof_live;
  std::vector<cudaEvent_t> ev_free;
  ft_profile prof_acc{};
  // prefill (lazy)
  ft::PrefillState* pf = nullptr;
  std::vector<ft_graph*> graphs;
};

namespace ft {

SlotLayout make_layout(int wtype, int H, int I) {
  SlotLayout l{};
  // weight bytes per element times 2: BF16 4, FP8 2, FP4 1
  const size_t e2 = wtype == FT_W_BF16 ? 4 : (wtype == FT_W_FP8_E4M3_B128 ? 2 : 1);  // FP4 formats: 1
  l.gate_b = (size_t)I * H * e2 / 2;
  l.down_b = (size_t)H * I * e2 / 2;
  l.gate = 0;
  l.up = l.gate_b;
  l.down = 2 * l.gate_b;
  size_t end = l.down + l.down_b;
  if (wtype == FT_W_FP8_E4M3_B128) {
    l.gs_b = (size_t)I * (H / 128) * 4;
    l.ds_b = (size_t)H * (I / 128) * 4;
  } else if (wtype == FT_W_NVFP4) {
    l.gs_b = (size_t)I * (H / 16);
    l.ds_b = (size_t)H * (I / 16);
  } else if (wtype == FT_W_MXFP4) {
    l.gs_b = (size_t)I * (H / 32);
    l.ds_b = (size_t)H * (I / 32);
  }
  l.gs = end;
  l.us = l.gs + l.gs_b;
  l.ds = l.us + l.gs_b;
  end = l.ds + l.ds_b;
  l.ts = end;
  if (wtype == FT_W_NVFP4) {
    l.ts_b = 16;
    end += l.ts_b;
  }
  l.used = end;
  l.stride = (end + 255) / 256 * 256;
  return l;
}

}  // namespace ft

namespace {

bool capturing(cudaStream_t s);

// Inside a capture an event becomes an event-record graph node only when recorded as
// external; otherwise it is a capture-internal dependency with no timestamp.
cudaError_t record_timing_event(cudaEvent_t e, cudaStream_t s) {
  return capturing(s) ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal) : cudaEventRecord(e, s);
}

ft_status prof_begin(ft_moe* h, cudaStream_t s, cudaEvent_t* out) {
  *out = nullptr;
  if (!h->prof) return FT_OK;
  cudaEvent_t e;
  if (!h->ev_free.empty()) {
    e = h->ev_free.back();
    h->ev_free.pop_back();
  } else {
    FT_CUDA(cudaEventCreate(&e));
  }
  FT_CUDA(record_timing_event(e, s));
  *out = e;
  return FT_OK;
}

ft_status prof_end(ft_moe* h, int kind, cudaStream_t s, cudaEvent_t a) {
  if (!h->prof || !a) return FT_OK;
  cudaEvent_t e;
  if (!h->ev_free.empty()) {
    e = h->ev_free.back();
    h->ev_free.pop_back();
  } else {
    FT_CUDA(cudaEventCreate(&e));
  }
  FT_CUDA(record_timing_event(e, s));
  h->prof_live.push_back({kind, a, e});
  return FT_OK;
}

bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &st);
  return st != cudaStreamCaptureStatusNone;
}

ft_status alloc_dev(ft_moe* h, void** p, size_t bytes) {
  cudaError_t e = dev_malloc(p, bytes < 16 ? 16 : bytes);
  if (e != cudaSuccess) return fail(FT_ERR_NOMEM, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
  h->allocs.push_back(*p);
  return FT_OK;
}

ft_status register_bank(HostBank& b, const void* p, size_t row, size_t n_rows) {
  b.host = static_cast<const uint8_t*>(p);
  b.row = row;
  b.bytes = row * n_rows;
  if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return fail(FT_ERR_INVALID, "host bank not 16-byte aligned");
  cudaPointerAttributes at{};
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  bool pinned = e == cudaSuccess && at.type == cudaMemoryTypeHost;
  cudaGetLastError();
  if (!pinned) {
    e = injected_failure(FT_INJECT_REGISTER)
            ? cudaErrorMemoryAllocation
            : cudaHostRegister(const_cast<void*>(p), b.bytes, cudaHostRegisterMapped | cudaHostRegisterPortable);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(FT_ERR_PIN, "cudaHostRegister(%zu bytes) failed: %s (no fallback path)", b.bytes,
                  cudaGetErrorString(e));
    }
    b.registered = true;
  }
  void* d = nullptr;
  e = cudaHostGetDevicePointer(&d, const_cast<void*>(p), 0);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(FT_ERR_PIN, "host bank is pinned but not mapped: %s", cudaGetErrorString(e));
  }
  b.dev = static_cast<const uint8_t*>(d);
  return FT_OK;
}

ft_status check_cfg(const ft_moe_config* c) {
  if (!c) return fail(FT_ERR_INVALID, "null config");
  if (c->n_layers < 1 || c->n_experts < 1 || c->n_experts > ft::kMaxE)
    return fail(FT_ERR_INVALID, "n_layers >= 1 and 1 <= n_experts <= %d required", ft::kMaxE);
  if (c->top_k < 1 || c->top_k > ft::kMaxK || c->top_k > c->n_experts)
    return fail(FT_ERR_INVALID, "1 <= top_k <= min(%d, n_experts) required", ft::kMaxK);
  if (c->wtype != FT_W_BF16 && c->wtype != FT_W_FP8_E4M3_B128 && c->wtype != FT_W_NVFP4 &&
      c->wtype != FT_W_MXFP4)
    return fail(FT_ERR_INVALID, "unknown wtype");
  const int hmul = c->wtype == FT_W_FP8_E4M3_B128 ? 512 : 256;
  if (c->hidden < hmul || c->hidden % hmul) return fail(FT_ERR_INVALID, "hidden must be a multiple of %d", hmul);
  if (c->inter < 128 || c->inter % 128) return fail(FT_ERR_INVALID, "inter must be a multiple of 128");
  if (c->max_batch < 1 || c->max_batch > ft::kMaxBatch)
    return fail(FT_ERR_INVALID, "1 <= max_batch <= %d required", ft::kMaxBatch);
  if (c->cache_slots < 1 || c->cache_slots > (1 << 20))
    return fail(FT_ERR_INVALID, "1 <= cache_slots <= 2^20 required");
  if (c->bh_gbps <= 0) return fail(FT_ERR_INVALID, "bh_gbps must be > 0");
  if (c->fill_mode != FT_FILL_KERNEL && c->fill_mode != FT_FILL_MEMCPY) return fail(FT_ERR_INVALID, "fill_mode");
  if (c->max_prefill_tokens < 0) return fail(FT_ERR_INVALID, "max_prefill_tokens < 0");
  if ((long long)c->n_layers * c->n_experts > (1LL << 30)) return fail(FT_ERR_INVALID, "too many experts");
  return FT_OK;
}

ft_status alloc_work(ft_moe* h) {
  const int B = h->cfg.max_batch, k = h->K, kc = h->kcap;
  const size_t npair = (size_t)B * k, nent = (size_t)kc + 1, ngp = npair + B;
  ft::DecodeWork& w = h->w;
  ft_status s;
#define A(ptr, n)                                                     \
  if ((s = alloc_dev(h, (void**)&(ptr), (n) * sizeof(*(ptr)))) != FT_OK) return s;
  A(w.sel, npair);
  A(w.gates, npair);
  A(w.slot_of_pair, npair);
  A(w.active, (size_t)kc);
  A(w.hit, (size_t)kc);
  A(w.miss, (size_t)kc);
  A(w.victims, (size_t)kc);
  A(w.copy_u, (size_t)kc);
  A(w.copy_slot, (size_t)kc);
  A(w.counts, (size_t)ft::C_NCOUNTS);
  A(w.g_w, nent);
  A(w.g_fill, nent);
  A(w.g_off, nent + 1);
  A(w.g_pair, ngp);
  A(w.h, ngp * h->I);
  A(w.ready, nent);
  A(w.rows, npair * h->H);
  A(w.shared_rows, (size_t)B * h->H);
  A(w.blk_count, (size_t)h->H / ft::kRowsPerItem2);
  A(w.ecopy, (size_t)2 * (2 + 2 * kc));
#undef A
  w.kmax = kc;
  FT_CUDA(cudaMemset(w.blk_count, 0, sizeof(uint32_t) * (h->H / ft::kRowsPerItem2)));
  FT_CUDA(cudaMemset(w.counts, 0, sizeof(int32_t) * ft::C_NCOUNTS));
  FT_CUDA(cudaMemset(w.ecopy, 0, sizeof(int32_t) * 2 * (2 + 2 * kc)));  // clock 0: no step
  return FT_OK;
}

// Enqueue one decode layer-step (control -> fill -> gate/up -> down+combine).
void CUDART_CB host_hook_call(void* arg) {
  auto* c = static_cast<std::pair<ft_moe*, std::pair<int, int>>*>(arg);
  ft_moe* h = c->first;
  if (h->hook) h->hook(h->hook_user, c->second.first, c->second.second, h->hk_sel, h->hk_gates, h->hk_slot, h->hk_rows);
}

ft_status enqueue_layer(ft_moe* h, int layer, int batch, const void* x, const float* logits,
                        const float* cpart, float* out, float* rows_out) {
  cudaStream_t cs = h->cs, ts = h->ts;
  ft::CtrlParams cp{};
  cp.logits = logits;
  cp.B = batch;
  cp.E = h->E;
  cp.k = h->K;
  cp.layer = layer;
  cp.S = h->S;
  cp.kcap = std::min(batch * h->K, h->E);
  cp.has_shared = h->cfg.has_shared;
  cp.gate = h->gate;
  cp.bp_mbs = h->bp_mbs;
  cp.bh_mbs = h->bh_mbs;
  cp.res = h->res;
  cp.owner = h->owner;
  cp.stamp = h->stamp;
  cp.st = h->st;
  cp.w = h->w;
  cp.pool = h->pool;
  cp.slot_stride = h->lay.stride;
  cp.shared_w = h->cfg.has_shared ? h->shared_w + (size_t)layer * h->lay.stride : nullptr;
  // In kernel-fill mode the whole layer is one chain of programmatic dependents on the
  // compute stream; the memcpy mode hands the fill to the transfer stream and back.
  const bool chain = h->cfg.fill_mode == FT_FILL_KERNEL;
  cp.pdl = chain;
  cp.logits_early = h->logits_early_next;
  h->logits_early_next = false;
  cudaEvent_t pa;
  ft_status s;
  if ((s = prof_begin(h, cs, &pa)) != FT_OK) return s;
  FT_CUDA(ft::launch_control(cp, cs));
  if ((s = prof_end(h, 0, cs, pa)) != FT_OK) return s;

  // in-step host branch for the C set: routing out, hook, rows back (stream order)
  const bool hooked = h->hook != nullptr;
  if (hooked) {
    const size_t np = (size_t)batch * h->K;
    FT_CUDA(cudaMemcpyAsync(h->hk_sel, h->w.sel, np * sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
    FT_CUDA(cudaMemcpyAsync(h->hk_gates, h->w.gates, np * sizeof(float), cudaMemcpyDeviceToHost, cs));
    FT_CUDA(cudaMemcpyAsync(h->hk_slot, h->w.slot_of_pair, np * sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
    FT_CUDA(cudaLaunchHostFunc(cs, host_hook_call, &h->hook_ctx[(size_t)layer * (h->cfg.max_batch + 1) + batch]));
    FT_CUDA(cudaMemcpyAsync(h->hk_rows_dev, h->hk_rows, np * h->H * sizeof(float), cudaMemcpyHostToDevice, cs));
    cpart = h->hk_rows_dev;
  }

  if (chain) {
    // fill kernel right after the control kernel on the compute stream
    ft::FillParams fp{};
    fp.counts = h->w.counts;
    fp.copy_u = h->w.copy_u;
    fp.copy_slot = h->w.copy_slot;
    fp.pool = h->pool;
    fp.lay = h->lay;
    fp.n_banks = h->n_banks;
    fp.pdl = !hooked;  // after the host branch's copies the fill follows a plain dependency
    fp.ecopy = h->w.ecopy;
    fp.st = h->st;
    fp.kmax = h->kcap;
    for (int j = 0; j < h->n_banks; ++j) {
      fp.src[j] = h->bank[j].dev;
      fp.src_row[j] = h->bank[j].row;
    }
    if ((s = prof_begin(h, cs, &pa)) != FT_OK) return s;
    FT_CUDA(ft::launch_fill(fp, h->grid_fill, cs));
    if ((s = prof_end(h, 1, cs, pa)) != FT_OK) return s;
  } else {
    // host-driven cudaMemcpyAsync fills on the transfer stream: read the copy list, then
    // one copy per bank per filled expert
    FT_CUDA(cudaEventRecord(h->ev_fork, cs));
    FT_CUDA(cudaStreamWaitEvent(ts, h->ev_fork, 0));
    FT_CUDA(cudaMemcpyAsync(h->counts_host, h->w.counts, sizeof(int32_t) * ft::C_NCOUNTS,
                            cudaMemcpyDeviceToHost, ts));
    FT_CUDA(cudaMemcpyAsync(h->copy_host, h->w.copy_u, sizeof(int32_t) * h->kcap, cudaMemcpyDeviceToHost, ts));
    FT_CUDA(cudaMemcpyAsync(h->copy_host + h->kcap, h->w.copy_slot, sizeof(int32_t) * h->kcap,
                            cudaMemcpyDeviceToHost, ts));
    FT_CUDA(cudaStreamSynchronize(ts));
    const int q = h->counts_host[ft::C_Q];
    const size_t seg[7] = {h->lay.gate, h->lay.up, h->lay.down, h->lay.gs, h->lay.us, h->lay.ds, h->lay.ts};
    if ((s = prof_begin(h, ts, &pa)) != FT_OK) return s;
    for (int i = 0; i < q; ++i) {
      const int u = h->copy_host[i], slot = h->copy_host[h->kcap + i];
      uint8_t* dst = h->pool + (size_t)slot * h->lay.stride;
      for (int j = 0; j < h->n_banks; ++j)
        FT_CUDA(cudaMemcpyAsync(dst + seg[j], h->bank[j].host + (size_t)u * h->bank[j].row, h->bank[j].row,
                                cudaMemcpyHostToDevice, ts));
    }
    if ((s = prof_end(h, 1, ts, pa)) != FT_OK) return s;
    FT_CUDA(cudaEventRecord(h->ev_join, ts));
    FT_CUDA(cudaStreamWaitEvent(cs, h->ev_join, 0));
  }

  ft::EvalParams ep{};
  ep.counts = h->w.counts;
  ep.g_w = h->w.g_w;
  ep.g_fill = h->w.g_fill;
  ep.g_off = h->w.g_off;
  ep.g_pair = h->w.g_pair;
  ep.gates = h->w.gates;
  ep.slot_of_pair = h->w.slot_of_pair;
  ep.x = static_cast<const uint16_t*>(x);
  ep.h = h->w.h;
  ep.ready = h->w.ready;
  ep.rows = rows_out ? rows_out : h->w.rows;
  ep.shared_rows = h->w.shared_rows;
  ep.c_partial = cpart;
  ep.out = out;
  ep.blk_count = h->w.blk_count;
  ep.error_word = &h->st->error_word;
  ep.lay = h->lay;
  ep.H = h->H;
  ep.I = h->I;
  ep.k = h->K;
  ep.B = batch;
  ep.has_shared = h->cfg.has_shared;
  ep.n_sm = chain ? h->n_sm - h->grid_fill : h->n_sm;  // the fill kernel's SMs are left to it
  ep.max_entries = h->kcap + 1;
  ep.pdl = chain;
  ep.allow_fused = h->fused_ok;
  ep.wait_extra = h->test_handoff_ns ? 1u : 0u;
  ep.wait_ns = h->test_handoff_ns ? h->test_handoff_ns : ft::kHandoffWaitNs;
  if ((s = prof_begin(h, cs, &pa)) != FT_OK) return s;
  FT_CUDA(ft::launch_gate_up(ep, h->cfg.wtype, h->grid_eval, cs));
  if ((s = prof_end(h, 2, cs, pa)) != FT_OK) return s;
  if (!ft::eval_fused(ep, h->cfg.wtype)) {
    if ((s = prof_begin(h, cs, &pa)) != FT_OK) return s;
    FT_CUDA(ft::launch_down_combine(ep, h->cfg.wtype, h->grid_eval, cs));
    if ((s = prof_end(h, 3, cs, pa)) != FT_OK) return s;
  }
  return FT_OK;
}

// Router kernel for n tokens of `layer` into z, on the compute stream.
ft_status enqueue_router(ft_moe* h, int layer, int n, const void* x, float* z, bool pdl) {
  ft::RouterParams rp{};
  rp.x = static_cast<const uint16_t*>(x);
  rp.w = h->router_w + (size_t)layer * h->E * h->H;
  rp.z = z;
  rp.T = n;
  rp.E = h->E;
  rp.H = h->H;
  ft::router_shape(n, h->E, h->H, &rp.tok_tile, &rp.e_per_warp);
  rp.pdl = pdl;
  cudaEvent_t pa;
  ft_status s;
  if ((s = prof_begin(h, h->cs, &pa)) != FT_OK) return s;
  FT_CUDA(ft::launch_router(rp, h->cs));
  return prof_end(h, 9, h->cs, pa);
}

ft_status check_router(ft_moe* h, int layer, int n, const void* x) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  if (!h->router_w) return fail(FT_ERR_STATE, "no router weights: call ft_moe_set_router first");
  if (layer < 0 || layer >= h->L) return fail(FT_ERR_INVALID, "layer %d out of range", layer);
  const int nmax = std::max(h->cfg.max_batch, h->cfg.max_prefill_tokens);
  if (n < 1 || n > nmax) return fail(FT_ERR_INVALID, "n_tokens %d outside [1, %d]", n, nmax);
  if (!x) return fail(FT_ERR_INVALID, "null x");
  if (reinterpret_cast<uintptr_t>(x) % 16) return fail(FT_ERR_INVALID, "x must be 16-byte aligned");
  return FT_OK;
}

ft_status check_step(ft_moe* h, int layer, int batch, const void* x, const float* logits, const float* cpart,
                     const float* out) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  if (layer < 0 || layer >= h->L) return fail(FT_ERR_INVALID, "layer %d out of range", layer);
  if (batch < 1 || batch > h->cfg.max_batch) return fail(FT_ERR_INVALID, "batch %d out of range", batch);
  if (!x || !logits || !out) return fail(FT_ERR_INVALID, "null x/logits/out");
  if (!cpart && !h->hook && h->bh_mbs > h->bp_mbs)
    return fail(FT_ERR_INVALID, "c_partial may be NULL only when B_H <= B_P (every miss filled)");
  if (h->pf) ft::prefill_interrupt(h->pf);
  return FT_OK;
}

}  // namespace

// ============================================================ ABI entry points
extern "C" {

ft_status ft_test_inject_failure(int kind, int nth) {
  if ((kind != FT_INJECT_MALLOC && kind != FT_INJECT_REGISTER) || nth < 0)
    return fail(FT_ERR_INVALID, "ft_test_inject_failure: unknown kind or negative count");
  std::lock_guard<std::mutex> lock(g_inject_mu);
  g_inject_kind = nth > 0 ? kind : 0;
  g_inject_left = nth;
  return FT_OK;
}

ft_status ft_host_alloc(size_t bytes, int flags, void** out) {
  if (!out || bytes == 0) return fail(FT_ERR_INVALID, "ft_host_alloc: null out or zero size");
  if (flags != FT_HOST_HUGE_PAGES && flags != FT_HOST_PINNED) return fail(FT_ERR_INVALID, "ft_host_alloc: flags");
  *out = nullptr;
  if (flags == FT_HOST_PINNED) {
    cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
      *out = nullptr;
      cudaGetLastError();
      return fail(FT_ERR_PIN, "cudaHostAlloc(%zu bytes) failed: %s", bytes, cudaGetErrorString(e));
    }
    std::lock_guard<std::mutex> lock(g_host_mu);
    g_host_maps[*out] = HostMap{nullptr, 0};
    return FT_OK;
  }
  const size_t huge = huge_page_bytes();
  const size_t span = (bytes + huge - 1) / huge * huge, len = span + huge;
  void* raw = mmap(nullptr, len, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (raw == MAP_FAILED) return fail(FT_ERR_NOMEM, "ft_host_alloc: mmap of %zu bytes failed", len);
  uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + huge - 1) / huge * huge);
  madvise(p, span, MADV_HUGEPAGE);  // no transparent huge pages: base pages, still correct
  cudaError_t e = cudaHostRegister(p, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable);
  if (e != cudaSuccess) {
    cudaGetLastError();
    munmap(raw, len);
    return fail(FT_ERR_PIN, "cudaHostRegister(%zu bytes) failed: %s", bytes, cudaGetErrorString(e));
  }
  std::lock_guard<std::mutex> lock(g_host_mu);
  g_host_maps[p] = HostMap{raw, len};
  *out = p;
  return FT_OK;
}

ft_status ft_host_free(void* p) {
  if (!p) return FT_OK;
  HostMap m{};
  {
    std::lock_guard<std::mutex> lock(g_host_mu);
    auto it = g_host_maps.find(p);
    if (it == g_host_maps.end()) return fail(FT_ERR_INVALID, "ft_host_free: not an ft_host_alloc address");
    m = it->second;
    g_host_maps.erase(it);
  }
  cudaError_t e = m.base ? cudaHostUnregister(p) : cudaFreeHost(p);
  if (m.base) munmap(m.base, m.len);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(FT_ERR_INVALID, "ft_host_free: %s", cudaGetErrorString(e));
  }
  return FT_OK;
}

const char* ft_last_error(void) { return g_last_error.c_str(); }

ft_status ft_split_misses(int m, double bp_gbps, double bh_gbps, int evictable, int* q_out) {
  if (!q_out || m < 0 || evictable < 0 || !(bp_gbps > 0) || !(bh_gbps > 0))
    return fail(FT_ERR_INVALID, "ft_split_misses: bad argument");
  const long long bp = to_mbps(bp_gbps), bh = to_mbps(bh_gbps);
  long long q;
  if (m == 0) {
    q = 0;
  } else if (bh <= bp) {
    q = m;
  } else {
    q = (2LL * m * bp + bh) / (2LL * bh);
    if (q < 1) q = 1;
  }
  q = std::min<long long>({q, (long long)m, (long long)evictable});
  *q_out = (int)q;
  return FT_OK;
}

ft_status ft_bench_bw(size_t bytes, int iters, double* bp_gbps) {
  if (!bp_gbps || bytes < 1024 || iters < 1) return fail(FT_ERR_INVALID, "ft_bench_bw: bad argument");
  void *hbuf = nullptr, *dbuf = nullptr;
  cudaStream_t s = nullptr;
  cudaEvent_t a = nullptr, b = nullptr;
  ft_status st = FT_OK;
  float ms = 0.f;
  if (cudaHostAlloc(&hbuf, bytes, cudaHostAllocDefault) != cudaSuccess) {
    st = fail(FT_ERR_PIN, "cudaHostAlloc(%zu) failed", bytes);
    goto done;
  }
  if (cudaMalloc(&dbuf, bytes) != cudaSuccess) {
    st = fail(FT_ERR_NOMEM, "cudaMalloc(%zu) failed", bytes);
    goto done;
  }
  memset(hbuf, 1, bytes);
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess || cudaEventCreate(&a) != cudaSuccess ||
      cudaEventCreate(&b) != cudaSuccess) {
    st = fail(FT_ERR_CUDA, "stream/event creation failed");
    goto done;
  }
  cudaMemcpyAsync(dbuf, hbuf, bytes, cudaMemcpyHostToDevice, s);  // warm-up
  cudaEventRecord(a, s);
  for (int i = 0; i < iters; ++i) cudaMemcpyAsync(dbuf, hbuf, bytes, cudaMemcpyHostToDevice, s);
  cudaEventRecord(b, s);
  if (cudaEventSynchronize(b) != cudaSuccess || cudaEventElapsedTime(&ms, a, b) != cudaSuccess || ms <= 0.f) {
    st = fail(FT_ERR_CUDA, "timing failed: %s", cudaGetErrorString(cudaGetLastError()));
    goto done;
  }
  *bp_gbps = (double)bytes * iters / (ms * 1e-3) / 1e9;
done:
  if (a) cudaEventDestroy(a);
  if (b) cudaEventDestroy(b);
  if (s) cudaStreamDestroy(s);
  if (dbuf) cudaFree(dbuf);
  if (hbuf) cudaFreeHost(hbuf);
  return st;
}

static ft_status init_body(ft_moe* h, const ft_moe_config* cfg, const ft_banks* host_pool, const ft_banks* shared) {
  const bool fp8 = cfg->wtype == FT_W_FP8_E4M3_B128;
  ft_status s;
  h->cfg = *cfg;
  h->dev = cfg->device;
  FT_CUDA(cudaSetDevice(h->dev));
  FT_CUDA(cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->dev));
  h->L = cfg->n_layers;
  h->E = cfg->n_experts;
  h->K = cfg->top_k;
  h->H = cfg->hidden;
  h->I = cfg->inter;
  h->S = cfg->cache_slots;
  h->kcap = std::min(cfg->max_batch * cfg->top_k, cfg->n_experts);
  h->lay = ft::make_layout(cfg->wtype, h->H, h->I);
  h->n_banks = cfg->wtype == FT_W_NVFP4 ? 7 : (fp8 || cfg->wtype == FT_W_MXFP4 ? 6 : 3);
  h->grid_eval = h->n_sm * 4;
  h->grid_fill = std::max(1, std::min(ft::kFillSms, h->n_sm / 4));
  if (cfg->compute_stream) {
    h->cs = (cudaStream_t)cfg->compute_stream;
  } else {
    FT_CUDA(cudaStreamCreateWithFlags(&h->cs, cudaStreamNonBlocking));
    h->own_cs = true;
  }
  if (cfg->transfer_stream) {
    h->ts = (cudaStream_t)cfg->transfer_stream;
  } else {
    FT_CUDA(cudaStreamCreateWithFlags(&h->ts, cudaStreamNonBlocking));
    h->own_ts = true;
  }
  FT_CUDA(cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming));
  FT_CUDA(cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming));
  FT_CUDA(cudaEventCreateWithFlags(&h->ev_ctrl, cudaEventDisableTiming));

  // bandwidths for the split rule (integer MB/s on the device)
  h->bh_gbps = cfg->bh_gbps;
  h->bp_gbps = cfg->bp_gbps;
  if (!(h->bp_gbps > 0) && (s = ft_bench_bw((size_t)256 << 20, 8, &h->bp_gbps)) != FT_OK) return s;
  h->bp_mbs = to_mbps(h->bp_gbps);
  h->bh_mbs = to_mbps(h->bh_gbps);

  // host pool: pin + map every bank
  const size_t nlog = (size_t)h->L * h->E;
  const bool fp4 = cfg->wtype == FT_W_NVFP4 || cfg->wtype == FT_W_MXFP4;
  const void* bp[7] = {host_pool->gate,
                       host_pool->up,
                       host_pool->down,
                       fp4 ? (const void*)host_pool->gate_bscale : host_pool->gate_scale,
                       fp4 ? (const void*)host_pool->up_bscale : host_pool->up_scale,
                       fp4 ? (const void*)host_pool->down_bscale : host_pool->down_scale,
                       host_pool->tensor_scale};
  const size_t rows[7] = {h->lay.gate_b, h->lay.gate_b, h->lay.down_b, h->lay.gs_b,
                          h->lay.gs_b,   h->lay.ds_b,   h->lay.ts_b};
  for (int j = 0; j < h->n_banks; ++j) {
    if (rows[j] % 16) return fail(FT_ERR_INVALID, "bank row bytes not a multiple of 16");
    if ((s = register_bank(h->bank[j], bp[j], rows[j], nlog)) != FT_OK) return s;
  }

  // HBM: slot pool, shared experts, state, work lists
  {
    cudaError_t e = dev_malloc((void**)&h->pool, (size_t)h->S * h->lay.stride);
    if (e != cudaSuccess)
      return fail(FT_ERR_NOMEM, "slot pool of %d x %zu bytes: %s", h->S, h->lay.stride, cudaGetErrorString(e));
  }
  if (cfg->has_shared) {
    FT_CUDA(dev_malloc((void**)&h->shared_w, (size_t)h->L * h->lay.stride));
    const void* sp[7] = {shared->gate,
                         shared->up,
                         shared->down,
                         fp4 ? (const void*)shared->gate_bscale : shared->gate_scale,
                         fp4 ? (const void*)shared->up_bscale : shared->up_scale,
                         fp4 ? (const void*)shared->down_bscale : shared->down_scale,
                         shared->tensor_scale};
    const size_t seg[7] = {h->lay.gate, h->lay.up, h->lay.down, h->lay.gs, h->lay.us, h->lay.ds, h->lay.ts};
    for (int l = 0; l < h->L; ++l)
      for (int j = 0; j < h->n_banks; ++j)
        FT_CUDA(cudaMemcpy(h->shared_w + (size_t)l * h->lay.stride + seg[j],
                           static_cast<const uint8_t*>(sp[j]) + (size_t)l * rows[j], rows[j], cudaMemcpyHostToDevice));
  }
  if ((s = alloc_dev(h, (void**)&h->res, sizeof(int32_t) * nlog)) != FT_OK) return s;
  if ((s = alloc_dev(h, (void**)&h->owner, sizeof(int32_t) * h->S)) != FT_OK) return s;
  if ((s = alloc_dev(h, (void**)&h->stamp, sizeof(uint32_t) * h->S)) != FT_OK) return s;
  if ((s = alloc_dev(h, (void**)&h->st, sizeof(ft::DevState))) != FT_OK) return s;
  FT_CUDA(cudaMemset(h->res, 0xff, sizeof(int32_t) * nlog));
  FT_CUDA(cudaMemset(h->owner, 0xff, sizeof(int32_t) * h->S));
  FT_CUDA(cudaMemset(h->stamp, 0, sizeof(uint32_t) * h->S));
  FT_CUDA(cudaMemset(h->st, 0, sizeof(ft::DevState)));
  if ((s = alloc_work(h)) != FT_OK) return s;
  FT_CUDA(cudaHostAlloc((void**)&h->counts_host, sizeof(int32_t) * ft::C_NCOUNTS, cudaHostAllocDefault));
  FT_CUDA(cudaHostAlloc((void**)&h->copy_host, sizeof(int32_t) * 2 * h->kcap, cudaHostAllocDefault));
  FT_CUDA(ft::prepare_kernels(h->cfg.wtype, h->H, h->I));
  FT_CUDA(ft::prepare_control());
  FT_CUDA(ft::prepare_router());
  // The batch-1 persistent GEMV hands h rows between its CTAs, so every CTA of its grid must
  // be resident at once: one CTA per SM on the SMs the fill kernel leaves.  When the kernel
  // does not fit on an SM, batch 1 runs the batched kernels instead (ft_stats.batch1_fused).
  h->fused_ok = ft::fused_gemv_fits(h->cfg.wtype, h->H, h->I, h->kcap + 1, h->n_sm - h->grid_fill);
  FT_CUDA(cudaDeviceSynchronize());
  return FT_OK;
}

ft_status ft_moe_init(const ft_moe_config* cfg, const ft_banks* host_pool, const ft_banks* shared, ft_moe** out) {
  ft_status s = check_cfg(cfg);
  if (s != FT_OK) return s;
  if (!out || !host_pool || !host_pool->gate || !host_pool->up || !host_pool->down)
    return fail(FT_ERR_INVALID, "null host pool / out");
  const bool fp8 = cfg->wtype == FT_W_FP8_E4M3_B128, nv4 = cfg->wtype == FT_W_NVFP4, mx4 = cfg->wtype == FT_W_MXFP4;
  auto scales_ok = [&](const ft_banks* b) {
    if (fp8) return b->gate_scale && b->up_scale && b->down_scale;
    if (nv4) return b->gate_bscale && b->up_bscale && b->down_bscale && b->tensor_scale;
    if (mx4) return b->gate_bscale && b->up_bscale && b->down_bscale;
    return true;
  };
  if (!scales_ok(host_pool)) return fail(FT_ERR_INVALID, "FP8 / NVFP4 banks need their scale arrays");
  if (cfg->has_shared && (!shared || !shared->gate || !shared->up || !shared->down || !scales_ok(shared)))
    return fail(FT_ERR_INVALID, "has_shared set but shared banks missing");
  *out = nullptr;
  ft_moe* h = new ft_moe();
  s = init_body(h, cfg, host_pool, shared);
  if (s != FT_OK) {
    std::string keep = g_last_error;
    ft_moe_destroy(h);
    g_last_error = keep;
    return s;
  }
  *out = h;
  return FT_OK;
}

ft_status ft_moe_decode_step(ft_moe* h, int layer, int batch, const void* x_bf16, const float* logits,
                             const float* c_partial, float* out, float* rows_out) {
  ft_status s = check_step(h, layer, batch, x_bf16, logits, c_partial, out);
  if (s != FT_OK) return s;
  if (h->cfg.fill_mode == FT_FILL_MEMCPY && capturing(h->cs))
    return fail(FT_ERR_STATE, "FT_FILL_MEMCPY steps cannot be captured into a graph");
  FT_CUDA(cudaSetDevice(h->dev));
  return enqueue_layer(h, layer, batch, x_bf16, logits, c_partial, out, rows_out);
}

ft_status ft_moe_set_router(ft_moe* h, const void* w_router_bf16, int gate) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  if (gate != FT_GATE_SOFTMAX_TOPK && gate != FT_GATE_SOFTMAX_ALL && gate != FT_GATE_SIGMOID_TOPK)
    return fail(FT_ERR_INVALID, "unknown gate function %d", gate);
  if (capturing(h->cs)) return fail(FT_ERR_STATE, "cannot change the router during capture");
  FT_CUDA(cudaSetDevice(h->dev));
  FT_CUDA(cudaStreamSynchronize(h->cs));
  if (w_router_bf16) {
    const size_t bytes = (size_t)h->L * h->E * h->H * sizeof(uint16_t);
    if (!h->router_w) {
      cudaError_t e = dev_malloc((void**)&h->router_w, bytes);
      if (e != cudaSuccess) {
        h->router_w = nullptr;
        return fail(e == cudaErrorMemoryAllocation ? FT_ERR_NOMEM : FT_ERR_CUDA, "router weights: %s",
                    cudaGetErrorString(e));
      }
      const size_t zb = (size_t)std::max(h->cfg.max_batch, h->cfg.max_prefill_tokens) * h->E * sizeof(float);
      e = dev_malloc((void**)&h->router_z, zb);
      if (e != cudaSuccess) {
        cudaFree(h->router_w);
        h->router_w = nullptr;
        h->router_z = nullptr;
        return fail(e == cudaErrorMemoryAllocation ? FT_ERR_NOMEM : FT_ERR_CUDA, "router logits: %s",
                    cudaGetErrorString(e));
      }
    }
    FT_CUDA(cudaMemcpy(h->router_w, w_router_bf16, bytes, cudaMemcpyHostToDevice));
  }
  h->gate = gate;
  return FT_OK;
}

ft_status ft_moe_router_logits(ft_moe* h, int layer, int n_tokens, const void* x_bf16, float* logits_out) {
  ft_status s = check_router(h, layer, n_tokens, x_bf16);
  if (s != FT_OK) return s;
  if (!logits_out) return fail(FT_ERR_INVALID, "null logits_out");
  FT_CUDA(cudaSetDevice(h->dev));
  return enqueue_router(h, layer, n_tokens, x_bf16, logits_out, false);
}

ft_status ft_moe_decode_step_hidden(ft_moe* h, int layer, int batch, const void* x_bf16, const float* c_partial,
                                    float* out, float* rows_out, float* logits_out) {
  ft_status s = check_router(h, layer, batch, x_bf16);
  if (s != FT_OK) return s;
  float* z = logits_out ? logits_out : h->router_z;
  if ((s = check_step(h, layer, batch, x_bf16, z, c_partial, out)) != FT_OK) return s;
  if (h->cfg.fill_mode == FT_FILL_MEMCPY && capturing(h->cs))
    return fail(FT_ERR_STATE, "FT_FILL_MEMCPY steps cannot be captured into a graph");
  FT_CUDA(cudaSetDevice(h->dev));
  // the router joins the step's chain of programmatic dependents (kernel-fill mode)
  if ((s = enqueue_router(h, layer, batch, x_bf16, z, h->cfg.fill_mode == FT_FILL_KERNEL)) != FT_OK) return s;
  return enqueue_layer(h, layer, batch, x_bf16, z, c_partial, out, rows_out);
}

ft_status ft_moe_decode_layers(ft_moe* h, int first_layer, int n_layers, int batch, const void* x_bf16,
                               const float* logits, const float* c_partial, float* out, float* rows_out) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  if (n_layers < 1 || first_layer < 0 || first_layer + n_layers > h->L)
    return fail(FT_ERR_INVALID, "layer range [%d, %d) out of range", first_layer, first_layer + n_layers);
  const size_t H = h->H, E = h->E, K = h->K;
  for (int i = 0; i < n_layers; ++i) {
    const size_t b = (size_t)i * batch;
    // layers after the first: their logits were written before this call's first kernel
    h->logits_early_next = i > 0;
    ft_status s = ft_moe_decode_step(
        h, first_layer + i, batch, static_cast<const uint16_t*>(x_bf16) + b * H, logits + b * E,
        c_partial ? c_partial + b * K * H : nullptr, out + b * H, rows_out ? rows_out + b * K * H : nullptr);
    h->logits_early_next = false;
    if (s != FT_OK) return s;
  }
  return FT_OK;
}

ft_status ft_moe_graph_capture_decode(ft_moe* h, int first_layer, int n_layers, int batch, const void* x_bf16,
                                      const float* logits, const float* c_partial, float* out, float* rows_out,
                                      ft_graph** g) {
  if (!h || !g) return fail(FT_ERR_INVALID, "null handle/graph");
  if (h->cfg.fill_mode != FT_FILL_KERNEL) return fail(FT_ERR_STATE, "graph capture needs FT_FILL_KERNEL");
  FT_CUDA(cudaSetDevice(h->dev));
  std::unique_ptr<ft_graph> gr(new ft_graph());
  gr->owner = h;
  const size_t n_prof0 = h->prof_live.size();
  FT_CUDA(cudaStreamBeginCapture(h->cs, cudaStreamCaptureModeThreadLocal));
  ft_status s = ft_moe_decode_layers(h, first_layer, n_layers, batch, x_bf16, logits, c_partial, out, rows_out);
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(h->cs, &graph);
  if (s != FT_OK) {
    if (graph) cudaGraphDestroy(graph);
    return s;
  }
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "capture failed: %s", cudaGetErrorString(e));
  gr->graph = graph;
  gr->prof.assign(h->prof_live.begin() + n_prof0, h->prof_live.end());
  h->prof_live.resize(n_prof0);
  e = cudaGraphInstantiate(&gr->exec, graph, 0);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
  *g = gr.release();
  h->graphs.push_back(*g);
  return FT_OK;
}

ft_status ft_graph_launch(ft_graph* g) {
  if (!g || !g->exec) return fail(FT_ERR_INVALID, "null graph");
  if (!g->owner) return fail(FT_ERR_STATE, "graph belongs to a resized or destroyed handle");
  if (g->owner->pf) ft::prefill_interrupt(g->owner->pf);
  FT_CUDA(cudaGraphLaunch(g->exec, g->owner->cs));
  ++g->pending;
  return FT_OK;
}

ft_status ft_graph_destroy(ft_graph* g) {
  if (!g) return FT_OK;
  if (g->owner) {
    auto& v = g->owner->graphs;
    v.erase(std::remove(v.begin(), v.end(), g), v.end());
  }
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  for (auto& r : g->prof) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  delete g;
  return FT_OK;
}

ft_status ft_moe_decode_layers_host(ft_moe* h, int first_layer, int n_layers, int batch, const void* x_host,
                                    const float* logits_host, const float* c_partial_host, float* out_host,
                                    int use_graph) {
  if (!h || !x_host || !logits_host) return fail(FT_ERR_INVALID, "null argument");
  if (n_layers < 1 || first_layer < 0 || first_layer + n_layers > h->L)
    return fail(FT_ERR_INVALID, "layer range out of range");
  if (batch < 1 || batch > h->cfg.max_batch) return fail(FT_ERR_INVALID, "batch out of range");
  FT_CUDA(cudaSetDevice(h->dev));
  const size_t L = h->L, B = h->cfg.max_batch, H = h->H, E = h->E, K = h->K;
  if (!h->stg_x) {
    ft_status s;
    if ((s = alloc_dev(h, (void**)&h->stg_x, sizeof(uint16_t) * L * B * H)) != FT_OK) return s;
    if ((s = alloc_dev(h, (void**)&h->stg_logits, sizeof(float) * L * B * E)) != FT_OK) return s;
    if ((s = alloc_dev(h, (void**)&h->stg_cp, sizeof(float) * L * B * K * H)) != FT_OK) return s;
    if ((s = alloc_dev(h, (void**)&h->stg_out, sizeof(float) * L * B * H)) != FT_OK) return s;
  }
  const size_t nb = (size_t)n_layers * batch;
  FT_CUDA(cudaMemcpyAsync(h->stg_x, x_host, sizeof(uint16_t) * nb * H, cudaMemcpyHostToDevice, h->cs));
  FT_CUDA(cudaMemcpyAsync(h->stg_logits, logits_host, sizeof(float) * nb * E, cudaMemcpyHostToDevice, h->cs));
  if (c_partial_host)
    FT_CUDA(cudaMemcpyAsync(h->stg_cp, c_partial_host, sizeof(float) * nb * K * H, cudaMemcpyHostToDevice, h->cs));
  const float* cp = c_partial_host ? h->stg_cp : nullptr;
  ft_status s;
  if (use_graph && h->cfg.fill_mode == FT_FILL_KERNEL && !h->prof) {
    auto key = std::make_tuple(first_layer, n_layers, batch * 2 + (cp ? 1 : 0));
    auto it = h->host_graphs.find(key);
    ft_graph* g = nullptr;
    if (it == h->host_graphs.end()) {
      s = ft_moe_graph_capture_decode(h, first_layer, n_layers, batch, h->stg_x, h->stg_logits, cp, h->stg_out,
                                      nullptr, &g);
      if (s != FT_OK) return s;
      h->host_graphs[key] = g;
    } else {
      g = it->second;
    }
    if ((s = ft_graph_launch(g)) != FT_OK) return s;
  } else {
    s = ft_moe_decode_layers(h, first_layer, n_layers, batch, h->stg_x, h->stg_logits, cp, h->stg_out, nullptr);
    if (s != FT_OK) return s;
  }
  if (out_host)
    FT_CUDA(cudaMemcpyAsync(out_host, h->stg_out, sizeof(float) * nb * H, cudaMemcpyDeviceToHost, h->cs));
  FT_CUDA(cudaStreamSynchronize(h->cs));
  return FT_OK;
}

ft_status ft_moe_synchronize(ft_moe* h) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  FT_CUDA(cudaSetDevice(h->dev));
  FT_CUDA(cudaStreamSynchronize(h->ts));
  FT_CUDA(cudaStreamSynchronize(h->cs));
  return FT_OK;
}

ft_status ft_moe_get_stats(ft_moe* h, ft_stats* out) {
  if (!h || !out) return fail(FT_ERR_INVALID, "null argument");
  ft_status s = ft_moe_synchronize(h);
  if (s != FT_OK) return s;
  ft::DevState d{};
  FT_CUDA(cudaMemcpy(&d, h->st, sizeof d, cudaMemcpyDeviceToHost));
  out->hits = d.hits;
  out->misses = d.misses;
  out->fills = d.fills;
  out->cpu_execs = d.cpu_execs;
  out->evictions = d.evictions;
  out->decode_steps = d.decode_steps;
  out->prefill_layers = d.prefill_layers;
  out->eval_entries = d.eval_entries;
  out->eval_pairs = d.eval_pairs;
  out->error_word = d.error_word;
  out->clock = d.clock;
  out->bp_gbps = h->bp_gbps;
  out->bh_gbps = h->bh_gbps;
  out->cache_slots = h->S;
  out->batch1_fused = h->fused_ok ? 1 : 0;
  return FT_OK;
}

ft_status ft_moe_reset_error(ft_moe* h) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  if (capturing(h->cs)) return fail(FT_ERR_STATE, "reset during capture");
  ft_status s = ft_moe_synchronize(h);
  if (s != FT_OK) return s;
  FT_CUDA(cudaMemset(&h->st->error_word, 0, sizeof(uint32_t)));
  FT_CUDA(cudaDeviceSynchronize());
  return FT_OK;
}

ft_status ft_moe_test_control(ft_moe* h, int what, long long value) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  if (what != FT_TEST_HANDOFF_TIMEOUT_NS || value < 0) return fail(FT_ERR_INVALID, "unknown test control");
  h->test_handoff_ns = (uint64_t)value;
  return FT_OK;
}

ft_status ft_moe_get_step_trace(ft_moe* h, ft_step_trace* t) {
  if (!h || !t) return fail(FT_ERR_INVALID, "null argument");
  ft_status s = ft_moe_synchronize(h);
  if (s != FT_OK) return s;
  int32_t c[ft::C_NCOUNTS];
  FT_CUDA(cudaMemcpy(c, h->w.counts, sizeof c, cudaMemcpyDeviceToHost));
  t->layer = c[ft::C_LAYER];
  t->batch = c[ft::C_BATCH];
  t->q = c[ft::C_Q];
  t->n_active = c[ft::C_NACTIVE];
  t->n_hit = c[ft::C_NHIT];
  t->n_miss = c[ft::C_NMISS];
  t->n_victims = c[ft::C_NVICT];
  t->n_cpu = c[ft::C_NMISS] - c[ft::C_Q];
  t->clock = (uint32_t)c[ft::C_CLOCK];
  const size_t np = (size_t)t->batch * h->K;
  if (t->sel) FT_CUDA(cudaMemcpy(t->sel, h->w.sel, np * 4, cudaMemcpyDeviceToHost));
  if (t->gates) FT_CUDA(cudaMemcpy(t->gates, h->w.gates, np * 4, cudaMemcpyDeviceToHost));
  if (t->slot_of_pair) FT_CUDA(cudaMemcpy(t->slot_of_pair, h->w.slot_of_pair, np * 4, cudaMemcpyDeviceToHost));
  if (t->active && t->n_active) FT_CUDA(cudaMemcpy(t->active, h->w.active, (size_t)t->n_active * 4, cudaMemcpyDeviceToHost));
  if (t->hit && t->n_hit) FT_CUDA(cudaMemcpy(t->hit, h->w.hit, (size_t)t->n_hit * 4, cudaMemcpyDeviceToHost));
  if (t->miss && t->n_miss) FT_CUDA(cudaMemcpy(t->miss, h->w.miss, (size_t)t->n_miss * 4, cudaMemcpyDeviceToHost));
  if (t->victims && t->n_victims)
    FT_CUDA(cudaMemcpy(t->victims, h->w.victims, (size_t)t->n_victims * 4, cudaMemcpyDeviceToHost));
  return FT_OK;
}

ft_status ft_moe_get_state(ft_moe* h, int32_t* res, int32_t* owner, uint32_t* stamp, uint32_t* clock) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  ft_status s = ft_moe_synchronize(h);
  if (s != FT_OK) return s;
  if (res) FT_CUDA(cudaMemcpy(res, h->res, sizeof(int32_t) * h->L * h->E, cudaMemcpyDeviceToHost));
  if (owner) FT_CUDA(cudaMemcpy(owner, h->owner, sizeof(int32_t) * h->S, cudaMemcpyDeviceToHost));
  if (stamp) FT_CUDA(cudaMemcpy(stamp, h->stamp, sizeof(uint32_t) * h->S, cudaMemcpyDeviceToHost));
  if (clock) {
    ft::DevState d{};
    FT_CUDA(cudaMemcpy(&d, h->st, sizeof d, cudaMemcpyDeviceToHost));
    *clock = d.clock;
  }
  return FT_OK;
}

ft_status ft_moe_set_profiling(ft_moe* h, int enable) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  ft_status s = ft_moe_synchronize(h);
  if (s != FT_OK) return s;
  h->prof = enable != 0;
  return FT_OK;
}

ft_status ft_moe_get_profile(ft_moe* h, ft_profile* out, int reset) {
  if (!h || !out) return fail(FT_ERR_INVALID, "null argument");
  ft_status s = ft_moe_synchronize(h);
  if (s != FT_OK) return s;
  for (auto& r : h->prof_live) {
    float ms = 0.f;
    FT_CUDA(cudaEventElapsedTime(&ms, r.a, r.b));
    h->prof_acc.launches[r.kind] += 1;
    h->prof_acc.total_ms[r.kind] += ms;
    h->ev_free.push_back(r.a);
    h->ev_free.push_back(r.b);
  }
  h->prof_live.clear();
  // graphs captured with profiling on: their event nodes hold the last replay's times
  for (ft_graph* g : h->graphs) {
    if (!g->pending || g->prof.empty()) continue;
    for (auto& r : g->prof) {
      float ms = 0.f;
      FT_CUDA(cudaEventElapsedTime(&ms, r.a, r.b));
      h->prof_acc.launches[r.kind] += 1;
      h->prof_acc.total_ms[r.kind] += ms;
    }
    g->pending = 0;
  }
  *out = h->prof_acc;
  if (reset) h->prof_acc = ft_profile{};
  return FT_OK;
}

ft_status ft_moe_set_stream(ft_moe* h, void* compute_stream) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  ft_status s = ft_moe_synchronize(h);
  if (s != FT_OK) return s;
  if (h->own_cs && h->cs) cudaStreamDestroy(h->cs);
  if (compute_stream) {
    h->cs = (cudaStream_t)compute_stream;
    h->own_cs = false;
  } else {
    FT_CUDA(cudaStreamCreateWithFlags(&h->cs, cudaStreamNonBlocking));
    h->own_cs = true;
  }
  return FT_OK;
}

ft_status ft_moe_prefill_chunk(ft_moe* h, int layer, int n_tokens, const void* x_bf16, const float* logits,
                               float* out) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  if (layer < 0 || layer >= h->L) return fail(FT_ERR_INVALID, "layer %d out of range", layer);
  if (n_tokens < 1 || n_tokens > h->cfg.max_prefill_tokens)
    return fail(FT_ERR_INVALID, "n_tokens %d outside [1, max_prefill_tokens=%d]", n_tokens, h->cfg.max_prefill_tokens);
  if (!x_bf16 || !logits || !out) return fail(FT_ERR_INVALID, "null x/logits/out");
  if (capturing(h->cs)) return fail(FT_ERR_STATE, "prefill chunks are not capturable");
  FT_CUDA(cudaSetDevice(h->dev));
  ft::PrefillCtx c{};
  c.cs = h->cs;
  c.ts = h->ts;
  c.L = h->L;
  c.E = h->E;
  c.K = h->K;
  c.H = h->H;
  c.I = h->I;
  c.S = h->S;
  c.has_shared = h->cfg.has_shared;
  c.max_tokens = h->cfg.max_prefill_tokens;
  c.n_sm = h->n_sm;
  c.lay = h->lay;
  c.pool = h->pool;
  c.shared_w = h->shared_w;
  c.res = h->res;
  c.owner = h->owner;
  c.stamp = h->stamp;
  c.st = h->st;
  c.n_banks = h->n_banks;
  c.wtype = h->cfg.wtype;
  for (int j = 0; j < h->n_banks; ++j) {
    c.bank_host[j] = h->bank[j].host;
    c.bank_dev[j] = static_cast<const uint8_t*>(h->bank[j].dev);
    c.bank_row[j] = h->bank[j].row;
  }
  c.prof = h->prof;
  c.overlap = h->pf_overlap;
  c.gate = h->gate;
  if (!h->pf) {
    cudaError_t e = ft::prefill_create(&h->pf, c);
    if (e != cudaSuccess) return fail(e == cudaErrorMemoryAllocation ? FT_ERR_NOMEM : FT_ERR_CUDA,
                                      "prefill buffers: %s", cudaGetErrorString(e));
  }
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> ev;
  std::string err;
  // two full-layer buffers when the pool holds them, else experts on demand
  const bool streamed = h->S >= 2 * h->E;
  cudaError_t e =
      streamed ? ft::prefill_layer(h->pf, c, layer, n_tokens, static_cast<const uint16_t*>(x_bf16), logits, out,
                                   h->prof ? &ev : nullptr, &err)
               : ft::prefill_layer_on_demand(h->pf, c, layer, n_tokens, static_cast<const uint16_t*>(x_bf16), logits,
                                             out, h->prof ? &ev : nullptr, &err);
  for (auto& r : ev) h->prof_live.push_back({r.first, r.second.first, r.second.second});
  if (e == cudaErrorNotSupported && err.rfind("capacity", 0) == 0)
    return fail(FT_ERR_CAPACITY, "prefill layer %d: %s", layer, err.c_str());
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "prefill layer %d: %s %s", layer, cudaGetErrorString(e), err.c_str());
  return FT_OK;
}

ft_status ft_moe_prefill_chunk_hidden(ft_moe* h, int layer, int n_tokens, const void* x_bf16, float* out) {
  ft_status s = check_router(h, layer, n_tokens, x_bf16);
  if (s != FT_OK) return s;
  if (n_tokens > h->cfg.max_prefill_tokens)
    return fail(FT_ERR_INVALID, "n_tokens %d above max_prefill_tokens=%d", n_tokens, h->cfg.max_prefill_tokens);
  if (!out) return fail(FT_ERR_INVALID, "null out");
  // the checks of ft_moe_prefill_chunk that do not depend on the logits, before any work
  if (capturing(h->cs)) return fail(FT_ERR_STATE, "prefill chunks are not capturable");
  FT_CUDA(cudaSetDevice(h->dev));
  if ((s = enqueue_router(h, layer, n_tokens, x_bf16, h->router_z, false)) != FT_OK) return s;
  return ft_moe_prefill_chunk(h, layer, n_tokens, x_bf16, h->router_z, out);
}

ft_status ft_moe_set_host_hook(ft_moe* h, ft_host_hook fn, void* user) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  if (capturing(h->cs)) return fail(FT_ERR_STATE, "cannot change the host hook during capture");
  FT_CUDA(cudaSetDevice(h->dev));
  if (fn && !h->hk_sel) {
    const size_t np = (size_t)h->cfg.max_batch * h->K;
    FT_CUDA(cudaMallocHost(&h->hk_sel, np * sizeof(int32_t)));
    FT_CUDA(cudaMallocHost(&h->hk_slot, np * sizeof(int32_t)));
    FT_CUDA(cudaMallocHost(&h->hk_gates, np * sizeof(float)));
    FT_CUDA(cudaMallocHost(&h->hk_rows, np * h->H * sizeof(float)));
    FT_CUDA(cudaMalloc(&h->hk_rows_dev, np * h->H * sizeof(float)));
    h->hook_ctx.resize((size_t)h->L * (h->cfg.max_batch + 1));
    for (int l = 0; l < h->L; ++l)
      for (int b = 0; b <= h->cfg.max_batch; ++b)
        h->hook_ctx[(size_t)l * (h->cfg.max_batch + 1) + b] = {h, {l, b}};
  }
  const ft_status st = ft_moe_synchronize(h);  // no step of the old hook is in flight
  if (st != FT_OK) return st;
  h->hook = fn;
  h->hook_user = user;
  return FT_OK;
}

ft_status ft_moe_set_prefill_overlap(ft_moe* h, int on) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  h->pf_overlap = on != 0;
  return FT_OK;
}

ft_status ft_cache_resize(ft_moe* h, int new_slots) {
  if (!h) return fail(FT_ERR_INVALID, "null handle");
  if (new_slots < 1 || new_slots > (1 << 20)) return fail(FT_ERR_INVALID, "new_slots out of range");
  if (capturing(h->cs)) return fail(FT_ERR_STATE, "resize during capture");
  ft_status s = ft_moe_synchronize(h);
  if (s != FT_OK) return s;
  if (h->pf) ft::prefill_interrupt(h->pf), ft_moe_synchronize(h);
  const int S = h->S, n = new_slots;
  const size_t nlog = (size_t)h->L * h->E;
  std::vector<int32_t> res(nlog), owner(S);
  std::vector<uint32_t> stamp(S);
  FT_CUDA(cudaMemcpy(res.data(), h->res, nlog * 4, cudaMemcpyDeviceToHost));
  FT_CUDA(cudaMemcpy(owner.data(), h->owner, (size_t)S * 4, cudaMemcpyDeviceToHost));
  FT_CUDA(cudaMemcpy(stamp.data(), h->stamp, (size_t)S * 4, cudaMemcpyDeviceToHost));
  const size_t stride = h->lay.stride;
  // every new buffer first: a refused allocation leaves the handle as it was
  uint8_t* np = nullptr;
  int32_t* nowner = nullptr;
  uint32_t* nstamp = nullptr;
  {
    cudaError_t e = n >= S ? dev_malloc((void**)&np, (size_t)n * stride) : cudaSuccess;
    if (e == cudaSuccess) e = dev_malloc((void**)&nowner, (size_t)n * 4);
    if (e == cudaSuccess) e = dev_malloc((void**)&nstamp, (size_t)n * 4);
    if (e != cudaSuccess) {
      if (np) cudaFree(np);
      if (nowner) cudaFree(nowner);
      cudaGetLastError();
      return fail(FT_ERR_NOMEM, "resize to %d slots: %s", n, cudaGetErrorString(e));
    }
  }
  if (n >= S) {
    FT_CUDA(cudaMemcpy(np, h->pool, (size_t)S * stride, cudaMemcpyDeviceToDevice));
    cudaFree(h->pool);
    h->pool = np;
    owner.resize(n, -1);
    stamp.resize(n, 0u);
  } else {
    // keep the n most recent entries (stamp desc, slot asc)
    std::vector<int> occ;
    for (int sl = 0; sl < S; ++sl)
      if (owner[sl] >= 0) occ.push_back(sl);
    std::stable_sort(occ.begin(), occ.end(), [&](int a, int b) {
      return stamp[a] != stamp[b] ? stamp[a] > stamp[b] : a < b;
    });
    std::vector<char> keep(S, 0);
    for (size_t i = 0; i < occ.size() && (int)i < n; ++i) keep[occ[i]] = 1;
    for (int sl = 0; sl < S; ++sl)
      if (owner[sl] >= 0 && !keep[sl]) {
        res[owner[sl]] = -1;
        owner[sl] = -1;
        stamp[sl] = 0;
      }
    std::vector<int> movers, freeb;
    for (int sl = n; sl < S; ++sl)
      if (keep[sl]) movers.push_back(sl);
    for (int sl = 0; sl < n; ++sl)
      if (!keep[sl]) freeb.push_back(sl);
    for (size_t i = 0; i < movers.size(); ++i) {
      const int src = movers[i], dst = freeb[i];
      FT_CUDA(cudaMemcpyAsync(h->pool + (size_t)dst * stride, h->pool + (size_t)src * stride, h->lay.used,
                              cudaMemcpyDeviceToDevice, h->cs));
      owner[dst] = owner[src];
      stamp[dst] = stamp[src];
      res[owner[dst]] = dst;
    }
    owner.resize(n);
    stamp.resize(n);
    FT_CUDA(cudaStreamSynchronize(h->cs));
  }
  FT_CUDA(cudaMemcpy(nowner, owner.data(), (size_t)n * 4, cudaMemcpyHostToDevice));
  FT_CUDA(cudaMemcpy(nstamp, stamp.data(), (size_t)n * 4, cudaMemcpyHostToDevice));
  FT_CUDA(cudaMemcpy(h->res, res.data(), nlog * 4, cudaMemcpyHostToDevice));
  for (auto& p : h->allocs) {
    if (p == h->owner) p = nowner;
    if (p == h->stamp) p = nstamp;
  }
  cudaFree(h->owner);
  cudaFree(h->stamp);
  h->owner = nowner;
  h->stamp = nstamp;
  h->S = n;
  h->cfg.cache_slots = n;
  // graphs captured earlier hold old pointers and sizes: drop them
  for (auto& kv : h->host_graphs) ft_graph_destroy(kv.second);
  h->host_graphs.clear();
  for (ft_graph* g : h->graphs) g->owner = nullptr;
  h->graphs.clear();
  if (h->pf) {
    ft::prefill_destroy(h->pf);
    h->pf = nullptr;
  }
  return FT_OK;
}

ft_status ft_moe_destroy(ft_moe* h) {
  if (!h) return FT_OK;
  cudaSetDevice(h->dev);
  if (h->cs) cudaStreamSynchronize(h->cs);
  if (h->ts) cudaStreamSynchronize(h->ts);
  for (auto& kv : h->host_graphs) ft_graph_destroy(kv.second);
  for (ft_graph* g : h->graphs) g->owner = nullptr;
  if (h->pf) ft::prefill_destroy(h->pf);
  for (auto& r : h->prof_live) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : h->ev_free) cudaEventDestroy(e);
  for (void* p : h->allocs) cudaFree(p);
  if (h->pool) cudaFree(h->pool);
  if (h->shared_w) cudaFree(h->shared_w);
  if (h->router_w) cudaFree(h->router_w);
  if (h->router_z) cudaFree(h->router_z);
  if (h->counts_host) cudaFreeHost(h->counts_host);
  if (h->copy_host) cudaFreeHost(h->copy_host);
  if (h->hk_sel) cudaFreeHost(h->hk_sel);
  if (h->hk_slot) cudaFreeHost(h->hk_slot);
  if (h->hk_gates) cudaFreeHost(h->hk_gates);
  if (h->hk_rows) cudaFreeHost(h->hk_rows);
  if (h->hk_rows_dev) cudaFree(h->hk_rows_dev);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->ev_ctrl) cudaEventDestroy(h->ev_ctrl);
  for (auto& b : h->bank)
    if (b.registered) cudaHostUnregister(const_cast<uint8_t*>(b.host));
  if (h->own_cs && h->cs) cudaStreamDestroy(h->cs);
  if (h->own_ts && h->ts) cudaStreamDestroy(h->ts);
  delete h;
  return FT_OK;
}

}  // extern "C"
