// The C ABI declared in include/fwmoe.h: argument checks, device memory of a
// handle, the one-time repack, and dispatch to the decode (T <= decode_T_max)
// or prefill kernels. No entry point synchronises the stream except init,
// free, status and the host-buffer forward.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>
#include <vector>

#include "internal.cuh"

namespace fw {
namespace {

thread_local char g_err[512] = "";
std::mutex g_live_mu;
std::unordered_set<Handle*> g_live;

fw_status fail(fw_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

fw_status cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? FW_ENOMEM : FW_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
              cudaGetErrorString(e));
}

bool live(Handle* h) {
  std::lock_guard<std::mutex> g(g_live_mu);
  return h && g_live.count(h) && h->magic == kHandleMagic;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Test hook: FWMOE_TEST_FAIL_ALLOC=n makes the n-th device allocation of the
// next fw_moe_init fail, to exercise the clean-up path.
struct Allocator {
  std::vector<void*> blocks;
  long fail_at = -1, count = 0;
  Allocator() {
    const char* s = getenv("FWMOE_TEST_FAIL_ALLOC");
    if (s && *s) fail_at = atol(s);
  }
  template <typename T>
  cudaError_t get(T** p, size_t bytes) {
    *p = nullptr;
    if (++count == fail_at) return cudaErrorMemoryAllocation;
    void* q = nullptr;
    cudaError_t e = cudaMalloc(&q, bytes < 256 ? 256 : bytes);
    if (e != cudaSuccess) return e;
    blocks.push_back(q);
    *p = static_cast<T*>(q);
    return cudaSuccess;
  }
  void release() {
    for (void* q : blocks) cudaFree(q);
    blocks.clear();
  }
};

void free_handle_memory(Handle* h) {
  void* ptrs[] = {h->q_gu, h->q_dc, h->st_d, h->t_gu, h->t_d, h->wr3, h->wr, h->bias, h->ids, h->gates,
                  h->logits, h->counts, h->offsets, h->perm, h->inv, h->row_token, h->row_gate, h->uinfo,
                  h->hist, h->minfo, h->minfo_m, h->minfo_s, h->xperm, h->hbuf, h->yp, h->partial, h->zpart, h->meta,
                  h->x_dev, h->out_dev, h->ids_dev};
  for (void* p : ptrs)
    if (p) cudaFree(p);
}

fw_status check_config(const fw_moe_config* c) {
  if (c->H <= 0 || c->H % 64) return fail(FW_EUNSUPPORTED, "H=%d must be a positive multiple of 64", c->H);
  if (c->I <= 0 || c->I % 64) return fail(FW_EUNSUPPORTED, "I=%d must be a positive multiple of 64", c->I);
  if (c->E < 1 || c->E > 256) return fail(FW_EUNSUPPORTED, "E=%d must be in [1, 256]", c->E);
  if (c->k < 1 || c->k > c->E || c->k > kMaxK) return fail(FW_EINVAL, "k=%d must be in [1, min(E, 16)]", c->k);
  if (c->n_shared != 0 && c->n_shared != 1) return fail(FW_EINVAL, "n_shared=%d must be 0 or 1", c->n_shared);
  if (c->T_max < 1 || c->T_max > (1 << 20)) return fail(FW_EINVAL, "T_max=%d must be in [1, 2^20]", c->T_max);
  if (c->decode_T_max < 0 || c->decode_T_max > kMaxDecodeT)
    return fail(FW_EINVAL, "decode_T_max=%d must be in [0, 16]", c->decode_T_max);
  if (c->act_q8 != 0 && c->act_q8 != 1) return fail(FW_EINVAL, "act_q8=%d must be 0 or 1", c->act_q8);
  return FW_OK;
}

int decode_limit(const Handle* h) { return h->cfg.decode_T_max ? h->cfg.decode_T_max : kMaxDecodeT; }

// T tokens take the decode kernel: T within the handle's decode limit and a
// shape that kernel holds; any other T takes the prefill path.
bool use_decode(const Handle* h, int T) { return T <= decode_limit(h) && decode_supported(h->cfg.H, T); }

// Some T in [1, T_max] takes the prefill path (its tensor maps and buffers are needed).
bool needs_prefill(const Handle* h) {
  const int Tm = h->cfg.T_max;
  return Tm > decode_limit(h) || !decode_supported(h->cfg.H, 1) || (Tm > 1 && !decode_supported(h->cfg.H, 2));
}

}  // namespace

// Record the text of a failed call for fw_moe_last_error (other source files).
fw_status set_error(fw_status st, const char* text) { return fail(st, "%s", text); }

}  // namespace fw

using namespace fw;

extern "C" {

const char* fw_moe_last_error(void) { return g_err; }

fw_status fw_moe_init(const fw_moe_config* cfg, const fw_moe_weights* w, void* stream, fw_moe_handle** out) {
  if (!cfg || !w || !out) return fail(FW_EINVAL, "fw_moe_init: null argument");
  *out = nullptr;
  fw_status st = check_config(cfg);
  if (st != FW_OK) return st;
  if (!w->router_w || !w->w_gate || !w->w_up || !w->w_down)
    return fail(FW_EINVAL, "fw_moe_init: router_w, w_gate, w_up and w_down are required");
  if (cfg->n_shared == 1 && (!w->shared_gate || !w->shared_up || !w->shared_down))
    return fail(FW_EINVAL, "fw_moe_init: n_shared=1 needs shared_gate, shared_up and shared_down");
  if (!aligned(w->router_w, 16) || (w->router_bias && !aligned(w->router_bias, 4)))
    return fail(FW_EINVAL, "fw_moe_init: router_w must be 16-byte aligned");
  const uint8_t* mats[] = {w->w_gate, w->w_up, w->w_down, w->shared_gate, w->shared_up, w->shared_down};
  for (const uint8_t* m : mats)
    if (m && !aligned(m, 2)) return fail(FW_EINVAL, "fw_moe_init: Q8_0 buffers must be 2-byte aligned");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FW_EUNSUPPORTED, "fw_moe_init: no CUDA device (%s)", cudaGetErrorString(e));
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(FW_EUNSUPPORTED, "fw_moe_init: device %d is sm_%d%d; this library is built for sm_103a only", dev,
                prop.major, prop.minor);

  e = configure_route_kernels();
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_init: router kernel set-up (is the library built for this GPU?)");
  g_err[0] = 0;
  e = configure_decode_kernels();
  if (e != cudaSuccess) {
    if (g_err[0]) return FW_EUNSUPPORTED;  // the set-up left its own text
    return cuda_fail(e, "fw_moe_init: decode kernel set-up");
  }
  e = configure_prefill_kernels();
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_init: prefill kernel set-up");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Handle* h = new Handle();
  std::memset(static_cast<void*>(h), 0, sizeof(Handle));
  h->cfg = *cfg;
  h->S = cfg->n_shared;
  h->EU = cfg->E + h->S;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->last_T = -1;
  {
    const char* s = getenv("FWMOE_TEST_GRID_TIMEOUTS");
    h->test_grid_timeouts = (s && *s) ? atoi(s) : 0;
  }
  const bool pre = needs_prefill(h);
  h->has_prefill = pre ? 1 : 0;
  const int64_t H = cfg->H, I = cfg->I, E = cfg->E, EU = h->EU, k = cfg->k, Tm = cfg->T_max;
  h->rows_max = Tm * (k + h->S);

  Allocator A;
  const int64_t n_route_tiles = (Tm + kRouteTileM - 1) / kRouteTileM;
  const int64_t n_mtiles_max = h->rows_max / kTokTile + EU + 1;
  const size_t hbuf_bytes = pre ? (size_t)h->rows_max * I * 2 : 256;  // prefill h (bf16)
  const int64_t T_dec = std::min<int64_t>(Tm, kMaxDecodeT);
  struct {
    void** p;
    size_t bytes;
  } req[] = {
      {(void**)&h->q_gu, (size_t)(EU * 2 * I * row_bytes(H))},
      {(void**)&h->q_dc, (size_t)(EU * H * I)},
      {(void**)&h->st_d, (size_t)(EU * (I / 32) * H * 2)},
      {(void**)&h->t_gu, (size_t)(pre ? EU * gemm_plane_bytes(2 * I / kTileRows, H / kTileK) : 256)},
      {(void**)&h->t_d, (size_t)(pre ? EU * gemm_plane_bytes((H + kTileRows - 1) / kTileRows, I / kTileK) : 256)},
      {(void**)&h->wr, (size_t)(E * H * 4)},
      {(void**)&h->bias, (size_t)(E * 4)},
      {(void**)&h->wr3, (size_t)(pre ? 3 * E * H * 2 : 256)},
      {(void**)&h->ids, (size_t)(Tm * k * 4)},
      {(void**)&h->gates, (size_t)(Tm * k * 4)},
      {(void**)&h->logits, (size_t)(std::min<int64_t>(Tm, kMaxDecodeT) * E * 4)},
      {(void**)&h->counts, (size_t)(EU * 4)},
      {(void**)&h->offsets, (size_t)((EU + 1) * 4)},
      {(void**)&h->perm, (size_t)(h->rows_max * 4)},
      {(void**)&h->inv, (size_t)(h->rows_max * 4)},
      {(void**)&h->row_token, (size_t)(h->rows_max * 4)},
      {(void**)&h->row_gate, (size_t)(h->rows_max * 4)},
      {(void**)&h->uinfo, (size_t)(EU * 16)},
      {(void**)&h->hist, (size_t)(n_route_tiles * EU * 4)},
      {(void**)&h->minfo, (size_t)(n_mtiles_max * 16)},
      {(void**)&h->minfo_m, (size_t)(EU * 16)},
      {(void**)&h->minfo_s, (size_t)(EU * 16)},
      {(void**)&h->xperm, (size_t)(pre ? h->rows_max * H * 2 : 256)},
      {(void**)&h->hbuf, hbuf_bytes},
      {(void**)&h->yp, (size_t)(pre ? h->rows_max * H * 2 : 256)},
      {(void**)&h->partial, (size_t)(h->num_sms * T_dec * H * 4)},
      {(void**)&h->zpart, (size_t)(pre ? kRouterMaxSplit * Tm * E * 4 : 256)},
      {(void**)&h->meta, sizeof(Meta)},
      {(void**)&h->x_dev, (size_t)(Tm * H * 2)},
      {(void**)&h->out_dev, (size_t)(Tm * H * 2)},
      {(void**)&h->ids_dev, (size_t)(Tm * k * 4)},
  };
  for (auto& r : req) {
    e = A.get(r.p, r.bytes);
    if (e != cudaSuccess) {
      A.release();
      delete h;
      return fail(FW_ENOMEM, "fw_moe_init: device allocation of %zu bytes failed (%s)", r.bytes,
                  cudaGetErrorName(e));
    }
  }

  e = cudaMemcpyAsync(h->wr, w->router_w, E * H * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = w->router_bias ? cudaMemcpyAsync(h->bias, w->router_bias, E * 4, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(h->bias, 0, E * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->meta, 0, sizeof(Meta), s);
  // the scale pads of the code planes are never used, but keep them defined
  if (e == cudaSuccess) e = cudaMemsetAsync(h->q_gu, 0, EU * 2 * I * row_bytes(H), s);
  // rows of a last partial down tile (H % 128 != 0) are read and their results dropped: keep them defined
  if (e == cudaSuccess && pre)
    e = cudaMemsetAsync(h->t_d, 0, EU * gemm_plane_bytes((H + kTileRows - 1) / kTileRows, I / kTileK), s);
  if (e == cudaSuccess) e = launch_repack(h, 0, 0, (int)E, w->w_gate, s);
  if (e == cudaSuccess) e = launch_repack(h, 1, 0, (int)E, w->w_up, s);
  if (e == cudaSuccess) e = launch_repack(h, 2, 0, (int)E, w->w_down, s);
  if (e == cudaSuccess && h->S) {
    e = launch_repack(h, 0, (int)E, 1, w->shared_gate, s);
    if (e == cudaSuccess) e = launch_repack(h, 1, (int)E, 1, w->shared_up, s);
    if (e == cudaSuccess) e = launch_repack(h, 2, (int)E, 1, w->shared_down, s);
  }
  if (e == cudaSuccess && pre) {
    // rows past the valid ones of a tile are read (and masked); keep them finite
    e = cudaMemsetAsync(h->xperm, 0, (size_t)h->rows_max * H * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->hbuf, 0, hbuf_bytes, s);
    if (e == cudaSuccess) e = launch_split_router(h, s);
    if (e == cudaSuccess) e = prepare_prefill(h);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    A.release();
    delete h->maps;
    delete h;
    return cuda_fail(e, "fw_moe_init");
  }
  h->magic = kHandleMagic;
  {
    std::lock_guard<std::mutex> g(g_live_mu);
    g_live.insert(h);
  }
  *out = reinterpret_cast<fw_moe_handle*>(h);
  return FW_OK;
}

static fw_status check_call(Handle* h, const void* x, int32_t T, const char* who) {
  if (!live(h)) return fail(FW_EINVAL, "%s: not a live handle", who);
  if (T < 0 || T > h->cfg.T_max) return fail(FW_EINVAL, "%s: T=%d outside [0, T_max=%d]", who, T, h->cfg.T_max);
  if (T > 0 && (!x || !aligned(x, 16))) return fail(FW_EINVAL, "%s: x must be a 16-byte aligned device pointer", who);
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != h->device) return fail(FW_EINVAL, "%s: current device %d is not the handle's device %d", who, dev, h->device);
  return FW_OK;
}

fw_status fw_moe_route(fw_moe_handle* hh, const void* x, int32_t T, int32_t* expert_ids, float* gates,
                       void* stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  fw_status st = check_call(h, x, T, "fw_moe_route");
  if (st != FW_OK) return st;
  if (T > 0 && (!expert_ids || !aligned(expert_ids, 4) || (gates && !aligned(gates, 4))))
    return fail(FW_EINVAL, "fw_moe_route: expert_ids must be a 4-byte aligned device pointer");
  h->last_T = T;
  if (T == 0) return FW_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  cudaError_t e = use_decode(h, T) ? launch_route_decode(h, xb, T, expert_ids, gates, true, s)
                                   : launch_route_prefill(h, xb, T, expert_ids, gates, s);
  if (e != cudaSuccess) {
    h->last_T = -1;
    return cuda_fail(e, "fw_moe_route launch");
  }
  return FW_OK;
}

fw_status fw_moe_ffn(fw_moe_handle* hh, const void* x, int32_t T, void* out, void* stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  fw_status st = check_call(h, x, T, "fw_moe_ffn");
  if (st != FW_OK) return st;
  if (T != h->last_T)
    return fail(FW_ESTATE, "fw_moe_ffn: T=%d but the last fw_moe_route on this handle had T=%d", T, h->last_T);
  if (T == 0) return FW_OK;
  if (!out || !aligned(out, 16)) return fail(FW_EINVAL, "fw_moe_ffn: out must be a 16-byte aligned device pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
  cudaError_t e = use_decode(h, T) ? launch_ffn_decode(h, xb, T, ob, false, nullptr, nullptr, s)
                                   : launch_ffn_prefill(h, xb, T, ob, s);
  if (e == cudaErrorNotSupported) return fail(FW_EUNSUPPORTED, "fw_moe_ffn: prefill path not available in this build");
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_ffn launch");
  return FW_OK;
}

fw_status fw_moe_forward(fw_moe_handle* hh, const void* x, int32_t T, int32_t* expert_ids, float* gates, void* out,
                         void* stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  fw_status st = check_call(h, x, T, "fw_moe_forward");
  if (st != FW_OK) return st;
  if (T > 0 && (!expert_ids || !aligned(expert_ids, 4) || (gates && !aligned(gates, 4))))
    return fail(FW_EINVAL, "fw_moe_forward: expert_ids must be a 4-byte aligned device pointer");
  if (T > 0 && (!out || !aligned(out, 16)))
    return fail(FW_EINVAL, "fw_moe_forward: out must be a 16-byte aligned device pointer");
  if (!use_decode(h, T)) {
    st = fw_moe_route(hh, x, T, expert_ids, gates, stream);
    return st != FW_OK ? st : fw_moe_ffn(hh, x, T, out, stream);
  }
  h->last_T = T;
  if (T == 0) return FW_OK;
  // decode: the router only makes logits; the expert kernels select and group
  // (in shared memory) and the gate/up kernel publishes ids, gates and grouping
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  cudaError_t e = launch_route_decode(h, xb, T, expert_ids, gates, false, s);
  if (e == cudaSuccess)
    e = launch_ffn_decode(h, xb, T, static_cast<__nv_bfloat16*>(out), true, expert_ids, gates, s);
  if (e != cudaSuccess) {
    h->last_T = -1;
    return cuda_fail(e, "fw_moe_forward launch");
  }
  return FW_OK;
}

}  // extern "C"

namespace fw {
namespace {
constexpr uint32_t kGraphMagic = 0x4772614Du;  // "MarG"
struct Graph {
  uint32_t magic;
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};
std::unordered_set<Graph*> g_live_graphs;  // under g_live_mu; a pointer is checked here before it is read
bool live_graph(Graph* g) {
  std::lock_guard<std::mutex> lk(g_live_mu);
  return g && g_live_graphs.count(g) && g->magic == kGraphMagic;
}
}  // namespace
}  // namespace fw

extern "C" {

fw_status fw_moe_graph_create(fw_moe_handle* const* layers, int32_t n, int32_t T, const void* const* x,
                              void* const* out, int32_t* const* expert_ids, fw_moe_graph** graph) {
  if (!graph) return fail(FW_EINVAL, "fw_moe_graph_create: graph is null");
  *graph = nullptr;
  if (!layers || !x || !out || !expert_ids || n < 1 || T < 1)
    return fail(FW_EINVAL, "fw_moe_graph_create: needs n >= 1 layers, T >= 1 and the x, out and expert_ids arrays");
  for (int i = 0; i < n; ++i) {
    Handle* h = reinterpret_cast<Handle*>(layers[i]);
    if (!live(h)) return fail(FW_EINVAL, "fw_moe_graph_create: layer %d is not a live handle", i);
    if (T > h->cfg.T_max) return fail(FW_EINVAL, "fw_moe_graph_create: T=%d above layer %d's T_max=%d", T, i, h->cfg.T_max);
    if (!x[i] || !aligned(x[i], 16) || !out[i] || !aligned(out[i], 16) || !expert_ids[i] || !aligned(expert_ids[i], 4))
      return fail(FW_EINVAL, "fw_moe_graph_create: call %d: x and out must be 16-byte, expert_ids 4-byte aligned", i);
    if (h->timing) return fail(FW_ESTATE, "fw_moe_graph_create: layer %d is profiling", i);
  }
  cudaStream_t cs;
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_graph_create: stream");
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) {
    cudaStreamDestroy(cs);
    return cuda_fail(e, "fw_moe_graph_create: begin capture");
  }
  fw_status st = FW_OK;
  char why[sizeof(g_err) + 64] = "";
  for (int i = 0; i < n && st == FW_OK; ++i) {
    st = fw_moe_forward(layers[i], x[i], T, expert_ids[i], nullptr, out[i], cs);
    if (st != FW_OK) snprintf(why, sizeof(why), "fw_moe_graph_create: call %d: %s", i, g_err);
  }
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(cs, &g);  // ends the capture whatever happened inside it
  cudaStreamDestroy(cs);
  if (st != FW_OK || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    if (st != FW_OK) return fail(st, "%s", why);
    return cuda_fail(e, "fw_moe_graph_create: end capture");
  }
  cudaGraphExec_t ge = nullptr;
  e = cudaGraphInstantiate(&ge, g, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    return cuda_fail(e, "fw_moe_graph_create: instantiate");
  }
  Graph* gr = new (std::nothrow) Graph{kGraphMagic, g, ge};
  if (!gr) {
    cudaGraphExecDestroy(ge);
    cudaGraphDestroy(g);
    return fail(FW_ENOMEM, "fw_moe_graph_create: out of host memory");
  }
  {
    std::lock_guard<std::mutex> lk(g_live_mu);
    g_live_graphs.insert(gr);
  }
  *graph = reinterpret_cast<fw_moe_graph*>(gr);
  return FW_OK;
}

fw_status fw_moe_graph_launch(fw_moe_graph* graph, void* stream) {
  Graph* g = reinterpret_cast<Graph*>(graph);
  if (!live_graph(g)) return fail(FW_EINVAL, "fw_moe_graph_launch: not a live graph");
  cudaError_t e = cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FW_OK : cuda_fail(e, "fw_moe_graph_launch");
}

fw_status fw_moe_graph_destroy(fw_moe_graph* graph) {
  Graph* g = reinterpret_cast<Graph*>(graph);
  if (!g) return FW_OK;
  {
    std::lock_guard<std::mutex> lk(g_live_mu);
    if (!g_live_graphs.erase(g)) return fail(FW_EINVAL, "fw_moe_graph_destroy: not a live graph");
  }
  g->magic = 0;
  cudaGraphExecDestroy(g->exec);
  cudaGraphDestroy(g->graph);
  delete g;
  return FW_OK;
}

fw_status fw_moe_forward_host(fw_moe_handle* hh, const void* x_host, int32_t T, int32_t* ids_host, void* out_host,
                              void* stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!live(h)) return fail(FW_EINVAL, "fw_moe_forward_host: not a live handle");
  if (T < 0 || T > h->cfg.T_max) return fail(FW_EINVAL, "fw_moe_forward_host: T=%d outside [0, T_max]", T);
  if (T == 0) {
    h->last_T = 0;
    return FW_OK;
  }
  if (!x_host || !ids_host || !out_host) return fail(FW_EINVAL, "fw_moe_forward_host: null host buffer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)T * h->cfg.H * 2, ib = (size_t)T * h->cfg.k * 4;
  cudaError_t e = cudaMemcpyAsync(h->x_dev, x_host, xb, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_forward_host H2D");
  fw_status st = fw_moe_forward(hh, h->x_dev, T, h->ids_dev, nullptr, h->out_dev, stream);
  if (st != FW_OK) return st;
  e = cudaMemcpyAsync(ids_host, h->ids_dev, ib, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out_host, h->out_dev, xb, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_forward_host");
  return FW_OK;
}

fw_status fw_moe_get_permutation(fw_moe_handle* hh, int32_t* offsets, int32_t* perm, int32_t* inv, void* stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!live(h)) return fail(FW_EINVAL, "fw_moe_get_permutation: not a live handle");
  if (h->last_T < 0) return fail(FW_ESTATE, "fw_moe_get_permutation: no route on this handle yet");
  if (!offsets || (h->last_T > 0 && !perm)) return fail(FW_EINVAL, "fw_moe_get_permutation: null output");
  cudaError_t e = launch_get_permutation(h, h->last_T, offsets, perm, inv, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_get_permutation");
  return FW_OK;
}

fw_status fw_moe_export_q8_0(fw_moe_handle* hh, int32_t expert, int32_t which, uint8_t* blocks, void* stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!live(h)) return fail(FW_EINVAL, "fw_moe_export_q8_0: not a live handle");
  if (expert < 0 || expert >= h->EU) return fail(FW_EINVAL, "fw_moe_export_q8_0: expert %d outside [0, %d)", expert, h->EU);
  if (which < 0 || which > 2) return fail(FW_EINVAL, "fw_moe_export_q8_0: which=%d must be 0, 1 or 2", which);
  if (!blocks || !aligned(blocks, 2)) return fail(FW_EINVAL, "fw_moe_export_q8_0: blocks must be 2-byte aligned");
  cudaError_t e = launch_export(h, which, expert, blocks, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_export_q8_0");
  return FW_OK;
}

fw_status fw_moe_status(fw_moe_handle* hh, void* stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!live(h)) return fail(FW_EINVAL, "fw_moe_status: not a live handle");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t word = 0, diag[4] = {0, 0, 0, 0};
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&word, &h->meta->status, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(diag, h->meta->diag, sizeof(diag), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(&h->meta->status, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(h->meta->diag, 0, sizeof(diag));
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_status");
  if (word & kStatusTimeout)
    return fail(FW_ETIMEOUT, "a kernel gave up a bounded wait (status 0x%x; site %d, block %d, stage %d, detail %d)",
                word, diag[0], diag[1], diag[2], diag[3]);
  if (word) return fail(FW_EDEVICE, "a kernel reported a failed check (status 0x%x)", word);
  return FW_OK;
}

static void drop_timing(Handle* h) {
  if (!h->timing) return;
  for (int i = 0; i < 2 * h->timing->cap; ++i) cudaEventDestroy(h->timing->ev[i]);
  delete[] h->timing->ev;
  delete[] h->timing->kind;
  delete h->timing;
  h->timing = nullptr;
}

fw_status fw_moe_profile_begin(fw_moe_handle* hh, int32_t max_launches) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!live(h)) return fail(FW_EINVAL, "fw_moe_profile_begin: not a live handle");
  if (max_launches < 1 || max_launches > (1 << 20))
    return fail(FW_EINVAL, "fw_moe_profile_begin: max_launches=%d outside [1, 2^20]", max_launches);
  drop_timing(h);
  Timing* t = new Timing();
  t->ev = new cudaEvent_t[2 * (size_t)max_launches];
  t->kind = new int[max_launches];
  for (int i = 0; i < 2 * max_launches; ++i) {
    cudaError_t e = cudaEventCreate(&t->ev[i]);
    if (e != cudaSuccess) {
      t->cap = i / 2;
      h->timing = t;
      drop_timing(h);
      return cuda_fail(e, "fw_moe_profile_begin");
    }
  }
  t->cap = max_launches;
  h->timing = t;
  return FW_OK;
}

fw_status fw_moe_profile_end(fw_moe_handle* hh, int32_t n_kinds, float* total_ms, int32_t* launches) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!live(h)) return fail(FW_EINVAL, "fw_moe_profile_end: not a live handle");
  if (!h->timing) return fail(FW_ESTATE, "fw_moe_profile_end: profiling was not begun");
  if (n_kinds < 0 || n_kinds > FW_KERNEL_KINDS || (n_kinds && (!total_ms || !launches)))
    return fail(FW_EINVAL, "fw_moe_profile_end: bad output arrays");
  for (int i = 0; i < n_kinds; ++i) {
    total_ms[i] = 0.f;
    launches[i] = 0;
  }
  Timing* t = h->timing;
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < t->next && e == cudaSuccess; ++i) {
    e = cudaEventSynchronize(t->ev[2 * i + 1]);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t->ev[2 * i], t->ev[2 * i + 1]);
    if (e == cudaSuccess && t->kind[i] < n_kinds) {
      total_ms[t->kind[i]] += ms;
      launches[t->kind[i]] += 1;
    }
  }
  drop_timing(h);
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_profile_end");
  return FW_OK;
}

fw_status fw_moe_free(fw_moe_handle* hh) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return FW_OK;
  {
    std::lock_guard<std::mutex> g(g_live_mu);
    if (!g_live.count(h)) return fail(FW_EINVAL, "fw_moe_free: not a live handle (freed twice?)");
    g_live.erase(h);
  }
  cudaError_t e = cudaDeviceSynchronize();
  drop_timing(h);
  free_handle_memory(h);
  delete h->maps;
  h->magic = kHandleFreed;
  delete h;
  if (e != cudaSuccess) return cuda_fail(e, "fw_moe_free");
  return FW_OK;
}

fw_status fw_q8_0_quantize(const float* w, int64_t rows, int64_t K, uint8_t* blocks, void* stream) {
  if (rows < 0 || K <= 0 || K % 32) return fail(FW_EINVAL, "fw_q8_0_quantize: need rows >= 0 and K %% 32 == 0");
  if (rows == 0) return FW_OK;
  if (!w || !blocks || !aligned(w, 16) || !aligned(blocks, 2))
    return fail(FW_EINVAL, "fw_q8_0_quantize: w must be 16-byte aligned and blocks 2-byte aligned");
  cudaError_t e = launch_quantize_q8_0(w, rows, K, blocks, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fw_q8_0_quantize");
  return FW_OK;
}

}  // extern "C"
