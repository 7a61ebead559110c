// fw_moe_route_noalloc: the decode router (logits, top-k with ties to the
// lower id, renormalised gates) for callers that cannot allocate device
// memory. Its only scratch (the logits and the last-CTA ticket) lives in a
// file-scope __device__ array that every GPU loading this library holds until
// process exit; nothing here calls cudaMalloc, cudaFree or any allocating
// routine.
#include <mutex>

#include "routing.cuh"

namespace fw {
namespace {

using namespace dev;

constexpr int kNaMaxT = kMaxDecodeT;  // 16 tokens
constexpr int kNaMaxE = kMaxE;        // 256 experts
constexpr int kNaThreads = 256;
constexpr size_t kNaLogitBytes = sizeof(float) * kNaMaxT * kNaMaxE;  // 16 KiB
constexpr size_t kNaScratchBytes = kNaLogitBytes + 256;              // + ticket

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaScratchBytes];

// Grid: E CTAs; CTA e computes z[t][e] for t < T into the scratch logits; the
// last CTA (atomic ticket on the scratch counter, no waiting) selects and
// gates every token and writes the caller's outputs.
__global__ void __launch_bounds__(kNaThreads)
    route_noalloc_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, const float* __restrict__ wr,
                         const float* __restrict__ bias, int E, int k, int32_t* __restrict__ ids_out,
                         float* __restrict__ gates_out, float* logits, unsigned int* ticket) {
  __shared__ float s_part[kNaThreads / 32][kNaMaxT];
  __shared__ bool s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e = blockIdx.x;
  float acc[kNaMaxT];
#pragma unroll
  for (int t = 0; t < kNaMaxT; ++t) acc[t] = 0.f;
  const float* wrow = wr + (int64_t)e * H;
  for (int h = 4 * tid; h < H; h += 4 * kNaThreads) {
    const float4 w = __ldg(reinterpret_cast<const float4*>(wrow + h));
#pragma unroll
    for (int t = 0; t < kNaMaxT; ++t) {
      if (t < T) {
        const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (int64_t)t * H + h));
        float x0, x1, x2, x3;
        bf16x2_to_f32(xv.x, x0, x1);
        bf16x2_to_f32(xv.y, x2, x3);
        acc[t] = fmaf(x0, w.x, acc[t]);
        acc[t] = fmaf(x1, w.y, acc[t]);
        acc[t] = fmaf(x2, w.z, acc[t]);
        acc[t] = fmaf(x3, w.w, acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kNaMaxT; ++t)
    if (t < T) {
      const float v = warp_sum(acc[t]);
      if (lane == 0) s_part[warp][t] = v;
    }
  __syncthreads();
  if (tid < T) {
    float z = 0.f;
#pragma unroll
    for (int w = 0; w < kNaThreads / 32; ++w) z += s_part[w][tid];
    logits[tid * E + e] = z + (bias ? bias[e] : 0.f);
    __threadfence();
  }
  __syncthreads();
  if (tid == 0) s_last = atomicInc(ticket, gridDim.x - 1) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int t = warp; t < T; t += kNaThreads / 32) {
    float zl[kMaxEPerLane];
#pragma unroll
    for (int m = 0; m < kMaxEPerLane; ++m) {
      const int ee = lane + 32 * m;
      zl[m] = ee < E ? __ldcg(logits + t * E + ee) : -INFINITY;
    }
    int id;
    float zv;
    warp_topk(zl, E, k, lane, &id, &zv);
    const float g = warp_gate(zv, k, lane);
    if (lane < k) {
      ids_out[t * k + lane] = id;
      if (gates_out) gates_out[t * k + lane] = g;
    }
  }
}

// Device address of the scratch array, looked up once per device with that
// device current (in host code the array's name is only a stand-in).
constexpr int kMaxDevices = 64;
std::mutex g_na_mu;
void* g_na_ptr[kMaxDevices] = {};

}  // namespace
}  // namespace fw

using namespace fw;

extern "C" fw_status fw_moe_route_noalloc(const void* x, int32_t T, int32_t H, const float* router_w,
                                          const float* router_bias, int32_t E, int32_t k, int32_t* expert_ids,
                                          float* gates, void* stream) {
  if (T < 0 || T > kNaMaxT)
    return set_error(FW_EINVAL, "fw_moe_route_noalloc: T must be in [0, 16] (the scratch holds 16 x 256 logits)");
  if (E < 1 || E > kNaMaxE || k < 1 || k > E || k > kMaxK)
    return set_error(FW_EINVAL, "fw_moe_route_noalloc: need 1 <= E <= 256 and 1 <= k <= min(E, 16)");
  if (H <= 0 || H % 4) return set_error(FW_EINVAL, "fw_moe_route_noalloc: H must be a positive multiple of 4");
  if (T == 0) return FW_OK;
  if (!x || !router_w || !expert_ids) return set_error(FW_EINVAL, "fw_moe_route_noalloc: null pointer");
  auto al = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
  if (!al(x, 8) || !al(router_w, 16) || !al(expert_ids, 4) || (gates && !al(gates, 4)) ||
      (router_bias && !al(router_bias, 4)))
    return set_error(FW_EINVAL, "fw_moe_route_noalloc: x needs 8-byte, router_w 16-byte, outputs 4-byte alignment");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return set_error(FW_ECUDA, "fw_moe_route_noalloc: no current CUDA device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (s) {  // the scratch address looked up below is the current device's: the stream must be on it
    int sdev = -1;
    if (cudaStreamGetDevice(s, &sdev) != cudaSuccess)
      return set_error(FW_EINVAL, "fw_moe_route_noalloc: stream is not a valid CUDA stream");
    if (sdev != dev)
      return set_error(FW_EINVAL, "fw_moe_route_noalloc: stream belongs to another device than the current one");
  }
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> g(g_na_mu);
    if (!g_na_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
        return set_error(FW_ECUDA, "fw_moe_route_noalloc: cudaGetSymbolAddress of the scratch array failed");
      g_na_ptr[dev] = p;
    }
    base = g_na_ptr[dev];
  }
  float* logits = static_cast<float*>(base);
  unsigned int* ticket = reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(base) + kNaLogitBytes);
  // the ticket must start at zero: clear it in stream order (no allocation)
  if (cudaMemsetAsync(ticket, 0, sizeof(unsigned int), s) != cudaSuccess)
    return set_error(FW_ECUDA, "fw_moe_route_noalloc: clearing the scratch ticket failed");
  route_noalloc_kernel<<<E, kNaThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(x), T, H, router_w, router_bias, E,
                                                k, expert_ids, gates, logits, ticket);
  if (cudaGetLastError() != cudaSuccess) return set_error(FW_ECUDA, "fw_moe_route_noalloc: launch failed");
  return FW_OK;
}
