// Decode path (T <= 16): the experts as grouped, HBM-bound GEMVs.
//
// The pages' runtime runs routed experts through grouped GPU kernels per
// quantisation format, Q8_0 among them (Flyweight README, §Quantization), and
// fuses the gate and up projections so they share one activation load (its
// CPU expert kernels, §Current limitations). Here every selected expert's Q8_0
// rows are streamed from HBM exactly once per call, with bulk asynchronous
// copies into a per-warp shared-memory ring, and dequantised in registers.
//
//   gate/up kernel: unit = (expert, i): gate row i and up row i share the
//     x loads; h = SiLU(g) * u for each of the expert's tokens -> hbuf (fp32,
//     one row per grouped (token, slot) pair).
//   down kernel: unit = 2 output rows; the warp walks every touched expert in
//     ascending id (the shared expert last), lane t accumulates
//     gate * (W_down h) for token t, and writes out[t] as bf16: the combine is
//     fused and its summation order is fixed (no atomics).
#include <algorithm>

#include "internal.cuh"

namespace fw {
namespace {

using namespace dev;

constexpr int kWarps = 8;

struct GateUpArgs {
  const int8_t* q;        // q_gu
  const uint8_t* s;       // s_gu
  const __nv_bfloat16* x;
  float* hbuf;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* row_token;
  const int32_t* uexp;
  Meta* meta;
  int H, I, EU;
  int stages;
  uint32_t stage_bytes;   // 2H + 2 pitch(H)
};

struct DownArgs {
  const int8_t* q;        // q_d
  const uint8_t* s;       // s_d
  const float* hbuf;
  __nv_bfloat16* out;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* row_token;
  const float* row_gate;
  const int32_t* uexp;
  Meta* meta;
  int H, I, T, EU;
  int stages;
  uint32_t stage_bytes;   // 2I + 2 pitch(I)
};

// sum_{i<16} q_i * x_i for 16 int8 codes (one uint4) and 16 floats.
__device__ __forceinline__ float dot16(const uint4 q, const float (&xv)[16]) {
  float c[16];
  i8x4_to_f32(q.x, c[0], c[1], c[2], c[3]);
  i8x4_to_f32(q.y, c[4], c[5], c[6], c[7]);
  i8x4_to_f32(q.z, c[8], c[9], c[10], c[11]);
  i8x4_to_f32(q.w, c[12], c[13], c[14], c[15]);
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    a0 = fmaf(c[i], xv[i], a0);
    a1 = fmaf(c[i + 1], xv[i + 1], a1);
  }
  return a0 + a1;
}

__device__ __forceinline__ void load_x16_bf16(const __nv_bfloat16* p, float (&xv)[16]) {
  uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
  bf16x2_to_f32(a.x, xv[0], xv[1]);
  bf16x2_to_f32(a.y, xv[2], xv[3]);
  bf16x2_to_f32(a.z, xv[4], xv[5]);
  bf16x2_to_f32(a.w, xv[6], xv[7]);
  bf16x2_to_f32(b.x, xv[8], xv[9]);
  bf16x2_to_f32(b.y, xv[10], xv[11]);
  bf16x2_to_f32(b.z, xv[12], xv[13]);
  bf16x2_to_f32(b.w, xv[14], xv[15]);
}

__device__ __forceinline__ void load_h16_f32(const float* p, float (&hv)[16]) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 v = __ldg(q + i);
    hv[4 * i] = v.x;
    hv[4 * i + 1] = v.y;
    hv[4 * i + 2] = v.z;
    hv[4 * i + 3] = v.w;
  }
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// This CTA's slice [lo, hi) of n units, balanced to within one unit.
__device__ __forceinline__ void cta_range(int64_t n, int64_t& lo, int64_t& hi) {
  lo = n * blockIdx.x / gridDim.x;
  hi = n * (blockIdx.x + 1) / gridDim.x;
}

// After a wait gave up at stage `from`, wait (each wait bounded) for every
// copy this warp still has in flight, so none lands in shared memory after the
// CTA has gone.
__device__ void drain_ring(uint64_t* bars, int stages, int64_t from, int64_t issued) {
  for (int64_t j = from; j < issued; ++j) mbar_wait(&bars[j % stages], (uint32_t)((j / stages) & 1));
}

// ------------------------------------------------------------- gate / up
__global__ void __launch_bounds__(kWarps * 32, 1) decode_gateup_kernel(GateUpArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t* ring = smem + (size_t)warp * a.stages * a.stage_bytes;
  const int H = a.H, I = a.I;
  const uint32_t pitch = (uint32_t)scale_pitch_bytes(H);
  if (lane == 0)
    for (int s = 0; s < a.stages; ++s) mbar_init(&bars[warp][s], 1);
  fence_mbar_init();
  __syncwarp();

  pdl_wait();  // routing of the previous kernel
  pdl_launch_dependents();
  const int n_unique = a.meta->n_unique;
  int64_t lo, hi;
  cta_range((int64_t)n_unique * I, lo, hi);
  // this warp's units: lo + warp, lo + warp + kWarps, ...
  const int64_t first = lo + warp;
  const int64_t n_mine = first < hi ? (hi - first + kWarps - 1) / kWarps : 0;

  auto issue = [&](int64_t j) {  // lane 0: stage j of this warp's sequence
    int64_t unit = first + j * kWarps;
    int u = (int)(unit / I), i = (int)(unit % I);
    int e = a.uexp[u];
    int64_t rg = (int64_t)e * 2 * I + gu_row_gate(i);
    int64_t ru = (int64_t)e * 2 * I + gu_row_up(i);
    uint8_t* st = ring + (size_t)(j % a.stages) * a.stage_bytes;
    uint64_t* bar = &bars[warp][j % a.stages];
    mbar_arrive_expect_tx(bar, a.stage_bytes);
    bulk_g2s(st, a.q + rg * H, H, bar);
    bulk_g2s(st + H, a.q + ru * H, H, bar);
    bulk_g2s(st + 2 * H, a.s + rg * pitch, pitch, bar);
    bulk_g2s(st + 2 * H + pitch, a.s + ru * pitch, pitch, bar);
  };

  int64_t issued = 0;
  if (lane == 0)
    for (; issued < n_mine && issued < a.stages; ++issued) issue(issued);
  issued = __shfl_sync(0xFFFFFFFFu, issued, 0);

  const int nseg = H / 16;
  for (int64_t j = 0; j < n_mine; ++j) {
    const int st_i = (int)(j % a.stages);
    if (!mbar_wait(&bars[warp][st_i], (uint32_t)((j / a.stages) & 1))) {
      if (lane == 0) {
        report(a.meta, kStatusTimeout);
        drain_ring(bars[warp], a.stages, j, issued);
      }
      return;
    }
    const uint8_t* st = ring + (size_t)st_i * a.stage_bytes;
    const int64_t unit = first + j * kWarps;
    const int u = (int)(unit / I), i = (int)(unit % I);
    const int e = a.uexp[u];
    const int n = a.counts[e], row0 = a.offsets[e];
    const uint16_t* sg = reinterpret_cast<const uint16_t*>(st + 2 * H);
    const uint16_t* su = reinterpret_cast<const uint16_t*>(st + 2 * H + pitch);
    for (int r = 0; r < n; ++r) {
      const int pos = row0 + r;
      const __nv_bfloat16* xrow = a.x + (int64_t)a.row_token[pos] * H;
      float accg = 0.f, accu = 0.f;
      for (int seg = lane; seg < nseg; seg += 32) {
        float xv[16];
        load_x16_bf16(xrow + seg * 16, xv);
        uint4 qg = *reinterpret_cast<const uint4*>(st + seg * 16);
        uint4 qu = *reinterpret_cast<const uint4*>(st + H + seg * 16);
        accg = fmaf(half_bits_to_f32(sg[seg >> 1]), dot16(qg, xv), accg);
        accu = fmaf(half_bits_to_f32(su[seg >> 1]), dot16(qu, xv), accu);
      }
      accg = warp_sum(accg);
      accu = warp_sum(accu);
      if (lane == 0) a.hbuf[(int64_t)pos * I + i] = silu(accg) * accu;
    }
    __syncwarp();
    if (lane == 0 && issued < n_mine) {
      fence_proxy_async_smem();
      issue(issued);
    }
    issued = __shfl_sync(0xFFFFFFFFu, issued < n_mine ? issued + 1 : issued, 0);
  }
}

// ------------------------------------------------------------- down + combine
constexpr int kDownRows = 2;

__global__ void __launch_bounds__(kWarps * 32, 1) decode_down_kernel(DownArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][16];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t* ring = smem + (size_t)warp * a.stages * a.stage_bytes;
  const int H = a.H, I = a.I;
  const uint32_t pitch = (uint32_t)scale_pitch_bytes(I);
  if (lane == 0)
    for (int s = 0; s < a.stages; ++s) mbar_init(&bars[warp][s], 1);
  fence_mbar_init();
  __syncwarp();

  pdl_wait();
  pdl_launch_dependents();
  const int n_unique = a.meta->n_unique;
  int64_t lo, hi;
  cta_range(H / kDownRows, lo, hi);
  const int64_t first = lo + warp;
  const int64_t n_units = first < hi ? (hi - first + kWarps - 1) / kWarps : 0;
  const int64_t n_stages = n_units * n_unique;  // (unit, expert) pairs, expert fastest

  auto issue = [&](int64_t j) {
    int64_t unit = first + (j / n_unique) * kWarps;
    int e = a.uexp[j % n_unique];
    int64_t row = (int64_t)e * H + unit * kDownRows;
    uint8_t* st = ring + (size_t)(j % a.stages) * a.stage_bytes;
    uint64_t* bar = &bars[warp][j % a.stages];
    mbar_arrive_expect_tx(bar, a.stage_bytes);
    bulk_g2s(st, a.q + row * I, kDownRows * I, bar);
    bulk_g2s(st + kDownRows * I, a.s + row * pitch, kDownRows * pitch, bar);
  };

  int64_t issued = 0;
  if (lane == 0)
    for (; issued < n_stages && issued < a.stages; ++issued) issue(issued);
  issued = __shfl_sync(0xFFFFFFFFu, issued, 0);

  const int nseg = I / 16;
  float acc[kDownRows];
#pragma unroll
  for (int r = 0; r < kDownRows; ++r) acc[r] = 0.f;
  for (int64_t j = 0; j < n_stages; ++j) {
    const int st_i = (int)(j % a.stages);
    if (!mbar_wait(&bars[warp][st_i], (uint32_t)((j / a.stages) & 1))) {
      if (lane == 0) {
        report(a.meta, kStatusTimeout);
        drain_ring(bars[warp], a.stages, j, issued);
      }
      return;
    }
    const uint8_t* st = ring + (size_t)st_i * a.stage_bytes;
    const int e = a.uexp[j % n_unique];
    const int n = a.counts[e], row0 = a.offsets[e];
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(st + kDownRows * I);
    for (int r = 0; r < n; ++r) {
      const int pos = row0 + r;
      const float* hrow = a.hbuf + (int64_t)pos * I;
      float d[kDownRows];
#pragma unroll
      for (int q = 0; q < kDownRows; ++q) d[q] = 0.f;
      for (int seg = lane; seg < nseg; seg += 32) {
        float hv[16];
        load_h16_f32(hrow + seg * 16, hv);
#pragma unroll
        for (int q = 0; q < kDownRows; ++q) {
          uint4 qq = *reinterpret_cast<const uint4*>(st + q * I + seg * 16);
          float sv = half_bits_to_f32(sc[q * (pitch / 2) + (seg >> 1)]);
          d[q] = fmaf(sv, dot16(qq, hv), d[q]);
        }
      }
      const float g = a.row_gate[pos];
      const int t = a.row_token[pos];
#pragma unroll
      for (int q = 0; q < kDownRows; ++q) {
        float v = warp_sum(d[q]);
        if (lane == t) acc[q] = fmaf(g, v, acc[q]);
      }
    }
    const bool unit_done = (j % n_unique) == n_unique - 1;
    if (unit_done) {
      const int64_t unit = first + (j / n_unique) * kWarps;
      if (lane < a.T) {
        __nv_bfloat162 v = __floats2bfloat162_rn(acc[0], acc[1]);
        *reinterpret_cast<__nv_bfloat162*>(a.out + (int64_t)lane * H + unit * kDownRows) = v;
      }
#pragma unroll
      for (int r = 0; r < kDownRows; ++r) acc[r] = 0.f;
    }
    __syncwarp();
    if (lane == 0 && issued < n_stages) {
      fence_proxy_async_smem();
      issue(issued);
    }
    issued = __shfl_sync(0xFFFFFFFFu, issued < n_stages ? issued + 1 : issued, 0);
  }
}

template <typename K, typename A>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, A args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

// Stages per warp so that the CTA's ring stays within ~200 KB.
int pick_stages(uint32_t stage_bytes, int max_stages) {
  int s = (int)((200u * 1024u) / (kWarps * stage_bytes));
  if (s > max_stages) s = max_stages;
  return s;
}

}  // namespace

cudaError_t configure_decode_kernels() {
  cudaError_t e = allow_max_dynamic_smem(decode_gateup_kernel);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(decode_down_kernel);
  return e;
}

cudaError_t launch_ffn_decode(Handle* h, const __nv_bfloat16* x, int T, __nv_bfloat16* out, cudaStream_t s) {
  const int H = h->cfg.H, I = h->cfg.I;
  cudaError_t err;
  {
    GateUpArgs a;
    a.q = h->q_gu;
    a.s = h->s_gu;
    a.x = x;
    a.hbuf = static_cast<float*>(h->hbuf);
    a.counts = h->counts;
    a.offsets = h->offsets;
    a.row_token = h->row_token;
    a.uexp = h->uexp;
    a.meta = h->meta;
    a.H = H;
    a.I = I;
    a.EU = h->EU;
    a.stage_bytes = (uint32_t)(2 * H + 2 * scale_pitch_bytes(H));
    a.stages = pick_stages(a.stage_bytes, 8);
    if (a.stages < 1) return cudaErrorInvalidConfiguration;
    size_t smem = (size_t)kWarps * a.stages * a.stage_bytes;
    int64_t max_units = (int64_t)std::min<int64_t>(h->EU, (int64_t)T * h->cfg.k + h->S) * I;
    int64_t grid = std::min<int64_t>(h->num_sms, (max_units + kWarps - 1) / kWarps);
    KernelTimer tm(h, FW_KERNEL_DECODE_GATEUP, s);
    err = launch_pdl(decode_gateup_kernel, dim3((unsigned)grid), dim3(kWarps * 32), smem, s, a);
    if (err != cudaSuccess) return err;
  }
  {
    DownArgs a;
    a.q = h->q_d;
    a.s = h->s_d;
    a.hbuf = static_cast<const float*>(h->hbuf);
    a.out = out;
    a.counts = h->counts;
    a.offsets = h->offsets;
    a.row_token = h->row_token;
    a.row_gate = h->row_gate;
    a.uexp = h->uexp;
    a.meta = h->meta;
    a.H = H;
    a.I = I;
    a.T = T;
    a.EU = h->EU;
    a.stage_bytes = (uint32_t)(kDownRows * I + kDownRows * scale_pitch_bytes(I));
    a.stages = pick_stages(a.stage_bytes, 16);
    size_t smem = (size_t)kWarps * a.stages * a.stage_bytes;
    int64_t units = H / kDownRows;
    int64_t grid = std::min<int64_t>(h->num_sms, (units + kWarps - 1) / kWarps);
    KernelTimer tm(h, FW_KERNEL_DECODE_DOWN, s);
    err = launch_pdl(decode_down_kernel, dim3((unsigned)grid), dim3(kWarps * 32), smem, s, a);
  }
  return err;
}

}  // namespace fw
