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

struct GateUpArgs {
  const int8_t* q;        // q_gu
  const uint8_t* s;       // s_gu
  const __nv_bfloat16* x;
  float* hbuf;
  const int32_t* row_token;
  const int4* uinfo;
  Meta* meta;
  int H, I, EU, T, rows;
  int stages;
  uint32_t stage_bytes;   // 2H + 2 pitch(H)
  int x_in_smem;          // x [T][H] bf16 staged in shared memory
};

struct DownArgs {
  const int8_t* q;        // q_d
  const uint8_t* s;       // s_d
  const float* hbuf;
  __nv_bfloat16* out;
  const int32_t* row_token;
  const float* row_gate;
  const int4* uinfo;
  Meta* meta;
  int H, I, T, EU, rows;
  int stages;
  uint32_t stage_bytes;   // I + pitch(I)
  int h_in_smem;          // hbuf [rows][I] fp32 staged in shared memory
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

__device__ __forceinline__ void unpack_x16(uint4 a, uint4 b, float (&xv)[16]) {
  bf16x2_to_f32(a.x, xv[0], xv[1]);
  bf16x2_to_f32(a.y, xv[2], xv[3]);
  bf16x2_to_f32(a.z, xv[4], xv[5]);
  bf16x2_to_f32(a.w, xv[6], xv[7]);
  bf16x2_to_f32(b.x, xv[8], xv[9]);
  bf16x2_to_f32(b.y, xv[10], xv[11]);
  bf16x2_to_f32(b.z, xv[12], xv[13]);
  bf16x2_to_f32(b.w, xv[14], xv[15]);
}

__device__ __forceinline__ void load_h16(const float* p, bool shared, float (&hv)[16]) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 v = shared ? q[i] : __ldg(q + i);
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

// The routing made by the router, copied once per CTA into shared memory:
// the table of experts with rows and, per grouped row, its token (and gate).
// All loads are independent: one round trip.
template <int NT>
__device__ __forceinline__ int load_routing(const Meta* meta, const int4* uinfo, int EU, const int32_t* row_token,
                                            const float* row_gate, int rows, int4* s_u, int* s_tok, float* s_gate) {
  const int n_unique = meta->n_unique;
  for (int i = threadIdx.x; i < EU; i += NT) s_u[i] = uinfo[i];
  for (int i = threadIdx.x; i < rows; i += NT) {
    s_tok[i] = row_token[i];
    if (s_gate) s_gate[i] = row_gate[i];
  }
  return n_unique;
}

constexpr int kMaxStages = 16;

// Shared memory carve-up shared by host and device: [uinfo][tokens][gates][act][rings].
struct DecodeSmem {
  uint32_t u_off, tok_off, gate_off, act_off, ring_off, total;
  __host__ __device__ DecodeSmem(int EU, int rows, uint32_t act_bytes, uint32_t ring_bytes) {
    u_off = 0;
    tok_off = (uint32_t)EU * 16;
    gate_off = tok_off + ((uint32_t)rows * 4 + 15) / 16 * 16;
    act_off = gate_off + ((uint32_t)rows * 4 + 15) / 16 * 16;
    ring_off = (act_off + act_bytes + 127) / 128 * 128;
    total = ring_off + ring_bytes;
  }
};

// ------------------------------------------------------------- gate / up
// Unit = (expert with rows, i): gate row i and up row i of that expert, streamed
// into this warp's ring; for each of the expert's rows (tokens) the warp forms
// g and u and writes h = SiLU(g) * u.
template <int W>
__global__ void __launch_bounds__(W * 32, 1) decode_gateup_kernel(GateUpArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[W][kMaxStages];
  __shared__ __align__(8) uint64_t xbar;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int H = a.H, I = a.I;
  const uint32_t pitch = (uint32_t)scale_pitch_bytes(H);
  DecodeSmem L(a.EU, a.rows, a.x_in_smem ? (uint32_t)a.T * H * 2 : 0, 0);
  int4* s_u = reinterpret_cast<int4*>(smem + L.u_off);
  int* s_tok = reinterpret_cast<int*>(smem + L.tok_off);
  const __nv_bfloat16* s_x = reinterpret_cast<const __nv_bfloat16*>(smem + L.act_off);
  uint8_t* ring = smem + L.ring_off + (size_t)warp * a.stages * a.stage_bytes;
  if (lane == 0)
    for (int s = 0; s < a.stages; ++s) mbar_init(&bars[warp][s], 1);
  if (threadIdx.x == 0) mbar_init(&xbar, 1);
  fence_mbar_init();

  pdl_wait();  // the router's results
  pdl_launch_dependents();
  if (threadIdx.x == 0 && a.x_in_smem) {
    mbar_arrive_expect_tx(&xbar, (uint32_t)a.T * H * 2);
    bulk_g2s(smem + L.act_off, a.x, (uint32_t)a.T * H * 2, &xbar);
  }
  const int n_unique = load_routing<W * 32>(a.meta, a.uinfo, a.EU, a.row_token, nullptr, a.rows, s_u, s_tok,
                                            nullptr);
  __syncthreads();
  int64_t lo, hi;
  cta_range((int64_t)n_unique * I, lo, hi);
  const int64_t first = lo + warp;
  const int64_t n_mine = first < hi ? (hi - first + W - 1) / W : 0;

  auto issue = [&](int64_t j) {  // lane 0: stage j of this warp's sequence
    int64_t unit = first + j * W;
    int u = (int)(unit / I), i = (int)(unit % I);
    int e = s_u[u].x;
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

  bool ok = true;
  if (a.x_in_smem) ok = mbar_wait(&xbar, 0);
  const int nseg = H / 16;
  for (int64_t j = 0; j < n_mine && ok; ++j) {
    const int st_i = (int)(j % a.stages);
    if (!mbar_wait(&bars[warp][st_i], (uint32_t)((j / a.stages) & 1))) {
      ok = false;
      if (lane == 0) drain_ring(bars[warp], a.stages, j, issued);
      break;
    }
    const uint8_t* st = ring + (size_t)st_i * a.stage_bytes;
    const int64_t unit = first + j * W;
    const int u = (int)(unit / I), i = (int)(unit % I);
    const int4 ui = s_u[u];
    const uint16_t* sg = reinterpret_cast<const uint16_t*>(st + 2 * H);
    const uint16_t* su = reinterpret_cast<const uint16_t*>(st + 2 * H + pitch);
    for (int r = 0; r < ui.z; ++r) {
      const int pos = ui.y + r;
      const int t = s_tok[pos];
      float accg = 0.f, accu = 0.f;
      for (int seg = lane; seg < nseg; seg += 32) {
        uint4 x0, x1;
        if (a.x_in_smem) {
          const uint4* xp = reinterpret_cast<const uint4*>(s_x + (size_t)t * H + seg * 16);
          x0 = xp[0];
          x1 = xp[1];
        } else {
          const uint4* xp = reinterpret_cast<const uint4*>(a.x + (size_t)t * H + seg * 16);
          x0 = __ldg(xp);
          x1 = __ldg(xp + 1);
        }
        float xv[16];
        unpack_x16(x0, x1, xv);
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
  if (!ok && lane == 0) report(a.meta, kStatusTimeout);
}

// ------------------------------------------------------------- down + combine
// Unit = one output row o: the warp walks every expert with rows in ascending
// id (the shared expert last), streaming row o of each W_down; lane t
// accumulates gate * (W_down h) for token t and writes out[t][o].
template <int W>
__global__ void __launch_bounds__(W * 32, 1) decode_down_kernel(DownArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[W][kMaxStages];
  __shared__ __align__(8) uint64_t hbar;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int H = a.H, I = a.I;
  const uint32_t pitch = (uint32_t)scale_pitch_bytes(I);
  const uint32_t h_bytes = (uint32_t)a.rows * I * 4;
  DecodeSmem L(a.EU, a.rows, a.h_in_smem ? h_bytes : 0, 0);
  int4* s_u = reinterpret_cast<int4*>(smem + L.u_off);
  int* s_tok = reinterpret_cast<int*>(smem + L.tok_off);
  float* s_gate = reinterpret_cast<float*>(smem + L.gate_off);
  const float* hsrc = a.h_in_smem ? reinterpret_cast<const float*>(smem + L.act_off) : a.hbuf;
  uint8_t* ring = smem + L.ring_off + (size_t)warp * a.stages * a.stage_bytes;
  if (lane == 0)
    for (int s = 0; s < a.stages; ++s) mbar_init(&bars[warp][s], 1);
  if (threadIdx.x == 0) mbar_init(&hbar, 1);
  fence_mbar_init();

  pdl_wait();  // h from the gate/up kernel
  pdl_launch_dependents();
  if (threadIdx.x == 0 && a.h_in_smem) {
    mbar_arrive_expect_tx(&hbar, h_bytes);
    bulk_g2s(smem + L.act_off, a.hbuf, h_bytes, &hbar);
  }
  const int n_unique = load_routing<W * 32>(a.meta, a.uinfo, a.EU, a.row_token, a.row_gate, a.rows, s_u, s_tok,
                                            s_gate);
  __syncthreads();
  int64_t lo, hi;
  cta_range(H, lo, hi);
  const int64_t first = lo + warp;
  const int64_t n_units = first < hi ? (hi - first + W - 1) / W : 0;
  const int64_t n_stages = n_units * n_unique;  // (unit, expert) pairs, expert fastest

  auto issue = [&](int64_t j) {
    int64_t o = first + (j / n_unique) * W;
    int e = s_u[j % n_unique].x;
    int64_t row = (int64_t)e * H + o;
    uint8_t* st = ring + (size_t)(j % a.stages) * a.stage_bytes;
    uint64_t* bar = &bars[warp][j % a.stages];
    mbar_arrive_expect_tx(bar, a.stage_bytes);
    bulk_g2s(st, a.q + row * I, I, bar);
    bulk_g2s(st + I, a.s + row * pitch, pitch, bar);
  };

  int64_t issued = 0;
  if (lane == 0)
    for (; issued < n_stages && issued < a.stages; ++issued) issue(issued);
  issued = __shfl_sync(0xFFFFFFFFu, issued, 0);

  bool ok = true;
  if (a.h_in_smem) ok = mbar_wait(&hbar, 0);
  const int nseg = I / 16;
  float acc = 0.f;
  for (int64_t j = 0; j < n_stages && ok; ++j) {
    const int st_i = (int)(j % a.stages);
    if (!mbar_wait(&bars[warp][st_i], (uint32_t)((j / a.stages) & 1))) {
      ok = false;
      if (lane == 0) drain_ring(bars[warp], a.stages, j, issued);
      break;
    }
    const uint8_t* st = ring + (size_t)st_i * a.stage_bytes;
    const int4 ui = s_u[j % n_unique];
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(st + I);
    for (int r = 0; r < ui.z; ++r) {
      const int pos = ui.y + r;
      const float* hrow = hsrc + (size_t)pos * I;
      float d = 0.f;
      for (int seg = lane; seg < nseg; seg += 32) {
        float hv[16];
        load_h16(hrow + seg * 16, a.h_in_smem != 0, hv);
        uint4 qq = *reinterpret_cast<const uint4*>(st + seg * 16);
        d = fmaf(half_bits_to_f32(sc[seg >> 1]), dot16(qq, hv), d);
      }
      d = warp_sum(d);
      if (lane == s_tok[pos]) acc = fmaf(s_gate[pos], d, acc);
    }
    if ((j % n_unique) == n_unique - 1) {  // all experts of this output row done
      const int64_t o = first + (j / n_unique) * W;
      if (lane < a.T) a.out[(int64_t)lane * H + o] = __float2bfloat16_rn(acc);
      acc = 0.f;
    }
    __syncwarp();
    if (lane == 0 && issued < n_stages) {
      fence_proxy_async_smem();
      issue(issued);
    }
    issued = __shfl_sync(0xFFFFFFFFu, issued < n_stages ? issued + 1 : issued, 0);
  }
  if (!ok && lane == 0) report(a.meta, kStatusTimeout);
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

int g_smem_optin = 0;  // usable dynamic shared memory per block (set at configure time)

// Warps per CTA and ring stages per warp for a stage size, given the bytes
// already taken; prefers 16 warps with at least 2 stages.
bool pick_shape(uint32_t stage_bytes, uint32_t fixed_bytes, int max_stages, int* warps, int* stages) {
  const int64_t budget = (int64_t)g_smem_optin - fixed_bytes - 1024;
  for (int W : {16, 8}) {
    int64_t s = budget / ((int64_t)W * stage_bytes);
    if (s > max_stages) s = max_stages;
    if (s >= 2 || (W == 8 && s >= 1)) {
      *warps = W;
      *stages = (int)s;
      return true;
    }
  }
  return false;
}

constexpr uint32_t kActSmemMax = 96 * 1024;  // x or h staged in shared memory up to this size

}  // namespace

cudaError_t configure_decode_kernels() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) g_smem_optin -= 4096;  // static barriers and slack
  if (e == cudaSuccess) e = allow_max_dynamic_smem(decode_gateup_kernel<16>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(decode_gateup_kernel<8>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(decode_down_kernel<16>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(decode_down_kernel<8>);
  return e;
}

cudaError_t launch_ffn_decode(Handle* h, const __nv_bfloat16* x, int T, __nv_bfloat16* out, cudaStream_t s) {
  const int H = h->cfg.H, I = h->cfg.I;
  const int rows = T * (h->cfg.k + h->S);
  cudaError_t err;
  {
    GateUpArgs a;
    a.q = h->q_gu;
    a.s = h->s_gu;
    a.x = x;
    a.hbuf = static_cast<float*>(h->hbuf);
    a.row_token = h->row_token;
    a.uinfo = h->uinfo;
    a.meta = h->meta;
    a.H = H;
    a.I = I;
    a.EU = h->EU;
    a.T = T;
    a.rows = rows;
    a.stage_bytes = (uint32_t)(2 * H + 2 * scale_pitch_bytes(H));
    a.x_in_smem = (uint32_t)T * H * 2 <= kActSmemMax;
    DecodeSmem L(h->EU, rows, a.x_in_smem ? (uint32_t)T * H * 2 : 0, 0);
    int W = 0;
    if (!pick_shape(a.stage_bytes, L.ring_off, kMaxStages, &W, &a.stages)) return cudaErrorInvalidConfiguration;
    size_t smem = L.ring_off + (size_t)W * a.stages * a.stage_bytes;
    int64_t max_units = (int64_t)std::min<int64_t>(h->EU, (int64_t)T * h->cfg.k + h->S) * I;
    int64_t grid = std::min<int64_t>(h->num_sms, (max_units + W - 1) / W);
    KernelTimer tm(h, FW_KERNEL_DECODE_GATEUP, s);
    err = W == 16 ? launch_pdl(decode_gateup_kernel<16>, dim3((unsigned)grid), dim3(16 * 32), smem, s, a)
                  : launch_pdl(decode_gateup_kernel<8>, dim3((unsigned)grid), dim3(8 * 32), smem, s, a);
    if (err != cudaSuccess) return err;
  }
  {
    DownArgs a;
    a.q = h->q_d;
    a.s = h->s_d;
    a.hbuf = static_cast<const float*>(h->hbuf);
    a.out = out;
    a.row_token = h->row_token;
    a.row_gate = h->row_gate;
    a.uinfo = h->uinfo;
    a.meta = h->meta;
    a.H = H;
    a.I = I;
    a.T = T;
    a.EU = h->EU;
    a.rows = rows;
    a.stage_bytes = (uint32_t)(I + scale_pitch_bytes(I));
    const uint32_t h_bytes = (uint32_t)rows * I * 4;
    a.h_in_smem = h_bytes <= kActSmemMax;
    DecodeSmem L(h->EU, rows, a.h_in_smem ? h_bytes : 0, 0);
    int W = 0;
    if (!pick_shape(a.stage_bytes, L.ring_off, kMaxStages, &W, &a.stages)) return cudaErrorInvalidConfiguration;
    size_t smem = L.ring_off + (size_t)W * a.stages * a.stage_bytes;
    int64_t grid = std::min<int64_t>(h->num_sms, H);
    KernelTimer tm(h, FW_KERNEL_DECODE_DOWN, s);
    err = W == 16 ? launch_pdl(decode_down_kernel<16>, dim3((unsigned)grid), dim3(16 * 32), smem, s, a)
                  : launch_pdl(decode_down_kernel<8>, dim3((unsigned)grid), dim3(8 * 32), smem, s, a);
  }
  return err;
}

}  // namespace fw
