// Decode path (T <= 16): the experts as grouped, HBM-bound GEMVs.
//
// The pages' runtime runs routed experts through grouped GPU kernels per
// quantisation format, Q8_0 among them (Flyweight README, §Quantization), and
// fuses the gate and up projections so they share one activation load (its
// CPU expert kernels, §Current limitations). Here every selected expert's Q8_0
// rows are streamed from HBM exactly once per call, in large bulk asynchronous
// copies (many contiguous rows per copy) into a shared-memory ring fed by one
// producer warp, and dequantised in registers by eight consumer warps.
//
// Both kernels first rebuild the batch's routing from the router logits in
// shared memory (top-k, gates and grouping are deterministic, so every CTA
// gets the same answer) instead of waiting for a published table.
//
//   gate/up kernel: unit = (expert, i): gate row i and up row i share the
//     x loads; h = SiLU(g) * u for each of the expert's tokens -> hbuf (fp32).
//     With `publish`, CTA 0 also writes the routing outputs.
//   down kernel: each CTA owns a block of output rows; it routes and starts
//     streaming W_down rows *before* waiting for the gate/up kernel
//     (programmatic dependent launch), then visits the touched experts in
//     ascending id (shared last): lane t accumulates gate * (W_down h) for
//     token t, so the combine is fused and its order fixed (no atomics).
#include <algorithm>

#include "routing.cuh"

namespace fw {
namespace {

using namespace dev;

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kProducer = kConsumerWarps;            // warp index of the producer
constexpr int kMaxStages = 16;
constexpr int kDownRowBlock = 16;                    // output rows per down stage
constexpr int kMaxDownBlocks = 4;                    // row blocks a CTA may own

struct GateUpArgs {
  const int8_t* q;        // q_gu
  const uint8_t* s;       // s_gu
  const __nv_bfloat16* x;
  const float* logits;
  float* hbuf;
  RoutingOut out;         // routing outputs (publish only; meta always)
  int H, I, E, k, S, T;
  int publish;
  int stages;
  int units_per_stage;    // consecutive i of one expert per stage (divides 64)
  uint32_t stage_bytes;
  int x_in_smem;
};

struct DownArgs {
  const int8_t* q;        // q_d
  const uint8_t* s;       // s_d
  const float* logits;
  const float* hbuf;
  __nv_bfloat16* out;
  Meta* meta;
  int H, I, E, k, S, T;
  int stages;
  uint32_t stage_bytes;   // kDownRowBlock * (I + pitch(I))
  int h_in_smem;
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

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Dynamic shared memory: [activation (x or h)][ring], 128-byte aligned.
__host__ __device__ inline uint32_t ring_offset(uint32_t act_bytes) { return (act_bytes + 127) / 128 * 128; }

// ------------------------------------------------------------- gate / up
// CTA c takes units [lo, hi) of the (expert with rows) x I unit space; a stage
// is up to R = units_per_stage consecutive units of one expert (R divides 64,
// so a stage never crosses a 64-row gate/up group): 4 bulk copies (gate codes,
// up codes, gate scales, up scales). Unit g goes to consumer warp g % 8,
// which arrives on its stage's empty barrier with a weight chosen so that each
// stage's arrivals sum to R.
__global__ void __launch_bounds__(kThreads, 1) decode_gateup_kernel(GateUpArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], xbar;
  __shared__ SmemRouting r;
  __shared__ int s_fail;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, I = a.I, T = a.T;
  const uint32_t pitch = (uint32_t)scale_pitch_bytes(H);
  const uint32_t x_bytes = a.x_in_smem ? (uint32_t)T * H * 2 : 0;
  const __nv_bfloat16* s_x = reinterpret_cast<const __nv_bfloat16*>(smem);
  uint8_t* ring = smem + ring_offset(x_bytes);
  const int R = a.units_per_stage;
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], R);
    }
    mbar_init(&xbar, 1);
    s_fail = 0;
    fence_mbar_init();
  }
  pdl_wait();  // the router's logits
  if (tid == 0 && x_bytes) {
    mbar_arrive_expect_tx(&xbar, x_bytes);
    bulk_g2s(smem, a.x, x_bytes, &xbar);
  }
  route_in_smem<kThreads>(a.logits, T, a.E, a.k, a.S, r);
  pdl_launch_dependents();
  if (a.publish && blockIdx.x == 0) publish_routing<kThreads>(r, T, a.E, a.k, a.S, a.out);

  const int64_t n_units = (int64_t)r.n_unique * I;
  const int64_t lo = n_units * blockIdx.x / gridDim.x, hi = n_units * (blockIdx.x + 1) / gridDim.x;
  const int64_t b0 = lo / R;  // stage j covers [max(lo, R(b0+j)), min(hi, R(b0+j+1)))
  const int64_t n_stages = hi > lo ? (hi + R - 1) / R - b0 : 0;

  if (warp == kProducer) {
    if (lane == 0) {
      int64_t j = 0;
      for (; j < n_stages; ++j) {
        const int st = (int)(j % a.stages);
        if (j >= a.stages && !mbar_wait(&empty[st], (uint32_t)(((j / a.stages) - 1) & 1))) {
          s_fail = 1;
          break;
        }
        const int64_t u0 = std::max<int64_t>(lo, (b0 + j) * R), u1 = std::min<int64_t>(hi, (b0 + j + 1) * R);
        const int n = (int)(u1 - u0);
        const int e = r.u[u0 / I].x, i0 = (int)(u0 % I);
        const int64_t rg = (int64_t)e * 2 * I + gu_row_gate(i0), ru = (int64_t)e * 2 * I + gu_row_up(i0);
        uint8_t* sb = ring + (size_t)st * a.stage_bytes;
        const uint32_t qb = (uint32_t)n * H, sbb = (uint32_t)n * pitch;
        mbar_arrive_expect_tx(&full[st], 2 * qb + 2 * sbb);
        bulk_g2s(sb, a.q + rg * H, qb, &full[st]);
        bulk_g2s(sb + (size_t)R * H, a.q + ru * H, qb, &full[st]);
        bulk_g2s(sb + (size_t)2 * R * H, a.s + rg * pitch, sbb, &full[st]);
        bulk_g2s(sb + (size_t)2 * R * H + (size_t)R * pitch, a.s + ru * pitch, sbb, &full[st]);
      }
      // every copy issued has landed before the CTA may leave
      for (int64_t q = std::max<int64_t>(0, j - a.stages); q < j; ++q)
        mbar_wait(&full[q % a.stages], (uint32_t)((q / a.stages) & 1));
    }
  } else {
    bool ok = !x_bytes || mbar_wait(&xbar, 0);
    const int nseg = H / 16;
    for (int64_t g = lo + warp; g < hi && ok; g += kConsumerWarps) {
      const int64_t j = g / R - b0;
      const int st = (int)(j % a.stages);
      if (!mbar_wait(&full[st], (uint32_t)((j / a.stages) & 1))) {
        ok = false;
        break;
      }
      const int64_t u0 = std::max<int64_t>(lo, (b0 + j) * R), u1 = std::min<int64_t>(hi, (b0 + j + 1) * R);
      const size_t off = (size_t)(g - u0);
      const uint8_t* sb = ring + (size_t)st * a.stage_bytes;
      const uint8_t* qg_row = sb + off * H;
      const uint8_t* qu_row = sb + (size_t)R * H + off * H;
      const uint16_t* sg = reinterpret_cast<const uint16_t*>(sb + (size_t)2 * R * H + off * pitch);
      const uint16_t* su = reinterpret_cast<const uint16_t*>(sb + (size_t)2 * R * H + (size_t)R * pitch + off * pitch);
      const int4 ui = r.u[g / I];
      const int i = (int)(g % I);
      for (int rr = 0; rr < ui.z; ++rr) {
        const int pos = ui.y + rr;
        const int t = r.tok[pos];
        float accg = 0.f, accu = 0.f;
        for (int seg = lane; seg < nseg; seg += 32) {
          uint4 x0, x1;
          if (x_bytes) {
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
          const uint4 qg = *reinterpret_cast<const uint4*>(qg_row + seg * 16);
          const uint4 qu = *reinterpret_cast<const uint4*>(qu_row + seg * 16);
          accg = fmaf(half_bits_to_f32(sg[seg >> 1]), dot16(qg, xv), accg);
          accu = fmaf(half_bits_to_f32(su[seg >> 1]), dot16(qu, xv), accu);
        }
        accg = warp_sum(accg);
        accu = warp_sum(accu);
        if (lane == 0) a.hbuf[(int64_t)pos * I + i] = silu(accg) * accu;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt(&empty[st], g == u0 ? (uint32_t)(R - (u1 - u0) + 1) : 1u);
    }
    if (!ok && lane == 0) s_fail = 1;
  }
  __syncthreads();
  if (tid == 0 && s_fail) report(a.out.meta, kStatusTimeout);
}

// ------------------------------------------------------------- down + combine
// CTA c owns output rows [o0, o1) in blocks of up to 16; a stage is one block
// of rows of one touched expert (2 bulk copies: codes, scales). Consumer warp
// w owns rows w and w + 8 of every block and keeps their per-token sums in
// registers (lane t: token t) across all experts.
__global__ void __launch_bounds__(kThreads, 1) decode_down_kernel(DownArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], hbar;
  __shared__ SmemRouting r;
  __shared__ int s_fail;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, I = a.I, T = a.T;
  const uint32_t pitch = (uint32_t)scale_pitch_bytes(I);
  const int rows_all = T * (a.k + a.S);
  const uint32_t h_bytes = a.h_in_smem ? (uint32_t)rows_all * I * 4 : 0;
  const float* hsrc = h_bytes ? reinterpret_cast<const float*>(smem) : a.hbuf;
  uint8_t* ring = smem + ring_offset(h_bytes);
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(&hbar, 1);
    s_fail = 0;
    fence_mbar_init();
  }
  // The router finished before the gate/up kernel let this grid start, so its
  // logits are final: route and start streaming W_down before h exists.
  route_in_smem<kThreads>(a.logits, T, a.E, a.k, a.S, r);
  const int o0 = (int)((int64_t)H * blockIdx.x / gridDim.x), o1 = (int)((int64_t)H * (blockIdx.x + 1) / gridDim.x);
  const int n_blocks = (o1 - o0 + kDownRowBlock - 1) / kDownRowBlock;
  const int nU = r.n_unique;
  const int64_t n_stages = (int64_t)nU * n_blocks;  // (expert, block), block fastest

  if (warp == kProducer) {
    if (lane == 0) {
      int64_t j = 0;
      for (; j < n_stages; ++j) {
        const int st = (int)(j % a.stages);
        if (j >= a.stages && !mbar_wait(&empty[st], (uint32_t)(((j / a.stages) - 1) & 1))) {
          s_fail = 1;
          break;
        }
        const int e = r.u[j / n_blocks].x, blk = (int)(j % n_blocks);
        const int r0 = o0 + blk * kDownRowBlock, nr = ::min(kDownRowBlock + 0, o1 - r0);
        const int64_t row = (int64_t)e * H + r0;
        uint8_t* sb = ring + (size_t)st * a.stage_bytes;
        mbar_arrive_expect_tx(&full[st], (uint32_t)nr * (I + pitch));
        bulk_g2s(sb, a.q + row * I, (uint32_t)nr * I, &full[st]);
        bulk_g2s(sb + (size_t)kDownRowBlock * I, a.s + row * pitch, (uint32_t)nr * pitch, &full[st]);
      }
      for (int64_t q = std::max<int64_t>(0, j - a.stages); q < j; ++q)
        mbar_wait(&full[q % a.stages], (uint32_t)((q / a.stages) & 1));
    }
  }
  pdl_wait();  // h from the gate/up kernel
  pdl_launch_dependents();
  if (tid == 0 && h_bytes) {
    mbar_arrive_expect_tx(&hbar, h_bytes);
    bulk_g2s(smem, a.hbuf, h_bytes, &hbar);
  }
  if (warp != kProducer) {
    bool ok = !h_bytes || mbar_wait(&hbar, 0);
    const int nseg = I / 16;
    float acc[kMaxDownBlocks][2];
#pragma unroll
    for (int b = 0; b < kMaxDownBlocks; ++b) acc[b][0] = acc[b][1] = 0.f;
    for (int64_t j = 0; j < n_stages && ok; ++j) {
      const int st = (int)(j % a.stages);
      if (!mbar_wait(&full[st], (uint32_t)((j / a.stages) & 1))) {
        ok = false;
        break;
      }
      const int4 ui = r.u[j / n_blocks];
      const int blk = (int)(j % n_blocks);
      const int nr = ::min(kDownRowBlock + 0, o1 - (o0 + blk * kDownRowBlock));
      const uint8_t* sb = ring + (size_t)st * a.stage_bytes;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int rr = warp + q * kConsumerWarps;
        if (rr >= nr) continue;
        const uint8_t* qrow = sb + (size_t)rr * I;
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(sb + (size_t)kDownRowBlock * I + (size_t)rr * pitch);
        for (int m = 0; m < ui.z; ++m) {
          const int pos = ui.y + m;
          const float* hrow = hsrc + (size_t)pos * I;
          float d = 0.f;
          for (int seg = lane; seg < nseg; seg += 32) {
            float hv[16];
            load_h16(hrow + seg * 16, h_bytes != 0, hv);
            const uint4 qq = *reinterpret_cast<const uint4*>(qrow + seg * 16);
            d = fmaf(half_bits_to_f32(sc[seg >> 1]), dot16(qq, hv), d);
          }
          d = warp_sum(d);
#pragma unroll
          for (int b = 0; b < kMaxDownBlocks; ++b)
            if (b == blk && lane == r.tok[pos]) acc[b][q] = fmaf(r.rg[pos], d, acc[b][q]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (ok && lane < T) {
#pragma unroll
      for (int b = 0; b < kMaxDownBlocks; ++b) {
        if (b >= n_blocks) break;
        const int r0 = o0 + b * kDownRowBlock, nr = ::min(kDownRowBlock + 0, o1 - r0);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int rr = warp + q * kConsumerWarps;
          if (rr < nr) a.out[(int64_t)lane * H + r0 + rr] = __float2bfloat16_rn(acc[b][q]);
        }
      }
    }
    if (!ok && lane == 0) s_fail = 1;
  }
  __syncthreads();
  if (tid == 0 && s_fail) report(a.meta, kStatusTimeout);
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

// The gate/up and down CTAs are sized to fit on one SM together (so the down
// kernel can start streaming while gate/up runs): each takes at most this
// much dynamic shared memory.
constexpr uint32_t kDynSmemEach = 96 * 1024;
constexpr uint32_t kActSmemMax = 32 * 1024;  // x or h staged in shared memory up to this size

}  // namespace

cudaError_t configure_decode_kernels() {
  cudaError_t e = allow_max_dynamic_smem(decode_gateup_kernel);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(decode_down_kernel);
  return e;
}

cudaError_t launch_ffn_decode(Handle* h, const __nv_bfloat16* x, int T, __nv_bfloat16* out, bool publish,
                              int32_t* ids_out, float* gates_out, cudaStream_t s) {
  const int H = h->cfg.H, I = h->cfg.I, k = h->cfg.k, S = h->S;
  const int rows = T * (k + S);
  if ((H + h->num_sms - 1) / h->num_sms > kDownRowBlock * kMaxDownBlocks) return cudaErrorNotSupported;
  cudaError_t err;
  {
    GateUpArgs a;
    a.q = h->q_gu;
    a.s = h->s_gu;
    a.x = x;
    a.logits = h->logits;
    a.hbuf = static_cast<float*>(h->hbuf);
    a.out = RoutingOut{ids_out, gates_out, h->ids,      h->gates,    h->counts, h->offsets,
                       h->perm, h->inv,    h->row_token, h->row_gate, h->uinfo,  h->meta};
    a.H = H;
    a.I = I;
    a.E = h->cfg.E;
    a.k = k;
    a.S = S;
    a.T = T;
    a.publish = publish ? 1 : 0;
    const uint32_t x_bytes = (uint32_t)T * H * 2;
    a.x_in_smem = x_bytes <= kActSmemMax;
    const uint32_t act = a.x_in_smem ? x_bytes : 0;
    const uint32_t unit_bytes = (uint32_t)(2 * H + 2 * scale_pitch_bytes(H));
    int R = 8;
    while (R > 1 && (uint64_t)R * unit_bytes * 3 > kDynSmemEach - ring_offset(act)) R /= 2;
    a.units_per_stage = R;
    a.stage_bytes = (uint32_t)R * unit_bytes;
    const uint32_t ring_off = ring_offset(act);
    a.stages = (int)std::min<int64_t>(kMaxStages, (kDynSmemEach - ring_off) / a.stage_bytes);
    if (a.stages < 2) return cudaErrorInvalidConfiguration;
    size_t smem = ring_off + (size_t)a.stages * a.stage_bytes;
    KernelTimer tm(h, FW_KERNEL_DECODE_GATEUP, s);
    err = launch_pdl(decode_gateup_kernel, dim3((unsigned)h->num_sms), dim3(kThreads), smem, s, a);
    if (err != cudaSuccess) return err;
  }
  {
    DownArgs a;
    a.q = h->q_d;
    a.s = h->s_d;
    a.logits = h->logits;
    a.hbuf = static_cast<const float*>(h->hbuf);
    a.out = out;
    a.meta = h->meta;
    a.H = H;
    a.I = I;
    a.E = h->cfg.E;
    a.k = k;
    a.S = S;
    a.T = T;
    const uint32_t h_bytes = (uint32_t)rows * I * 4;
    a.h_in_smem = h_bytes <= kActSmemMax;
    a.stage_bytes = (uint32_t)(kDownRowBlock * (I + scale_pitch_bytes(I)));
    const uint32_t ring_off = ring_offset(a.h_in_smem ? h_bytes : 0);
    a.stages = (int)std::min<int64_t>(kMaxStages, (kDynSmemEach - ring_off) / a.stage_bytes);
    if (a.stages < 2) return cudaErrorInvalidConfiguration;
    size_t smem = ring_off + (size_t)a.stages * a.stage_bytes;
    KernelTimer tm(h, FW_KERNEL_DECODE_DOWN, s);
    err = launch_pdl(decode_down_kernel, dim3((unsigned)std::min(h->num_sms, H)), dim3(kThreads), smem, s, a);
  }
  return err;
}

}  // namespace fw
