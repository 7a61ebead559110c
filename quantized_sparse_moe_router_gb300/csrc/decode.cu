// Decode path (T <= 16): the experts of one call as one fused, HBM-bound
// kernel: gate/up, SiLU, down and the gate-weighted combine.
//
// The pages' runtime runs routed experts through grouped GPU kernels per
// quantisation format, Q8_0 among them (Flyweight README, §Quantization), and
// fuses the gate and up projections so they share one activation load (its
// CPU expert kernels, §Current limitations). Here every selected expert's
// Q8_0 bytes are streamed from HBM exactly once per call, in large bulk
// asynchronous copies into a shared-memory ring fed by one producer warp.
//
// The work is cut along I into chunks of 16 units of one expert: the chunk's
// 16 gate and 16 up rows, and the matching 16 columns of its down matrix
// (split-K over I). One persistent CTA per SM takes a contiguous range of
// chunks and, for each, computes h = SiLU(W_gate x) * (W_up x) for the
// chunk's units and then gate * W_down[:, chunk] h into a partial output of
// the CTA. So the down projection streams alongside gate/up, and the one
// grid-wide wait left is for the partial outputs: after it each CTA sums its
// rows of them over the CTAs in a fixed order (deterministic, no atomics).
//
// Gate/up dot products run on integer dot-product instructions: each token's
// x is held, per 16-element segment, as a 16-bit fixed-point number scaled to
// the segment's largest exponent (exact for every element within 2^7 of the
// segment's largest; smaller ones are rounded at 2^-15 of it), split into a
// signed high and an unsigned low byte plane; the Q8_0 codes (offset binary)
// multiply both planes with dp4a, and one fp32 multiply-add per segment
// applies the weight scale and the segment's power of two. The down
// projection multiplies fp32 h by the exactly dequantised codes in fp32.
//
// One CTA per SM, all resident (see launch()):
//   0. x -> fixed-point planes in shared memory (before the router finishes);
//   1. after the router's grid completes (programmatic dependent launch), the
//      batch's routing rebuilt from the logits in shared memory
//      (deterministic, so every CTA agrees); CTA 0 publishes it;
//   2. the CTA's chunks: gate/up stages -> h (shared memory), then down
//      stages -> the CTA's partial output (fp32: shared memory for one token,
//      registers for several);
//   3. partial outputs to global memory, grid-wide arrival and bounded wait;
//   4. each CTA's output rows summed over the CTAs' partials, bf16.
#include <algorithm>
#include <cstdio>

#include "routing.cuh"

namespace fw {
namespace {

using namespace dev;

constexpr int kCW = 16;                    // consumer warps
constexpr int kCT = kCW * 32;              // consumer threads
constexpr int kThreads = kCT + 32;         // + one producer warp
constexpr int kProducer = kCW;
constexpr int kMaxStages = 16;
constexpr int kChunk = 16;                 // units of I per chunk (one 16-byte segment of a down row)
constexpr int kRowsMulti = 4;              // several tokens: down rows per consumer thread (H <= 2048)
constexpr int kMaxHMulti = kRowsMulti * kCT;
constexpr int kMaxHOne = 16384;            // one token: the partial output row fits in shared memory
constexpr int kDnRowsMax = 2048;           // down rows per stage at most
constexpr uint32_t kConsumerBarrier = 1;   // named barrier of the 16 consumer warps
constexpr uint32_t kStageTarget = 36 * 1024;
constexpr int kRedBatch = 10;              // partial loads in flight per lane in the final sums
constexpr int kMaxGrid = 256;              // CTAs (one per SM) the per-CTA token masks have room for

struct DecodeArgs {
  const uint8_t* q_gu;   // [EU][2I] rows of row_bytes(H): codes + 128, then binary16 scales
  const uint8_t* q_dc;   // [EU][I/16][H][16] down codes (+ 128) by 16-column groups
  const uint16_t* st_d;  // [EU][I/32][H] down scales
  const __nv_bfloat16* x;
  const float* logits;
  float* partial;        // [grid][T][H] fp32 partial outputs
  __nv_bfloat16* out;
  RoutingOut ro;
  Meta* meta;
  int H, I, E, k, S, T;
  int publish;
  int R;                 // gate/up units per stage (even, divides kChunk)
  int Dr;                // down rows per stage (multiple of 16)
  uint32_t stage_bytes;
  int stages;
  uint32_t off_info, off_acc, off_h, off_ring;  // dynamic shared memory layout (bytes)
  uint32_t grid_extra;   // arrivals the grid wait expects beyond the grid (0; > 0 only to test the bound)
  uint64_t grid_wait_ns; // bound of the grid-wide wait
};

// ------------------------------------------------------------- helpers
typedef unsigned long long f2;

__device__ __forceinline__ f2 f2_pack(float a, float b) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ f2 f2_pack_bits(uint32_t a, uint32_t b) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float f2_hsum(f2 v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return a + b;
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Four offset-binary codes of a word times four h values (two pairs), added
// to a pair accumulator: the byte permute makes the float 2^23 + q + 128 and
// one packed subtraction leaves q exactly.
__device__ __forceinline__ f2 dot4(uint32_t w, f2 x01, f2 x23, f2 acc) {
  const f2 bias = f2_pack(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
  const f2 m01 = f2_pack_bits(__byte_perm(w, 0x4B000000u, 0x7650), __byte_perm(w, 0x4B000000u, 0x7651));
  const f2 m23 = f2_pack_bits(__byte_perm(w, 0x4B000000u, 0x7652), __byte_perm(w, 0x4B000000u, 0x7653));
  acc = f2_fma(f2_add(m01, bias), x01, acc);
  return f2_fma(f2_add(m23, bias), x23, acc);
}

// sum_{i<16} q_i h_i for one 16-code segment; h as 8 pairs.
__device__ __forceinline__ float dot16(const uint4 q, const f2 (&h)[8]) {
  f2 a = dot4(q.x, h[0], h[1], 0ull);
  f2 b = dot4(q.y, h[2], h[3], 0ull);
  a = dot4(q.z, h[4], h[5], a);
  b = dot4(q.w, h[6], h[7], b);
  return f2_hsum(f2_add(a, b));
}

// The same with h read from shared memory (a broadcast) one pair of words at
// a time, so that few registers hold h.
__device__ __forceinline__ float dot16_smem(const uint4 q, const float* h) {
  const float4* hp = reinterpret_cast<const float4*>(h);
  float4 v0 = hp[0], v1 = hp[1];
  f2 a = dot4(q.x, f2_pack(v0.x, v0.y), f2_pack(v0.z, v0.w), 0ull);
  f2 b = dot4(q.y, f2_pack(v1.x, v1.y), f2_pack(v1.z, v1.w), 0ull);
  v0 = hp[2];
  v1 = hp[3];
  a = dot4(q.z, f2_pack(v0.x, v0.y), f2_pack(v0.z, v0.w), a);
  b = dot4(q.w, f2_pack(v1.x, v1.y), f2_pack(v1.z, v1.w), b);
  return f2_hsum(f2_add(a, b));
}

__device__ __forceinline__ void load_h16(const float* p, f2 (&h)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = reinterpret_cast<const float4*>(p)[i];
    h[2 * i] = f2_pack(v.x, v.y);
    h[2 * i + 1] = f2_pack(v.z, v.w);
  }
}

// Integer dot products of four code bytes (unsigned, q + 128) with four
// signed / unsigned activation bytes, added to c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// sum_i (q_i + 128) * xf_i over a 16-code segment, xf = 256 hi + lo.
__device__ __forceinline__ int seg_dot_i(const uint4 q, const uint4 hi, const uint4 lo) {
  int sh = dp4a_us(q.x, hi.x, 0);
  uint32_t sl = dp4a_uu(q.x, lo.x, 0u);
  sh = dp4a_us(q.y, hi.y, sh);
  sl = dp4a_uu(q.y, lo.y, sl);
  sh = dp4a_us(q.z, hi.z, sh);
  sl = dp4a_uu(q.z, lo.z, sl);
  sh = dp4a_us(q.w, hi.w, sh);
  sl = dp4a_uu(q.w, lo.w, sl);
  return sh * 256 + (int)sl;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"r"(kConsumerBarrier), "r"(kCT) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__host__ __device__ inline uint32_t align128(uint32_t v) { return (v + 127) / 128 * 128; }

// One 16-element segment of bf16 x -> 16-bit fixed point at the segment's
// largest exponent: hi/lo byte planes, the power of two that undoes the
// scaling, and 128 * sum(xf) (the codes are stored as q + 128). Segments whose
// largest magnitude is below 2^-112 count as zero.
__device__ __forceinline__ void x_segment_to_planes(const uint4 a, const uint4 b, uint4& hi, uint4& lo, int2& info) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t emax = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) emax = max(emax, max((w[i] >> 7) & 0xFFu, (w[i] >> 23) & 0xFFu));
  if (emax < 15u) {
    hi = lo = make_uint4(0u, 0u, 0u, 0u);
    info = make_int2(0, 0);
    return;
  }
  const float mult = __uint_as_float((268u - emax) << 23);  // 2^(14 - e), e = emax - 127
  int xf[16];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    xf[2 * i] = __float2int_rn(__uint_as_float(w[i] << 16) * mult);
    xf[2 * i + 1] = __float2int_rn(__uint_as_float(w[i] & 0xFFFF0000u) * mult);
    sum += xf[2 * i] + xf[2 * i + 1];
  }
  uint32_t h4[4], l4[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    h4[j] = 0u;
    l4[j] = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      h4[j] |= ((uint32_t)(xf[4 * j + i] >> 8) & 0xFFu) << (8 * i);
      l4[j] |= ((uint32_t)xf[4 * j + i] & 0xFFu) << (8 * i);
    }
  }
  hi = make_uint4(h4[0], h4[1], h4[2], h4[3]);
  lo = make_uint4(l4[0], l4[1], l4[2], l4[3]);
  info = make_int2((int)((emax - 14u) << 23), 128 * sum);  // float bits of 2^(e - 14), offset term
}

// ------------------------------------------------------------- the kernel
// kMulti: several tokens (T <= 16, H <= 2048; partial output in registers);
// otherwise one token (partial output in shared memory).
template <bool kMulti>
__global__ void __launch_bounds__(kThreads, 1) decode_experts_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages];
  __shared__ SmemRouting r;
  __shared__ uint32_t s_emask[kMaxE + 1];  // per touched expert (ascending): its tokens
  __shared__ uint32_t s_pm[kMaxGrid];       // per CTA: the tokens its partial output covers
  __shared__ volatile int s_abort;  // a consumer gave up a wait: the others stop waiting too
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, I = a.I, T = kMulti ? a.T : 1, R = a.R, Dr = a.Dr;
  const int nseg = H / 16;
  const uint32_t rb_h = (uint32_t)row_bytes(H);
  uint8_t* xhi = smem;                                              // [T][H] int8
  uint8_t* xlo = smem + (size_t)T * H;                              // [T][H] uint8
  int2* xinfo = reinterpret_cast<int2*>(smem + a.off_info);         // [T][H/16]
  float* acc_s = reinterpret_cast<float*>(smem + a.off_acc);        // [H] (one token)
  float* hbuf = reinterpret_cast<float*>(smem + a.off_h);           // [2][T][16]
  uint8_t* ring = smem + a.off_ring;
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp != kProducer) {
    // x was written before the router kernel started (that launch waits for
    // the whole stream): staged while the router still runs
    for (int c = tid; c < T * nseg; c += kCT) {
      const uint4* src = reinterpret_cast<const uint4*>(a.x) + 2 * c;
      uint4 hi, lo;
      int2 info;
      x_segment_to_planes(__ldg(src), __ldg(src + 1), hi, lo, info);
      reinterpret_cast<uint4*>(xhi)[c] = hi;
      reinterpret_cast<uint4*>(xlo)[c] = lo;
      xinfo[c] = info;
    }
    if (!kMulti)
      for (int o = tid; o < H; o += kCT) acc_s[o] = 0.f;
  }
  pdl_wait();  // the router's logits (and its reset of the grid counter)
  float* zbuf = reinterpret_cast<float*>(ring);  // the ring is not yet in use
  if (kMulti)
    route_in_smem<kThreads>(a.logits, T, a.E, a.k, a.S, r, zbuf);
  else
    route_one_in_smem<kThreads>(a.logits, a.E, a.k, a.S, r, zbuf);
  if (a.publish && blockIdx.x == 0) publish_routing<kThreads>(r, T, a.E, a.k, a.S, a.ro);

  // this CTA's chunks: [c0, c1) of the nU * I/16 chunks, expert-major
  const int G = I / kChunk;
  const int n_ch = r.n_unique * G;
  // (32-bit: a 64-bit division is a long software routine; n_ch * grid < 2^32)
  const int c0 = (int)((uint32_t)n_ch * blockIdx.x / gridDim.x);
  const int c1 = (int)((uint32_t)n_ch * (blockIdx.x + 1) / gridDim.x);
  const int n_gu = kChunk / R;            // gate/up stages per chunk
  const int n_dn = (H + Dr - 1) / Dr;     // down stages per chunk
  // Tokens each CTA's partial output covers (the CTAs' chunk ranges follow
  // from the routing, which every CTA has): per touched expert, then per CTA.
  for (int u = tid; u < r.n_unique; u += kThreads) {
    const int4 ui = r.u[u];
    uint32_t m = 0;
    for (int p = ui.y; p < ui.y + ui.z; ++p) m |= 1u << r.tok[p];
    s_emask[u] = m;
  }
  __syncthreads();
  for (int c = tid; c < (int)gridDim.x; c += kThreads) {
    const int b0 = (int)((uint32_t)n_ch * c / gridDim.x), b1 = (int)((uint32_t)n_ch * (c + 1) / gridDim.x);
    uint32_t m = 0;
    if (b1 > b0)
      for (int u = b0 / G; u <= (b1 - 1) / G; ++u) m |= s_emask[u];
    s_pm[c] = m;
  }
  __syncthreads();
  const uint32_t cta_mask = s_pm[blockIdx.x];

  if (warp == kProducer) {
    // ------------------------------------------------------ producer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      int j = 0;  // stages issued
      bool ok = true;
      const int per_ch = n_gu + n_dn, n_st = (c1 - c0) * per_ch;
      // Stage x of this CTA (chunk c0 + x / per_ch, step x % per_ch): global
      // source and bytes of its (first) copy.
      auto stage_src = [&](int x, const uint8_t*& src, uint32_t& bytes) {
        const int ch = c0 + x / per_ch, q = x - (x / per_ch) * per_ch;
        const int u = ch / G, g = ch - u * G;
        const int e = r.u[u].x;
        if (q < n_gu) {
          const int i0 = g * kChunk + q * R;
          src = a.q_gu + ((int64_t)e * 2 * I + 2 * i0) * rb_h;
          bytes = (uint32_t)(2 * R) * rb_h;
        } else {
          const int r0 = (q - n_gu) * Dr, nr = ::min(Dr, H - r0);
          src = a.q_dc + (((int64_t)e * G + g) * H + r0) * kChunk;
          bytes = (uint32_t)nr * kChunk;
        }
      };
      // (no L2 prefetch ahead of the ring: measured, it only lengthens the
      // queue the ring's own copies wait in)
      for (int x = 0; x < n_st && ok; ++x) {
        if (j >= a.stages && !mbar_wait(&empty[st], ph ^ 1u)) {
          report_wait(a.meta, kSiteGuEmpty, j, x);
          ok = false;
          break;
        }
        uint8_t* sb = ring + (size_t)st * a.stage_bytes;
        const uint8_t* src;
        uint32_t bytes;
        stage_src(x, src, bytes);
        const int q = x % per_ch;
        if (q < n_gu) {  // rows 2 i0 .. 2 (i0 + R) of the interleaved gate/up plane
          mbar_arrive_expect_tx(&full[st], bytes);
          bulk_g2s(sb, src, bytes, &full[st]);
        } else {  // down rows [r0, r0 + nr) of the chunk's column group: codes, then their scales
          const int ch = c0 + x / per_ch;
          const int u = ch / G, g = ch - u * G, e = r.u[u].x;
          const int r0 = (q - n_gu) * Dr, nr = (int)(bytes / kChunk);
          mbar_arrive_expect_tx(&full[st], (uint32_t)nr * 18u);
          bulk_g2s(sb, src, bytes, &full[st]);
          bulk_g2s(sb + (size_t)nr * kChunk, a.st_d + ((int64_t)e * (I / 32) + g / 2) * H + r0, (uint32_t)nr * 2u,
                   &full[st]);
        }
        ++j;
        if (++st == a.stages) {
          st = 0;
          ph ^= 1u;
        }
      }
      // every copy issued has landed before the ring is reused or the CTA leaves
      for (int q = ::max(0, j - a.stages); q < j; ++q)
        if (!mbar_wait(&full[q % a.stages], (uint32_t)((q / a.stages) & 1))) break;
    }
  } else {
    // ------------------------------------------------------ consumers
    // After a wait gives up (ok = false) a warp skips the rest of its waits,
    // work and arrivals but still passes every consumer barrier, so that the
    // other warps are never left waiting at one.
    bool ok = true;
    float acc[kMulti ? kRowsMulti : 1][kMulti ? kMaxDecodeT : 1];
#pragma unroll
    for (int jr = 0; jr < (kMulti ? kRowsMulti : 1); ++jr)
#pragma unroll
      for (int t = 0; t < (kMulti ? kMaxDecodeT : 1); ++t) acc[jr][t] = 0.f;
    int st = 0;
    uint32_t ph = 0;
    int jj = 0;  // stages consumed
    for (int ch = c0; ch < c1; ++ch) {
      const int4 ui = r.u[ch / G];  // (expert, first grouped row, rows, 0)
      float* hb = hbuf + ((ch - c0) & 1) * (kMulti ? kMaxDecodeT : 1) * kChunk;
      // ---- gate/up: unit q of the chunk is computed by warp q, in stage q / R
      for (int q = 0; q < n_gu; ++q) {
        ok = ok && !s_abort;
        if (ok && !mbar_wait(&full[st], ph)) {
          report_wait(a.meta, kSiteGuFull, jj, warp);
          ok = false;
          s_abort = 1;
        }
        if (ok && warp / R == q) {
          const int off = warp - q * R;  // unit within the stage
          const uint8_t* grow = ring + (size_t)st * a.stage_bytes +
                                (size_t)((off / kGUGroup) * 2 * kGUGroup + off % kGUGroup) * rb_h;
          const uint8_t* urow = grow + (size_t)kGUGroup * rb_h;
          const uint16_t* sg = reinterpret_cast<const uint16_t*>(grow + H);
          const uint16_t* su = reinterpret_cast<const uint16_t*>(urow + H);
          for (int m = 0; m < (kMulti ? ui.z : 1); ++m) {
            const int t = kMulti ? r.tok[ui.y + m] : 0;
            const uint8_t* xh = xhi + (size_t)t * H;
            const uint8_t* xl = xlo + (size_t)t * H;
            const int2* xi = xinfo + (size_t)t * nseg;
            float ag = 0.f, au = 0.f;
#pragma unroll(kMulti ? 1 : 2)
            for (int s = lane; s < nseg; s += 32) {
              const uint4 qg = *reinterpret_cast<const uint4*>(grow + s * 16);
              const uint4 qu = *reinterpret_cast<const uint4*>(urow + s * 16);
              const uint4 vh = *reinterpret_cast<const uint4*>(xh + s * 16);
              const uint4 vl = *reinterpret_cast<const uint4*>(xl + s * 16);
              const int2 inf = xi[s];
              const float f = __int_as_float(inf.x);
              const int Sg = seg_dot_i(qg, vh, vl) - inf.y;
              const int Su = seg_dot_i(qu, vh, vl) - inf.y;
              ag = fmaf((float)Sg, half_bits_to_f32(sg[s >> 1]) * f, ag);
              au = fmaf((float)Su, half_bits_to_f32(su[s >> 1]) * f, au);
            }
            ag = warp_sum(ag);
            au = warp_sum(au);
            if (lane == 0) hb[m * kChunk + warp] = silu(ag) * au;
          }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(&empty[st]);
        ++jj;
        if (++st == a.stages) {
          st = 0;
          ph ^= 1u;
        }
      }
      consumer_sync();  // the chunk's h is complete
      // ---- down: thread tid takes rows tid, tid + 512, ... of each stage
      for (int q = 0; q < n_dn; ++q) {
        ok = ok && !s_abort;
        if (ok && !mbar_wait(&full[st], ph)) {
          report_wait(a.meta, kSiteDnFull, jj, warp);
          ok = false;
          s_abort = 1;
        }
        if (ok) {
          const uint8_t* sb = ring + (size_t)st * a.stage_bytes;
          const int r0 = q * Dr, nr = ::min(Dr, H - r0);
          const uint16_t* sc = reinterpret_cast<const uint16_t*>(sb + (size_t)nr * kChunk);
          if (kMulti) {
            // all rows in this one stage (H <= 2048); the expert's tokens ascending
            uint32_t emask = 0;
            for (int p = ui.y; p < ui.y + ui.z; ++p) emask |= 1u << r.tok[p];
#pragma unroll
            for (int tt = 0; tt < kMaxDecodeT; ++tt) {
              if ((emask >> tt) & 1u) {
                const int m = __popc(emask & ((1u << tt) - 1u));
                const float gate = r.gates[r.slot[ui.y + m]];
                const float* hm = hb + m * kChunk;
#pragma unroll
                for (int jr = 0; jr < kRowsMulti; ++jr) {
                  const int rr = tid + kCT * jr;
                  if (rr < nr) {
                    const uint4 qq = *reinterpret_cast<const uint4*>(sb + (size_t)rr * kChunk);
                    acc[jr][tt] = fmaf(gate * half_bits_to_f32(sc[rr]), dot16_smem(qq, hm), acc[jr][tt]);
                  }
                }
              }
            }
          } else {
            const float gate = r.gates[r.slot[ui.y]];
            f2 hv[8];
            load_h16(hb, hv);
            for (int rr = tid; rr < nr; rr += kCT) {
              const uint4 qq = *reinterpret_cast<const uint4*>(sb + (size_t)rr * kChunk);
              acc_s[r0 + rr] = fmaf(gate * half_bits_to_f32(sc[rr]), dot16(qq, hv), acc_s[r0 + rr]);
            }
          }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(&empty[st]);
        ++jj;
        if (++st == a.stages) {
          st = 0;
          ph ^= 1u;
        }
      }
    }
    // ---- partial output of this CTA to global memory
    float* part = a.partial + (size_t)blockIdx.x * T * H;
    if (kMulti) {
#pragma unroll
      for (int tt = 0; tt < kMaxDecodeT; ++tt)
        if ((cta_mask >> tt) & 1u) {
#pragma unroll
          for (int jr = 0; jr < kRowsMulti; ++jr) {
            const int rr = tid + kCT * jr;
            if (rr < H) __stcg(part + (size_t)tt * H + rr, acc[jr][tt]);
          }
        }
    } else {
      consumer_sync();  // every row of acc_s is final
      if (cta_mask)
        for (int o = tid; o < H; o += kCT) __stcg(part + o, acc_s[o]);
    }
    // ---- grid-wide: every partial is written before any CTA sums them. The
    // arrival is a release (ordering the CTA's partial stores, which the
    // consumer barrier ordered before it), the poll an acquire.
    consumer_sync();
    if (tid == 0) {
      unsigned long long* gb = reinterpret_cast<unsigned long long*>(&a.meta->gbar);
      const unsigned long long target = (unsigned long long)gridDim.x + a.grid_extra;
      asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(gb) : "memory");
      if (ld_acquire_u64(gb) < target) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_u64(gb) < target) {
          if (globaltimer_ns() - t0 > a.grid_wait_ns) {
            report_wait(a.meta, kSiteGrid, 0, gridDim.x);
            break;
          }
        }
      }
    }
    consumer_sync();
    // ---- this CTA's output rows [o0, o1): warp w sums the partials of CTAs
    // [w cpw, (w + 1) cpw), lane = row; then the 16 warp sums in order.
    float* red = reinterpret_cast<float*>(ring);  // [kCW][T][rows]
    const int o0 = (int)((uint32_t)H * blockIdx.x / gridDim.x), o1 = (int)((uint32_t)H * (blockIdx.x + 1) / gridDim.x);
    const int nrow = o1 - o0;
    const int cpw = ((int)gridDim.x + kCW - 1) / kCW;
    const int cb = warp * cpw, ce = ::min((int)gridDim.x, cb + cpw);
    for (int rl = lane; rl < nrow; rl += 32) {
      for (int t = 0; t < T; ++t) {
        float v = 0.f;
        for (int c = cb; c < ce; c += kRedBatch) {  // the batch's loads all in flight, then summed in order
          float pv[kRedBatch];
#pragma unroll
          for (int q = 0; q < kRedBatch; ++q)
            pv[q] = (c + q < ce && ((s_pm[c + q] >> t) & 1u))
                        ? __ldcg(a.partial + ((size_t)(c + q) * T + t) * H + o0 + rl)
                        : 0.f;
#pragma unroll
          for (int q = 0; q < kRedBatch; ++q) v += pv[q];
        }
        red[((size_t)warp * T + t) * nrow + rl] = v;
      }
    }
    consumer_sync();
    for (int i = tid; i < T * nrow; i += kCT) {
      const int t = i / nrow, rl = i - t * nrow;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kCW; ++w) v += red[((size_t)w * T + t) * nrow + rl];
      a.out[(size_t)t * H + o0 + rl] = __float2bfloat16_rn(v);
    }
  }
  __syncthreads();
}

// The grid-wide wait needs every CTA resident: the grid is one CTA per SM
// and each CTA takes more than half of an SM's shared memory (checked at
// init), so once earlier work has drained all of them are; if something else
// holds SMs past the wait bound the call reports FW_ETIMEOUT instead of
// hanging.
cudaError_t launch(const DecodeArgs& a, bool multi, unsigned grid, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return multi ? cudaLaunchKernelEx(&cfg, decode_experts_kernel<true>, a)
               : cudaLaunchKernelEx(&cfg, decode_experts_kernel<false>, a);
}

int g_smem_optin = 0;  // dynamic shared memory per CTA the kernels may use

}  // namespace

bool decode_supported(int H, int T) { return T >= 1 && T <= kMaxDecodeT && (T == 1 ? H <= kMaxHOne : H <= kMaxHMulti); }

cudaError_t configure_decode_kernels() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa, fb;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, decode_experts_kernel<false>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fb, decode_experts_kernel<true>);
  if (e == cudaSuccess) g_smem_optin -= (int)std::max(fa.sharedSizeBytes, fb.sharedSizeBytes);
  const void* kern[2] = {(const void*)decode_experts_kernel<false>, (const void*)decode_experts_kernel<true>};
  for (int m = 0; m < 2 && e == cudaSuccess; ++m) {
    e = cudaFuncSetAttribute(kern[m], cudaFuncAttributeMaxDynamicSharedMemorySize, g_smem_optin);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern[m], cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
  }
  // one CTA per SM must fit with the least shared memory a launch asks for:
  // the grid-wide wait relies on every CTA of the grid being resident
  for (int m = 0; m < 2 && e == cudaSuccess; ++m) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern[m], kThreads, (size_t)g_smem_optin / 2 + 1024);
    if (e == cudaSuccess && n < 1) {
      cudaFuncAttributes f = m ? fb : fa;
      char msg[256];
      snprintf(msg, sizeof(msg),
               "decode kernel: no CTA of %d threads fits an SM (registers %d, static smem %zu, dynamic %d)",
               kThreads, f.numRegs, f.sharedSizeBytes, g_smem_optin / 2 + 1024);
      set_error(FW_EUNSUPPORTED, msg);
      e = cudaErrorInvalidConfiguration;
    }
  }
  return e;
}

cudaError_t launch_ffn_decode(Handle* h, const __nv_bfloat16* x, int T, __nv_bfloat16* out, bool publish,
                              int32_t* ids_out, float* gates_out, cudaStream_t s) {
  const int H = h->cfg.H, I = h->cfg.I, k = h->cfg.k, S = h->S;
  const bool multi = T > 1;
  const int tcap = multi ? kMaxDecodeT : 1;
  DecodeArgs a;
  a.q_gu = h->q_gu;
  a.q_dc = h->q_dc;
  a.st_d = h->st_d;
  a.x = x;
  a.logits = h->logits;
  a.partial = h->partial;
  a.out = out;
  a.ro = RoutingOut{ids_out, gates_out, h->ids,      h->gates,    h->counts, h->offsets,
                    h->perm, h->inv,    h->row_token, h->row_gate, h->uinfo,  h->meta};
  a.meta = h->meta;
  a.H = H;
  a.I = I;
  a.E = h->cfg.E;
  a.k = k;
  a.S = S;
  a.T = T;
  a.publish = publish ? 1 : 0;
  // stages: gate/up R units (2R rows of row_bytes(H)), down Dr rows x 18 bytes
  const uint32_t rb = (uint32_t)row_bytes(H);
  int R = kChunk;
  while (R > kGUGroup && (uint32_t)(2 * R) * rb > kStageTarget) R /= 2;
  a.R = R;
  const int nd = (H + kDnRowsMax - 1) / kDnRowsMax;
  a.Dr = multi ? H : ((H + nd - 1) / nd + 15) / 16 * 16;
  a.stage_bytes = std::max((uint32_t)(2 * R) * rb, align128((uint32_t)a.Dr * 18u));
  a.stage_bytes = align128(a.stage_bytes);
  // dynamic shared memory: x planes, segment info, the one-token partial row, h
  const uint32_t xb = align128((uint32_t)(2 * T * H));
  a.off_info = xb;
  a.off_acc = a.off_info + align128((uint32_t)(T * (H / 16) * 8));
  a.off_h = a.off_acc + (multi ? 0u : align128((uint32_t)H * 4u));
  a.off_ring = a.off_h + align128((uint32_t)(2 * tcap * kChunk * 4));
  const int64_t ring_bytes = (int64_t)g_smem_optin - a.off_ring - 256;
  a.stages = (int)std::min<int64_t>(kMaxStages, ring_bytes / a.stage_bytes);
  if (a.stages < 2) return cudaErrorInvalidConfiguration;
  const int grid = h->num_sms;
  // the ring also holds the logits while routing and the sums at the end
  if (grid > kMaxGrid) return cudaErrorInvalidConfiguration;
  const uint32_t need_end = (uint32_t)(kCW * T * ((H + grid - 1) / grid) * 4);
  if ((uint32_t)a.stages * a.stage_bytes < std::max<uint32_t>(need_end, (uint32_t)(T * h->cfg.E * 4)))
    return cudaErrorInvalidConfiguration;
  if (h->test_grid_timeouts > 0) {  // test hook: this call's grid-wide wait cannot be met and gives up fast
    --h->test_grid_timeouts;
    a.grid_extra = 1;
    a.grid_wait_ns = 1000000ull;
  } else {
    a.grid_extra = 0;
    a.grid_wait_ns = kWaitLimitNs;
  }
  // at least half the SM's shared memory, so that no two CTAs share an SM
  const size_t smem = std::max<size_t>(a.off_ring + (size_t)a.stages * a.stage_bytes,
                                       (size_t)g_smem_optin / 2 + 1024);
  KernelTimer tm(h, FW_KERNEL_DECODE_EXPERTS, s);
  return launch(a, multi, (unsigned)grid, smem, s);
}

}  // namespace fw
