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
// projection does the same with the chunk's h (16 fp32 values per token, made
// fixed point at their largest exponent: by every thread for one token, once
// per token into shared memory for several).
//
// Chunks are split over the CTAs in contiguous ranges: of equal count for one
// token; for several, of equal cost, a chunk costing its weight stream plus
// its expert's token count of arithmetic (a CTA whose range falls on experts
// with many tokens would otherwise finish last).
//
// One CTA per SM, all resident (see launch()):
//   0. x -> fixed-point planes in shared memory (before the router finishes);
//   1. after the router's grid completes (programmatic dependent launch), the
//      batch's routing rebuilt from the logits in shared memory
//      (deterministic, so every CTA agrees); CTA 0 publishes it;
//   2. the CTA's chunks: gate/up stages -> h (shared memory), then down
//      stages -> the CTA's partial output (fp32: shared memory for one token,
//      tensor memory for several);
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
constexpr int kMaxHOne = 14336;            // one token: x planes, the fp32 partial row and two ring stages fit in shared memory
constexpr int kDnRowsMax = 2048;           // down rows per stage at most
constexpr uint32_t kConsumerBarrier = 1;   // named barrier of the 16 consumer warps
constexpr uint32_t kStageTarget = 36 * 1024;
constexpr int kRedBatch = 10;              // partial loads in flight per lane in the final sums
constexpr int kMaxGrid = 256;              // CTAs (one per SM) the per-CTA token masks have room for
// Several tokens: the cost of a chunk is kChunkCost (its weight stream) plus
// kTokCost per token of its expert (the arithmetic). Measured at 16 tokens
// (per call): 1 + 1 n 112.6 us, 2 + n 120.6, 4 + n 135.7, 8 + n 151.1,
// 0 + n 128.5, 1 + 2 n 117.4, 1 + 4 n 122.0.
constexpr int kChunkCost = 1;
constexpr int kTokCost = 1;

// The chunk's h of one token as 16-bit fixed point (see h16_to_planes).
struct HPlanes {
  uint4 hi, lo;
  int2 info;
  int2 pad;
};

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
  uint32_t off_info, off_acc, off_h, off_hp, off_ring;  // dynamic shared memory layout (bytes)
  uint32_t grid_extra;   // arrivals the grid wait expects beyond the grid (0; > 0 only to test the bound)
  uint64_t grid_wait_ns; // bound of the grid-wide wait
};

// ------------------------------------------------------------- helpers
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

// The same with Q8 activations: one signed plane, sum_i (q_i + 128) * x8_i.
__device__ __forceinline__ int seg_dot_q8(const uint4 q, const uint4 x8) {
  int s = dp4a_us(q.x, x8.x, 0);
  s = dp4a_us(q.y, x8.y, s);
  s = dp4a_us(q.z, x8.z, s);
  return dp4a_us(q.w, x8.w, s);
}
template <bool kQ8>
__device__ __forceinline__ int seg_dot(const uint4 q, const uint4 hi, const uint4 lo) {
  if constexpr (kQ8)
    return seg_dot_q8(q, hi);
  else
    return seg_dot_i(q, hi, lo);
}

// Q8 code of v in a block of scale d (d > 0): round-half-away of the fp32
// quotient, clamped to [-127, 127].
__device__ __forceinline__ int q8_code(float v, float d) {
  return ::max(-127, ::min(127, (int)roundf(__fdiv_rn(v, d))));
}
__device__ __forceinline__ uint32_t pack_s8x4(int a, int b, int c, int d) {
  return ((uint32_t)a & 0xFFu) | (((uint32_t)b & 0xFFu) << 8) | (((uint32_t)c & 0xFFu) << 16) | ((uint32_t)d << 24);
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

// Q8 activations: one 32-value block of bf16 x (four 16-byte words) -> two
// segments of signed codes, each with the block's scale d = amax/127 (fp32
// division) as its float and 128 * sum(codes); an all-zero block: zeros.
__device__ __forceinline__ void x_block_to_q8(const uint4 a, const uint4 b, const uint4 c, const uint4 e, uint4& q0,
                                              uint4& q1, int2& i0, int2& i1) {
  const uint32_t w[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, e.x, e.y, e.z, e.w};
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
  if (amax == 0.f) {
    q0 = q1 = make_uint4(0u, 0u, 0u, 0u);
    i0 = i1 = make_int2(0, 0);
    return;
  }
  const float d = __fdiv_rn(amax, 127.0f);
  uint32_t p[8];
  int s0 = 0, s1 = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c0 = q8_code(__uint_as_float(w[2 * j] << 16), d), c1 = q8_code(__uint_as_float(w[2 * j] & 0xFFFF0000u), d);
    const int c2 = q8_code(__uint_as_float(w[2 * j + 1] << 16), d),
              c3 = q8_code(__uint_as_float(w[2 * j + 1] & 0xFFFF0000u), d);
    p[j] = pack_s8x4(c0, c1, c2, c3);
    if (j < 4) s0 += c0 + c1 + c2 + c3; else s1 += c0 + c1 + c2 + c3;
  }
  q0 = make_uint4(p[0], p[1], p[2], p[3]);
  q1 = make_uint4(p[4], p[5], p[6], p[7]);
  i0 = make_int2(__float_as_int(d), 128 * s0);
  i1 = make_int2(__float_as_int(d), 128 * s1);
}

// The chunk's h of one token (16 fp32 values in shared memory) -> the same
// 16-bit fixed point at its largest exponent as x (byte planes, 2^(e - 14),
// 128 * sum): the down codes then multiply it with dp4a. Two passes over the
// values (broadcast reads) keep few registers live. Largest magnitude below
// 2^-112: zero.
__device__ __forceinline__ void h16_to_planes(const float* h, uint4& hi, uint4& lo, int2& info) {
  const float4* h4 = reinterpret_cast<const float4*>(h);
  uint32_t emax = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 v = h4[j];
    emax = max(emax, max(max((__float_as_uint(v.x) >> 23) & 0xFFu, (__float_as_uint(v.y) >> 23) & 0xFFu),
                         max((__float_as_uint(v.z) >> 23) & 0xFFu, (__float_as_uint(v.w) >> 23) & 0xFFu)));
  }
  if (emax < 15u) {
    hi = lo = make_uint4(0u, 0u, 0u, 0u);
    info = make_int2(0, 0);
    return;
  }
  const float mult = __uint_as_float((268u - emax) << 23);  // 2^(14 - e)
  uint32_t hw[4], lw[4];
  int sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 v = h4[j];
    const int x0 = __float2int_rn(v.x * mult), x1 = __float2int_rn(v.y * mult), x2 = __float2int_rn(v.z * mult),
              x3 = __float2int_rn(v.w * mult);
    sum += x0 + x1 + x2 + x3;
    hw[j] = ((uint32_t)(x0 >> 8) & 0xFFu) | (((uint32_t)(x1 >> 8) & 0xFFu) << 8) | (((uint32_t)(x2 >> 8) & 0xFFu) << 16) |
            (((uint32_t)(x3 >> 8) & 0xFFu) << 24);
    lw[j] = ((uint32_t)x0 & 0xFFu) | (((uint32_t)x1 & 0xFFu) << 8) | (((uint32_t)x2 & 0xFFu) << 16) |
            (((uint32_t)x3 & 0xFFu) << 24);
  }
  hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  info = make_int2((int)((emax - 14u) << 23), 128 * sum);
}

// The same conversion by one warp (lane j < 16 holds value j), written to
// shared memory: the several-token path converts each token's h once per
// chunk instead of once per thread.
__device__ __forceinline__ void h16_to_planes_warp(const float* h, HPlanes* out, int lane) {
  const float v = lane < 16 ? h[lane] : 0.f;
  const uint32_t emax = __reduce_max_sync(0xFFFFFFFFu, (__float_as_uint(v) >> 23) & 0xFFu);
  int xi = 0;
  if (emax >= 15u) xi = __float2int_rn(v * __uint_as_float((268u - emax) << 23));  // 2^(14 - e)
  const int sum = __reduce_add_sync(0xFFFFFFFFu, xi);
  uint32_t hw = ((uint32_t)(xi >> 8) & 0xFFu) << ((lane & 3) * 8), lw = ((uint32_t)xi & 0xFFu) << ((lane & 3) * 8);
  hw |= __shfl_xor_sync(0xFFFFFFFFu, hw, 1);
  lw |= __shfl_xor_sync(0xFFFFFFFFu, lw, 1);
  hw |= __shfl_xor_sync(0xFFFFFFFFu, hw, 2);
  lw |= __shfl_xor_sync(0xFFFFFFFFu, lw, 2);
  if (lane < 16 && (lane & 3) == 0) {
    reinterpret_cast<uint32_t*>(&out->hi)[lane >> 2] = hw;
    reinterpret_cast<uint32_t*>(&out->lo)[lane >> 2] = lw;
  }
  if (lane == 0) out->info = emax >= 15u ? make_int2((int)((emax - 14u) << 23), 128 * sum) : make_int2(0, 0);
}

// Q8 activations: the chunk's h of one token (16 fp32 values) -> signed codes
// at d = amax/127, (float bits of d, 128 * sum); all zero: zeros.
__device__ __forceinline__ void h16_to_q8(const float* h, uint4& q, int2& info) {
  const float4* h4 = reinterpret_cast<const float4*>(h);
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 v = h4[j];
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  if (amax == 0.f) {
    q = make_uint4(0u, 0u, 0u, 0u);
    info = make_int2(0, 0);
    return;
  }
  const float d = __fdiv_rn(amax, 127.0f);
  uint32_t p[4];
  int sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 v = h4[j];
    const int c0 = q8_code(v.x, d), c1 = q8_code(v.y, d), c2 = q8_code(v.z, d), c3 = q8_code(v.w, d);
    sum += c0 + c1 + c2 + c3;
    p[j] = pack_s8x4(c0, c1, c2, c3);
  }
  q = make_uint4(p[0], p[1], p[2], p[3]);
  info = make_int2(__float_as_int(d), 128 * sum);
}
__device__ __forceinline__ void h16_to_q8_warp(const float* h, HPlanes* out, int lane) {
  const float v = lane < 16 ? h[lane] : 0.f;
  // |v| as unsigned bits orders like |v| itself
  const float amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(v) & 0x7FFFFFFFu));
  int c = 0;
  float d = 0.f;
  if (amax > 0.f) {
    d = __fdiv_rn(amax, 127.0f);
    c = lane < 16 ? q8_code(v, d) : 0;
  }
  const int sum = __reduce_add_sync(0xFFFFFFFFu, c);
  uint32_t qw = ((uint32_t)c & 0xFFu) << ((lane & 3) * 8);
  qw |= __shfl_xor_sync(0xFFFFFFFFu, qw, 1);
  qw |= __shfl_xor_sync(0xFFFFFFFFu, qw, 2);
  if (lane < 16 && (lane & 3) == 0) reinterpret_cast<uint32_t*>(&out->hi)[lane >> 2] = qw;
  if (lane == 0) out->info = make_int2(__float_as_int(d), 128 * sum);
}

// Four consecutive fp32 columns of this thread's tensor-memory lane (the
// several-token path keeps its partial output there: 64 per thread would not
// fit in registers beside the rest).
__device__ __forceinline__ float4 tmem_ld4(uint32_t taddr) {
  uint32_t r0, r1, r2, r3;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  return make_float4(__uint_as_float(r0), __uint_as_float(r1), __uint_as_float(r2), __uint_as_float(r3));
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, float4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(__float_as_uint(v.x)),
               "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)), "r"(__float_as_uint(v.w))
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
constexpr uint32_t kTmemCols = 512;  // several tokens: 16 warps x (16 tokens x 4 rows) fp32, by lane quarter

// ------------------------------------------------------------- the kernel
// kMulti: several tokens (T <= 16, H <= 2048; partial output in registers);
// otherwise one token (partial output in shared memory).
template <bool kMulti, bool kQ8>
__global__ void __launch_bounds__(kThreads, 1) decode_experts_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages];
  __shared__ SmemRouting r;
  __shared__ uint32_t s_emask[kMaxE + 1];  // per touched expert (ascending): its tokens
  __shared__ uint32_t s_pm[kMaxGrid];       // per CTA: the tokens its partial output covers
  __shared__ int s_c0[kMaxGrid + 1];         // per CTA: its first chunk (s_c0[grid] = all chunks)
  __shared__ uint32_t s_pref[kMaxE + 2];     // several tokens: chunk cost before each touched expert
  __shared__ volatile int s_abort;  // a consumer gave up a wait: the others stop waiting too
  __shared__ uint32_t s_tmem;        // several tokens: tensor-memory base of the partial outputs
  __shared__ HPlanes s_hq;           // one token, Q8 activations: the chunk's h codes
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, I = a.I, T = kMulti ? a.T : 1, R = a.R, Dr = a.Dr;
  const int nseg = H / 16;
  const uint32_t rb_h = (uint32_t)row_bytes(H);
  uint8_t* xhi = smem;                                              // [T][H] int8
  uint8_t* xlo = smem + (size_t)T * H;                              // [T][H] uint8
  int2* xinfo = reinterpret_cast<int2*>(smem + a.off_info);         // [T][H/16]
  float* acc_s = reinterpret_cast<float*>(smem + a.off_acc);        // [H] (one token)
  float* hbuf = reinterpret_cast<float*>(smem + a.off_h);           // [2][T][16]
  HPlanes* hpl = reinterpret_cast<HPlanes*>(smem + a.off_hp);       // [T] (several tokens)
  uint8_t* ring = smem + a.off_ring;
  // The next kernel in the stream (the next call's router) may launch at
  // once: it waits for this grid's completion before touching memory, and
  // meanwhile its CTAs, where they fit beside this one, prefetch their weights.
  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (kMulti && warp == 0) {  // one CTA per SM: the 512 columns are free
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp != kProducer) {
    // x is complete: the router lets this grid launch only after everything
    // before it in the stream has completed. Staged while the router still runs.
    if constexpr (kQ8 && kMulti) {
      // Q8 activations, one plane, several tokens: a thread per 32-value
      // block (two segments); the work is spread over all threads already
      for (int c = tid; c < T * nseg / 2; c += kCT) {
        const uint4* src = reinterpret_cast<const uint4*>(a.x) + 4 * c;
        uint4 q0, q1;
        int2 i0, i1;
        x_block_to_q8(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3), q0, q1, i0, i1);
        reinterpret_cast<uint4*>(xhi)[2 * c] = q0;
        reinterpret_cast<uint4*>(xhi)[2 * c + 1] = q1;
        xinfo[2 * c] = i0;
        xinfo[2 * c + 1] = i1;
      }
    } else if constexpr (kQ8) {
      // Q8 activations, one plane, one token: four values a thread (a block
      // a thread would leave most threads idle), a 32-value block
      // over eight lanes (its amax and each 16-value segment's code sum by
      // shuffles within the group); whole warps, so the trip count is uniform
      const int n4 = T * H / 4;
      for (int c0 = warp * 32; c0 < n4; c0 += kCW * 32) {
        const int c = c0 + lane;
        const bool in = c < n4;  // n4 is a multiple of 8: a group is all in or all out
        const uint2 v = in ? __ldg(reinterpret_cast<const uint2*>(a.x) + c) : make_uint2(0u, 0u);
        const float f0 = __uint_as_float(v.x << 16), f1 = __uint_as_float(v.x & 0xFFFF0000u),
                    f2 = __uint_as_float(v.y << 16), f3 = __uint_as_float(v.y & 0xFFFF0000u);
        float amax = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
        int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
        float d = 0.f;
        if (amax > 0.f) {
          d = __fdiv_rn(amax, 127.0f);
          q0 = q8_code(f0, d);
          q1 = q8_code(f1, d);
          q2 = q8_code(f2, d);
          q3 = q8_code(f3, d);
        }
        int sum = q0 + q1 + q2 + q3;
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);  // the 16-value segment's four lanes
        if (in) {
          reinterpret_cast<uint32_t*>(xhi)[c] = pack_s8x4(q0, q1, q2, q3);
          if ((lane & 3) == 0) xinfo[c >> 2] = make_int2(__float_as_int(d), 128 * sum);
        }
      }
    } else {
      for (int c = tid; c < T * nseg; c += kCT) {
        const uint4* src = reinterpret_cast<const uint4*>(a.x) + 2 * c;
        uint4 hi, lo;
        int2 info;
        x_segment_to_planes(__ldg(src), __ldg(src + 1), hi, lo, info);
        reinterpret_cast<uint4*>(xhi)[c] = hi;
        reinterpret_cast<uint4*>(xlo)[c] = lo;
        xinfo[c] = info;
      }
    }
    if (!kMulti)
      for (int o = tid; o < H; o += kCT) acc_s[o] = 0.f;
  }
  const int G = I / kChunk;
  const int n_gu = kChunk / R;            // gate/up stages per chunk
  const int n_dn = (H + Dr - 1) / Dr;     // down stages per chunk
  if (!kMulti) {
    // One token touches k + S experts whatever the logits, so its chunk ranges
    // (equal counts) and which CTAs' partial outputs hold it are known before
    // the routing is. (32-bit: n_ch * grid < 2^32.)
    const uint32_t n1 = (uint32_t)((a.k + a.S) * G);
    for (int c = tid; c < (int)gridDim.x; c += kThreads)
      s_pm[c] = n1 * (uint32_t)(c + 1) / gridDim.x > n1 * (uint32_t)c / gridDim.x ? 1u : 0u;
  }
  pdl_wait();  // the router's logits (and its reset of the grid counter)
  float* zbuf = reinterpret_cast<float*>(ring);  // the ring is not yet in use
  if (kMulti) {
    route_in_smem<kThreads>(a.logits, T, a.E, a.k, a.S, r, zbuf);
  } else {
    route_one_in_smem<kThreads>(a.logits, a.E, a.k, a.S, r);
    // the gates are first read in a down stage, after a consumer barrier
    if (warp == 0) route_one_gates(a.k, a.S, r, lane);
  }
  if (a.publish && blockIdx.x == 0) {
    if (!kMulti) {
      route_one_tables<kThreads>(a.E, a.k, a.S, r);
      __syncthreads();
    }
    publish_routing<kThreads>(r, T, a.E, a.k, a.S, a.ro);
  }

  // this CTA's chunks: [c0, c1) of the nU * I/16 chunks, expert-major
  const int n_ch = r.n_unique * G;
  int c0, c1;
  if (kMulti) {
    // Tokens each CTA's partial output covers (the CTAs' chunk ranges follow
    // from the routing, which every CTA has): per touched expert its token
    // mask, then per CTA.
    for (int u = tid; u < r.n_unique; u += kThreads) {
      const int e = r.u[u].x;
      s_emask[u] = e < a.E ? r.mask[e] : (1u << T) - 1u;
    }
    // A chunk costs its weight stream plus its expert's token count of
    // arithmetic: kChunkCost + kTokCost n. CTA b takes the chunks whose starting cost
    // lies in [b C / grid, (b + 1) C / grid), C the total. Prefix costs per
    // expert by one warp (C < 2^32), the bounds by a thread per CTA.
    if (warp == 0) {
      const int nu = r.n_unique, per = (nu + 31) / 32, u0 = lane * per;
      uint32_t run = 0;
      for (int u = u0; u < ::min(nu, u0 + per); ++u) run += (uint32_t)(kChunkCost + kTokCost * r.u[u].z) * G;
      uint32_t inc = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += v;
      }
      uint32_t p = inc - run;
      for (int u = u0; u < ::min(nu, u0 + per); ++u) {
        s_pref[u] = p;
        p += (uint32_t)(kChunkCost + kTokCost * r.u[u].z) * G;
      }
      if (lane == 31) s_pref[nu] = inc;
    }
    __syncthreads();
    const uint64_t C = s_pref[r.n_unique], grid = gridDim.x;
    for (int b = tid; b <= (int)grid; b += kThreads) {
      // first chunk c with cost(c) * grid >= b * C (once per call: 64-bit)
      const uint64_t target = (uint64_t)b * C;
      int lo = 0, hi = r.n_unique;  // expert: the last u with s_pref[u] * grid <= target
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pref[mid] * grid <= target) lo = mid; else hi = mid;
      }
      int c = n_ch;
      if (b < (int)grid && r.n_unique > 0) {
        // rem < w G: the quotient is at most G, and rem + w fits 32 bits
        const uint64_t w = (uint64_t)(kChunkCost + kTokCost * r.u[lo].z) * grid;
        const uint64_t rem = target - s_pref[lo] * grid;
        c = ::min(lo * G + (int)(((uint32_t)rem + (uint32_t)w - 1u) / (uint32_t)w), n_ch);
      }
      s_c0[b] = c;
    }
    __syncthreads();
    c0 = s_c0[blockIdx.x];
    c1 = s_c0[blockIdx.x + 1];
    for (int c = tid; c < (int)gridDim.x; c += kThreads) {
      const int b0 = s_c0[c], b1 = s_c0[c + 1];
      uint32_t m = 0;
      if (b1 > b0)
        for (int u = b0 / G; u <= (b1 - 1) / G; ++u) m |= s_emask[u];
      s_pm[c] = m;
    }
    __syncthreads();
  } else {
    c0 = (int)((uint32_t)n_ch * blockIdx.x / gridDim.x);
    c1 = (int)((uint32_t)n_ch * (blockIdx.x + 1) / gridDim.x);
  }
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
    // several tokens: this thread's partial output rows tid + 512 jr of token
    // t in its tensor-memory lane, column (warp / 4) 64 + 4 t + jr
    uint32_t tacc = 0;
    if (kMulti) {
      tc_fence_after();
      tacc = s_tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(warp >> 2) * 64u;
#pragma unroll 1
      for (int t = 0; t < kMaxDecodeT; ++t) tmem_st4(tacc + 4 * t, make_float4(0.f, 0.f, 0.f, 0.f));
    }
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
        ok = __all_sync(0xFFFFFFFFu, ok);  // warp-uniform (tensor-memory accesses are warp-wide)
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
              const uint4 vl = kQ8 ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(xl + s * 16);
              const int2 inf = xi[s];
              const float f = __int_as_float(inf.x);
              const int Sg = seg_dot<kQ8>(qg, vh, vl) - inf.y;
              const int Su = seg_dot<kQ8>(qu, vh, vl) - inf.y;
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
      if constexpr (!kMulti && kQ8) {  // one token, Q8: its h codes once, by one warp (sixteen divisions)
        if (warp == 0) h16_to_q8_warp(hb, &s_hq, lane);
        consumer_sync();
      }
      if (kMulti) {  // each token's h -> fixed-point planes, a warp per token
        for (int m = warp; m < ui.z; m += kCW) {
          if constexpr (kQ8)
            h16_to_q8_warp(hb + m * kChunk, hpl + m, lane);
          else
            h16_to_planes_warp(hb + m * kChunk, hpl + m, lane);
        }
        consumer_sync();
      }
      uint4 dhh = make_uint4(0u, 0u, 0u, 0u), dhl = dhh;  // one token: the chunk's h planes
      int2 dhinf = make_int2(0, 0);
      float dgf = 0.f;
      // ---- down: thread tid takes rows tid, tid + 512, ... of each stage
      for (int q = 0; q < n_dn; ++q) {
        ok = ok && !s_abort;
        if (ok && !mbar_wait(&full[st], ph)) {
          report_wait(a.meta, kSiteDnFull, jj, warp);
          ok = false;
          s_abort = 1;
        }
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (ok) {
          const uint8_t* sb = ring + (size_t)st * a.stage_bytes;
          const int r0 = q * Dr, nr = ::min(Dr, H - r0);
          const uint16_t* sc = reinterpret_cast<const uint16_t*>(sb + (size_t)nr * kChunk);
          if (kMulti) {
            // all rows in this one stage (H <= 2048); the expert's tokens in
            // ascending order: the row products, then the token's four
            // partial sums read, added to and written back to tensor memory
            for (int m = 0; m < ui.z; ++m) {
              const int t = r.tok[ui.y + m];
              const uint4 hh = hpl[m].hi, hl = hpl[m].lo;
              const int2 inf = hpl[m].info;
              const float gf = r.gates[r.slot[ui.y + m]] * __int_as_float(inf.x);
              float d[kRowsMulti];
#pragma unroll
              for (int jr = 0; jr < kRowsMulti; ++jr) {
                const int rr = tid + kCT * jr;
                d[jr] = 0.f;
                if (rr < nr) {
                  const uint4 qq = *reinterpret_cast<const uint4*>(sb + (size_t)rr * kChunk);
                  d[jr] = (float)(seg_dot<kQ8>(qq, hh, hl) - inf.y) * (gf * half_bits_to_f32(sc[rr]));
                }
              }
              float4 v = tmem_ld4(tacc + 4 * t);
              v.x += d[0];
              v.y += d[1];
              v.z += d[2];
              v.w += d[3];
              tmem_st4(tacc + 4 * t, v);
            }
          } else {
            // (the chunk's h planes: the same in every down stage of the chunk)
            if (q == 0) {
              if constexpr (kQ8) {  // quantised by warp 0 after the chunk's gate/up
                dhh = s_hq.hi;
                dhinf = s_hq.info;
              } else {
                h16_to_planes(hb, dhh, dhl, dhinf);
              }
              dgf = r.gates[r.slot[ui.y]] * __int_as_float(dhinf.x);
            }
            for (int rr = tid; rr < nr; rr += kCT) {
              const uint4 qq = *reinterpret_cast<const uint4*>(sb + (size_t)rr * kChunk);
              const int S = seg_dot<kQ8>(qq, dhh, dhl) - dhinf.y;
              acc_s[r0 + rr] = fmaf((float)S, dgf * half_bits_to_f32(sc[rr]), acc_s[r0 + rr]);
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
      for (int tt = 0; tt < kMaxDecodeT; ++tt)
        if ((cta_mask >> tt) & 1u) {
          const float4 v = tmem_ld4(tacc + 4 * tt);
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int jr = 0; jr < kRowsMulti; ++jr) {
            const int rr = tid + kCT * jr;
            if (rr < H) __stcg(part + (size_t)tt * H + rr, vv[jr]);
          }
        }
    } else {
      consumer_sync();  // every row of acc_s is final
      if (cta_mask)
        for (int o = tid; o < H; o += kCT) __stcg(part + o, acc_s[o]);
    }
    // ---- this CTA's output rows [o0, o1) (summed after the grid-wide wait).
    // For each token, the CTAs whose partials hold it (ascending), made here
    // while other CTAs still stream (the ring is free: every stage is consumed;
    // the sums clamp the CTA index all the same, should a wait have given up
    // with a copy still in flight)
    const int o0 = (int)((uint32_t)H * blockIdx.x / gridDim.x), o1 = (int)((uint32_t)H * (blockIdx.x + 1) / gridDim.x);
    const int nrow = o1 - o0, pairs = T * nrow;
    const int P = ::max(1, ::min(kCW, kCT / ::max(1, pairs)));
    float* red = reinterpret_cast<float*>(ring);                       // [P][pairs]: P pairs <= max(kCT, pairs)
    int* lists = reinterpret_cast<int*>(ring) + ::max(kCT, pairs);     // [T][grid]
    __shared__ int s_len[kMaxDecodeT];
    for (int t = warp; t < T; t += kCW) {  // a warp per token: its CTAs by ballot, ascending
      int n = 0;
      for (int c0 = 0; c0 < (int)gridDim.x; c0 += 32) {
        const int c = c0 + lane;
        const bool has = c < (int)gridDim.x && ((s_pm[c] >> t) & 1u);
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, has);
        if (has) lists[t * gridDim.x + n + __popc(bal & ((1u << lane) - 1u))] = c;
        n += __popc(bal);
      }
      if (lane == 0) s_len[t] = n;
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
    // ---- each (token, row) pair of this CTA's rows is summed over its
    // token's list by P threads taking consecutive parts of it (a part's loads
    // all in flight, then added in order), then the P part sums in order.
    for (int i = tid; i < P * pairs; i += kCT) {
      const int part = i / pairs, pr = i - part * pairs;
      const int t = pr / nrow, rl = pr - t * nrow;
      const int len = s_len[t], q0 = len * part / P, q1 = len * (part + 1) / P;
      const int* lt = lists + t * gridDim.x;
      float v = 0.f;
      for (int q = q0; q < q1; q += kRedBatch) {
        float pv[kRedBatch];
#pragma unroll
        for (int j = 0; j < kRedBatch; ++j)
          pv[j] = q + j < q1 ? __ldcg(a.partial + ((size_t)::min((unsigned)lt[q + j], gridDim.x - 1u) * T + t) * H + o0 + rl)
                             : 0.f;
#pragma unroll
        for (int j = 0; j < kRedBatch; ++j) v += pv[j];
      }
      red[part * pairs + pr] = v;
    }
    consumer_sync();
    for (int i = tid; i < pairs; i += kCT) {
      const int t = i / nrow, rl = i - t * nrow;
      float v = 0.f;
      for (int part = 0; part < P; ++part) v += red[part * pairs + i];
      a.out[(size_t)t * H + o0 + rl] = __float2bfloat16_rn(v);
    }
  }
  if (kMulti) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(s_tmem), "r"(kTmemCols) : "memory");
  } else {
    __syncthreads();
  }
}

// The grid-wide wait needs every CTA resident: the grid is one CTA per SM
// and each CTA takes more than half of an SM's shared memory (checked at
// init), so once earlier work has drained all of them are; if something else
// holds SMs past the wait bound the call reports FW_ETIMEOUT instead of
// hanging.
cudaError_t launch(const DecodeArgs& a, bool multi, bool q8, unsigned grid, size_t smem, cudaStream_t s) {
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
  if (q8)
    return multi ? cudaLaunchKernelEx(&cfg, decode_experts_kernel<true, true>, a)
                 : cudaLaunchKernelEx(&cfg, decode_experts_kernel<false, true>, a);
  return multi ? cudaLaunchKernelEx(&cfg, decode_experts_kernel<true, false>, a)
               : cudaLaunchKernelEx(&cfg, decode_experts_kernel<false, false>, a);
}

int g_smem_optin = 0;  // dynamic shared memory per CTA the kernels may use

}  // namespace

bool decode_supported(int H, int T) { return T >= 1 && T <= kMaxDecodeT && (T == 1 ? H <= kMaxHOne : H <= kMaxHMulti); }

cudaError_t configure_decode_kernels() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const void* kern[4] = {(const void*)decode_experts_kernel<false, false>,
                         (const void*)decode_experts_kernel<true, false>,
                         (const void*)decode_experts_kernel<false, true>, (const void*)decode_experts_kernel<true, true>};
  cudaFuncAttributes fk[4];
  size_t static_max = 0;
  for (int m = 0; m < 4 && e == cudaSuccess; ++m) {
    e = cudaFuncGetAttributes(&fk[m], kern[m]);
    static_max = std::max(static_max, fk[m].sharedSizeBytes);
  }
  if (e == cudaSuccess) g_smem_optin -= (int)static_max;
  for (int m = 0; m < 4 && e == cudaSuccess; ++m) {
    e = cudaFuncSetAttribute(kern[m], cudaFuncAttributeMaxDynamicSharedMemorySize, g_smem_optin);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern[m], cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
  }
  // one CTA per SM must fit with the least shared memory a launch asks for:
  // the grid-wide wait relies on every CTA of the grid being resident
  for (int m = 0; m < 4 && e == cudaSuccess; ++m) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern[m], kThreads, (size_t)g_smem_optin / 2 + 1024);
    if (e == cudaSuccess && n < 1) {
      const cudaFuncAttributes& f = fk[m];
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
  const bool q8 = h->cfg.act_q8 != 0;  // Q8 activations: one code plane instead of two
  const uint32_t xb = align128((uint32_t)((q8 ? 1 : 2) * T * H));
  a.off_info = xb;
  a.off_acc = a.off_info + align128((uint32_t)(T * (H / 16) * 8));
  a.off_h = a.off_acc + (multi ? 0u : align128((uint32_t)H * 4u));
  a.off_hp = a.off_h + align128((uint32_t)(2 * tcap * kChunk * 4));
  a.off_ring = a.off_hp + (multi ? align128((uint32_t)(tcap * sizeof(HPlanes))) : 0u);
  const int64_t ring_bytes = (int64_t)g_smem_optin - a.off_ring - 256;
  a.stages = (int)std::min<int64_t>(kMaxStages, ring_bytes / a.stage_bytes);
  if (a.stages < 2) return cudaErrorInvalidConfiguration;
  const int grid = h->num_sms;
  if (!multi) {
    // One token: a CTA streams about ceil((k + S) I/16 / grid) chunks of
    // n_gu + n_dn stages. A ring deeper than a third of that only front-loads
    // the requests: every CTA's first stages then queue behind everyone's
    // later ones (1-token call at H = 2048, nine stages a CTA: ring of 2
    // stages 20.0 us, 3: 18.0, 4: 18.3, 5: 18.4; at H = 7168, 96 stages a
    // CTA, the deepest ring is fastest).
    const int64_t per_cta = ((int64_t)(k + S) * (I / kChunk) + grid - 1) / grid * (kChunk / R + (H + a.Dr - 1) / a.Dr);
    a.stages = (int)std::min<int64_t>(a.stages, std::max<int64_t>(3, (per_cta + 2) / 3));
  }
  // the ring also holds the logits while routing and the sums at the end
  if (grid > kMaxGrid) return cudaErrorInvalidConfiguration;
  // the final sums: part sums (at most max(kCT, T rows) floats), then the per-token CTA lists
  const uint32_t need_end = (uint32_t)((std::max(kCT, T * ((H + grid - 1) / grid)) + T * grid) * 4);
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
  return launch(a, multi, q8, (unsigned)grid, smem, s);
}

}  // namespace fw
