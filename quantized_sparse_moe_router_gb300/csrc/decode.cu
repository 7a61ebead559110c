// Decode path (T <= 16): the experts of one call as one fused, HBM-bound
// grouped GEMV kernel.
//
// The pages' runtime runs routed experts through grouped GPU kernels per
// quantisation format, Q8_0 among them (Flyweight README, §Quantization), and
// fuses the gate and up projections so they share one activation load (its
// CPU expert kernels, §Current limitations). Here every selected expert's
// Q8_0 rows are streamed from HBM exactly once per call, in large bulk
// asynchronous copies into a shared-memory ring fed by one producer warp, and
// dequantised in registers by sixteen consumer warps.
//
// One persistent CTA per SM (all resident at once, see launch()):
//   0. after the router's grid completes (programmatic dependent launch), each
//      CTA rebuilds the batch's routing from the logits in shared memory
//      (top-k by rank; deterministic, so every CTA agrees); CTA 0 publishes
//      it;
//   1. gate/up: the CTA's slice of the (touched expert, i) units; for each of
//      the expert's tokens h = SiLU(g) * u -> hbuf (fp32, grouped row order);
//   2. grid-wide barrier (every h written) -- meanwhile the producer keeps
//      streaming this CTA's W_down rows into the ring;
//   3. down + combine: the CTA's output rows in blocks of 16, per block every
//      touched expert in ascending id (shared last); each lane keeps partial
//      sums of gate * (W_down h) per token across the experts, one warp
//      reduction per (row, token) at the end of the block; out[t] (bf16) in a
//      fixed order, no atomics.
#include <algorithm>

#include "routing.cuh"

namespace fw {
namespace {

using namespace dev;

constexpr int kCW = 16;                    // consumer warps
constexpr int kThreads = (kCW + 1) * 32;   // + one producer warp
constexpr int kProducer = kCW;
constexpr int kMaxStages = 16;
constexpr int kRowBlock = 16;              // output rows per W_down block
constexpr int kMaxPer = 2;                 // experts' blocks per W_down stage
constexpr int kMaxRowsOne = 128;           // output rows per CTA of the one-token instantiation
constexpr int kStaticChunks = 2;           // gate/up chunks per CTA assigned without a ticket
constexpr uint32_t kConsumerBarrier = 1;   // named barrier of the 16 consumer warps
constexpr int64_t kL2PrefetchMax = 40ll << 20;  // W_down bytes per call prefetched into L2 (L2 is 129 MB)

enum XMode { kXGlobal = 0, kXSmemF32 = 1, kXSmemBf16 = 2 };

struct DecodeArgs {
  const uint8_t* q_gu;   // rows of row_bytes(H): codes + 128, then binary16 scales
  const uint8_t* q_d;    // rows of row_bytes(I)
  const __nv_bfloat16* x;
  const float* logits;
  float* hbuf;           // [rows][I] fp32
  __nv_bfloat16* out;
  RoutingOut ro;
  Meta* meta;
  int H, I, E, k, S, T;
  int publish;
  int R;                 // gate/up units per stage (a multiple of kGUGroup dividing 32)
  int n_per;             // experts per W_down stage (each a block of <= 16 rows), <= kMaxPer
  uint32_t stage_bytes;  // ring slot size (max of a gate/up and a down stage)
  int stages;
  int x_mode;
  int h_smem;            // h staged in shared memory (fp32)
  uint32_t act_bytes;    // shared-memory area for x, then for h
};
// (smem layouts of x and h: see x16_from_f32_t)

// ------------------------------------------------------------- packed fp32
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

// Four offset-binary codes of a word times four x values (two pairs), added
// to a pair accumulator: the byte permute makes the float 2^23 + q + 128 and
// one packed subtraction leaves q exactly.
__device__ __forceinline__ f2 dot4(uint32_t w, f2 x01, f2 x23, f2 acc) {
  const f2 bias = f2_pack(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
  const f2 m01 = f2_pack_bits(__byte_perm(w, 0x4B000000u, 0x7650), __byte_perm(w, 0x4B000000u, 0x7651));
  const f2 m23 = f2_pack_bits(__byte_perm(w, 0x4B000000u, 0x7652), __byte_perm(w, 0x4B000000u, 0x7653));
  acc = f2_fma(f2_add(m01, bias), x01, acc);
  return f2_fma(f2_add(m23, bias), x23, acc);
}

// sum_{i<16} q_i x_i for one 16-code segment; x as 8 pairs.
__device__ __forceinline__ float dot16(const uint4 q, const f2 (&x)[8]) {
  f2 a = dot4(q.x, x[0], x[1], 0ull);
  f2 b = dot4(q.y, x[2], x[3], 0ull);
  a = dot4(q.z, x[4], x[5], a);
  b = dot4(q.w, x[6], x[7], b);
  return f2_hsum(f2_add(a, b));
}

// Shared-memory vectors (x, h) are stored "segment-transposed" so that lane l
// reading its 16-element segment l touches consecutive 16-byte words in each
// of its loads (no bank conflicts): fp32 element e = 16 seg + 4 i + j of a
// length-K vector sits at i * K/4 + 4 seg + j; bf16 element e = 16 seg + 8 i + j
// at i * K/2 + 8 seg + j.
__device__ __forceinline__ void x16_from_f32_t(const float* v, int K, int seg, f2 (&x)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 w = *reinterpret_cast<const float4*>(v + i * (K / 4) + seg * 4);
    x[2 * i] = f2_pack(w.x, w.y);
    x[2 * i + 1] = f2_pack(w.z, w.w);
  }
}

__device__ __forceinline__ void x16_from_bf16(uint4 a, uint4 b, f2 (&x)[8]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = f2_pack_bits(w[i] << 16, w[i] & 0xFFFF0000u);
}

// h written by other CTAs during this kernel: coherent (L2) loads, not the
// read-only path.
__device__ __forceinline__ void x16_from_f32_global(const float* p, f2 (&x)[8]) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = __ldcg(q + i);
    x[2 * i] = f2_pack(v.x, v.y);
    x[2 * i + 1] = f2_pack(v.z, v.w);
  }
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"r"(kConsumerBarrier), "r"(kCW * 32) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__host__ __device__ inline uint32_t align128(uint32_t v) { return (v + 127) / 128 * 128; }

// ------------------------------------------------------------- the kernel
// kOne: the single-token instantiation (T = 1, x in shared memory as fp32):
// its hot code is the T = 1 paths only, which keeps it small for the
// instruction cache.
template <bool kOne>
__global__ void __launch_bounds__(kThreads, 1) decode_experts_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages];
  __shared__ SmemRouting r;
  __shared__ int2 stage_units[kMaxStages];  // gate/up units [x, y) held by each ring stage (x < 0: no more)
  __shared__ float s_half[2][kMaxRowsOne];   // (one token) the two halves of each output row
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, I = a.I, T = kOne ? 1 : a.T, R = a.R;
  const int x_mode = kOne ? (int)kXSmemF32 : a.x_mode;
  const uint32_t rb_h = (uint32_t)row_bytes(H), rb_i = (uint32_t)row_bytes(I);
  uint8_t* ring = smem + align128(a.act_bytes);
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    fence_mbar_init();
  }
  if (warp != kProducer) {
    // x was written before the router kernel started (that launch waits for
    // the whole stream), so it is staged while the router still runs.
    // segment-transposed, fp32 or bf16 in shared memory (else read from global)
    if (x_mode == kXSmemF32) {
      float* xs = reinterpret_cast<float*>(smem);
      for (int c = tid; c < T * H / 8; c += kCW * 32) {  // c: 8 bf16 = half a segment
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x) + c);
        const int t = c / (H / 8), cc = c % (H / 8), seg = cc >> 1, half = cc & 1;
        float4 lo4, hi4;
        bf16x2_to_f32(v.x, lo4.x, lo4.y);
        bf16x2_to_f32(v.y, lo4.z, lo4.w);
        bf16x2_to_f32(v.z, hi4.x, hi4.y);
        bf16x2_to_f32(v.w, hi4.z, hi4.w);
        float* base = xs + (size_t)t * H + seg * 4;
        *reinterpret_cast<float4*>(base + (2 * half) * (H / 4)) = lo4;
        *reinterpret_cast<float4*>(base + (2 * half + 1) * (H / 4)) = hi4;
      }
    } else if (x_mode == kXSmemBf16) {
      __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);
      for (int c = tid; c < T * H / 8; c += kCW * 32) {
        const int t = c / (H / 8), cc = c % (H / 8), seg = cc >> 1, half = cc & 1;
        *reinterpret_cast<uint4*>(xs + (size_t)t * H + half * (H / 2) + seg * 8) =
            __ldg(reinterpret_cast<const uint4*>(a.x) + c);
      }
    }
  }
  pdl_wait();  // the router's logits (and its reset of the grid barrier)
  if (kOne)
    route_one_in_smem<kThreads>(a.logits, a.E, a.k, a.S, r);
  else
    route_in_smem<kThreads>(a.logits, T, a.E, a.k, a.S, r);
  if (a.publish && blockIdx.x == 0) publish_routing<kThreads>(r, T, a.E, a.k, a.S, a.ro);

  const int nU = r.n_unique;
  // gate/up work, in stages of at most R consecutive units of the nU x I unit
  // space (never across an expert, since R divides I: a stage is one run of
  // consecutive interleaved rows of one expert, one copy).
  //  * one token: the units are split evenly, each CTA a contiguous range
  //    starting and ending on a kGUGroup boundary (every unit costs the same);
  //  * several tokens: the cost of a unit is its expert's token count, so
  //    R-unit chunks are handed out -- CTA b's first kStaticChunks are b,
  //    b + grid, ..., the rest come from a ticket counter.
  // (32-bit indices throughout the loops: a 64-bit division is a long
  // software routine, and these run once per stage in every warp)
  const int n_units = nU * I;
  const int64_t n_grp = n_units / kGUGroup;
  const int lo = (int)(n_grp * blockIdx.x / gridDim.x) * kGUGroup;
  const int hi = (int)(n_grp * (blockIdx.x + 1) / gridDim.x) * kGUGroup;
  // down stages: output rows [o0, o1), blocks of 16 rows; per block every touched expert
  const int o0 = (int)((int64_t)H * blockIdx.x / gridDim.x), o1 = (int)((int64_t)H * (blockIdx.x + 1) / gridDim.x);
  // (a down stage holds the same 16-row block of up to n_per experts, so that
  // a warp's dot products for those experts overlap)
  const int n_blk = (o1 - o0 + kRowBlock - 1) / kRowBlock;
  const int n_ge = (nU + a.n_per - 1) / a.n_per;
  const int n_dn = n_ge * n_blk;

  if (warp == kProducer) {
    // ------------------------------------------------------ producer
    if (lane == 0) {
      // Once the ring is full of gate/up stages, ask L2 for all of this CTA's
      // W_down rows, so that they stream from HBM alongside gate/up instead
      // of after it -- when the call's W_down fits comfortably in L2.
      bool pf = (int64_t)nU * H * rb_i <= kL2PrefetchMax;
      // (several tokens) chunk of the current stage and of the next two: the
      // ticket for the second is requested two stages ahead, so its round
      // trip overlaps copies
      int j = 0, c = blockIdx.x, q0 = blockIdx.x + gridDim.x, q1 = 0;
      if (!kOne) q1 = (int)atomicAdd(&a.meta->chunk_ctr, 1u) + kStaticChunks * (int)gridDim.x;
      int su = lo;      // (one token) next unit of the CTA's range
      bool gu = true;   // still issuing gate/up stages
      int st = 0;       // j % stages
      uint32_t ph = 0;  // (j / stages) & 1
      int ge = 0, blk = 0;  // down stage jd: expert group, row block
      for (int jd = 0; gu || jd < n_dn;) {
        if (pf && j == a.stages) {  // the ring is full: the TMA unit has time for it
          pf = false;
          for (int u = 0; u < nU; ++u) {
            const int64_t row = (int64_t)r.u[u].x * H + o0;
            prefetch_l2(a.q_d + row * rb_i, (uint32_t)(o1 - o0) * rb_i);
          }
        }
        if (j >= a.stages && !mbar_wait(&empty[st], ph ^ 1u)) {
          report_wait(a.meta, kSiteGuEmpty, j, n_dn);
          break;
        }
        uint8_t* sb = ring + (size_t)st * a.stage_bytes;
        if (gu) {
          int u0, u1;
          if (kOne) {
            u0 = su;
            u1 = ::min(hi, (su / R + 1) * R);
            su = u1;
          } else {
            u0 = c * R;
            u1 = u0 + R;
            c = q0;
            q0 = q1;
            q1 = (int)atomicAdd(&a.meta->chunk_ctr, 1u) + kStaticChunks * (int)gridDim.x;
          }
          if (u0 >= (kOne ? hi : n_units)) {
            gu = false;
            if (kOne) continue;  // the consumers know the count: this slot goes to the down stages
            stage_units[st] = make_int2(-1, -1);  // ticketed work: an empty stage tells the consumers
            mbar_arrive(&full[st]);
          } else {
            stage_units[st] = make_int2(u0, u1);
            const int eu = u0 / I;  // a stage never spans two experts (R divides I)
            const int e = r.u[eu].x, i0 = u0 - eu * I;
            const uint32_t bytes = (uint32_t)(u1 - u0) * 2 * rb_h;
            mbar_arrive_expect_tx(&full[st], bytes);
            bulk_g2s(sb, a.q_gu + ((int64_t)e * 2 * I + 2 * i0) * rb_h, bytes, &full[st]);
          }
        } else {
          // block-major: all expert groups of block 0, then block 1, ...
          const int e0 = ge * a.n_per, e1 = ::min(nU, e0 + a.n_per);
          const int r0 = o0 + blk * kRowBlock, nr = ::min(kRowBlock + 0, o1 - r0);
          mbar_arrive_expect_tx(&full[st], (uint32_t)(e1 - e0) * nr * rb_i);
          for (int u = e0; u < e1; ++u)
            bulk_g2s(sb + (size_t)(u - e0) * kRowBlock * rb_i, a.q_d + ((int64_t)r.u[u].x * H + r0) * rb_i,
                     (uint32_t)nr * rb_i, &full[st]);
          ++jd;
          if (++ge == n_ge) {
            ge = 0;
            ++blk;
          }
        }
        ++j;
        if (++st == a.stages) {
          st = 0;
          ph ^= 1u;
        }
      }
      // every copy issued has landed before the CTA may leave
      for (int q = ::max(0, j - a.stages); q < j; ++q)
        mbar_wait(&full[q % a.stages], (uint32_t)((q / a.stages) & 1));
    }
  } else {
    // ------------------------------------------------------ consumers
    bool ok = true;  // (x is visible: route_in_smem ends with a CTA barrier)

    // ---- phase 1: gate/up. Every consumer warp passes every stage in order
    // (no wait is ever more than one phase ahead of its barrier) and computes
    // its units of the stage's chunk, until the empty stage.
    const int nseg_h = H / 16;
    // stages of gate/up work this CTA took (ticketed work: then one empty stage)
    int n_gu = kOne ? (hi > lo ? (hi + R - 1) / R - lo / R : 0) : 0;
    int st = 0;       // j % stages
    uint32_t ph = 0;  // (j / stages) & 1
    for (int j = 0; ok && (!kOne || j < n_gu); ++j) {
      if (!mbar_wait(&full[st], ph)) {
        report_wait(a.meta, kSiteGuFull, j, warp);
        ok = false;
        break;
      }
      const int2 su = stage_units[st];
      if (su.x < 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        n_gu = j + 1;
        break;
      }
      const int u0 = su.x, u1 = su.y;
      const uint8_t* sb = ring + (size_t)st * a.stage_bytes;
      const int eu = u0 / I;  // the stage's expert (a stage never spans two)
      const int4 ui = r.u[eu];
      // units alternate over the warps from stage to stage: unit q of stage j
      // goes to warp (j R + q) mod 16
      for (int g = u0 + ((warp - j * R) % kCW + kCW) % kCW; g < u1; g += kCW) {
        // the stage holds rows 2 i0 .. 2 i1 of the expert: per group, kGUGroup
        // gate rows then their up rows; u0 is group-aligned
        const int off = (int)(g - u0);
        const uint8_t* qg_row = sb + (size_t)((off / kGUGroup) * 2 * kGUGroup + off % kGUGroup) * rb_h;
        const uint8_t* qu_row = qg_row + (size_t)kGUGroup * rb_h;
        const uint16_t* sg = reinterpret_cast<const uint16_t*>(qg_row + H);
        const uint16_t* su = reinterpret_cast<const uint16_t*>(qu_row + H);
        const int i = g - eu * I;
        auto load_x = [&](int t, int seg, f2(&xv)[8]) {
          if (x_mode == kXSmemF32) {
            x16_from_f32_t(reinterpret_cast<const float*>(smem) + (size_t)t * H, H, seg, xv);
          } else if (x_mode == kXSmemBf16) {
            const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(smem) + (size_t)t * H;
            x16_from_bf16(*reinterpret_cast<const uint4*>(xb + seg * 8), *reinterpret_cast<const uint4*>(xb + H / 2 + seg * 8),
                          xv);
          } else {
            const uint4* xp = reinterpret_cast<const uint4*>(a.x + (size_t)t * H + seg * 16);
            x16_from_bf16(__ldg(xp), __ldg(xp + 1), xv);
          }
        };
        if (T == 1) {
          // one row: two segments per pass, independent accumulators
          float ag0 = 0.f, au0 = 0.f, ag1 = 0.f, au1 = 0.f;
          int seg = lane;
          for (; seg + 32 < nseg_h; seg += 64) {
            f2 x0[8], x1[8];
            load_x(0, seg, x0);
            load_x(0, seg + 32, x1);
            const uint4 g0 = *reinterpret_cast<const uint4*>(qg_row + seg * 16);
            const uint4 v0 = *reinterpret_cast<const uint4*>(qu_row + seg * 16);
            const uint4 g1 = *reinterpret_cast<const uint4*>(qg_row + (seg + 32) * 16);
            const uint4 v1 = *reinterpret_cast<const uint4*>(qu_row + (seg + 32) * 16);
            ag0 = fmaf(half_bits_to_f32(sg[seg >> 1]), dot16(g0, x0), ag0);
            au0 = fmaf(half_bits_to_f32(su[seg >> 1]), dot16(v0, x0), au0);
            ag1 = fmaf(half_bits_to_f32(sg[(seg + 32) >> 1]), dot16(g1, x1), ag1);
            au1 = fmaf(half_bits_to_f32(su[(seg + 32) >> 1]), dot16(v1, x1), au1);
          }
          if (seg < nseg_h) {
            f2 x0[8];
            load_x(0, seg, x0);
            const uint4 g0 = *reinterpret_cast<const uint4*>(qg_row + seg * 16);
            const uint4 v0 = *reinterpret_cast<const uint4*>(qu_row + seg * 16);
            ag0 = fmaf(half_bits_to_f32(sg[seg >> 1]), dot16(g0, x0), ag0);
            au0 = fmaf(half_bits_to_f32(su[seg >> 1]), dot16(v0, x0), au0);
          }
          const float accg = warp_sum(ag0 + ag1), accu = warp_sum(au0 + au1);
          if (lane == 0) a.hbuf[(int64_t)ui.y * I + i] = silu(accg) * accu;
        } else {
          for (int rr = 0; rr < ui.z; ++rr) {
            const int pos = ui.y + rr;
            const int t = r.tok[pos];
            float accg = 0.f, accu = 0.f;
            for (int seg = lane; seg < nseg_h; seg += 32) {
              f2 xv[8];
              load_x(t, seg, xv);
              const uint4 qg = *reinterpret_cast<const uint4*>(qg_row + seg * 16);
              const uint4 qu = *reinterpret_cast<const uint4*>(qu_row + seg * 16);
              accg = fmaf(half_bits_to_f32(sg[seg >> 1]), dot16(qg, xv), accg);
              accu = fmaf(half_bits_to_f32(su[seg >> 1]), dot16(qu, xv), accu);
            }
            accg = warp_sum(accg);
            accu = warp_sum(accu);
            if (lane == 0) a.hbuf[(int64_t)pos * I + i] = silu(accg) * accu;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (++st == a.stages) {
        st = 0;
        ph ^= 1u;
      }
    }

    // ---- phase 2: every CTA's h is written before any CTA reads it. The
    // arrival is a release (ordering this CTA's h stores, which the consumer
    // barrier ordered before it), the poll an acquire.
    consumer_sync();
    if (tid == 0) {
      unsigned long long* gb = reinterpret_cast<unsigned long long*>(&a.meta->gbar);
      asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(gb) : "memory");
      if (ld_acquire_u64(gb) < gridDim.x) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_u64(gb) < gridDim.x) {
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            report_wait(a.meta, kSiteGrid, 0, gridDim.x);
            break;
          }
        }
      }
    }
    consumer_sync();
    if (a.h_smem) {  // x is no longer read: the area now takes h, segment-transposed
      float* hs = reinterpret_cast<float*>(smem);
      const int q4 = I / 4;
      for (int c = tid; c < r.rows * q4; c += kCW * 32) {  // c: 4 floats
        const int pos = c / q4, cc = c % q4, seg = cc >> 2, i = cc & 3;
        *reinterpret_cast<float4*>(hs + (size_t)pos * I + i * (I / 4) + seg * 4) =
            __ldcg(reinterpret_cast<const float4*>(a.hbuf) + c);
      }
      consumer_sync();
    }

    // ---- phase 3: down + combine. Warp w owns row w of every 16-row block;
    // per block it visits every touched expert (ascending id, shared last)
    // keeping per-lane partial sums per token, and reduces across the warp
    // once, at the end of the block. The experts of a stage are processed
    // together (independent dot products in flight).
    const float* hsrc = a.h_smem ? reinterpret_cast<const float*>(smem) : a.hbuf;
    const int nseg_i = I / 16;
    float part[kMaxDecodeT];
#pragma unroll
    for (int t = 0; t < kMaxDecodeT; ++t) part[t] = 0.f;
    st = n_gu % a.stages;  // ring position of stage n_gu + jd
    ph = (uint32_t)(n_gu / a.stages) & 1u;
    int ge = 0, blk = 0;  // expert group and row block of down stage jd
    for (int jd = 0; jd < n_dn && ok; ++jd) {
      if (!mbar_wait(&full[st], ph)) {
        report_wait(a.meta, kSiteDnFull, n_gu + jd, warp);
        ok = false;
        break;
      }
      const int e0 = ge * a.n_per, ne = ::min(nU, e0 + a.n_per) - e0;
      const int r0 = o0 + blk * kRowBlock;
      const int nr = ::min(kRowBlock + 0, o1 - r0);
      if (kOne) {
        // one token: warp w takes rows ra = w & 7 and ra + 8 of the block and
        // the segments of parity w >> 3, so an h segment is loaded once for
        // two rows; the two halves of a row are added after the loop
        const int ra = warp & 7, hf = warp >> 3;
        if (ra < nr) {
          const bool has_b = ra + 8 < nr;
          const uint8_t* sa = ring + (size_t)st * a.stage_bytes + (size_t)ra * rb_i;
          float da[kMaxPer], db[kMaxPer];
          const float* hrow[kMaxPer];
#pragma unroll
          for (int el = 0; el < kMaxPer; ++el) {
            da[el] = 0.f;
            db[el] = 0.f;
            hrow[el] = hsrc + (size_t)(el < ne ? r.u[e0 + el].y : 0) * I;
          }
          for (int seg = 2 * lane + hf; seg < nseg_i; seg += 64) {
#pragma unroll
            for (int el = 0; el < kMaxPer; ++el) {
              if (el < ne) {
                const uint8_t* qa = sa + (size_t)el * kRowBlock * rb_i;
                f2 hv[8];
                if (a.h_smem)
                  x16_from_f32_t(hrow[el], I, seg, hv);
                else
                  x16_from_f32_global(hrow[el] + seg * 16, hv);
                const uint4 qq = *reinterpret_cast<const uint4*>(qa + seg * 16);
                da[el] = fmaf(half_bits_to_f32(reinterpret_cast<const uint16_t*>(qa + I)[seg >> 1]), dot16(qq, hv),
                              da[el]);
                if (has_b) {
                  const uint8_t* qb = qa + (size_t)8 * rb_i;
                  const uint4 qr = *reinterpret_cast<const uint4*>(qb + seg * 16);
                  db[el] = fmaf(half_bits_to_f32(reinterpret_cast<const uint16_t*>(qb + I)[seg >> 1]), dot16(qr, hv),
                                db[el]);
                }
              }
            }
          }
#pragma unroll
          for (int el = 0; el < kMaxPer; ++el)
            if (el < ne) {
              const float g = r.gates[r.slot[r.u[e0 + el].y]];
              part[0] = fmaf(g, da[el], part[0]);
              part[1] = fmaf(g, db[el], part[1]);
            }
        }
      } else if (warp < nr) {
        const uint8_t* sb = ring + (size_t)st * a.stage_bytes + (size_t)warp * rb_i;
        if (T == 1) {        } else {
          for (int el = 0; el < ne; ++el) {
            const int4 ui = r.u[e0 + el];
            const uint8_t* qrow = sb + (size_t)el * kRowBlock * rb_i;
            const uint16_t* sc = reinterpret_cast<const uint16_t*>(qrow + I);
            for (int m = 0; m < ui.z; ++m) {
              const int pos = ui.y + m;
              const float* hr = hsrc + (size_t)pos * I;
              float d = 0.f;
              for (int seg = lane; seg < nseg_i; seg += 32) {
                f2 hv[8];
                if (a.h_smem)
                  x16_from_f32_t(hr, I, seg, hv);
                else
                  x16_from_f32_global(hr + seg * 16, hv);
                const uint4 qq = *reinterpret_cast<const uint4*>(qrow + seg * 16);
                d = fmaf(half_bits_to_f32(sc[seg >> 1]), dot16(qq, hv), d);
              }
              const float g = r.gates[r.slot[pos]];
              const int t = r.tok[pos];
#pragma unroll
              for (int tt = 0; tt < kMaxDecodeT; ++tt)
                if (tt == t) part[tt] = fmaf(g, d, part[tt]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (ge == n_ge - 1 && kOne) {  // block done: this warp's halves of its two rows
        const float va = warp_sum(part[0]), vb = warp_sum(part[1]);
        const int ra = warp & 7, hf = warp >> 3, rr = blk * kRowBlock + ra;
        if (lane == 0 && ra < nr) s_half[hf][rr] = va;
        if (lane == 0 && ra + 8 < nr) s_half[hf][rr + 8] = vb;
        part[0] = 0.f;
        part[1] = 0.f;
      } else if (ge == n_ge - 1) {  // block done: one reduction per token, lane t writes token t
        if (warp < nr) {
          float mine = 0.f;
#pragma unroll
          for (int tt = 0; tt < kMaxDecodeT; ++tt) {
            if (tt < T) {
              const float v = warp_sum(part[tt]);
              if (lane == tt) mine = v;
            }
            part[tt] = 0.f;
          }
          if (lane < T) a.out[(int64_t)lane * H + r0 + warp] = __float2bfloat16_rn(mine);
        }
      }
      if (++ge == n_ge) {
        ge = 0;
        ++blk;
      }
      if (++st == a.stages) {
        st = 0;
        ph ^= 1u;
      }
    }
    if (kOne) {  // every consumer warp gets here (a timed-out wait ends the loop, not the warp)
      consumer_sync();
      for (int i = tid; i < o1 - o0; i += kCW * 32) a.out[o0 + i] = __float2bfloat16_rn(s_half[0][i] + s_half[1][i]);
    }
  }
  __syncthreads();
}

// The grid-wide barrier needs every CTA resident: the grid is one CTA per SM
// and each CTA takes most of an SM's shared memory, so once earlier work has
// drained all of them are; if something else holds SMs past the wait limit
// the call reports FW_ETIMEOUT instead of hanging.
cudaError_t launch(const DecodeArgs& a, unsigned grid, size_t smem, cudaStream_t s) {
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
  const bool one = a.T == 1 && a.x_mode == kXSmemF32 && (a.H + (int)grid - 1) / (int)grid <= kMaxRowsOne;
  return one ? cudaLaunchKernelEx(&cfg, decode_experts_kernel<true>, a)
             : cudaLaunchKernelEx(&cfg, decode_experts_kernel<false>, a);
}

int g_smem_optin = 0;
constexpr uint32_t kActMax = 80 * 1024;     // x or h in shared memory up to this size
constexpr uint32_t kStageTarget = 36 * 1024;  // one bulk copy per stage: fewer, larger copies stream faster

}  // namespace

cudaError_t configure_decode_kernels() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  // the dynamic budget is what the larger static footprint of the two
  // instantiations leaves (the one-token one also holds the row halves)
  cudaFuncAttributes fa, fb;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, decode_experts_kernel<false>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fb, decode_experts_kernel<true>);
  if (e == cudaSuccess) {
    g_smem_optin -= (int)std::max(fa.sharedSizeBytes, fb.sharedSizeBytes);
    e = cudaFuncSetAttribute(decode_experts_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, g_smem_optin);
  }
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_experts_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, g_smem_optin);
  return e;
}

cudaError_t launch_ffn_decode(Handle* h, const __nv_bfloat16* x, int T, __nv_bfloat16* out, bool publish,
                              int32_t* ids_out, float* gates_out, cudaStream_t s) {
  const int H = h->cfg.H, I = h->cfg.I, k = h->cfg.k, S = h->S;
  const int rows = T * (k + S);
  const int grid = h->num_sms;
  DecodeArgs a;
  a.q_gu = h->q_gu;
  a.q_d = h->q_d;
  a.x = x;
  a.logits = h->logits;
  a.hbuf = static_cast<float*>(h->hbuf);
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
  const uint32_t x32 = (uint32_t)T * H * 4, x16 = (uint32_t)T * H * 2, hb = (uint32_t)rows * I * 4;
  a.x_mode = x32 <= 32 * 1024 ? kXSmemF32 : (x16 <= kActMax ? kXSmemBf16 : kXGlobal);
  a.h_smem = hb <= kActMax;
  const uint32_t xb = a.x_mode == kXSmemF32 ? x32 : (a.x_mode == kXSmemBf16 ? x16 : 0);
  a.act_bytes = std::max(xb, a.h_smem ? hb : 0u);
  const uint32_t unit = (uint32_t)(2 * row_bytes(H));
  int R = 32;
  while (R > kGUGroup && (uint32_t)R * unit > kStageTarget) R /= 2;
  a.R = R;
  const uint32_t dn_block = (uint32_t)(kRowBlock * row_bytes(I));
  a.n_per = (int)std::max<uint32_t>(1, std::min<uint32_t>(kMaxPer, (uint32_t)R * unit / dn_block));
  a.stage_bytes = std::max((uint32_t)R * unit, (uint32_t)a.n_per * dn_block);
  const int64_t ring_bytes = (int64_t)g_smem_optin - align128(a.act_bytes) - 256;
  a.stages = (int)std::min<int64_t>(kMaxStages, ring_bytes / a.stage_bytes);
  if (a.stages < 2) return cudaErrorInvalidConfiguration;
  // at least half the SM's shared memory, so that no two CTAs share an SM
  const size_t smem = std::max<size_t>(align128(a.act_bytes) + (size_t)a.stages * a.stage_bytes,
                                       (size_t)g_smem_optin / 2 + 1024);
  KernelTimer tm(h, FW_KERNEL_DECODE_EXPERTS, s);
  return launch(a, (unsigned)grid, smem, s);
}

}  // namespace fw
