// Prefill path (T > decode_T_max): the experts as grouped GEMMs on the
// tcgen05 tensor cores, with the Q8_0 weights dequantised to bf16 in shared
// memory.
//
// The pages' runtime has a tensor-core GEMM that dequantises stored Q8_0 in
// place against bf16 activations (Flyweight README, §Image generation,
// "balanced" mode), and block-table kernels for prompt-time routed experts
// (§Runtime controls); its NVFP4 prefill path needs Blackwell (0.5.1 page).
// This path keeps bf16 activations and Q8_0 weights rounded to bf16 on their
// way into the MMA, with fp32 accumulation in tensor memory.
//
//   gather:   xperm[pos] = x[token of grouped row pos]           (bf16 rows)
//   GEMM 1:   per (expert, 128-row tile, 256-column tile of the interleaved
//             gate/up rows): acc = X_tile . deq(W_gu)^T; epilogue
//             h = SiLU(gate) * up -> hbuf (bf16, grouped order)
//   GEMM 2:   per (expert, 128-row tile, 256 output columns):
//             Yp = gate_of_row * (h . deq(W_down)^T)  -> yp (bf16)
//   combine:  out[t] = sum_j Yp[inv[t*k + j]] (+ shared row), fixed order
//
// One persistent CTA per SM, 14 warps: 0-3 epilogue (TMEM lane quarters),
// 4 TMA producer, 5 MMA issuer (and TMEM owner), 6-13 dequantisers.
#include <cudaTypedefs.h>

#include <algorithm>

#include "internal.cuh"

namespace fw {
namespace {

using namespace dev;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 3;
constexpr int kEpiWarps = 4, kProducerWarp = 4, kMmaWarp = 5, kDeqWarp0 = 6, kDeqWarps = 8;
constexpr int kThreads = (kDeqWarp0 + kDeqWarps) * 32;  // 448
constexpr uint32_t kABytes = BM * BK * 2;    // 16 KB bf16 A tile
constexpr uint32_t kBBytes = BN * BK * 2;    // 32 KB bf16 B tile
constexpr uint32_t kQBytes = BN * BK;        // 16 KB int8 codes
constexpr uint32_t kSBytes = BN * 2 * 2;     // 1 KB: 2 scale blocks x 256 rows
constexpr uint32_t kSmemBytes = kStages * (kABytes + kBBytes + kQBytes + kSBytes) + 1024;
constexpr uint32_t kTmemCols = 512;          // two 128 x 256 fp32 accumulators

enum Epi { kEpiSwiGLU = 0, kEpiDownScale = 1 };

struct GemmArgs {
  const int4* minfo;      // per 128-row tile: (expert, first row, valid rows, 0)
  const Meta* meta;
  const float* row_gate;  // kEpiDownScale
  __nv_bfloat16* outp;    // hbuf (SwiGLU, [rows][I]) or yp ([rows][H])
  int K;                  // reduction length (H or I)
  int prows;              // weight rows per expert in the code plane (2I or H)
  int n_ntiles;           // ceil(prows / 256)
  int out_cols;           // I (SwiGLU) or H
};

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 operand tile stored with
// the 128-byte swizzle: rows of 128 B (64 bf16 along K), 8-row groups 1024 B
// apart (stride byte offset), descriptor version 1, swizzle mode 2 (128B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// ------------------------------------------------------------- the GEMM
template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_s, GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t a_full[kStages], q_full[kStages], b_full[kStages];
  __shared__ __align__(8) uint64_t ab_empty[kStages], q_empty[kStages];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* base = smem_raw + pad;
  uint8_t* sA = base;
  uint8_t* sB = sA + kStages * kABytes;
  uint8_t* sQ = sB + kStages * kBBytes;
  uint8_t* sS = sQ + kStages * kQBytes;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&q_full[i], 1);
      mbar_init(&b_full[i], kDeqWarps);
      mbar_init(&ab_empty[i], 1);
      mbar_init(&q_empty[i], kDeqWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
    }
    mbar_init(&mma_done, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;

  const int n_tiles = a.meta->n_mtiles * a.n_ntiles;
  const int KT = a.K / BK;
  const int nb = a.K / 32;  // scale blocks per weight row
  bool ok = true;

  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_wait(bar, parity)) return true;
    if (atomicExch(&s_abort, 1) == 0) report_wait(const_cast<Meta*>(a.meta), kSiteGemm, warp, (int)parity);
    return false;
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int4 mi = a.minfo[tile / a.n_ntiles];
        const int n0 = (tile % a.n_ntiles) * BN;
        for (int kb = 0; kb < KT && ok; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!(ok = wait(&ab_empty[s], ph ^ 1))) break;
          if (!(ok = wait(&q_empty[s], ph ^ 1))) break;
          mbar_arrive_expect_tx(&a_full[s], kABytes);
          tma_load_2d(sA + s * kABytes, &map_a, kb * BK, mi.y, &a_full[s]);
          mbar_arrive_expect_tx(&q_full[s], kQBytes + kSBytes);
          tma_load_2d(sQ + s * kQBytes, &map_q, kb * BK, mi.x * a.prows + n0, &q_full[s]);
          tma_load_2d(sS + s * kSBytes, &map_s, n0, mi.x * nb + kb * 2, &q_full[s]);
        }
      }
      // copies still in flight after an abort land before the CTA leaves
      for (uint32_t j = it > kStages ? it - kStages : 0; j < it; ++j) {
        mbar_wait(&a_full[j % kStages], (j / kStages) & 1);
        mbar_wait(&q_full[j % kStages], (j / kStages) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, BN);
      uint32_t it = 0, tc = 0;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tc) {
        const int b = tc & 1;
        if (!(ok = wait(&acc_empty[b], ((tc >> 1) & 1) ^ 1))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * BN;
        for (int kb = 0; kb < KT; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!(ok = wait(&a_full[s], ph))) break;
          if (!(ok = wait(&b_full[s], ph))) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kABytes), b0 = smem_u32(sB + s * kBBytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16(d_tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc, (kb | k) != 0);
          mma_commit(&ab_empty[s]);
        }
        if (ok) mma_commit(&acc_full[b]);
      }
      // every MMA this thread issued has finished before TMEM is released
      mma_commit(&mma_done);
      mbar_wait(&mma_done, 0);
    }
  } else if (warp >= kDeqWarp0) {
    // ------------------------------------------------ dequantisers: int8 x scale -> bf16, swizzled
    const int dt = threadIdx.x - kDeqWarp0 * 32;  // 0..255
    uint32_t it = 0;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      for (int kb = 0; kb < KT && ok; ++kb, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!(ok = wait(&q_full[s], ph))) break;
        if (!(ok = wait(&ab_empty[s], ph ^ 1))) break;
        const uint8_t* q = sQ + s * kQBytes;
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(sS + s * kSBytes);
        uint8_t* bt = sB + s * kBBytes;
#pragma unroll
        for (int i = 0; i < (BN * BK / 16) / 256; ++i) {
          const int item = dt + 256 * i;
          const int r = item >> 2, c = item & 3;
          const uint4 qv = *reinterpret_cast<const uint4*>(q + r * BK + c * 16);
          const float d = half_bits_to_f32(sc[(c >> 1) * BN + r]);
          float f[16];
          u8x4_to_f32(qv.x, f[0], f[1], f[2], f[3]);
          u8x4_to_f32(qv.y, f[4], f[5], f[6], f[7]);
          u8x4_to_f32(qv.z, f[8], f[9], f[10], f[11]);
          u8x4_to_f32(qv.w, f[12], f[13], f[14], f[15]);
          uint4 lo, hi;
          lo.x = pack_bf16x2(f[0] * d, f[1] * d);
          lo.y = pack_bf16x2(f[2] * d, f[3] * d);
          lo.z = pack_bf16x2(f[4] * d, f[5] * d);
          lo.w = pack_bf16x2(f[6] * d, f[7] * d);
          hi.x = pack_bf16x2(f[8] * d, f[9] * d);
          hi.y = pack_bf16x2(f[10] * d, f[11] * d);
          hi.z = pack_bf16x2(f[12] * d, f[13] * d);
          hi.w = pack_bf16x2(f[14] * d, f[15] * d);
          const int sw = r & 7;
          *reinterpret_cast<uint4*>(bt + r * 128 + (((2 * c) ^ sw) << 4)) = lo;
          *reinterpret_cast<uint4*>(bt + r * 128 + (((2 * c + 1) ^ sw) << 4)) = hi;
        }
        fence_proxy_async_smem();  // the generic-proxy stores must be visible to the tensor cores
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&b_full[s]);
          mbar_arrive(&q_empty[s]);
        }
      }
    }
  } else {
    // ------------------------------------------------ epilogue: TMEM -> registers -> global
    const int m = warp * 32 + lane;  // row of the tile = TMEM lane
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tc) {
      const int4 mi = a.minfo[tile / a.n_ntiles];
      const int n0 = (tile % a.n_ntiles) * BN;
      const int b = tc & 1;
      if (!(ok = wait(&acc_full[b], (tc >> 1) & 1))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + b * BN + ((uint32_t)(warp * 32) << 16);
      const bool valid = m < mi.z;
      const int64_t row = (int64_t)mi.y + m;
      if (EPI == kEpiSwiGLU) {
        // columns of the 256-row weight tile: groups of kGUGroup gate rows,
        // then the up rows of the same i; 32 columns give 16 consecutive i
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(taddr + c0, v);
          const int i0 = (n0 + c0) / 2;
          if (valid && i0 < a.out_cols) {
            uint32_t hw[8];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              const int q0 = (j / kGUGroup) * 2 * kGUGroup + j % kGUGroup;
              const int q1 = ((j + 1) / kGUGroup) * 2 * kGUGroup + (j + 1) % kGUGroup;
              hw[j / 2] = pack_bf16x2(silu(v[q0]) * v[q0 + kGUGroup], silu(v[q1]) * v[q1 + kGUGroup]);
            }
            uint4* dst = reinterpret_cast<uint4*>(a.outp + row * a.out_cols + i0);
            dst[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            dst[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
          }
        }
      } else {
        const float gate = valid ? a.row_gate[row] : 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(taddr + c0, v);
          if (valid && n0 + c0 < a.out_cols) {
            uint4* dst = reinterpret_cast<uint4*>(a.outp + row * a.out_cols + n0 + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 w;
              w.x = pack_bf16x2(gate * v[8 * q + 0], gate * v[8 * q + 1]);
              w.y = pack_bf16x2(gate * v[8 * q + 2], gate * v[8 * q + 3]);
              w.z = pack_bf16x2(gate * v[8 * q + 4], gate * v[8 * q + 5]);
              w.w = pack_bf16x2(gate * v[8 * q + 6], gate * v[8 * q + 7]);
              dst[q] = w;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
}

// ------------------------------------------------------------- gather, combine
// xperm[pos] = x[row_token[pos]], 16 bytes per thread.
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ row_token,
                                   int rows, int H, __nv_bfloat16* __restrict__ xperm) {
  const int chunks = H / 8;
  const int64_t n = (int64_t)rows * chunks;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t pos = i / chunks;
    const int c = (int)(i % chunks);
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (int64_t)row_token[pos] * H) + c);
    reinterpret_cast<uint4*>(xperm + pos * H)[c] = v;
  }
}

// out[t] = sum over the token's slots j (ascending) of Yp[inv[t*k + j]], then
// the shared expert's row; fp32 sum, one bf16 rounding.
__global__ void combine_kernel(const __nv_bfloat16* __restrict__ yp, const int32_t* __restrict__ inv, int T, int k,
                               int S, int H, __nv_bfloat16* __restrict__ out) {
  const int chunks = H / 8;
  const int64_t n = (int64_t)T * chunks;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / chunks), c = (int)(i % chunks);
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int j = 0; j < k + S; ++j) {
      const int slot = j < k ? t * k + j : T * k + t;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(yp + (int64_t)inv[slot] * H) + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float lo, hi;
        bf16x2_to_f32(w[q], lo, hi);
        acc[2 * q] += lo;
        acc[2 * q + 1] += hi;
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(out + (int64_t)t * H)[c] = o;
  }
}

// ------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* gaddr, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz,
                      CUtensorMapL2promotion l2) {
  if (!g_encode) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, gaddr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

unsigned grid_for(int64_t n, int threads, int cap) {
  int64_t g = (n + threads - 1) / threads;
  if (g > cap) g = cap;
  return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t configure_prefill_kernels() {
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e != cudaSuccess ? e : cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cudaError_t e = allow_max_dynamic_smem(grouped_gemm_kernel<kEpiSwiGLU>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(grouped_gemm_kernel<kEpiDownScale>);
  return e;
}

cudaError_t prepare_prefill(Handle* h) {
  const uint64_t H = h->cfg.H, I = h->cfg.I, EU = h->EU, R = h->rows_max;
  PrefillMaps* m = new PrefillMaps();
  h->maps = m;
  cudaError_t e = encode_2d(&m->a_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->xperm, H, R, H * 2, BK, BM,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e == cudaSuccess)
    e = encode_2d(&m->a_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->hbuf, I, R, I * 2, BK, BM,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e == cudaSuccess)
    e = encode_2d(&m->q_gu, CU_TENSOR_MAP_DATA_TYPE_UINT8, h->q_gu, H, EU * 2 * I, row_bytes(H), BK, BN,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e == cudaSuccess)
    e = encode_2d(&m->s_gu, CU_TENSOR_MAP_DATA_TYPE_UINT16, h->st_gu, 2 * I, EU * (H / 32), 2 * I * 2, BN, 2,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e == cudaSuccess)
    e = encode_2d(&m->q_d, CU_TENSOR_MAP_DATA_TYPE_UINT8, h->q_d, I, EU * H, row_bytes(I), BK, BN, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e == cudaSuccess)
    e = encode_2d(&m->s_d, CU_TENSOR_MAP_DATA_TYPE_UINT16, h->st_d, H, EU * (I / 32), H * 2, BN, 2,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  return e;
}

cudaError_t launch_ffn_prefill(Handle* h, const __nv_bfloat16* x, int T, __nv_bfloat16* out, cudaStream_t s) {
  if (!h->maps) return cudaErrorNotSupported;
  const int H = h->cfg.H, I = h->cfg.I, k = h->cfg.k, S = h->S;
  const int rows = T * (k + S);
  cudaError_t err;
  {
    KernelTimer tm(h, FW_KERNEL_PREFILL_GATHER, s);
    gather_rows_kernel<<<grid_for((int64_t)rows * (H / 8), 256, h->num_sms * 8), 256, 0, s>>>(x, h->row_token, rows,
                                                                                            H, h->xperm);
  }
  GemmArgs g;
  g.minfo = h->minfo;
  g.meta = h->meta;
  g.row_gate = h->row_gate;
  {
    g.outp = static_cast<__nv_bfloat16*>(h->hbuf);
    g.K = H;
    g.prows = 2 * I;
    g.n_ntiles = (2 * I + BN - 1) / BN;
    g.out_cols = I;
    KernelTimer tm(h, FW_KERNEL_PREFILL_GATEUP, s);
    grouped_gemm_kernel<kEpiSwiGLU><<<h->num_sms, kThreads, kSmemBytes, s>>>(h->maps->a_x, h->maps->q_gu,
                                                                             h->maps->s_gu, g);
  }
  {
    g.outp = h->yp;
    g.K = I;
    g.prows = H;
    g.n_ntiles = (H + BN - 1) / BN;
    g.out_cols = H;
    KernelTimer tm(h, FW_KERNEL_PREFILL_DOWN, s);
    grouped_gemm_kernel<kEpiDownScale><<<h->num_sms, kThreads, kSmemBytes, s>>>(h->maps->a_h, h->maps->q_d,
                                                                                h->maps->s_d, g);
  }
  {
    KernelTimer tm(h, FW_KERNEL_PREFILL_COMBINE, s);
    combine_kernel<<<grid_for((int64_t)T * (H / 8), 256, h->num_sms * 8), 256, 0, s>>>(h->yp, h->inv, T, k, S, H,
                                                                                     out);
  }
  err = cudaGetLastError();
  return err;
}

}  // namespace fw
