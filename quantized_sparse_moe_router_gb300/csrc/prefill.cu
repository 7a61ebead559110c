// Prefill path (T > decode_T_max): the experts as grouped GEMMs on the
// tcgen05 tensor cores, with the Q8_0 weights dequantised to bf16 straight
// into tensor memory.
//
// The pages' runtime has a tensor-core GEMM that dequantises stored Q8_0 in
// place against bf16 activations (Flyweight README, §Image generation,
// "balanced" mode), and block-table kernels for prompt-time routed experts
// (§Runtime controls); its NVFP4 prefill path needs Blackwell (0.5.1 page).
// This path keeps bf16 activations and Q8_0 weights rounded to bf16 on their
// way into the MMA, with fp32 accumulation in tensor memory.
//
//   gather:   xperm[pos] = x[token of grouped row pos]           (bf16 rows)
//   GEMM 1:   per (token tile of one expert, 128 interleaved gate/up rows):
//             D = deq(W_gu rows) . X_tile^T; epilogue h = SiLU(gate) * up
//             -> hbuf (bf16, grouped order)
//   GEMM 2:   per (token tile, 128 output features):
//             Yp = deq(W_down rows) . h_tile^T -> yp (bf16)
//   combine:  out[t] = sum_j g[t, j] Yp[inv[t*k + j]] (+ shared row), fixed order
//
// The weights are the MMA's A operand (M = 128 rows, read from tensor
// memory, written there by the dequantising warps with tcgen05.st); the
// tokens are B (N = the tile's rows rounded up to 16; K-major bf16 in shared
// memory, 128-byte swizzle, loaded by TMA). So the bf16 weights never pass
// through shared memory, and a partial token tile costs only the MMA columns
// it uses. Three shapes of the kernel, by the rows of the token tile (up to
// 192, 96 or 64), against one or two 128-row weight blocks per CTA.
//
// One persistent CTA per SM, 15 warps: 0-3 epilogue (TMEM lane quarters), 4
// TMA producer, 5 MMA issuer (and TMEM owner), 6-13 dequantisers (two groups
// of four, one per lane quarter, taking alternate stages; a thread converts
// the 64 codes of its weight row in each block of the stage), 14 the second
// MMA issuer of the two-block shapes.
#include <cudaTypedefs.h>

#include <algorithm>

#include "routing.cuh"

namespace fw {
namespace {

using namespace dev;

constexpr int BM = 128, BK = 64;
constexpr int kEpiWarps = 4, kProducerWarp = 4, kMmaWarp = 5, kDeqWarp0 = 6, kDeqWarps = 8;
constexpr int kMmaWarp2 = kDeqWarp0 + kDeqWarps;        // the second MMA issuer (two-block shape)
constexpr int kThreads = (kMmaWarp2 + 1) * 32;          // 480
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSmemLimit = 227 * 1024; // dynamic shared memory a CTA may have

// The three shapes of the grouped GEMM, by the rows of the token tile. A
// stage brings a K step of the token tile and of MB weight tiles; the SM
// takes in at most about 65 GB/s from L2 whatever the mix, so the fewer token
// bytes per weight byte, the closer the weights stream to the HBM rate:
//   kBig   (tiles of 97..192 rows): one 128-row weight block per CTA -- the
//          compute-heavy tiles (an expert's full 192-row tiles);
//   kMid   (65..96 rows): two weight blocks per CTA (12 KB of tokens for
//          17 KB of codes);
//   kSmall (1..64 rows): two weight blocks per CTA (8 KB for 17 KB).
// Accumulators are double-buffered; the rest of tensor memory holds A stages.
enum TileShape { kBig = 0, kMid = 1, kSmall = 2 };

template <int SH>
struct Shape {
  static constexpr int MB = SH == kBig ? 1 : 2;                  // 128-row weight blocks per CTA
  static constexpr int BN = SH == kBig ? kTokTile : (SH == kMid ? kMidTile : kSmallTile);  // MMA N <= BN
  // token rows per TMA box
  static constexpr int XBox = SH == kBig ? BN / 2 : BN;
  static constexpr uint32_t XBytes = BN * BK * 2;                // bf16 token tile slot
  static constexpr uint32_t WBytes = MB * kTileBytes;            // MB weight tiles: codes, then scales
  static constexpr uint32_t StageBytes = XBytes + WBytes;
  static constexpr int Stages = (int)((kSmemLimit - 2048) / StageBytes) & ~1;
  static constexpr uint32_t SmemBytes = Stages * StageBytes + 1024;
  static constexpr uint32_t AccCols = MB * BN;                   // one accumulator buffer (MB blocks)
  static constexpr uint32_t ACol0 = 2 * AccCols;                 // A stages after the two buffers
  static constexpr uint32_t ACols = MB * BK / 2;                 // one A stage: 64 bf16 per row per block
  static constexpr int AStages = (int)((kTmemCols - ACol0) / ACols) & ~1;
  static_assert(AStages >= 2 && ACol0 + AStages * ACols <= kTmemCols, "tensor memory budget");
  static_assert(BN % XBox == 0 && BN % 16 == 0 && BN <= 256 && XBox % 8 == 0, "token tile");
  static_assert(BM == kTileRows && BK == kTileK, "a stage holds whole weight tiles");
  static_assert(Stages >= 4 && Stages % 2 == 0, "the two dequantising groups own alternate stages");
};

enum Epi { kEpiSwiGLU = 0, kEpiDown = 1 };

struct GemmArgs {
  const uint8_t* wt;      // the projection's weight tiles [EU][n_mb][K/64]
  const int4* minfo;      // per token tile: (expert, first grouped row, valid rows, 0)
  const int32_t* n_mtiles; // number of tiles in minfo (written by the scan kernel)
  const Meta* meta;
  __nv_bfloat16* outp;    // hbuf (SwiGLU, [rows][I]) or yp ([rows][H])
  int K;                  // reduction length (H or I)
  int prows;              // weight rows per expert in the code plane (2I or H)
  int n_mb;               // ceil(prows / 128): weight tiles per expert and K step
  int out_cols;           // I (SwiGLU) or H
  int wait_prev;          // launched as a dependent that reads its predecessor's output (the gather's)
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

// D (tensor memory) [+]= A (tensor memory, lane = row) x B (shared memory descriptor)
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (tensor memory) [+]= A (shared memory descriptor) x B (shared memory descriptor)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
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

// 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}


__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

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

// The code byte placed by a byte permute in bits 8..15 of the float
// 2^23 + 256 (q + 128); with d' = d / 256, fma(m, d', -(2^15 + 2^7) d) is
// q d exactly (every product and the constant fit in fp32's 24 bits), then
// one rounding to bf16: one packed op fewer than subtract-then-multiply.
__device__ __forceinline__ uint32_t deq_pair_fma(uint32_t bits_lo, uint32_t bits_hi, f2 dd, f2 cc) {
  f2 m = f2_pack_bits(bits_lo, bits_hi), w;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(w) : "l"(m), "l"(dd), "l"(cc));
  uint32_t r;
  asm("{\n\t.reg .f32 a, b;\n\tmov.b64 {a, b}, %1;\n\tcvt.rn.bf16x2.f32 %0, b, a;\n\t}" : "=r"(r) : "l"(w));
  return r;
}

// ------------------------------------------------------------- the GEMM
template <int EPI, int SH>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_b, GemmArgs a) {
  using G = Shape<SH>;
  constexpr int MB = G::MB;
  constexpr int kStages = G::Stages, kAStages = G::AStages;
  constexpr int kIssuers = MB;  // MMA-issuing threads: one per weight block
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], a_full[kAStages], a_empty[kAStages];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the next GEMM of the call may start on SMs this grid leaves (its tiles
  // are independent of this grid's; see launch_gemm) -- once this grid's own
  // inputs are complete
  if (a.wait_prev) pdl_wait();
  pdl_launch_dependents();
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* base = smem_raw + pad;
  uint8_t* sX = base;                            // [kStages][BN rows][128 B], 128B swizzle
  uint8_t* sW = sX + kStages * G::XBytes;        // [kStages][MB] weight tiles: [128 rows][64 B] swizzled, [2][128] scales

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kIssuers);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&a_full[i], kDeqWarps / 2);  // one group of four warps per stage
      mbar_init(&a_empty[i], kIssuers);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], kIssuers);
      mbar_init(&acc_empty[i], kEpiWarps);
    }
    mbar_init(&mma_done, kIssuers);
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

  // tiles: (token tile, group of MB weight blocks), token-tile-major, so the
  // CTAs working on one token tile at the same time read it from L2 (a block
  // past the matrix is neither loaded nor stored)
  const int n_mbg = (a.n_mb + MB - 1) / MB;
  const int n_tiles = *a.n_mtiles * n_mbg;
  const int cid = blockIdx.x, ncl = gridDim.x;
  const int KT = a.K / BK;
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
      int4 mi_next = cid < n_tiles ? a.minfo[cid / n_mbg] : make_int4(0, 0, 0, 0);
      for (int tile = cid; tile < n_tiles && ok; tile += ncl) {
        const int4 mi = mi_next;
        const int mb0 = (tile % n_mbg) * MB;  // this CTA's first weight block
        const int nw = ::max(0, ::min(MB, a.n_mb - mb0));  // blocks within the matrix (the rest: no copy, no store)
        const int nx = (mi.z + G::XBox - 1) / G::XBox;
        if (tile + ncl < n_tiles) mi_next = a.minfo[(tile + ncl) / n_mbg];  // in flight during this tile
        const uint8_t* wsrc = a.wt + gemm_tile_offset(mi.x, mb0, 0, a.n_mb, KT);
        for (int kb = 0; kb < KT && ok; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!(ok = wait(&empty[s], ph ^ 1))) break;
          mbar_arrive_expect_tx(&full[s], (uint32_t)nx * G::XBox * BK * 2 + (uint32_t)nw * kTileBytes);
          for (int x = 0; x < nx; ++x)
            tma_load_2d(sX + s * G::XBytes + x * G::XBox * 128, &map_b, kb * BK, mi.y + x * G::XBox, &full[s]);
          for (int b = 0; b < nw; ++b)  // tile (expert, mb0 + b, kb): one contiguous copy
            bulk_g2s(sW + s * G::WBytes + b * kTileBytes, wsrc + ((int64_t)b * KT + kb) * kTileBytes, kTileBytes,
                     &full[s]);
        }
      }
      // copies still in flight after an abort land before the CTA leaves
      for (uint32_t j = it > kStages ? it - kStages : 0; j < it; ++j) mbar_wait(&full[j % kStages], (j / kStages) & 1);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp2) {
    // ------------------------------------------------ MMA issuers
    // At the small tiles' N <= 64 one thread's MMAs and commits keep the
    // tensor pipe busy less than half of the time, two issuing threads reach
    // its peak: with two weight blocks each block has its own issuing warp
    // (both wait for the same stages; the barriers the MMAs release count
    // both commits).
    if (lane == 0 && (warp == kMmaWarp || kIssuers == 2)) {
      const int q = warp == kMmaWarp ? 0 : 1;
      uint32_t it = 0, tc = 0;
      int4 mi_next = cid < n_tiles ? a.minfo[cid / n_mbg] : make_int4(0, 0, 0, 0);
      for (int tile = cid; tile < n_tiles && ok; tile += ncl, ++tc) {
        const int4 mi = mi_next;
        if (tile + ncl < n_tiles) mi_next = a.minfo[(tile + ncl) / n_mbg];
        const int n_mma = (mi.z + 15) / 16 * 16;
        const uint32_t idesc = idesc_bf16(BM, n_mma);
        const int b = tc & 1;
        if (!(ok = wait(&acc_empty[b], ((tc >> 1) & 1) ^ 1))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * G::AccCols;
        for (int kb = 0; kb < KT; ++kb, ++it) {
          const int s = it % kStages, sa = it % kAStages;
          if (!(ok = wait(&full[s], (it / kStages) & 1))) break;
          if (!(ok = wait(&a_full[sa], (it / kAStages) & 1))) break;
          tc_fence_after();
          const uint32_t b0 = smem_u32(sX + s * G::XBytes);
          const uint32_t a0 = tmem_base + G::ACol0 + sa * G::ACols;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)  // block q
            mma_tmem_a(d_tmem + q * G::BN, a0 + q * (BK / 2) + k * 8, sw128_desc(b0 + k * 32), idesc, (kb | k) != 0);
          mma_commit(&empty[s]);
          mma_commit(&a_empty[sa]);
        }
        if (ok) mma_commit(&acc_full[b]);
      }
      // every MMA either issuer issued has finished before TMEM is released
      mma_commit(&mma_done);
      mbar_wait(&mma_done, 0);
    }
  } else if (warp >= kDeqWarp0 && warp < kDeqWarp0 + kDeqWarps) {
    // ------------------------------------------------ dequantisers: int8 x scale -> bf16 -> TMEM (A)
    // Two groups of four warps (one per TMEM lane quarter) take alternate
    // stages, so the conversion of one stage overlaps the next; a thread
    // converts the 64 codes (two Q8_0 blocks) of its row in each weight block.
    const int quarter = warp & 3, group = (warp - kDeqWarp0) >> 2;
    const int r = quarter * 32 + lane;  // weight row of the tile = TMEM lane
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int sw = (r >> 1) & 3;                        // 64-byte swizzle of this row
    uint32_t it = 0;
    for (int tile = cid; tile < n_tiles && ok; tile += ncl) {
      for (int kb = 0; kb < KT && ok; ++kb, ++it) {
        if ((int)(it & 1) != group) continue;
        const int s = it % kStages, sa = it % kAStages;
        if (!(ok = wait(&full[s], (it / kStages) & 1))) break;
        // the MMAs that last read A stage sa have completed
        if (!(ok = wait(&a_empty[sa], ((it / kAStages) & 1) ^ 1))) break;
#pragma unroll 1
        for (int mb = 0; mb < MB; ++mb) {  // row r of each of the CTA's weight blocks
          const uint8_t* wtile = sW + s * G::WBytes + mb * kTileBytes;
          const uint8_t* qrow = wtile + r * 64;
          uint4 c[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) c[q] = *reinterpret_cast<const uint4*>(qrow + ((q ^ sw) << 4));
          const uint16_t* sc = reinterpret_cast<const uint16_t*>(wtile + kTileCodeBytes);
          const float d0 = half_bits_to_f32(sc[r]), d1 = half_bits_to_f32(sc[BM + r]);
          uint32_t out[32];
          const float e0 = d0 * 0.00390625f, e1 = d1 * 0.00390625f;       // d / 256
          const float k0 = d0 * -32896.0f, k1 = d1 * -32896.0f;           // -(2^15 + 2^7) d
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const f2 dd = q < 2 ? f2_pack(e0, e0) : f2_pack(e1, e1);
            const f2 cc = q < 2 ? f2_pack(k0, k0) : f2_pack(k1, k1);
            const uint32_t w4[4] = {c[q].x, c[q].y, c[q].z, c[q].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t w = w4[i];
              out[8 * q + 2 * i] = deq_pair_fma(__byte_perm(w, 0x4B000000u, 0x7504), __byte_perm(w, 0x4B000000u, 0x7514),
                                                dd, cc);
              out[8 * q + 2 * i + 1] = deq_pair_fma(__byte_perm(w, 0x4B000000u, 0x7524),
                                                    __byte_perm(w, 0x4B000000u, 0x7534), dd, cc);
            }
          }
          tmem_st32(tmem_base + lane_addr + G::ACol0 + sa * G::ACols + mb * (BK / 2), out);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[sa]);
      }
    }
  } else {
    // ------------------------------------------------ epilogue: TMEM -> registers -> global
    uint32_t tc = 0;
    int4 mi_next = cid < n_tiles ? a.minfo[cid / n_mbg] : make_int4(0, 0, 0, 0);
    for (int tile = cid; tile < n_tiles && ok; tile += ncl, ++tc) {
      const int4 mi = mi_next;
      if (tile + ncl < n_tiles) mi_next = a.minfo[(tile + ncl) / n_mbg];
      const int m0 = (tile % n_mbg) * MB * BM;
      const int b = tc & 1;
      if (!(ok = wait(&acc_full[b], (tc >> 1) & 1))) break;
      tc_fence_after();
#pragma unroll 1
      for (int mb = 0; mb < MB; ++mb) {
        const uint32_t taddr = tmem_base + b * G::AccCols + mb * G::BN + ((uint32_t)(warp * 32) << 16);
        const int prow = m0 + mb * BM + warp * 32 + lane;  // weight row (interleaved gate/up for SwiGLU)
        for (int c0 = 0; c0 < mi.z; c0 += 32) {
          float v[32];
          tmem_ld32(taddr + c0, v);
          if (EPI == kEpiSwiGLU) {
            // lanes 4g, 4g+1 hold the gate rows of i = 2(prow/4) + {0,1}, lanes
            // 4g+2, 4g+3 the matching up rows. Partners (lane ^ 2) swap halves:
            // a gate lane computes tokens 0..15 of the chunk, an up lane 16..31,
            // so every lane makes 16 distinct outputs.
            const bool gate_lane = (lane & 2) == 0;
            const int i = (prow >> 2) * 2 + (lane & 1);
            const int jt = gate_lane ? 0 : 16;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float mine = gate_lane ? v[j] : v[16 + j];
              const float other = __shfl_xor_sync(0xFFFFFFFFu, gate_lane ? v[16 + j] : v[j], 2);
              const float g = gate_lane ? mine : other, u = gate_lane ? other : mine;
              const float hv = __fdividef(g, 1.0f + __expf(-g)) * u;  // h is rounded to bf16 next
              const float hn = __shfl_xor_sync(0xFFFFFFFFu, hv, 1);
              const int c = c0 + jt + j;
              if ((lane & 1) == 0 && c < mi.z && i < a.out_cols)
                *reinterpret_cast<uint32_t*>(a.outp + (int64_t)(mi.y + c) * a.out_cols + i) = pack_bf16x2(hv, hn);
            }
          } else {
            // (the row gates are applied in the combine)
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const bool valid = c0 + j < mi.z;
              const float y = v[j];
              const float yn = __shfl_down_sync(0xFFFFFFFFu, y, 1);
              if ((lane & 1) == 0 && valid && prow < a.out_cols)
                *reinterpret_cast<uint32_t*>(a.outp + (int64_t)(mi.y + c0 + j) * a.out_cols + prow) = pack_bf16x2(y, yn);
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


// ------------------------------------------------------------- router on the tensor cores
// Logits z = x W_r^T + b for 128 tokens per CTA, then the top-k, the gates and
// the per-32-token expert counts the scan kernel takes (the same outputs as
// the tiled fp32 router). W_r is split once into three bf16 planes whose sum
// is exactly W_r (each holds the next 8 significant bits); x is bf16. So every
// product is exact, and the three MMAs of a K step add them into one fp32
// accumulator in tensor memory.
constexpr int kRM = 128, kRK = 64, kRStages = 3;
constexpr int kRThreads = 192;  // warp 0 TMA, warp 1 MMA (TMEM owner), warps 2-5 epilogue (lane quarters 2,3,0,1)
constexpr int kRMaxE = 256;
constexpr int kRPassE = 128;    // experts per pass over x (E > 128: two passes, N = 128 each)

struct RouteMmaArgs {
  const float* bias;
  float* zpart;   // K split over gridDim.y > 1: partial logits [gridDim.y][T][E] (no bias); else null
  int T, H, E, k;
  int32_t* ids;
  float* gates;
  int32_t* ids_out;
  float* gates_out;
  int32_t* hist;  // [ceil(T/32)][E]
  Meta* meta;
};

// Insert (v, e) into the descending list (tv, ti) of length KS, behind any
// equal value (ids arrive in ascending order, so ties keep the lower id).
// Branch-free: every slot compares against the old list, so the KS selects
// are independent of one another.
template <int KS>
__device__ __forceinline__ void topk_insert(float (&tv)[KS], int (&ti)[KS], float v, int e) {
  bool c[KS];
#pragma unroll
  for (int m = 0; m < KS; ++m) c[m] = v > tv[m];
#pragma unroll
  for (int m = KS - 1; m > 0; --m) {
    const float nv = c[m - 1] ? tv[m - 1] : (c[m] ? v : tv[m]);
    const int ni = c[m - 1] ? ti[m - 1] : (c[m] ? e : ti[m]);
    tv[m] = nv;
    ti[m] = ni;
  }
  tv[0] = c[0] ? v : tv[0];
  ti[0] = c[0] ? e : ti[0];
}

// KS: length of the per-token list, the smallest of 8 and 16 that holds k.
template <int KS>
__global__ void __launch_bounds__(kRThreads, 1)
    route_mma_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                     RouteMmaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kRStages], empty[kRStages], acc_full;
  __shared__ uint32_t s_tmem;
  __shared__ int s_cnt[4][kRMaxE];
  __shared__ float s_bias[kRMaxE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, k = a.k, t0 = blockIdx.x * kRM;
  pdl_launch_dependents();  // the select kernel may start early: it waits for this grid before reading
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* sX = smem_raw + pad;                 // [kRStages][128 tokens][128 B]
  const int BR = E < kRPassE ? E : kRPassE;      // W_r rows per pass
  const int n_pass = (E + kRPassE - 1) / kRPassE;
  uint8_t* sW = sX + kRStages * kRM * kRK * 2;  // [kRStages][3 planes][BR rows][128 B]
  const uint32_t wstage = 3u * BR * kRK * 2;
  for (int i = threadIdx.x; i < 4 * kRMaxE; i += kRThreads) (&s_cnt[0][0])[i] = 0;
  for (int i = threadIdx.x; i < E; i += kRThreads) s_bias[i] = a.bias[i];
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&acc_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kRMaxE)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // this CTA's K steps: [kbeg, kbeg + KT) of the H / 64 (the K split is blockIdx.y)
  const int KT_all = a.H / kRK;
  const int kbeg = KT_all * blockIdx.y / gridDim.y;
  const int KT = KT_all * (blockIdx.y + 1) / gridDim.y - kbeg;
  const int NI = n_pass * KT;  // pipeline iterations: (pass, K step)
  // each CTA starts its K loop at its own offset, so the CTAs do not all ask
  // the same L2 lines for the same W_r tile at the same time
  const int kb0 = (int)(((int64_t)blockIdx.x * KT) / gridDim.x);
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < NI && ok; ++i) {
        const int s = i % kRStages, ps = i / KT, kb = i % KT;
        const int kk = kbeg + (kb + kb0 < KT ? kb + kb0 : kb + kb0 - KT);
        if (!(ok = mbar_wait(&empty[s], ((i / kRStages) & 1) ^ 1))) {
          report_wait(a.meta, kSiteGemm, i, 0);
          break;
        }
        mbar_arrive_expect_tx(&full[s], (uint32_t)kRM * kRK * 2 + wstage);
        tma_load_2d(sX + s * kRM * kRK * 2, &map_x, kk * kRK, t0, &full[s]);
        for (int p = 0; p < 3; ++p)
          tma_load_2d(sW + s * wstage + p * BR * kRK * 2, &map_w, kk * kRK, p * E + ps * kRPassE, &full[s]);
      }
      for (int j = ::max(0, NI - kRStages); j < NI; ++j) mbar_wait(&full[j % kRStages], (j / kRStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < NI && ok; ++i) {
        const int s = i % kRStages, ps = i / KT, kb = i % KT;
        const int np = E - ps * kRPassE < kRPassE ? E - ps * kRPassE : kRPassE;  // this pass's experts
        const uint32_t idesc = idesc_bf16(kRM, np);
        if (!(ok = mbar_wait(&full[s], (i / kRStages) & 1))) {
          report_wait(a.meta, kSiteGemm, i, 1);
          break;
        }
        tc_fence_after();
        const uint32_t x0 = smem_u32(sX + s * kRM * kRK * 2), w0 = smem_u32(sW + s * wstage);
        const uint32_t d = tmem + ps * kRPassE;  // the pass's accumulator columns
#pragma unroll
        for (int kk = 0; kk < kRK / 16; ++kk)
#pragma unroll
          for (int p = 2; p >= 0; --p)  // smallest plane first
            mma_ss(d, sw128_desc(x0 + kk * 32), sw128_desc(w0 + p * BR * kRK * 2 + kk * 32), idesc,
                   (kb | kk | (2 - p)) != 0);
        mma_commit(&empty[s]);
      }
      mma_commit(&acc_full);  // (also when aborted: the epilogue then reads what is there)
    }
  } else {
    // epilogue: thread = token row (TMEM lane); top-k kept sorted in registers
    const int q = warp & 3, row = q * 32 + lane, t = t0 + row;
    if (!mbar_wait(&acc_full, 0)) report_wait(a.meta, kSiteGemm, 0, 2);
    tc_fence_after();
    if (a.zpart) {  // a K split: this CTA's partial logits, summed (in split order) by the select kernel
      float* zp = a.zpart + ((size_t)blockIdx.y * a.T + t) * E;
      for (int c0 = 0; c0 < E; c0 += 32) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
        if (t < a.T) {
          const int n = c0 + 32 <= E ? 32 : 16;  // E is a multiple of 16
          for (int j = 0; j < n; j += 4) *reinterpret_cast<float4*>(zp + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      }
    } else {
    float tv[KS];
    int ti[KS];
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      tv[j] = -INFINITY;
      ti[j] = j;  // valid ids even if nothing is inserted
    }
    for (int c0 = 0; c0 < E; c0 += 32) {  // E is a multiple of 16, so only the last chunk is partial
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
      if (c0 + 32 <= E) {
#pragma unroll
        for (int j = 0; j < 32; ++j) topk_insert<KS>(tv, ti, v[j] + s_bias[c0 + j], c0 + j);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) topk_insert<KS>(tv, ti, v[j] + s_bias[c0 + j], c0 + j);
      }
    }
    if (t < a.T) {
      float ex[KS], sum = 0.f;
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        ex[j] = j < k ? expf(tv[j] - tv[0]) : 0.f;
        sum += ex[j];
      }
#pragma unroll
      for (int j = 0; j < KS; ++j)
        if (j < k) {
          const float g = ex[j] / sum;
          a.ids[t * k + j] = ti[j];
          a.gates[t * k + j] = g;
          a.ids_out[t * k + j] = ti[j];
          if (a.gates_out) a.gates_out[t * k + j] = g;
          atomicAdd(&s_cnt[q][ti[j]], 1);
        }
    }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (!a.zpart)
    for (int i = threadIdx.x; i < 4 * E; i += kRThreads) {
      const int q = i / E, e = i % E, tile = blockIdx.x * 4 + q;
      if (tile * 32 < a.T) a.hist[(int64_t)tile * E + e] = s_cnt[q][e];
    }
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kRMaxE) : "memory");
}

// After a K-split router: per token (a warp) the logits summed over the
// splits in order, plus the bias; the top-k (ties to the lower id), the gates,
// and the CTA's per-expert counts of its 32 tokens for the scan kernel.
constexpr int kSelTokens = 32;
__global__ void __launch_bounds__(kSelTokens * 32) route_select_kernel(RouteMmaArgs a, int ks) {
  __shared__ int s_cnt[kRMaxE];
  pdl_wait();  // the partial logits
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, E = a.E, k = a.k;
  const int t = blockIdx.x * kSelTokens + warp;
  for (int i = threadIdx.x; i < E; i += kSelTokens * 32) s_cnt[i] = 0;
  __syncthreads();
  if (t < a.T) {
    // the K splits summed in order, then the bias; a split's loads for all of
    // the lane's experts in flight together
    float zl[kMaxEPerLane];
#pragma unroll
    for (int m = 0; m < kMaxEPerLane; ++m) zl[m] = 0.f;
    for (int q = 0; q < ks; ++q) {
      const float* zq = a.zpart + ((size_t)q * a.T + t) * E;
      float v[kMaxEPerLane];
#pragma unroll
      for (int m = 0; m < kMaxEPerLane; ++m) v[m] = lane + 32 * m < E ? __ldg(zq + lane + 32 * m) : 0.f;
#pragma unroll
      for (int m = 0; m < kMaxEPerLane; ++m) zl[m] += v[m];
    }
#pragma unroll
    for (int m = 0; m < kMaxEPerLane; ++m) zl[m] = lane + 32 * m < E ? zl[m] + a.bias[lane + 32 * m] : -INFINITY;
    int id;
    float zv;
    warp_topk(zl, E, k, lane, &id, &zv);
    const float g = warp_gate(zv, k, lane);
    if (lane < k) {
      a.ids[t * k + lane] = id;
      a.gates[t * k + lane] = g;
      a.ids_out[t * k + lane] = id;
      if (a.gates_out) a.gates_out[t * k + lane] = g;
      atomicAdd(&s_cnt[id], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kSelTokens * 32) a.hist[(int64_t)blockIdx.x * E + e] = s_cnt[e];
}

// W_r (fp32) -> three bf16 planes hi, mid, lo with hi + mid + lo == W_r exactly.
__global__ void split_router_kernel(const float* __restrict__ wr, int64_t n, __nv_bfloat16* __restrict__ w3) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float w = wr[i];
  const __nv_bfloat16 hi = __float2bfloat16_rn(w);
  const float r1 = w - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(mid);
  w3[i] = hi;
  w3[n + i] = mid;
  w3[2 * n + i] = __float2bfloat16_rn(r2);
}

// ------------------------------------------------------------- gather, combine
// One warp per row, 16 bytes per lane per step (no per-element division).
constexpr int kRowThreads = 256;
constexpr int kGatherBatch = 8;  // 16-byte chunks of a row a lane has in flight

// xperm[pos] = x[row_token[pos]].
__global__ void __launch_bounds__(kRowThreads) gather_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                                  const int32_t* __restrict__ row_token, int rows,
                                                                  int H, __nv_bfloat16* __restrict__ xperm) {
  const int chunks = H / 8, lane = threadIdx.x & 31;
  pdl_wait();  // the scatter's row tokens
  pdl_launch_dependents();
  // warp w copies rows w, w + nw, ...: their tokens 32 at a time (one load a
  // lane, then shuffles), and each row's 16-byte chunks kGatherBatch a lane
  // in flight before any store
  const int nw = gridDim.x * (kRowThreads / 32);
  for (int p0 = blockIdx.x * (kRowThreads / 32) + (threadIdx.x >> 5); p0 < rows; p0 += 32 * nw) {
    const int mine = p0 + lane * nw;
    const int tok_l = mine < rows ? row_token[mine] : 0;
    const int nr = ::min(32, (rows - p0 + nw - 1) / nw);
    for (int i = 0; i < nr; ++i) {
      const int tok = __shfl_sync(0xFFFFFFFFu, tok_l, i);
      const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)tok * H);
      uint4* dst = reinterpret_cast<uint4*>(xperm + (int64_t)(p0 + i * nw) * H);
      for (int c0 = lane; c0 < chunks; c0 += 32 * kGatherBatch) {
        uint4 v[kGatherBatch];
#pragma unroll
        for (int u = 0; u < kGatherBatch; ++u)
          if (c0 + 32 * u < chunks) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
        for (int u = 0; u < kGatherBatch; ++u)
          if (c0 + 32 * u < chunks) dst[c0 + 32 * u] = v[u];
      }
    }
  }
}

// out[t] = sum over the token's slots j (ascending) of g[t, j] Yp[inv[t*k + j]],
// then the shared expert's row (weight 1); fp32 sum, one bf16 rounding. (The
// gate is applied here rather than in the down GEMM's epilogue, which is on
// the GEMM's critical path.) One CTA per token: its rows and gates into shared
// memory, then a thread per 16-byte chunk with all of the chunk's k + S <= kN
// row loads in flight before the sum (in slot order).
template <int kN>
__global__ void __launch_bounds__(kRowThreads) combine_kernel(const __nv_bfloat16* __restrict__ yp,
                                                              const int32_t* __restrict__ inv,
                                                              const float* __restrict__ gates, int T, int k, int S,
                                                              int H, __nv_bfloat16* __restrict__ out) {
  __shared__ int s_row[kN];
  __shared__ float s_g[kN];
  const int chunks = H / 8, n = k + S;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (threadIdx.x < n) {
      const int j = threadIdx.x, slot = j < k ? t * k + j : T * k + t;
      s_row[j] = inv[slot];
      s_g[j] = j < k ? gates[slot] : 1.0f;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < chunks; c += kRowThreads) {
      uint4 v[kN];
#pragma unroll
      for (int j = 0; j < kN; ++j)
        if (j < n) v[j] = __ldg(reinterpret_cast<const uint4*>(yp + (int64_t)s_row[j] * H) + c);
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
      for (int j = 0; j < kN; ++j) {
        if (j < n) {
          const float g = s_g[j];
          const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float lo, hi;
            bf16x2_to_f32(w[q], lo, hi);
            acc[2 * q] = fmaf(g, lo, acc[2 * q]);
            acc[2 * q + 1] = fmaf(g, hi, acc[2 * q + 1]);
          }
        }
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      reinterpret_cast<uint4*>(out + (int64_t)t * H)[c] = o;
    }
    __syncthreads();  // s_row and s_g are rewritten for the next token
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



template <int EPI, int SH>
cudaError_t launch_gemm(const CUtensorMap& mb, const GemmArgs& g, int num_sms, bool overlap, cudaStream_t s) {
  // One persistent CTA per SM (its shared memory admits no second). With
  // `overlap` the launch is a programmatic dependent of the kernel before it:
  // its CTAs take the SMs that grid's CTAs leave while the last of them still
  // run. The mid and small GEMMs of a projection follow the GEMM before them
  // and read nothing it writes (disjoint tiles and outputs), so they do not
  // wait; the gate/up big-tile GEMM follows the gather and waits for it
  // (wait_prev) before anything else. The down big-tile GEMM is an ordinary
  // launch: it reads the h of all three gate/up GEMMs.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Shape<SH>::SmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<EPI, SH>, mb, g);
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
  cudaError_t e = allow_max_dynamic_smem(grouped_gemm_kernel<kEpiSwiGLU, kBig>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(grouped_gemm_kernel<kEpiDown, kBig>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(grouped_gemm_kernel<kEpiSwiGLU, kMid>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(grouped_gemm_kernel<kEpiDown, kMid>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(grouped_gemm_kernel<kEpiSwiGLU, kSmall>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(grouped_gemm_kernel<kEpiDown, kSmall>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(route_mma_kernel<8>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(route_mma_kernel<16>);
  return e;
}

cudaError_t prepare_prefill(Handle* h) {
  const uint64_t H = h->cfg.H, I = h->cfg.I, R = h->rows_max;
  PrefillMaps* m = new PrefillMaps();
  h->maps = m;
  cudaError_t e = encode_2d(&m->a_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->xperm, H, R, H * 2, BK, Shape<kBig>::XBox,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e == cudaSuccess)
    e = encode_2d(&m->a_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->hbuf, I, R, I * 2, BK, Shape<kBig>::XBox,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e == cudaSuccess)
    e = encode_2d(&m->a_xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->xperm, H, R, H * 2, BK, Shape<kMid>::XBox,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e == cudaSuccess)
    e = encode_2d(&m->a_hm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->hbuf, I, R, I * 2, BK, Shape<kMid>::XBox,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e == cudaSuccess)
    e = encode_2d(&m->a_xs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->xperm, H, R, H * 2, BK, Shape<kSmall>::XBox,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e == cudaSuccess)
    e = encode_2d(&m->a_hs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->hbuf, I, R, I * 2, BK, Shape<kSmall>::XBox,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e == cudaSuccess && h->wr3)
    e = encode_2d(&m->w3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->wr3, H, 3 * (uint64_t)h->cfg.E, H * 2, kRK,
                  (uint32_t)std::min(h->cfg.E, kRPassE), CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  return e;
}

bool route_prefill_mma_available(const Handle* h) {
  return h->maps && h->wr3 && h->cfg.E <= kRMaxE && h->cfg.E % 16 == 0 && h->cfg.E >= 16;
}

cudaError_t launch_split_router(Handle* h, cudaStream_t s) {
  const int64_t n = (int64_t)h->cfg.E * h->cfg.H;
  split_router_kernel<<<grid_for(n, 256, 1 << 20), 256, 0, s>>>(h->wr, n, h->wr3);
  return cudaGetLastError();
}

cudaError_t launch_route_prefill_mma(Handle* h, const __nv_bfloat16* x, int T, int32_t* ids_out, float* gates_out,
                                     cudaStream_t s) {
  const int H = h->cfg.H, E = h->cfg.E;
  CUtensorMap map_x;  // x is the caller's buffer: its map is made per call
  cudaError_t e = encode_2d(&map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<__nv_bfloat16*>(x), H, T, H * 2,
                            kRK, kRM, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e != cudaSuccess) return e;
  RouteMmaArgs a;
  a.bias = h->bias;
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = h->cfg.k;
  a.ids = h->ids;
  a.gates = h->gates;
  a.ids_out = ids_out;
  a.gates_out = gates_out;
  a.hist = h->hist;
  a.meta = h->meta;
  const size_t smem = (size_t)kRStages * (kRM * kRK * 2 + 3 * std::min(E, kRPassE) * kRK * 2) + 1024;
  const int tiles = (T + kRM - 1) / kRM;
  // split K when the token tiles alone leave most SMs idle (a partial-logit
  // pass, then a select kernel); the splits are summed in a fixed order
  int ks = std::min(std::min(h->num_sms / tiles, kRouterMaxSplit), H / kRK);
  if (ks < 2) ks = 1;
  a.zpart = ks > 1 ? h->zpart : nullptr;
  const dim3 grid((unsigned)tiles, (unsigned)ks);
  if (a.k <= 8)
    route_mma_kernel<8><<<grid, kRThreads, smem, s>>>(map_x, h->maps->w3, a);
  else
    route_mma_kernel<16><<<grid, kRThreads, smem, s>>>(map_x, h->maps->w3, a);
  cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess && ks > 1)
    err = launch_dependent(route_select_kernel, dim3((unsigned)((T + kSelTokens - 1) / kSelTokens)),
                           dim3(kSelTokens * 32), 0, s, a, ks);
  return err;
}

cudaError_t launch_ffn_prefill(Handle* h, const __nv_bfloat16* x, int T, __nv_bfloat16* out, cudaStream_t s) {
  if (!h->maps) return cudaErrorNotSupported;
  const int H = h->cfg.H, I = h->cfg.I, k = h->cfg.k, S = h->S;
  const int rows = T * (k + S);
  cudaError_t err;
  {
    KernelTimer tm(h, FW_KERNEL_PREFILL_GATHER, s);
    err = launch_dependent(gather_rows_kernel, dim3(grid_for(rows, kRowThreads / 32, h->num_sms * 8)),
                           dim3(kRowThreads), 0, s, x, (const int32_t*)h->row_token, rows, H, h->xperm);
  }
  if (err != cudaSuccess) return err;
  // each projection: the big tiles, the mid ones, then the small ones
  GemmArgs g;
  g.wt = h->t_gu;
  g.meta = h->meta;
  g.outp = static_cast<__nv_bfloat16*>(h->hbuf);
  g.K = H;
  g.prows = 2 * I;
  g.n_mb = (2 * I + BM - 1) / BM;
  g.out_cols = I;
  g.wait_prev = 0;
  auto lists = [&](GemmArgs base, int shape) {
    base.minfo = shape == kBig ? h->minfo : (shape == kMid ? h->minfo_m : h->minfo_s);
    base.n_mtiles = shape == kBig ? &h->meta->n_mtiles : (shape == kMid ? &h->meta->n_midtiles : &h->meta->n_stiles);
    return base;
  };
  {
    KernelTimer tm(h, FW_KERNEL_PREFILL_GATEUP, s);
    GemmArgs gb = lists(g, kBig);
    gb.wait_prev = 1;
    err = launch_gemm<kEpiSwiGLU, kBig>(h->maps->a_x, gb, h->num_sms, true, s);
  }
  {
    KernelTimer tm(h, FW_KERNEL_PREFILL_GATEUP_MID, s);
    if (err == cudaSuccess) err = launch_gemm<kEpiSwiGLU, kMid>(h->maps->a_xm, lists(g, kMid), h->num_sms, true, s);
  }
  {
    KernelTimer tm(h, FW_KERNEL_PREFILL_GATEUP_SMALL, s);
    if (err == cudaSuccess) err = launch_gemm<kEpiSwiGLU, kSmall>(h->maps->a_xs, lists(g, kSmall), h->num_sms, true, s);
  }
  g.outp = h->yp;
  g.wt = h->t_d;
  g.K = I;
  g.prows = H;
  g.n_mb = (H + BM - 1) / BM;
  g.out_cols = H;
  {
    KernelTimer tm(h, FW_KERNEL_PREFILL_DOWN, s);
    if (err == cudaSuccess) err = launch_gemm<kEpiDown, kBig>(h->maps->a_h, lists(g, kBig), h->num_sms, false, s);
  }
  {
    KernelTimer tm(h, FW_KERNEL_PREFILL_DOWN_MID, s);
    if (err == cudaSuccess) err = launch_gemm<kEpiDown, kMid>(h->maps->a_hm, lists(g, kMid), h->num_sms, true, s);
  }
  {
    KernelTimer tm(h, FW_KERNEL_PREFILL_DOWN_SMALL, s);
    if (err == cudaSuccess) err = launch_gemm<kEpiDown, kSmall>(h->maps->a_hs, lists(g, kSmall), h->num_sms, true, s);
  }
  if (err != cudaSuccess) return err;
  {
    KernelTimer tm(h, FW_KERNEL_PREFILL_COMBINE, s);
    const unsigned cgrid = (unsigned)std::min(T, h->num_sms * 16);
    if (k + S <= 9)
      combine_kernel<9><<<cgrid, kRowThreads, 0, s>>>(h->yp, h->inv, h->gates, T, k, S, H, out);
    else
      combine_kernel<kMaxK + 1><<<cgrid, kRowThreads, 0, s>>>(h->yp, h->inv, h->gates, T, k, S, H, out);
  }
  return cudaGetLastError();
}

}  // namespace fw
