// Q8_0 on the device: the quantiser, and the one-time repack of GGUF-style
// 34-byte blocks into the handle's aligned planes (and back, for checking).
//
// Q8_0 is named on the pages as one of the GGUF tensor formats the grouped
// routed-expert kernels read (Flyweight README, §Quantization); its layout is
// the GGUF one: per 32 consecutive values of a row, a binary16 scale d then 32
// int8 codes, value = d * q.
#include "internal.cuh"

namespace fw {
namespace {

// One thread per 32-value block. The decisions (d and every code) are taken in
// fp64: d = amax/127, q = w/d rounded to the nearest integer with halves away
// from zero (the C library's round(), as CUDA provides it for double), clamped
// to +-127; d is stored rounded to binary16 (nearest even).
__global__ void quantize_q8_0_kernel(const float* __restrict__ w, int64_t nblocks, uint8_t* __restrict__ out) {
  int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= nblocks) return;
  const float4* src = reinterpret_cast<const float4*>(w + blk * kQBlock);
  float v[kQBlock];
#pragma unroll
  for (int i = 0; i < kQBlock / 4; ++i) {
    float4 f = src[i];
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kQBlock; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const double d = (double)amax / 127.0;
  uint16_t* dst = reinterpret_cast<uint16_t*>(out + blk * kQBlockBytes);  // 34-byte blocks are 2-byte aligned
  dst[0] = __half_as_ushort(__double2half(d));
#pragma unroll
  for (int i = 0; i < kQBlock; i += 2) {
    int q0 = 0, q1 = 0;
    if (amax > 0.0f) {
      q0 = max(-127, min(127, (int)round((double)v[i] / d)));
      q1 = max(-127, min(127, (int)round((double)v[i + 1] / d)));
    }
    dst[1 + i / 2] = (uint16_t)((q0 & 0xFF) | ((q1 & 0xFF) << 8));
  }
}

// Where one matrix kind of an expert lives after the repack.
struct PlaneView {
  uint8_t* q;      // gate/up: decode rows [EU][2I] of row_bytes(H) (codes, then scales), interleaved; else null
  uint8_t* qc;     // down: decode codes by 16-column groups [EU][I/16][H][16]; else null
  uint16_t* st;    // down: decode scales [EU][I/32][H]; else null
  uint8_t* tiles;  // GEMM tiles of this projection (gate/up share one plane), or null without a prefill path
  int64_t rows;    // rows of one expert's matrix (I for gate/up, H for down)
  int64_t prows;   // rows of one expert in the GEMM plane (2I for gate/up, H for down)
  int64_t K;       // row length (H for gate/up, I for down)
  int which;       // 0 gate, 1 up, 2 down
};

__device__ __forceinline__ int64_t plane_row(const PlaneView& p, int64_t r) {
  return p.which == 0 ? gu_row_gate(r) : (p.which == 1 ? gu_row_up(r) : r);
}

// One thread per GGUF block of one expert range: the block's codes (stored as
// q + 128, offset binary: q XOR 0x80, which the decode kernel multiplies as
// unsigned bytes and the GEMM turns into floats with a byte permute and one
// fused multiply-add) and scale go to the decode plane of
// the kind and to the GEMM tile that holds its row and K step.
__global__ void repack_kernel(PlaneView p, int expert0, int64_t nblocks, const uint8_t* __restrict__ src) {
  int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= nblocks) return;
  const int64_t nb = p.K / kQBlock;
  const int64_t per_expert = p.rows * nb;
  const int64_t e = expert0 + blk / per_expert;
  const int64_t r = (blk % per_expert) / nb;
  const int64_t b = blk % nb;
  const uint16_t* in = reinterpret_cast<const uint16_t*>(src + blk * kQBlockBytes);
  uint32_t words[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) words[i] = ((uint32_t)in[1 + 2 * i] | ((uint32_t)in[2 + 2 * i] << 16)) ^ 0x80808080u;
  const uint4 lo = make_uint4(words[0], words[1], words[2], words[3]);
  const uint4 hi = make_uint4(words[4], words[5], words[6], words[7]);
  const int64_t pr = plane_row(p, r);
  if (p.q) {  // decode gate/up row: codes, then its scales
    uint8_t* row = p.q + (e * p.prows + pr) * row_bytes(p.K);
    reinterpret_cast<uint4*>(row + b * kQBlock)[0] = lo;
    reinterpret_cast<uint4*>(row + b * kQBlock)[1] = hi;
    reinterpret_cast<uint16_t*>(row + p.K)[b] = in[0];
  }
  if (p.qc) {  // decode down: the two 16-column groups of the block, and the scale
    *reinterpret_cast<uint4*>(p.qc + ((e * (p.K / 16) + 2 * b) * p.rows + r) * 16) = lo;
    *reinterpret_cast<uint4*>(p.qc + ((e * (p.K / 16) + 2 * b + 1) * p.rows + r) * 16) = hi;
    p.st[(e * nb + b) * p.rows + r] = in[0];
  }
  if (!p.tiles) return;  // no prefill path on this handle
  // GEMM tile (e, row block, K step b / 2): row pr % 128, 16-byte chunks 2 (b & 1) and 2 (b & 1) + 1
  const int64_t n_mb = (p.prows + kTileRows - 1) / kTileRows, KT = p.K / kTileK;
  const int rr = (int)(pr % kTileRows), half = (int)(b & 1);
  uint8_t* t = p.tiles + gemm_tile_offset(e, pr / kTileRows, b / 2, n_mb, KT);
  *reinterpret_cast<uint4*>(t + tile_code_offset(rr, 2 * half)) = lo;
  *reinterpret_cast<uint4*>(t + tile_code_offset(rr, 2 * half + 1)) = hi;
  reinterpret_cast<uint16_t*>(t + kTileCodeBytes)[half * kTileRows + rr] = in[0];
}

// GGUF blocks of one matrix of one expert, back from the decode planes.
__global__ void export_kernel(PlaneView p, int expert, int64_t nblocks, uint8_t* __restrict__ dst) {
  int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= nblocks) return;
  const int64_t nb = p.K / kQBlock;
  const int64_t r = blk / nb, b = blk % nb, e = expert;
  uint4 lo, hi;
  uint16_t d;
  if (p.q) {
    const uint8_t* row = p.q + (e * p.prows + plane_row(p, r)) * row_bytes(p.K);
    lo = reinterpret_cast<const uint4*>(row + b * kQBlock)[0];
    hi = reinterpret_cast<const uint4*>(row + b * kQBlock)[1];
    d = reinterpret_cast<const uint16_t*>(row + p.K)[b];
  } else {
    lo = *reinterpret_cast<const uint4*>(p.qc + ((e * (p.K / 16) + 2 * b) * p.rows + r) * 16);
    hi = *reinterpret_cast<const uint4*>(p.qc + ((e * (p.K / 16) + 2 * b + 1) * p.rows + r) * 16);
    d = p.st[(e * nb + b) * p.rows + r];
  }
  uint32_t words[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint16_t* out = reinterpret_cast<uint16_t*>(dst + blk * kQBlockBytes);
  out[0] = d;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w = words[i] ^ 0x80808080u;  // back from offset binary
    out[1 + 2 * i] = (uint16_t)(w & 0xFFFF);
    out[2 + 2 * i] = (uint16_t)(w >> 16);
  }
}

PlaneView view_of(const Handle* h, int which) {
  PlaneView p;
  const int64_t H = h->cfg.H, I = h->cfg.I;
  p.which = which;
  if (which == 2) {
    p.q = nullptr;
    p.qc = h->q_dc;
    p.st = h->st_d;
    p.tiles = h->has_prefill ? h->t_d : nullptr;
    p.rows = H;
    p.prows = H;
    p.K = I;
  } else {
    p.q = h->q_gu;
    p.qc = nullptr;
    p.st = nullptr;
    p.tiles = h->has_prefill ? h->t_gu : nullptr;
    p.rows = I;
    p.prows = 2 * I;
    p.K = H;
  }
  return p;
}

unsigned grid_1d(int64_t n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

cudaError_t launch_quantize_q8_0(const float* w, int64_t rows, int64_t K, uint8_t* blocks, cudaStream_t s) {
  int64_t nblocks = rows * (K / kQBlock);
  if (nblocks == 0) return cudaSuccess;
  quantize_q8_0_kernel<<<grid_1d(nblocks, 256), 256, 0, s>>>(w, nblocks, blocks);
  return cudaGetLastError();
}

// Repack `count` consecutive experts starting at `expert0` (count experts of GGUF blocks at `blocks`).
cudaError_t launch_repack(const Handle* h, int which, int expert0, int count, const uint8_t* blocks,
                          cudaStream_t s) {
  PlaneView p = view_of(h, which);
  int64_t nblocks = (int64_t)count * p.rows * (p.K / kQBlock);
  if (nblocks == 0) return cudaSuccess;
  repack_kernel<<<grid_1d(nblocks, 256), 256, 0, s>>>(p, expert0, nblocks, blocks);
  return cudaGetLastError();
}

cudaError_t launch_export(const Handle* h, int which, int expert, uint8_t* blocks, cudaStream_t s) {
  PlaneView p = view_of(h, which);
  int64_t nblocks = p.rows * (p.K / kQBlock);
  export_kernel<<<grid_1d(nblocks, 256), 256, 0, s>>>(p, expert, nblocks, blocks);
  return cudaGetLastError();
}

}  // namespace fw
