// Router, top-k, gates and the token-to-expert grouping.
//
// The pages name the router only in passing (the vOOM README lists it among
// the substeps its profiler brackets, and keeps routers in the checkpoint
// dtype; the Flyweight README lists dynamic MoE routing among the places its
// runtime still synchronises with the host, §Current limitations). The reading
// used: fp32 logits z = x Wr^T + b, the k largest per token with ties to the
// lower id, ordered by descending z, gates = softmax restricted to the k and
// renormalised; then the (token, slot) pairs grouped by expert, stable in
// token order, with every count and offset kept on the device.
#include "internal.cuh"

namespace fw {
namespace {

using namespace dev;

constexpr int kMaxE = 256;               // experts supported by the register layouts below
constexpr int kMaxEPerLane = kMaxE / 32;

// --------------------------------------------------------------- top-k
// One warp selects the k largest of z[0..E) (lane l holds z[l + 32 m]),
// ties to the lower id, in descending order; lane j < k ends with
// (id_j, z_j) in (*out_id, *out_z).
__device__ __forceinline__ void warp_topk(const float (&zl)[kMaxEPerLane], int E, int k, int lane, int* out_id,
                                          float* out_z) {
  uint32_t taken = 0;  // bit m: z[lane + 32 m] already selected
  int my_id = -1;
  float my_z = 0.0f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int m = 0; m < kMaxEPerLane; ++m) {
      int e = lane + 32 * m;
      if (e < E && !((taken >> m) & 1u)) {
        float v = zl[m];
        if (v > bv || (v == bv && e < bi)) {
          bv = v;
          bi = e;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_id = bi;
      my_z = bv;
    }
  }
  *out_id = my_id;
  *out_z = my_z;
}

// Gates of the selection held by lanes 0..k-1: exp(z_j - z_0) / sum.
__device__ __forceinline__ float warp_gate(float my_z, int k, int lane) {
  float z0 = __shfl_sync(0xFFFFFFFFu, my_z, 0);
  float ex = lane < k ? expf(my_z - z0) : 0.0f;
  float sum = warp_sum(ex);
  return ex / sum;
}

// Exclusive scan of n ints in shared memory by the whole block of NT threads.
// Returns the total.
template <int NT>
__device__ int block_exclusive_scan(int* v, int n, int* warp_tot) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (n + NT - 1) / NT;
  const int b = tid * per, e = min(n, b + per);
  int s = 0;
  for (int i = b; i < e; ++i) s += v[i];
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  int wbase = 0, total = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    if (i < w) wbase += warp_tot[i];
    total += warp_tot[i];
  }
  int run = wbase + incl - s;
  for (int i = b; i < e; ++i) {
    int c = v[i];
    v[i] = run;
    run += c;
  }
  __syncthreads();
  return total;
}

// ------------------------------------------------------ decode router
struct RouteArgs {
  const __nv_bfloat16* x;
  const float* wr;
  const float* bias;
  int T, H, E, k, S;
  float* logits;
  int32_t* ids;        // internal [T][k]
  float* gates;        // internal [T][k]
  int32_t* ids_out;    // caller [T][k]
  float* gates_out;    // caller [T][k] or null
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* row_token;
  float* row_gate;
  int4* uinfo;
  Meta* meta;
};

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteUnroll = 8;  // float4 loads of the router row in flight per lane

// Grid: E CTAs of 8 warps; CTA e computes z[t][e] for the T <= 16 tokens, its
// warps splitting H with all of a lane's loads issued before any use. The
// last CTA to finish (atomic ticket, no waiting) selects, makes the gates and
// groups the (token, slot) pairs for all tokens.
__global__ void __launch_bounds__(kRouteThreads) route_decode_kernel(RouteArgs a) {
  __shared__ float s_part[kRouteWarps][kMaxDecodeT];
  __shared__ int s_cnt[kMaxE + 2];
  __shared__ int s_c2[kMaxE + 1];
  __shared__ uint32_t s_mask[kMaxE + 1];
  __shared__ int s_nz[kMaxE + 2];
  __shared__ int s_ids[kMaxDecodeT * kMaxK];
  __shared__ float s_gates[kMaxDecodeT * kMaxK];
  __shared__ int s_wtot[kRouteWarps];
  __shared__ bool s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e = blockIdx.x;
  const int T = a.T, H = a.H;
  pdl_launch_dependents();  // the expert kernels wait for this grid's completion before reading
  {
    float acc[kMaxDecodeT];
#pragma unroll
    for (int t = 0; t < kMaxDecodeT; ++t) acc[t] = 0.0f;
    const float* wrow = a.wr + (int64_t)e * H;
    for (int base = 4 * tid; base < H; base += 4 * kRouteThreads * kRouteUnroll) {
      float4 w[kRouteUnroll];
#pragma unroll
      for (int u = 0; u < kRouteUnroll; ++u) {
        int h = base + 4 * kRouteThreads * u;
        w[u] = h < H ? __ldg(reinterpret_cast<const float4*>(wrow + h)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kRouteUnroll; ++u) {
        int h = base + 4 * kRouteThreads * u;
        if (h < H) {
#pragma unroll
          for (int t = 0; t < kMaxDecodeT; ++t) {
            if (t < T) {
              uint2 xv = __ldg(reinterpret_cast<const uint2*>(a.x + (int64_t)t * H + h));
              float x0, x1, x2, x3;
              bf16x2_to_f32(xv.x, x0, x1);
              bf16x2_to_f32(xv.y, x2, x3);
              acc[t] = fmaf(x0, w[u].x, acc[t]);
              acc[t] = fmaf(x1, w[u].y, acc[t]);
              acc[t] = fmaf(x2, w[u].z, acc[t]);
              acc[t] = fmaf(x3, w[u].w, acc[t]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kMaxDecodeT; ++t) {
      if (t < T) {
        float v = warp_sum(acc[t]);
        if (lane == 0) s_part[warp][t] = v;
      }
    }
  }
  __syncthreads();
  if (tid < T) {
    float z = 0.f;
#pragma unroll
    for (int w = 0; w < kRouteWarps; ++w) z += s_part[w][tid];
    a.logits[tid * a.E + e] = z + a.bias[e];
    __threadfence();
  }
  __syncthreads();
  if (tid == 0) s_last = atomicInc(&a.meta->ticket, gridDim.x - 1) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- selection and gates: one warp per token
  const int k = a.k, E = a.E;
  for (int t = warp; t < T; t += kRouteWarps) {
    float zl[kMaxEPerLane];
#pragma unroll
    for (int m = 0; m < kMaxEPerLane; ++m) {
      int ee = lane + 32 * m;
      zl[m] = ee < E ? __ldcg(a.logits + t * E + ee) : -INFINITY;
    }
    int id;
    float zv;
    warp_topk(zl, E, k, lane, &id, &zv);
    float g = warp_gate(zv, k, lane);
    if (lane < k) {
      s_ids[t * k + lane] = id;
      s_gates[t * k + lane] = g;
      a.ids[t * k + lane] = id;
      a.gates[t * k + lane] = g;
      a.ids_out[t * k + lane] = id;
      if (a.gates_out) a.gates_out[t * k + lane] = g;
    }
  }
  // ---- grouping: counts, offsets, stable ranks via per-expert token masks
  const int EU = E + a.S;
  for (int i = tid; i < EU + 1; i += kRouteThreads) s_cnt[i] = 0;
  for (int i = tid; i < EU; i += kRouteThreads) s_mask[i] = 0;
  __syncthreads();
  for (int p = tid; p < T * k; p += kRouteThreads) {
    int ee = s_ids[p];
    atomicAdd(&s_cnt[ee], 1);
    atomicOr(&s_mask[ee], 1u << (p / k));
  }
  if (a.S && tid == 0) s_cnt[E] = T;
  __syncthreads();
  for (int i = tid; i < EU; i += kRouteThreads) {
    a.counts[i] = s_cnt[i];
    s_c2[i] = s_cnt[i];
    s_nz[i] = s_cnt[i] > 0;
  }
  __syncthreads();
  block_exclusive_scan<kRouteThreads>(s_cnt, EU + 1, s_wtot);  // s_cnt[EU] = total rows
  for (int i = tid; i < EU + 1; i += kRouteThreads) a.offsets[i] = s_cnt[i];
  for (int p = tid; p < T * k; p += kRouteThreads) {
    int t = p / k, ee = s_ids[p];
    int pos = s_cnt[ee] + __popc(s_mask[ee] & ((1u << t) - 1u));
    a.perm[pos] = p;
    a.inv[p] = pos;
    a.row_token[pos] = t;
    a.row_gate[pos] = s_gates[p];
  }
  if (a.S) {
    for (int t = tid; t < T; t += kRouteThreads) {
      int pos = s_cnt[E] + t;
      a.perm[pos] = T * k + t;
      a.inv[T * k + t] = pos;
      a.row_token[pos] = t;
      a.row_gate[pos] = 1.0f;
    }
  }
  __syncthreads();
  int n_unique = block_exclusive_scan<kRouteThreads>(s_nz, EU, s_wtot);
  for (int i = tid; i < EU; i += kRouteThreads)
    if (s_c2[i] > 0) a.uinfo[s_nz[i]] = make_int4(i, s_cnt[i], s_c2[i], 0);
  if (tid == 0) {
    a.meta->n_unique = n_unique;
    a.meta->T = T;
  }
}

// ------------------------------------------------------ prefill router
// Tiled fp32 router: each CTA owns 32 tokens and all E (<= 256) experts; the
// K loop stages 32-wide slices of x and Wr in shared memory; every thread keeps
// 4 tokens x ceil(E/32) experts of accumulators. Then one warp per 4 tokens
// selects, and the CTA writes its per-expert counts.
constexpr int kKC = 32;

template <int EM>
__global__ void __launch_bounds__(256) route_tiles_kernel(RouteArgs a, int32_t* hist) {
  extern __shared__ float smem[];
  float* xs = smem;                       // [32][kKC + 1]
  float* ws = xs + kRouteTileM * (kKC + 1);  // [EM*32][kKC + 1], later z [32][EM*32 + 1]
  __shared__ int s_cnt[kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ty = tid >> 5, tx = tid & 31;
  const int T = a.T, H = a.H, E = a.E, k = a.k;
  const int t0 = blockIdx.x * kRouteTileM;
  float acc[4][EM];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int m = 0; m < EM; ++m) acc[i][m] = 0.0f;

  for (int h0 = 0; h0 < H; h0 += kKC) {
    // x slice: 32 tokens x 32 values, 4 per thread (bf16 -> f32)
    {
      int r = tid >> 3, c = (tid & 7) * 4;
      int t = t0 + r;
      float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
      if (t < T) {
        uint2 xv = __ldg(reinterpret_cast<const uint2*>(a.x + (int64_t)t * H + h0 + c));
        bf16x2_to_f32(xv.x, v0, v1);
        bf16x2_to_f32(xv.y, v2, v3);
      }
      float* d = xs + r * (kKC + 1) + c;
      d[0] = v0;
      d[1] = v1;
      d[2] = v2;
      d[3] = v3;
    }
    // Wr slice: EM*32 rows x 32 values
    for (int idx = tid; idx < EM * 32 * (kKC / 4); idx += 256) {
      int r = idx / (kKC / 4), c = (idx % (kKC / 4)) * 4;
      float4 w = r < E ? __ldg(reinterpret_cast<const float4*>(a.wr + (int64_t)r * H + h0 + c))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      float* d = ws + r * (kKC + 1) + c;
      d[0] = w.x;
      d[1] = w.y;
      d[2] = w.z;
      d[3] = w.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKC; ++kk) {
      float xv[4], wv[EM];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = xs[(ty * 4 + i) * (kKC + 1) + kk];
#pragma unroll
      for (int m = 0; m < EM; ++m) wv[m] = ws[(tx + 32 * m) * (kKC + 1) + kk];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < EM; ++m) acc[i][m] = fmaf(xv[i], wv[m], acc[i][m]);
    }
    __syncthreads();
  }
  // logits to shared memory (z[token][expert])
  float* zs = ws;
  const int zp = EM * 32 + 1;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int m = 0; m < EM; ++m) {
      int ee = tx + 32 * m;
      zs[(ty * 4 + i) * zp + ee] = ee < E ? acc[i][m] + a.bias[ee] : -INFINITY;
    }
  for (int i = tid; i < kMaxE; i += 256) s_cnt[i] = 0;
  __syncthreads();
  for (int i = 0; i < 4; ++i) {
    int tl = warp * 4 + i, t = t0 + tl;
    if (t >= T) break;
    float zl[kMaxEPerLane];
#pragma unroll
    for (int m = 0; m < kMaxEPerLane; ++m) zl[m] = m < EM ? zs[tl * zp + lane + 32 * m] : -INFINITY;
    int id;
    float zv;
    warp_topk(zl, E, k, lane, &id, &zv);
    float g = warp_gate(zv, k, lane);
    if (lane < k) {
      a.ids[t * k + lane] = id;
      a.gates[t * k + lane] = g;
      a.ids_out[t * k + lane] = id;
      if (a.gates_out) a.gates_out[t * k + lane] = g;
      atomicAdd(&s_cnt[id], 1);
    }
  }
  __syncthreads();
  for (int i = tid; i < E; i += 256) hist[(int64_t)blockIdx.x * E + i] = s_cnt[i];
}

// One CTA: per-expert totals over the tiles, offsets (shared expert last),
// per-tile absolute bases (in place of the tile counts), the list of experts
// with rows, and the list of 128-row tiles per expert for the prefill GEMMs.
__global__ void __launch_bounds__(256) route_scan_kernel(RouteArgs a, int32_t* hist, int n_tiles,
                                                         int32_t* mtiles) {
  __shared__ int s_off[kMaxE + 2];
  __shared__ int s_nz[kMaxE + 2];
  __shared__ int s_nt[kMaxE + 2];
  const int E = a.E, EU = E + a.S, T = a.T, tid = threadIdx.x;
  for (int e = tid; e < EU + 1; e += 256) s_off[e] = 0;
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    int run = 0;
    for (int c = 0; c < n_tiles; ++c) {
      int v = hist[(int64_t)c * E + e];
      hist[(int64_t)c * E + e] = run;
      run += v;
    }
    s_off[e] = run;
  }
  if (a.S && tid == 0) s_off[E] = T;
  __syncthreads();
  for (int e = tid; e < EU; e += 256) {
    a.counts[e] = s_off[e];
    s_nz[e] = s_off[e] > 0;
    s_nt[e] = (s_off[e] + 127) / 128;
  }
  if (tid == 0) {
    // tiny serial scans (EU <= 257) kept simple: one thread
    int run = 0, nz = 0, nt = 0;
    for (int e = 0; e < EU; ++e) {
      int c = s_off[e];
      s_off[e] = run;
      run += c;
      int z = s_nz[e];
      s_nz[e] = nz;
      nz += z;
      int t = s_nt[e];
      s_nt[e] = nt;
      nt += t;
    }
    s_off[EU] = run;
    s_nz[EU] = nz;
    s_nt[EU] = nt;
    a.meta->n_unique = nz;
    a.meta->n_mtiles = nt;
    a.meta->T = T;
  }
  __syncthreads();
  for (int e = tid; e < EU + 1; e += 256) a.offsets[e] = s_off[e];
  for (int e = tid; e < EU; e += 256) {
    int cnt = a.counts[e];
    if (cnt > 0) a.uinfo[s_nz[e]] = make_int4(e, s_off[e], cnt, 0);
    int nt = (cnt + 127) / 128;
    for (int i = 0; i < nt; ++i) mtiles[s_nt[e] + i] = (e << 16) | i;
  }
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    int base = s_off[e];
    for (int c = 0; c < n_tiles; ++c) hist[(int64_t)c * E + e] += base;
  }
}

// One CTA per 32-token tile: stable scatter of the tile's (token, slot) pairs.
__global__ void __launch_bounds__(256) route_scatter_kernel(RouteArgs a, const int32_t* hist) {
  __shared__ uint32_t s_mask[kMaxE];
  __shared__ int s_ids[kRouteTileM * kMaxK];
  const int tid = threadIdx.x, T = a.T, k = a.k, E = a.E;
  const int t0 = blockIdx.x * kRouteTileM;
  const int nt = min(kRouteTileM, T - t0);
  for (int i = tid; i < E; i += 256) s_mask[i] = 0;
  __syncthreads();
  for (int p = tid; p < nt * k; p += 256) {
    int ee = a.ids[t0 * k + p];
    s_ids[p] = ee;
    atomicOr(&s_mask[ee], 1u << (p / k));
  }
  __syncthreads();
  for (int p = tid; p < nt * k; p += 256) {
    int tl = p / k, ee = s_ids[p];
    int pos = hist[(int64_t)blockIdx.x * E + ee] + __popc(s_mask[ee] & ((1u << tl) - 1u));
    int slot = t0 * k + p;
    a.perm[pos] = slot;
    a.inv[slot] = pos;
    a.row_token[pos] = t0 + tl;
    a.row_gate[pos] = a.gates[slot];
  }
  if (a.S) {
    for (int tl = tid; tl < nt; tl += 256) {
      int t = t0 + tl, pos = T * k + t;
      a.perm[pos] = pos;
      a.inv[pos] = pos;
      a.row_token[pos] = t;
      a.row_gate[pos] = 1.0f;
    }
  }
}

RouteArgs route_args(Handle* h, const __nv_bfloat16* x, int T, int32_t* ids_out, float* gates_out) {
  RouteArgs a;
  a.x = x;
  a.wr = h->wr;
  a.bias = h->bias;
  a.T = T;
  a.H = h->cfg.H;
  a.E = h->cfg.E;
  a.k = h->cfg.k;
  a.S = h->S;
  a.logits = h->logits;
  a.ids = h->ids;
  a.gates = h->gates;
  a.ids_out = ids_out;
  a.gates_out = gates_out;
  a.counts = h->counts;
  a.offsets = h->offsets;
  a.perm = h->perm;
  a.inv = h->inv;
  a.row_token = h->row_token;
  a.row_gate = h->row_gate;
  a.uinfo = h->uinfo;
  a.meta = h->meta;
  return a;
}

template <int EM>
cudaError_t launch_tiles(RouteArgs a, int32_t* hist, int n_tiles, cudaStream_t s) {
  size_t smem = sizeof(float) * (kRouteTileM * (kKC + 1) + (size_t)EM * 32 * (kKC + 1));
  size_t zsmem = sizeof(float) * (kRouteTileM * (kKC + 1) + (size_t)kRouteTileM * (EM * 32 + 1));
  if (zsmem > smem) smem = zsmem;
  route_tiles_kernel<EM><<<n_tiles, 256, smem, s>>>(a, hist);
  return cudaGetLastError();
}

}  // namespace

cudaError_t configure_route_kernels() {
  cudaError_t e = allow_max_dynamic_smem(route_tiles_kernel<1>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(route_tiles_kernel<2>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(route_tiles_kernel<3>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(route_tiles_kernel<4>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(route_tiles_kernel<5>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(route_tiles_kernel<6>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(route_tiles_kernel<7>);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(route_tiles_kernel<8>);
  return e;
}

cudaError_t launch_route_decode(Handle* h, const __nv_bfloat16* x, int T, int32_t* ids_out, float* gates_out,
                                cudaStream_t s) {
  RouteArgs a = route_args(h, x, T, ids_out, gates_out);
  KernelTimer tm(h, FW_KERNEL_ROUTE_DECODE, s);
  route_decode_kernel<<<h->cfg.E, kRouteThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_route_prefill(Handle* h, const __nv_bfloat16* x, int T, int32_t* ids_out, float* gates_out,
                                 cudaStream_t s) {
  RouteArgs a = route_args(h, x, T, ids_out, gates_out);
  const int n_tiles = (T + kRouteTileM - 1) / kRouteTileM;
  const int EM = (h->cfg.E + 31) / 32;
  cudaError_t err;
  {
  KernelTimer tm(h, FW_KERNEL_ROUTE_TILES, s);
  switch (EM) {
    case 1: err = launch_tiles<1>(a, h->hist, n_tiles, s); break;
    case 2: err = launch_tiles<2>(a, h->hist, n_tiles, s); break;
    case 3: err = launch_tiles<3>(a, h->hist, n_tiles, s); break;
    case 4: err = launch_tiles<4>(a, h->hist, n_tiles, s); break;
    case 5: err = launch_tiles<5>(a, h->hist, n_tiles, s); break;
    case 6: err = launch_tiles<6>(a, h->hist, n_tiles, s); break;
    case 7: err = launch_tiles<7>(a, h->hist, n_tiles, s); break;
    default: err = launch_tiles<8>(a, h->hist, n_tiles, s); break;
  }
  }
  if (err != cudaSuccess) return err;
  {
    KernelTimer tm(h, FW_KERNEL_ROUTE_SCAN, s);
    route_scan_kernel<<<1, 256, 0, s>>>(a, h->hist, n_tiles, h->mtiles);
  }
  {
    KernelTimer tm(h, FW_KERNEL_ROUTE_SCATTER, s);
    route_scatter_kernel<<<n_tiles, 256, 0, s>>>(a, h->hist);
  }
  return cudaGetLastError();
}

cudaError_t launch_get_permutation(const Handle* h, int T, int32_t* offsets, int32_t* perm, int32_t* inv,
                                   cudaStream_t s) {
  const int E = h->cfg.E, k = h->cfg.k;
  cudaError_t err = cudaMemcpyAsync(offsets, h->offsets, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToDevice, s);
  if (err == cudaSuccess && T > 0)
    err = cudaMemcpyAsync(perm, h->perm, sizeof(int32_t) * (size_t)T * k, cudaMemcpyDeviceToDevice, s);
  if (err == cudaSuccess && inv && T > 0)
    err = cudaMemcpyAsync(inv, h->inv, sizeof(int32_t) * (size_t)T * k, cudaMemcpyDeviceToDevice, s);
  return err;
}

}  // namespace fw
