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
#include "routing.cuh"

namespace fw {
namespace {

using namespace dev;

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
constexpr int kRouteXStage = 64 * 1024;  // x staged in shared memory by one bulk copy when it fits
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteUnroll = 8;  // float4 loads of the router row in flight per lane

// Grid: E CTAs of kNT / 32 warps; CTA e computes z[t][e] for the T <= kT
// tokens, its warps splitting H with all of a lane's loads issued before any
// use. With kSelect (the route-only entry point), the last CTA to finish
// (atomic ticket, no waiting) also selects, makes the gates and groups the
// (token, slot) pairs and publishes them; without it the logits are the only
// output (the expert kernels rebuild the routing from them), and the kernel
// holds no routing tables in shared memory.
//
// kNT = 128 (one or two tokens, H <= kSmallRouterH, no selection): four
// warps of two accumulators a thread and four row loads in flight a lane, at
// most 32 registers. So sized, two of its CTAs fit in what a one-token
// expert CTA leaves of an SM (the registers of each scheduler's share of
// warps included), which lets them launch, and prefetch their rows, while
// that kernel still runs. At larger H the eight-warp form, though it cannot
// launch early, is faster (7,168: 3.5 against 5.6 us after the wait).
constexpr int kSmallRouterH = 2048;
template <bool kSelect, int kT, int kNT>
__global__ void __launch_bounds__(kNT, kNT == 128 ? 16 : 1) route_decode_kernel(RouteArgs a, int staged) {
  static_assert(kT == 2 || kT == kMaxDecodeT, "two tokens, or the decode limit");
  static_assert(kNT == kRouteThreads || (kNT == 128 && kT == 2 && !kSelect), "the small form: two tokens, no selection");
  constexpr int kNW = kNT / 32, kU = kNT == 128 ? 4 : kRouteUnroll;
  extern __shared__ __align__(128) uint8_t x_s[];  // [T][H] bf16 when staged
  __shared__ float s_part[kNW][kT];
  __shared__ __align__(8) uint64_t xbar;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e = blockIdx.x;
  const int T = a.T, H = a.H;
  // Launched as a programmatic dependent of whatever came before it (the
  // previous call's expert kernel, typically): wait for it to complete before
  // touching memory (x may be its output; the grid counter is its own), and
  // only then let this call's expert kernel start (it stages x before its own
  // wait for this grid). The router row is a weight, written by nothing in
  // the stream: it starts coming into L2 before the wait.
  if (tid == 0) prefetch_l2(a.wr + (int64_t)e * H, (uint32_t)(H * 4));
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x == 0 && tid == 0) {  // fresh grid barrier and chunk tickets for this call's expert kernel
    a.meta->gbar = 0;
    a.meta->chunk_ctr = 0;
  }
  // Several tokens: all of x (up to 64 KB) into shared memory by one bulk
  // copy; read from there by every warp (as loads of 8 bytes from global
  // memory by each thread it took 7.5 us at 16 tokens, the copy about 1).
  const __nv_bfloat16* xs = a.x;
  if (staged) {
    const uint32_t bytes = (uint32_t)(T * H * 2);
    if (tid == 0) {
      mbar_init(&xbar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&xbar, bytes);
      bulk_g2s(x_s, a.x, bytes, &xbar);
    }
    __syncthreads();
    if (!mbar_wait(&xbar, 0)) {  // bounded: report, and leave the logits as they are
      if (tid == 0) report_wait(a.meta, kSiteRouteX, blockIdx.x, 0);
      return;
    }
    xs = reinterpret_cast<const __nv_bfloat16*>(x_s);
  }
  {
    float acc[kT];
#pragma unroll
    for (int t = 0; t < kT; ++t) acc[t] = 0.0f;
    const float* wrow = a.wr + (int64_t)e * H;
    for (int base = 4 * tid; base < H; base += 4 * kNT * kU) {
      float4 w[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        int h = base + 4 * kNT * u;
        w[u] = h < H ? __ldg(reinterpret_cast<const float4*>(wrow + h)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        int h = base + 4 * kNT * u;
        if (h < H) {
#pragma unroll
          for (int t = 0; t < kT; ++t) {
            if (t < T) {
              const uint2 xv = staged ? *reinterpret_cast<const uint2*>(xs + (int64_t)t * H + h)
                                      : __ldg(reinterpret_cast<const uint2*>(xs + (int64_t)t * H + h));
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
    if (kT == 2 || T <= 2) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (t < T) {
          float v = warp_sum(acc[t]);
          if (lane == 0) s_part[warp][t] = v;
        }
      }
    } else if constexpr (kT == kMaxDecodeT) {
      // the 16 sums of the warp by recursive halving: at each step a lane
      // keeps one half of its values (by its lane bit), sends the other to
      // its partner and adds what it receives -- 16 shuffles, not 16 x 5;
      // lane pair (2 t', 2 t' + 1) ends with token t's sum, t from the lane bits
#pragma unroll
      for (int m = 16, half = 8; m >= 2; m >>= 1, half >>= 1) {
        const bool hi = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = hi ? acc[i] : acc[i + half];
          const float keep = hi ? acc[i + half] : acc[i];
          acc[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, m);
        }
      }
      acc[0] += __shfl_xor_sync(0xFFFFFFFFu, acc[0], 1);
      const int t = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
      if ((lane & 1) == 0 && t < T) s_part[warp][t] = acc[0];
    }
  }
  __syncthreads();
  if (tid < T) {
    float z = 0.f;
#pragma unroll
    for (int w = 0; w < kNW; ++w) z += s_part[w][tid];
    a.logits[tid * a.E + e] = z + a.bias[e];
    if (kSelect) __threadfence();
  }
  if constexpr (kSelect) {
    __shared__ bool s_last;
    __syncthreads();
    if (tid == 0) s_last = atomicInc(&a.meta->ticket, gridDim.x - 1) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    __shared__ SmemRouting r;
    __shared__ __align__(16) float zbuf[kMaxDecodeT * kMaxE];
    route_in_smem<kNT>(a.logits, T, a.E, a.k, a.S, r, zbuf);
    RoutingOut o{a.ids_out, a.gates_out, a.ids,      a.gates,    a.counts, a.offsets,
                 a.perm,    a.inv,       a.row_token, a.row_gate, a.uinfo,  a.meta};
    publish_routing<kNT>(r, T, a.E, a.k, a.S, o);
  }
}

// ------------------------------------------------------ prefill router
// Tiled fp32 router: each CTA owns 32 tokens and all E (<= 256) experts; the
// 32 tokens x all experts per CTA (256 threads: warp w owns tokens 4w..4w+3,
// lane l experts l + 32m). The K loop runs over 32-wide slices of x (bf16 ->
// fp32) and Wr, double-buffered in shared memory: the next slice's global
// loads are in registers while the current one is multiplied, so one barrier
// per slice. Rows are padded to 36 floats, which makes each lane's 128-bit
// read of its expert row conflict-free; the token reads are broadcasts. Then
// one warp per 4 tokens selects, and the CTA writes its per-expert counts.
constexpr int kKC = 32;
constexpr int kKP = kKC + 4;  // padded row (floats)

template <int EM>
__global__ void __launch_bounds__(256) route_tiles_kernel(RouteArgs a, int32_t* hist) {
  extern __shared__ __align__(16) float smem[];
  float* xs = smem;                             // [2][32][kKP]
  float* ws = xs + 2 * kRouteTileM * kKP;       // [2][EM*32][kKP]; later z [32][EM*32 + 1]
  __shared__ int s_cnt[kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ty = warp, tx = lane;
  const int T = a.T, H = a.H, E = a.E, k = a.k;
  const int t0 = blockIdx.x * kRouteTileM;
  constexpr int kWPer = EM * 32 * (kKC / 4) / 256;  // float4 of the Wr slice per thread (= EM)
  float acc[4][EM];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int m = 0; m < EM; ++m) acc[i][m] = 0.0f;

  // this thread's share of a slice: x row xr, columns xc..xc+3; Wr rows wr_q
  const int xr = tid >> 3, xc = (tid & 7) * 4;
  const bool xok = t0 + xr < T;
  const __nv_bfloat16* xsrc = a.x + (int64_t)(t0 + xr) * H + xc;
  uint2 xreg;
  float4 wreg[kWPer];
  auto load = [&](int h0) {
    xreg = xok ? __ldg(reinterpret_cast<const uint2*>(xsrc + h0)) : make_uint2(0u, 0u);
#pragma unroll
    for (int q = 0; q < kWPer; ++q) {
      const int idx = tid + 256 * q, r = idx >> 3, c = (idx & 7) * 4;
      wreg[q] = r < E ? __ldg(reinterpret_cast<const float4*>(a.wr + (int64_t)r * H + h0 + c))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto store = [&](int b) {
    float4 xv;
    bf16x2_to_f32(xreg.x, xv.x, xv.y);
    bf16x2_to_f32(xreg.y, xv.z, xv.w);
    *reinterpret_cast<float4*>(xs + (b * kRouteTileM + xr) * kKP + xc) = xv;
#pragma unroll
    for (int q = 0; q < kWPer; ++q) {
      const int idx = tid + 256 * q, r = idx >> 3, c = (idx & 7) * 4;
      *reinterpret_cast<float4*>(ws + (b * EM * 32 + r) * kKP + c) = wreg[q];
    }
  };

  const int nS = H / kKC;
  load(0);
  store(0);
  __syncthreads();
  for (int sl = 0; sl < nS; ++sl) {
    const int b = sl & 1;
    if (sl + 1 < nS) load((sl + 1) * kKC);
    const float* xb = xs + (b * kRouteTileM + ty * 4) * kKP;
    const float* wb = ws + (b * EM * 32 + tx) * kKP;
#pragma unroll
    for (int kk = 0; kk < kKC; kk += 4) {
      float4 xv[4], wv[EM];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = *reinterpret_cast<const float4*>(xb + i * kKP + kk);
#pragma unroll
      for (int m = 0; m < EM; ++m) wv[m] = *reinterpret_cast<const float4*>(wb + m * 32 * kKP + kk);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < EM; ++m) {
          acc[i][m] = fmaf(xv[i].x, wv[m].x, acc[i][m]);
          acc[i][m] = fmaf(xv[i].y, wv[m].y, acc[i][m]);
          acc[i][m] = fmaf(xv[i].z, wv[m].z, acc[i][m]);
          acc[i][m] = fmaf(xv[i].w, wv[m].w, acc[i][m]);
        }
    }
    if (sl + 1 < nS) store(b ^ 1);  // the other buffer: last read before the previous barrier
    __syncthreads();
  }
  // logits to shared memory (z[token][expert]); the slices are no longer read
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
// with rows, and the list of token tiles (kTokTile rows) per expert for the
// prefill GEMMs.
// The per-expert walks over the tiles batch their loads 16 deep; the three
// scans over the experts run in one warp, in registers.
constexpr int kScanBatch = 16;

// An expert's token tiles: full kTokTile-row tiles, then the rest -- which
// goes to the small-tile list when it has at most kSmallTile rows, to the
// mid-tile list when it has at most kMidTile, else it is a big tile too.
// When the batch has fewer mid tiles than `mid_min` (less than one tile per
// SM in the mid-tile GEMMs) they join the big tiles instead: a launch that
// gives each SM at most one tile costs a whole tile's latency, which a few
// more tiles among the big ones do not.
__device__ __forceinline__ int big_tiles(int c) {
  const int r = c % kTokTile;
  return c / kTokTile + (r > kMidTile ? 1 : 0);
}
__device__ __forceinline__ int mid_tiles(int c) {
  const int r = c % kTokTile;
  return r > kSmallTile && r <= kMidTile ? 1 : 0;
}
__device__ __forceinline__ int small_tiles(int c) {
  const int r = c % kTokTile;
  return r > 0 && r <= kSmallTile ? 1 : 0;
}

constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) route_scan_kernel(RouteArgs a, int32_t* hist, int n_tiles,
                                                                  int4* minfo, int4* minfo_m, int4* minfo_s,
                                                                  int mid_min) {
  __shared__ int s_cnt[kMaxE + 2];
  __shared__ int s_off[kMaxE + 2];
  __shared__ int s_nz[kMaxE + 2];
  __shared__ int s_nt[kMaxE + 2];
  __shared__ int s_ns[kMaxE + 2];
  __shared__ int s_nm[kMaxE + 2];
  __shared__ int s_nbm[kMaxE + 2];  // big + mid tiles before the expert (mid tiles merged)
  __shared__ int s_merge;
  __shared__ int s_part[kScanThreads];  // [part][expert]: the part's count (pass 1)
  pdl_wait();  // the per-tile counts of the router
  pdl_launch_dependents();
  const int E = a.E, EU = E + a.S, T = a.T, tid = threadIdx.x, lane = tid & 31;
  // thread (part, expert): the experts' per-tile counts are summed by P
  // threads each over consecutive tile ranges (a few batched loads instead
  // of n_tiles / 16 round trips)
  int ep = 32;
  while (ep < E) ep *= 2;
  const int P = kScanThreads / ep, part = tid / ep, e_me = tid % ep;
  const int per = (n_tiles + P - 1) / P, c_lo = ::min(n_tiles, part * per), c_hi = ::min(n_tiles, c_lo + per);
  {
    int run = 0;
    if (e_me < E)
      for (int c0 = c_lo; c0 < c_hi; c0 += kScanBatch) {
        int v[kScanBatch];
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) v[u] = c0 + u < c_hi ? hist[(int64_t)(c0 + u) * E + e_me] : 0;
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) run += v[u];
      }
    s_part[tid] = run;
  }
  __syncthreads();
  for (int e = tid; e < E; e += kScanThreads) {
    int run = 0;
    for (int q = 0; q < P; ++q) run += s_part[q * ep + e];
    s_cnt[e] = run;
  }
  if (a.S && tid == 0) s_cnt[E] = T;
  __syncthreads();
  if (tid < 32) {
    constexpr int kPer = (kMaxE + 1 + 31) / 32;
    const int per = (EU + 31) / 32, b0 = lane * per;
    int cn[kPer];
    int sc = 0, sn = 0, st = 0, ss = 0, sm = 0;
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int i = b0 + m;
      cn[m] = (m < per && i < EU) ? s_cnt[i] : 0;
      sc += cn[m];
      sn += cn[m] > 0;
      st += big_tiles(cn[m]);
      ss += small_tiles(cn[m]);
      sm += mid_tiles(cn[m]);
    }
    int ic = sc, in = sn, it = st, is = ss, im = sm;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int uc = __shfl_up_sync(0xFFFFFFFFu, ic, o), un = __shfl_up_sync(0xFFFFFFFFu, in, o),
                ut = __shfl_up_sync(0xFFFFFFFFu, it, o), us = __shfl_up_sync(0xFFFFFFFFu, is, o),
                um = __shfl_up_sync(0xFFFFFFFFu, im, o);
      if (lane >= o) {
        ic += uc;
        in += un;
        it += ut;
        is += us;
        im += um;
      }
    }
    int rc = ic - sc, rn = in - sn, rt = it - st, rs = is - ss, rm = im - sm;
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int i = b0 + m;
      if (m < per && i < EU) {
        s_off[i] = rc;
        s_nz[i] = rn;
        s_nt[i] = rt;
        s_ns[i] = rs;
        s_nm[i] = rm;
        s_nbm[i] = rt + rm;
        rc += cn[m];
        rn += cn[m] > 0;
        rt += big_tiles(cn[m]);
        rs += small_tiles(cn[m]);
        rm += mid_tiles(cn[m]);
      }
    }
    if (lane == 31) {
      const bool merge = im < mid_min;
      s_merge = merge;
      s_off[EU] = ic;
      a.meta->n_unique = in;
      a.meta->n_mtiles = merge ? it + im : it;
      a.meta->n_stiles = is;
      a.meta->n_midtiles = merge ? 0 : im;
      a.meta->T = T;
    }
  }
  __syncthreads();
  for (int e = tid; e < EU + 1; e += kScanThreads) a.offsets[e] = s_off[e];
  for (int e = tid; e < EU; e += kScanThreads) {
    const int cnt = s_cnt[e];
    a.counts[e] = cnt;
    if (cnt > 0) a.uinfo[s_nz[e]] = make_int4(e, s_off[e], cnt, 0);
    const bool merge = s_merge;
    const int nt = big_tiles(cnt) + (merge ? mid_tiles(cnt) : 0), t0 = merge ? s_nbm[e] : s_nt[e];
    for (int i = 0; i < nt; ++i)
      minfo[t0 + i] = make_int4(e, s_off[e] + kTokTile * i, min(kTokTile, cnt - kTokTile * i), 0);
    const int r0 = cnt / kTokTile * kTokTile;
    if (small_tiles(cnt)) minfo_s[s_ns[e]] = make_int4(e, s_off[e] + r0, cnt - r0, 0);
    if (!merge && mid_tiles(cnt)) minfo_m[s_nm[e]] = make_int4(e, s_off[e] + r0, cnt - r0, 0);
  }
  // per-tile bases: thread (part, expert) starts after the parts before it
  if (e_me < E) {
    int run = s_off[e_me];
    for (int q = 0; q < part; ++q) run += s_part[q * ep + e_me];
    for (int c0 = c_lo; c0 < c_hi; c0 += kScanBatch) {
      int v[kScanBatch];
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) v[u] = c0 + u < c_hi ? hist[(int64_t)(c0 + u) * E + e_me] : 0;
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u)
        if (c0 + u < c_hi) {
          hist[(int64_t)(c0 + u) * E + e_me] = run;
          run += v[u];
        }
    }
  }
}

// One CTA per 32-token tile: stable scatter of the tile's (token, slot) pairs.
__global__ void __launch_bounds__(256) route_scatter_kernel(RouteArgs a, const int32_t* hist) {
  __shared__ uint32_t s_mask[kMaxE];
  __shared__ int s_ids[kRouteTileM * kMaxK];
  pdl_wait();  // the scan's offsets and per-tile bases
  pdl_launch_dependents();
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
  size_t smem = sizeof(float) * (2 * kRouteTileM * kKP + 2 * (size_t)EM * 32 * kKP);
  size_t zsmem = sizeof(float) * (2 * kRouteTileM * kKP + (size_t)kRouteTileM * (EM * 32 + 1));
  if (zsmem > smem) smem = zsmem;
  route_tiles_kernel<EM><<<n_tiles, 256, smem, s>>>(a, hist);
  return cudaGetLastError();
}

}  // namespace

cudaError_t configure_route_kernels() {
  // The decode router runs on the SMs that the expert kernel (all of shared
  // memory) takes next: with the same carve-out an SM need not be
  // reconfigured between the two.
  void (*const routers[5])(RouteArgs, int) = {
      route_decode_kernel<false, 2, 128>, route_decode_kernel<false, 2, kRouteThreads>,
      route_decode_kernel<true, 2, kRouteThreads>, route_decode_kernel<false, kMaxDecodeT, kRouteThreads>,
      route_decode_kernel<true, kMaxDecodeT, kRouteThreads>};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 5 && e == cudaSuccess; ++i) {
    e = cudaFuncSetAttribute(routers[i], cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(routers[i], cudaFuncAttributeMaxDynamicSharedMemorySize, kRouteXStage);
  }
  if (e == cudaSuccess) e = allow_max_dynamic_smem(route_tiles_kernel<1>);
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
                                bool select, cudaStream_t s) {
  RouteArgs a = route_args(h, x, T, ids_out, gates_out);
  KernelTimer tm(h, FW_KERNEL_ROUTE_DECODE, s);
  // x by one bulk copy into shared memory for several tokens (16-byte aligned, fits)
  const size_t xbytes = (size_t)T * h->cfg.H * 2;
  const int staged = T > 1 && xbytes <= (size_t)kRouteXStage && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  const dim3 grid(h->cfg.E);
  const size_t dyn = staged ? xbytes : 0;
  const dim3 block(kRouteThreads);
  if (T <= 2 && !select && h->cfg.H <= kSmallRouterH)
    return launch_dependent(route_decode_kernel<false, 2, 128>, grid, dim3(128), dyn, s, a, staged);
  if (T <= 2)
    return select ? launch_dependent(route_decode_kernel<true, 2, kRouteThreads>, grid, block, dyn, s, a, staged)
                  : launch_dependent(route_decode_kernel<false, 2, kRouteThreads>, grid, block, dyn, s, a, staged);
  return select ? launch_dependent(route_decode_kernel<true, kMaxDecodeT, kRouteThreads>, grid, block, dyn, s, a, staged)
                : launch_dependent(route_decode_kernel<false, kMaxDecodeT, kRouteThreads>, grid, block, dyn, s, a,
                                   staged);
}

cudaError_t launch_route_prefill(Handle* h, const __nv_bfloat16* x, int T, int32_t* ids_out, float* gates_out,
                                 cudaStream_t s) {
  RouteArgs a = route_args(h, x, T, ids_out, gates_out);
  const int n_tiles = (T + kRouteTileM - 1) / kRouteTileM;
  const int EM = (h->cfg.E + 31) / 32;
  cudaError_t err;
  if (route_prefill_mma_available(h)) {
    KernelTimer tm(h, FW_KERNEL_ROUTE_TILES, s);
    err = launch_route_prefill_mma(h, x, T, ids_out, gates_out, s);
  } else {
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
    // the mid-tile GEMMs take two 128-row weight blocks per SM and tile
    const int64_t mb_gu = (2 * (int64_t)h->cfg.I + 127) / 128, mb_d = ((int64_t)h->cfg.H + 127) / 128;
    const int n_mbg = (int)::min((mb_gu + 1) / 2, (mb_d + 1) / 2);
    const int mid_min = (h->num_sms + n_mbg - 1) / n_mbg;
    err = launch_dependent(route_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, a, h->hist, n_tiles, h->minfo,
                           h->minfo_m, h->minfo_s, mid_min);
  }
  if (err != cudaSuccess) return err;
  {
    KernelTimer tm(h, FW_KERNEL_ROUTE_SCATTER, s);
    err = launch_dependent(route_scatter_kernel, dim3(n_tiles), dim3(256), 0, s, a, (const int32_t*)h->hist);
  }
  return err;
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
