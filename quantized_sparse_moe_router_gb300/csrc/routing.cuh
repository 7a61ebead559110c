// Selection, gates and grouping of a decode batch (T <= 16 tokens) computed by
// one CTA in shared memory from the router logits. The decode router's last
// CTA uses it to publish the routing; the decode expert kernels use it to
// rebuild the same routing locally (it is deterministic) instead of waiting
// for a published table.
#pragma once

#include "internal.cuh"

namespace fw {
namespace dev {

constexpr int kMaxE = 256;               // experts supported by the register layouts below
constexpr int kMaxEPerLane = kMaxE / 32;
constexpr int kMaxRowsDecode = kMaxDecodeT * (kMaxK + 1);

// One warp selects the k largest of z[0..E) (lane l holds z[l + 32 m]), ties
// to the lower id, in descending order; lane j < k ends with (id_j, z_j).
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

// The routing of a decode batch in shared memory.
struct SmemRouting {
  int ids[kMaxDecodeT * kMaxK];
  float gates[kMaxDecodeT * kMaxK];
  int cnt[kMaxE + 2];     // per expert, then exclusive offsets (cnt[EU] = rows)
  int c2[kMaxE + 2];      // per-expert counts
  uint32_t mask[kMaxE + 1];
  int nz[kMaxE + 2];      // nonzero flags, then their exclusive scan
  int4 u[kMaxE + 1];      // (expert, first row, rows, 0) of experts with rows, ascending
  int tok[kMaxRowsDecode];
  float rg[kMaxRowsDecode];
  int slot[kMaxRowsDecode];  // grouped row -> slot id (perm)
  int wtot[32];
  int n_unique;
  int rows;
};

// Whole block (NT threads, NT >= 32 * min(T, NT/32)): selection for T tokens
// from logits [T][E] (global, written by an earlier kernel), gates, and the
// grouping. Ends with a __syncthreads; every field above is then valid.
template <int NT>
__device__ void route_in_smem(const float* logits, int T, int E, int k, int S, SmemRouting& r) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int t = warp; t < T; t += NW) {
    float zl[kMaxEPerLane];
#pragma unroll
    for (int m = 0; m < kMaxEPerLane; ++m) {
      int ee = lane + 32 * m;
      zl[m] = ee < E ? __ldcg(logits + t * E + ee) : -INFINITY;
    }
    int id;
    float zv;
    warp_topk(zl, E, k, lane, &id, &zv);
    float g = warp_gate(zv, k, lane);
    if (lane < k) {
      r.ids[t * k + lane] = id;
      r.gates[t * k + lane] = g;
    }
  }
  const int EU = E + S;
  for (int i = tid; i < EU + 1; i += NT) r.cnt[i] = 0;
  for (int i = tid; i < EU; i += NT) r.mask[i] = 0;
  __syncthreads();
  for (int p = tid; p < T * k; p += NT) {
    int ee = r.ids[p];
    atomicAdd(&r.cnt[ee], 1);
    atomicOr(&r.mask[ee], 1u << (p / k));
  }
  if (S && tid == 0) r.cnt[E] = T;
  __syncthreads();
  for (int i = tid; i < EU; i += NT) {
    r.c2[i] = r.cnt[i];
    r.nz[i] = r.cnt[i] > 0;
  }
  __syncthreads();
  const int rows = block_exclusive_scan<NT>(r.cnt, EU + 1, r.wtot);
  for (int p = tid; p < T * k; p += NT) {
    int t = p / k, ee = r.ids[p];
    int pos = r.cnt[ee] + __popc(r.mask[ee] & ((1u << t) - 1u));
    r.tok[pos] = t;
    r.rg[pos] = r.gates[p];
    r.slot[pos] = p;
  }
  if (S)
    for (int t = tid; t < T; t += NT) {
      int pos = r.cnt[E] + t;
      r.tok[pos] = t;
      r.rg[pos] = 1.0f;
      r.slot[pos] = T * k + t;
    }
  const int n_unique = block_exclusive_scan<NT>(r.nz, EU, r.wtot);
  for (int i = tid; i < EU; i += NT)
    if (r.c2[i] > 0) r.u[r.nz[i]] = make_int4(i, r.cnt[i], r.c2[i], 0);
  if (tid == 0) {
    r.n_unique = n_unique;
    r.rows = rows;
  }
  __syncthreads();
}

// Publish a routing computed by route_in_smem (whole block).
struct RoutingOut {
  int32_t* ids_out;    // caller [T][k]
  float* gates_out;    // caller [T][k] or null
  int32_t* ids;        // workspace copies
  float* gates;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* row_token;
  float* row_gate;
  int4* uinfo;
  Meta* meta;
};

template <int NT>
__device__ void publish_routing(const SmemRouting& r, int T, int E, int k, int S, const RoutingOut& o) {
  const int tid = threadIdx.x, EU = E + S;
  for (int p = tid; p < T * k; p += NT) {
    if (o.ids_out) o.ids_out[p] = r.ids[p];
    if (o.gates_out) o.gates_out[p] = r.gates[p];
    o.ids[p] = r.ids[p];
    o.gates[p] = r.gates[p];
  }
  for (int i = tid; i < EU; i += NT) o.counts[i] = r.c2[i];
  for (int i = tid; i < EU + 1; i += NT) o.offsets[i] = r.cnt[i];
  for (int pos = tid; pos < r.rows; pos += NT) {
    o.perm[pos] = r.slot[pos];
    o.inv[r.slot[pos]] = pos;
    o.row_token[pos] = r.tok[pos];
    o.row_gate[pos] = r.rg[pos];
  }
  for (int i = tid; i < r.n_unique; i += NT) o.uinfo[i] = r.u[i];
  if (tid == 0) {
    o.meta->n_unique = r.n_unique;
    o.meta->T = T;
  }
}

}  // namespace dev
}  // namespace fw
