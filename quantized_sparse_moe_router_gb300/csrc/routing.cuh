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

// Compare-exchange of the register pairs (m, m ^ S) of one lane inside a
// bitonic stage of block size `size` (S < EPL: both elements are in this lane).
template <int EPL, int S>
__device__ __forceinline__ void bitonic_local(float (&z)[EPL], int (&id)[EPL], int lane, int size) {
  if constexpr (S < EPL) {
#pragma unroll
    for (int m = 0; m < EPL; ++m) {
      const int mm = m ^ S;
      if (mm > m) {
        const bool up = (((lane * EPL) + m) & size) == 0;
        const bool m_first = z[m] > z[mm] || (z[m] == z[mm] && id[m] < id[mm]);
        if (m_first != up) {
          const float tz = z[m];
          z[m] = z[mm];
          z[mm] = tz;
          const int ti = id[m];
          id[m] = id[mm];
          id[mm] = ti;
        }
      }
    }
  }
}

// Bitonic sort, within one warp, of 32*EPL (logit, id) pairs into "comes
// first" order: descending logit, equal logits by ascending id. Lane l holds
// positions l*EPL .. l*EPL+EPL-1. The stage loops stay rolled: this runs once
// per CTA, where instruction fetch, not arithmetic, is the cost.
template <int EPL>
__device__ __forceinline__ void warp_sort_desc(float (&z)[EPL], int (&id)[EPL], int lane) {
  constexpr int N = 32 * EPL;
#pragma unroll 1
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll 1
    for (int stride = size / 2; stride > 0; stride >>= 1) {
      if (stride >= EPL) {
        const int pl = stride / EPL;
        const bool lower = (lane & pl) == 0;
#pragma unroll
        for (int m = 0; m < EPL; ++m) {
          const float oz = __shfl_xor_sync(0xFFFFFFFFu, z[m], pl);
          const int oid = __shfl_xor_sync(0xFFFFFFFFu, id[m], pl);
          const bool up = ((((lane & ~pl) * EPL) + m) & size) == 0;
          const bool mine_first = z[m] > oz || (z[m] == oz && id[m] < oid);
          const bool keep = (lower == up) ? mine_first : !mine_first;
          if (!keep) {
            z[m] = oz;
            id[m] = oid;
          }
        }
      } else if (stride == 4) {
        bitonic_local<EPL, 4>(z, id, lane, size);
      } else if (stride == 2) {
        bitonic_local<EPL, 2>(z, id, lane, size);
      } else {
        bitonic_local<EPL, 1>(z, id, lane, size);
      }
    }
  }
}

// One warp: the top-k of logits z[0..E) (E <= 32*EPL), ties to the lower id,
// in descending order; lane j < k ends with (id_j, gate_j).
template <int EPL>
__device__ __forceinline__ void warp_select_sorted(const float* zrow, int E, int k, int lane, int* out_id,
                                                   float* out_gate) {
  float z[EPL];
  int id[EPL];
#pragma unroll
  for (int m = 0; m < EPL; ++m) {
    const int e = lane * EPL + m;
    z[m] = e < E ? __ldcg(zrow + e) : -INFINITY;
    id[m] = e < E ? e : 0x40000000 + e;  // padding sorts last
  }
  warp_sort_desc<EPL>(z, id, lane);
  int my_id = -1;
  float my_z = -INFINITY;
#pragma unroll
  for (int m = 0; m < EPL; ++m) {
    const float vz = __shfl_sync(0xFFFFFFFFu, z[m], lane / EPL);
    const int vi = __shfl_sync(0xFFFFFFFFu, id[m], lane / EPL);
    if (lane % EPL == m) {
      my_z = vz;
      my_id = vi;
    }
  }
  *out_id = my_id;
  *out_gate = warp_gate(my_z, k, lane);
}

__device__ __forceinline__ void warp_select_any(const float* zrow, int E, int k, int lane, int* id, float* g) {
  if (E <= 128)
    warp_select_sorted<4>(zrow, E, k, lane, id, g);
  else
    warp_select_sorted<8>(zrow, E, k, lane, id, g);
}

// One warp: exclusive scan of n <= 32*9 ints in place; returns the total.
__device__ __forceinline__ int warp_exclusive_scan(int* v, int n, int lane) {
  const int per = (n + 31) / 32;
  const int b = lane * per, e = min(n, b + per);
  int s = 0;
  for (int i = b; i < e; ++i) s += v[i];
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  int run = incl - s;
  for (int i = b; i < e; ++i) {
    const int c = v[i];
    v[i] = run;
    run += c;
  }
  return __shfl_sync(0xFFFFFFFFu, incl, 31);
}

// The routing of a decode batch in shared memory.
struct SmemRouting {
  int ids[kMaxDecodeT * kMaxK];
  float gates[kMaxDecodeT * kMaxK];
  int cnt[kMaxE + 2];     // per-expert counts (cnt[E] = T for the shared expert)
  int off[kMaxE + 2];     // exclusive offsets (off[EU] = rows)
  uint32_t mask[kMaxE + 1];
  int nz[kMaxE + 2];      // nonzero flags, then their exclusive scan
  int4 u[kMaxE + 1];      // (expert, first row, rows, 0) of experts with rows, ascending
  int tok[kMaxRowsDecode];
  float rg[kMaxRowsDecode];
  int slot[kMaxRowsDecode];  // grouped row -> slot id (perm)
  int n_unique;
  int rows;
};

// Whole block (NT threads, at least min(T, NT/32) warps): selection for T <= 16
// tokens from logits [T][E] (global, written by an earlier kernel; one warp per
// token, bitonic top-k), gates, and the grouping. Four block barriers; ends
// with one, after which every field is valid.
template <int NT>
__device__ void route_in_smem(const float* logits, int T, int E, int k, int S, SmemRouting& r) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int EU = E + S;
  for (int t = warp; t < T; t += NW) {
    int id;
    float g;
    warp_select_any(logits + t * E, E, k, lane, &id, &g);
    if (lane < k) {
      r.ids[t * k + lane] = id;
      r.gates[t * k + lane] = g;
    }
  }
  for (int i = tid; i < EU + 1; i += NT) {
    r.cnt[i] = 0;
    if (i < EU) r.mask[i] = 0;
  }
  __syncthreads();
  for (int p = tid; p < T * k; p += NT) {
    const int ee = r.ids[p];
    atomicAdd(&r.cnt[ee], 1);
    atomicOr(&r.mask[ee], 1u << (p / k));
  }
  if (S && tid == 0) r.cnt[E] = T;
  __syncthreads();
  if (warp == 0) {
    for (int i = lane; i < EU + 1; i += 32) {
      r.off[i] = i < EU ? r.cnt[i] : 0;
      r.nz[i] = i < EU ? (r.cnt[i] > 0) : 0;
    }
    __syncwarp();
    const int rows = warp_exclusive_scan(r.off, EU + 1, lane);
    __syncwarp();
    const int n_unique = warp_exclusive_scan(r.nz, EU, lane);
    __syncwarp();
    for (int i = lane; i < EU; i += 32)
      if (r.cnt[i] > 0) r.u[r.nz[i]] = make_int4(i, r.off[i], r.cnt[i], 0);
    if (lane == 0) {
      r.n_unique = n_unique;
      r.rows = rows;
    }
  }
  __syncthreads();
  for (int p = tid; p < T * k; p += NT) {
    const int t = p / k, ee = r.ids[p];
    const int pos = r.off[ee] + __popc(r.mask[ee] & ((1u << t) - 1u));
    r.tok[pos] = t;
    r.rg[pos] = r.gates[p];
    r.slot[pos] = p;
  }
  if (S)
    for (int t = tid; t < T; t += NT) {
      const int pos = r.off[E] + t;
      r.tok[pos] = t;
      r.rg[pos] = 1.0f;
      r.slot[pos] = T * k + t;
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
  for (int i = tid; i < EU; i += NT) o.counts[i] = r.cnt[i];
  for (int i = tid; i < EU + 1; i += NT) o.offsets[i] = r.off[i];
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
