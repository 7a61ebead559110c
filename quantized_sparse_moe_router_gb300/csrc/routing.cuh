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

// Order-preserving key of a logit: a larger float has a larger key, -0 keys
// as +0 (the two compare equal), and NaN keys as 1, with the padding past E,
// below every number (whose keys are at least that of -inf, 0x007FFFFF).
__device__ __forceinline__ uint32_t topk_key(float z) {
  uint32_t u = __float_as_uint(z);
  if (u == 0x80000000u) u = 0u;
  const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (u & 0x7FFFFFFFu) > 0x7F800000u ? 1u : key;
}
__device__ __forceinline__ float topk_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// One warp selects the k largest of z[0..E) (lane l holds z[l + 32 m], m <
// MPL), ties to the lower id, in descending order; lane j < k ends with
// (id_j, z_j). Per round two integer warp reductions: the largest key, then
// the lowest id holding it (each lane offers its lowest); the chosen entry's
// key becomes 0, below everything left (k <= E, so a key >= 1 always remains).
template <int MPL>
__device__ __forceinline__ void warp_topk_n(const float (&zl)[kMaxEPerLane], int E, int k, int lane, int* out_id,
                                            float* out_z) {
  uint32_t key[MPL];
#pragma unroll
  for (int m = 0; m < MPL; ++m) key[m] = lane + 32 * m < E ? topk_key(zl[m]) : 1u;
  int my_id = -1;
  float my_z = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint32_t best = key[0];
#pragma unroll
    for (int m = 1; m < MPL; ++m) best = max(best, key[m]);
    const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, best);
    uint32_t cand = 0xFFFFFFFFu;
#pragma unroll
    for (int m = MPL - 1; m >= 0; --m) cand = key[m] == top ? (uint32_t)(lane + 32 * m) : cand;
    const uint32_t id = __reduce_min_sync(0xFFFFFFFFu, cand);
    if (lane == j) {
      my_id = (int)id;
      my_z = topk_value(top);
    }
#pragma unroll
    for (int m = 0; m < MPL; ++m) key[m] = (uint32_t)(lane + 32 * m) == id ? 0u : key[m];
  }
  *out_id = my_id;
  *out_z = my_z;
}
__device__ __forceinline__ void warp_topk(const float (&zl)[kMaxEPerLane], int E, int k, int lane, int* out_id,
                                          float* out_z) {
  if (E <= 128)
    warp_topk_n<4>(zl, E, k, lane, out_id, out_z);
  else
    warp_topk_n<kMaxEPerLane>(zl, E, k, lane, out_id, out_z);
}

// Gates of the selection held by lanes 0..k-1: exp(z_j - z_0) / sum.
__device__ __forceinline__ float warp_gate(float my_z, int k, int lane) {
  float z0 = __shfl_sync(0xFFFFFFFFu, my_z, 0);
  float ex = lane < k ? expf(my_z - z0) : 0.0f;
  float sum = warp_sum(ex);
  return ex / sum;
}

// How many of a row's logits come before logit e (larger, or equal with a
// lower id), over the float4 words c, c + s, c + 2s, ... of the row (one of s
// lanes sharing expert e): the lanes with the same c read the same word, the
// s different c consecutive words, so the loads are free of bank conflicts.
__device__ __forceinline__ int rank_in_row(const float4* z4, int n4, int c, int s, int e) {
  const float z = reinterpret_cast<const float*>(z4)[e];
  int rank = 0;
#pragma unroll 4
  for (int i = c; i < n4; i += s) {
    const float4 v = z4[i];
    const int f = 4 * i;
    rank += (v.x > z) | ((v.x == z) & (f < e));
    rank += (v.y > z) | ((v.y == z) & (f + 1 < e));
    rank += (v.z > z) | ((v.z == z) & (f + 2 < e));
    rank += (v.w > z) | ((v.w == z) & (f + 3 < e));
  }
  return rank;
}

// The routing of a decode batch in shared memory. The batch's logits are
// staged in a separate buffer the caller provides (T * E floats), which is
// free again once the routing is made.
struct SmemRouting {
  float zsel[kMaxDecodeT * kMaxK];  // selected logits, in rank order
  int ids[kMaxDecodeT * kMaxK];
  float gates[kMaxDecodeT * (kMaxK + 1)];  // by slot; slot T k + t is token t's shared expert (1)
  int cnt[kMaxE + 2];     // per-expert counts (cnt[E] = T for the shared expert)
  int off[kMaxE + 2];     // exclusive offsets (off[EU] = rows)
  uint32_t mask[kMaxE + 1];  // per expert: bit t set when token t selected it
  int4 u[kMaxE + 1];      // (expert, first row, rows, 0) of experts with rows, ascending
  int tok[kMaxRowsDecode];
  int slot[kMaxRowsDecode];  // grouped row -> slot id (perm); its gate is gates[slot]
  int n_unique;
  int rows;
};

// Whole block (NT threads): selection for T <= 16 tokens from logits [T][E]
// (global, written by an earlier kernel), gates, and the grouping. Three
// block barriers; after the last one every field is valid.
//
// Selection: when T E is small (at least 4 lanes per pair), by rank -- every
// (token, expert) pair counts, split over a group of lanes, the logits that
// come before it (larger, or equal with a lower id); ranks below k are the
// top-k in order. Otherwise one warp per token takes the k largest in turn
// (warp_topk). Either way each selected pair sets its token's bit in its
// expert's mask. Then warp 0 alone groups the pairs (counts as popcounts of
// the masks, offsets, the table of touched experts, positions) while the
// other warps make the gates.
template <int NT>
__device__ void route_in_smem(const float* logits, int T, int E, int k, int S, SmemRouting& r, float* zbuf) {
  static_assert(NT % 32 == 0 && NT >= 64, "whole warps, at least two");
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int EU = E + S;
  const int P = T * E;
  const int E4 = (E + 3) & ~3;  // staged rows padded to whole float4 with -inf (never ranked ahead)
  const bool by_rank = 4 * P <= NT;
  if (by_rank)
    for (int i = tid; i < T * E4; i += NT) {
      const int t = i / E4, e = i - t * E4;
      zbuf[i] = e < E ? __ldcg(logits + t * E + e) : -INFINITY;
    }
  for (int i = tid; i < EU; i += NT) r.mask[i] = 0;
  __syncthreads();

  if (by_rank) {
    // s lanes per pair (a power of two, as many as the block allows), lane c
    // of a group taking the float4 words c, c + s, ... of the token's row
    int s = 32;
    while (s > 1 && P * s > NT) s >>= 1;
    const int gpw = 32 / s, c = lane & (s - 1);
    for (int b = warp * gpw; b < P; b += NW * gpw) {  // warp-uniform trip count
      const int p = b + lane / s;
      int rank = 0, t = 0, e = 0;
      float z = 0.f;
      if (p < P) {
        t = p / E;
        e = p - t * E;
        z = zbuf[t * E4 + e];
        rank = rank_in_row(reinterpret_cast<const float4*>(zbuf + t * E4), E4 / 4, c, s, e);
      }
      for (int o = 1; o < s; o <<= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o);
      if (p < P && c == 0 && rank < k) {
        r.ids[t * k + rank] = e;
        r.zsel[t * k + rank] = z;
        atomicOr(&r.mask[e], 1u << t);
      }
    }
  } else {
    for (int t = warp; t < T; t += NW) {
      float zl[kMaxEPerLane];
#pragma unroll
      for (int m = 0; m < kMaxEPerLane; ++m) {
        const int e = lane + 32 * m;
        zl[m] = e < E ? __ldcg(logits + t * E + e) : -INFINITY;
      }
      int id;
      float zv;
      warp_topk(zl, E, k, lane, &id, &zv);
      if (lane < k) {  // k distinct experts: no two lanes share a mask word
        r.ids[t * k + lane] = id;
        r.zsel[t * k + lane] = zv;
        atomicOr(&r.mask[id], 1u << t);
      }
    }
  }
  __syncthreads();

  if (warp == 0) {
    // lane l owns the consecutive experts [l per, l per + per), in registers;
    // both scans (rows and touched experts) in one pass of shuffles
    constexpr int kPer = (kMaxE + 1 + 31) / 32;
    const int per = (EU + 31) / 32, b0 = lane * per;
    int cn[kPer];
    int sc = 0, sn = 0;
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int i = b0 + m;
      cn[m] = (m < per && i < EU) ? (i < E ? __popc(r.mask[i]) : T) : 0;
      sc += cn[m];
      sn += cn[m] > 0;
    }
    int ic = sc, in = sn;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int uc = __shfl_up_sync(0xFFFFFFFFu, ic, o), un = __shfl_up_sync(0xFFFFFFFFu, in, o);
      if (lane >= o) {
        ic += uc;
        in += un;
      }
    }
    int rc = ic - sc, rn = in - sn;
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int i = b0 + m;
      if (m < per && i < EU) {
        r.cnt[i] = cn[m];
        r.off[i] = rc;
        if (cn[m] > 0) r.u[rn++] = make_int4(i, rc, cn[m], 0);
        rc += cn[m];
      }
    }
    if (lane == 31) {
      r.off[EU] = ic;
      r.rows = ic;
      r.n_unique = in;
    }
    __syncwarp();
    // grouped positions: within an expert, ascending token
    for (int p = lane; p < T * k; p += 32) {
      const int t = p / k, ee = r.ids[p];
      const int pos = r.off[ee] + __popc(r.mask[ee] & ((1u << t) - 1u));
      r.tok[pos] = t;
      r.slot[pos] = p;
    }
    if (S)
      for (int t = lane; t < T; t += 32) {
        const int pos = r.off[E] + t;
        r.tok[pos] = t;
        r.slot[pos] = T * k + t;
        r.gates[T * k + t] = 1.0f;
      }
  } else {
    for (int t = warp - 1; t < T; t += NW - 1) {
      const float zj = lane < k ? r.zsel[t * k + lane] : 0.f;
      const float g = warp_gate(zj, k, lane);
      if (lane < k) r.gates[t * k + lane] = g;
    }
  }
  __syncthreads();
}

// The same for one token (T = 1), with less work and code: warp 0 selects
// straight from the logits and sorts the k ids (each selected expert gets one
// grouped row), then one block barrier. The gates (route_one_gates) and the
// counts and offsets over all experts (route_one_tables, read only when the
// routing is published) are left to the caller, off the path to the first
// weight copy.
template <int NT>
__device__ void route_one_in_smem(const float* logits, int E, int k, int S, SmemRouting& r) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == 0) {
    float zl[kMaxEPerLane];
#pragma unroll
    for (int m = 0; m < kMaxEPerLane; ++m) {
      const int e = lane + 32 * m;
      zl[m] = e < E ? __ldcg(logits + e) : -INFINITY;
    }
    int id;
    float zv;
    warp_topk(zl, E, k, lane, &id, &zv);
    // lane j < k: the expert of rank j, its row among the k ids in ascending order
    const int e = lane < k ? id : 0x7FFFFFFF;
    int pos = 0;
    for (int m = 0; m < k; ++m) pos += __shfl_sync(0xFFFFFFFFu, e, m) < e;
    if (lane < k) {
      r.ids[lane] = id;
      r.zsel[lane] = zv;
      r.u[pos] = make_int4(e, pos, 1, 0);
      r.tok[pos] = 0;
      r.slot[pos] = lane;
    }
    if (lane == 0) {
      if (S) {
        r.u[k] = make_int4(E, k, 1, 0);
        r.tok[k] = 0;
        r.slot[k] = k;
      }
      r.n_unique = k + S;
      r.rows = k + S;
    }
  }
  __syncthreads();
}

// One warp, after route_one_in_smem: the gates of the k selected experts (and
// 1 for the shared expert's slot).
__device__ __forceinline__ void route_one_gates(int k, int S, SmemRouting& r, int lane) {
  const float g = warp_gate(lane < k ? r.zsel[lane] : 0.f, k, lane);
  if (lane < k) r.gates[lane] = g;
  if (S && lane == 0) r.gates[k] = 1.0f;
}

// Whole block, after route_one_in_smem: counts [E + S] and offsets [E + S + 1]
// over all experts, by comparison with the k ids (the shared expert's row
// comes after the k routed ones).
template <int NT>
__device__ void route_one_tables(int E, int k, int S, SmemRouting& r) {
  for (int i = threadIdx.x; i <= E + S; i += NT) {
    int before = 0, hit = 0;
    for (int m = 0; m < k; ++m) {
      const int em = r.ids[m];
      before += em < i;
      hit += em == i;
    }
    if (i >= E) {
      before = k + (i > E ? 1 : 0);
      hit = i == E ? 1 : 0;
    }
    r.off[i] = before;
    if (i < E + S) r.cnt[i] = hit;
  }
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
    o.row_gate[pos] = r.gates[r.slot[pos]];
  }
  for (int i = tid; i < r.n_unique; i += NT) o.uinfo[i] = r.u[i];
  if (tid == 0) {
    o.meta->n_unique = r.n_unique;
    o.meta->T = T;
  }
}

}  // namespace dev
}  // namespace fw
