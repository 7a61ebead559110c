// Internal declarations of the fwmoe library: the handle, the device layout of
// the repacked weights and workspace, and the small PTX helpers (mbarrier,
// bulk asynchronous copies, bounded waits) the kernels share.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/fwmoe.h"

namespace fw {

constexpr uint32_t kHandleMagic = 0x4D6F4531u;  // "1EoM"
constexpr uint32_t kHandleFreed = 0xDEADF00Du;
constexpr int kQBlock = 32;        // Q8_0 block length
constexpr int kQBlockBytes = 34;   // fp16 scale + 32 int8
constexpr int kGUGroup = 2;        // gate/up rows are interleaved in groups of 2
constexpr int kMaxK = 16;          // experts per token
constexpr int kMaxDecodeT = 16;    // decode path token limit (one lane per token in the combine)
constexpr int kRouteTileM = 32;    // tokens per CTA in the tiled router
constexpr int kTokTile = 192;      // prefill GEMM token tile (rows of one expert)
constexpr int kMidTile = 96;       // an expert's last tile of at most this many rows goes to the mid-tile GEMM
constexpr int kSmallTile = 64;     // ... of at most this many, to the small-tile GEMM
constexpr int kRouterMaxSplit = 8; // prefill router: K splits at most (partial logits [splits][T_max][E])

// Status bits written by kernels into the handle's device status word.
constexpr int kStatusTimeout = 1;
constexpr int kStatusBadIndex = 2;

// Scale rows are padded to a multiple of 16 bytes.
__host__ __device__ inline int64_t scale_pitch_bytes(int64_t K) { return ((K / kQBlock) * 2 + 15) / 16 * 16; }

// One row of a code plane: its K codes (offset binary), then its K/32 binary16
// scales padded to 16 bytes, so that any run of consecutive rows -- codes and
// scales -- is one contiguous, 16-byte aligned range.
__host__ __device__ inline int64_t row_bytes(int64_t K) { return K + scale_pitch_bytes(K); }

// The GEMMs' weight tiles: per (expert, block of 128 plane rows, K step of
// 64) one contiguous tile -- the 128 rows' 64 codes (+ 128), each row's four
// 16-byte chunks placed as a 64-byte-swizzled TMA copy would place them
// (chunk c of row r at position c ^ ((r >> 1) & 3)), then the two Q8_0 scale
// rows [2][128] binary16 -- so that a CTA's weights for one K step arrive in
// one bulk copy per block.
constexpr int kTileRows = 128;
constexpr int kTileK = 64;
constexpr int kTileCodeBytes = kTileRows * kTileK;               // 8192
constexpr int kTileBytes = kTileCodeBytes + 2 * kTileRows * 2;   // 8704
__host__ __device__ inline int64_t gemm_tile_offset(int64_t e, int64_t mb, int64_t kb, int64_t n_mb, int64_t KT) {
  return ((e * n_mb + mb) * KT + kb) * (int64_t)kTileBytes;
}
// bytes of one expert's tiles of a projection with n_mb row blocks and KT K steps
__host__ __device__ inline int64_t gemm_plane_bytes(int64_t n_mb, int64_t KT) { return n_mb * KT * (int64_t)kTileBytes; }
__host__ __device__ inline int tile_code_offset(int r, int chunk) { return r * kTileK + ((chunk ^ ((r >> 1) & 3)) << 4); }

// Row of gate/up matrix row i in the interleaved [2I] plane: groups of
// kGUGroup gate rows followed by the up rows of the same i, so the units
// i0..i1 (kGUGroup-aligned) are the consecutive rows 2 i0 .. 2 i1.
__host__ __device__ inline int64_t gu_row_gate(int64_t i) { return (i / kGUGroup) * 2 * kGUGroup + (i % kGUGroup); }
__host__ __device__ inline int64_t gu_row_up(int64_t i) { return gu_row_gate(i) + kGUGroup; }

// Device-side routing metadata (one small struct per handle, device memory).
struct Meta {
  unsigned long long gbar;  // decode grid-wide barrier: CTAs arrived (reset by the router)
  int32_t n_unique;     // experts with at least one row, shared included
  uint32_t ticket;      // last-CTA detection in the router (self-resetting)
  int32_t status;       // kStatus* bits
  int32_t T;            // T of the last route
  int32_t n_mtiles;     // prefill: token tiles of more than kMidTile rows (minfo)
  int32_t n_stiles;     // prefill: token tiles of at most kSmallTile rows (minfo_s)
  int32_t n_midtiles;   // prefill: token tiles of kSmallTile+1 .. kMidTile rows (minfo_m)
  uint32_t chunk_ctr;   // decode gate/up chunk tickets handed out (reset by the router)
  int32_t diag[4];      // first failed wait: (site, block, stage, detail); site 0 = none
};

// Host-side event pool of the optional per-kernel timing.
struct Timing {
  cudaEvent_t* ev = nullptr;  // 2 * cap events
  int* kind = nullptr;        // kind of each recorded pair
  int cap = 0;
  int next = 0;
};

// TMA descriptors of the prefill GEMMs (host copies, passed by value).
struct PrefillMaps {
  CUtensorMap a_x;    // xperm [rows_max][H] bf16, 128B swizzle, box 64 x (the big-tile GEMM's token box)
  CUtensorMap a_h;    // hbuf  [rows_max][I] bf16, likewise
  CUtensorMap a_xm;   // the same, box 64 x 96 (mid-tile GEMM)
  CUtensorMap a_hm;
  CUtensorMap a_xs;   // the same, box 64 x 64 (small-tile GEMM)
  CUtensorMap a_hs;
  CUtensorMap w3;     // router planes [3E][H] bf16, box 64 x min(E, 128), 128B swizzle (E <= 256)
};

struct Handle {
  uint32_t magic;
  Timing* timing;     // null unless profiling
  PrefillMaps* maps;  // null unless T_max exceeds the decode limit
  fw_moe_config cfg;
  int S, EU;          // shared experts, routed + shared
  int device;
  int num_sms;
  int last_T;         // T of the last fw_moe_route, -1 before any
  int has_prefill;    // some T in [1, T_max] takes the prefill path (its tiles and buffers exist)
  // ---- repacked weights (device)
  uint8_t* q_gu;      // decode: [EU][2I] rows of row_bytes(H): codes + 128 (offset binary), then scales;
                      // gate/up interleaved per kGUGroup rows
  uint8_t* q_dc;      // decode: [EU][I/16][H][16] down codes by 16-column groups
  uint16_t* st_d;     // decode: [EU][I/32][H] down scales
  uint8_t* t_gu;      // prefill: GEMM tiles of the interleaved gate/up rows, [EU][2I/128][H/64] tiles
  uint8_t* t_d;       // prefill: GEMM tiles of the down rows, [EU][ceil(H/128)][I/64] tiles
  float* wr;          // [E][H]
  float* bias;        // [E] (zeros when none)
  __nv_bfloat16* wr3; // [3][E][H] bf16 planes summing exactly to wr (prefill router), or null
  // ---- workspace (device), sized for T_max
  int64_t rows_max;   // T_max * (k + S)
  int32_t* ids;       // [T_max][k]
  float* gates;       // [T_max][k]
  float* logits;      // [T_max][E] (decode router)
  int32_t* counts;    // [EU]
  int32_t* offsets;   // [EU + 1]
  int32_t* perm;      // [rows_max]  slot of each grouped row (routed t*k+j, shared T*k+t)
  int32_t* inv;       // [rows_max]
  int32_t* row_token; // [rows_max]
  float* row_gate;    // [rows_max]
  int4* uinfo;        // [EU] (expert, first grouped row, rows, 0) of the experts with rows, ascending id
  int32_t* hist;      // [ceil(T_max/32)][EU] per-tile counts, then per-tile bases
  int4* minfo;        // [rows_max/kTokTile + EU] prefill token tiles: (expert, first row, valid rows, 0)
  int4* minfo_m;      // [EU] the tiles of kSmallTile+1 .. kMidTile rows (an expert's only or last tile)
  int4* minfo_s;      // [EU] the tiles of at most kSmallTile rows (an expert's only or last tile)
  __nv_bfloat16* xperm; // [rows_max][H] x gathered into grouped order (prefill)
  void* hbuf;         // [rows_max][I] fp32 (decode) or bf16 (prefill)
  __nv_bfloat16* yp;  // [rows_max][H] bf16 (prefill)
  float* zpart;       // [kRouterMaxSplit][T_max][E] prefill router: partial logits of a K split
  float* partial;     // [num_sms][min(T_max, 16)][H] decode: per-CTA partial outputs
  Meta* meta;
  int test_grid_timeouts;  // test hook (FWMOE_TEST_GRID_TIMEOUTS at init): decode calls whose grid wait must time out
  // ---- device staging for fw_moe_forward_host
  void* x_dev;
  void* out_dev;
  int32_t* ids_dev;
};

// Brackets one kernel launch with events when the handle is profiling.
struct KernelTimer {
  Timing* t;
  int slot;
  cudaStream_t s;
  KernelTimer(const Handle* h, int kind, cudaStream_t st) : t(h->timing), slot(-1), s(st) {
    if (t && t->next < t->cap) {
      slot = t->next++;
      t->kind[slot] = kind;
      cudaEventRecord(t->ev[2 * slot], s);
    }
  }
  ~KernelTimer() {
    if (slot >= 0) cudaEventRecord(t->ev[2 * slot + 1], s);
  }
};

// Allow a kernel the device's full opt-in shared memory (done at init, never on
// the launch path, so that launches stay legal inside stream capture).
template <typename K>
inline cudaError_t allow_max_dynamic_smem(K kernel) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
  return e;
}

// Record the text of a failed call for fw_moe_last_error; returns st.
fw_status set_error(fw_status st, const char* text);

// ---------------------------------------------------------------- launchers
cudaError_t configure_route_kernels();
cudaError_t configure_decode_kernels();
cudaError_t configure_prefill_kernels();
cudaError_t prepare_prefill(Handle* h);  // tensor maps; needs the planes and workspace allocated
// Each returns cudaGetLastError() of its launches.
// Whether T tokens take the decode kernel for hidden size H (several tokens:
// H <= 2048, the partial outputs live in registers).
bool decode_supported(int H, int T);
cudaError_t launch_quantize_q8_0(const float* w, int64_t rows, int64_t K, uint8_t* blocks, cudaStream_t s);
cudaError_t launch_repack(const Handle* h, int which, int expert0, int count, const uint8_t* blocks,
                          cudaStream_t s);
cudaError_t launch_export(const Handle* h, int which, int expert, uint8_t* blocks, cudaStream_t s);
// select: publish ids/gates/grouping from the router itself (standalone
// route); otherwise only logits, and the decode expert kernels route.
cudaError_t launch_route_decode(Handle* h, const __nv_bfloat16* x, int T, int32_t* ids_out, float* gates_out,
                                bool select, cudaStream_t s);
cudaError_t launch_route_prefill(Handle* h, const __nv_bfloat16* x, int T, int32_t* ids_out, float* gates_out,
                                 cudaStream_t s);
// publish: the gate/up kernel also writes ids (to ids_out/gates_out, which may
// be null) and the grouping, for a forward whose router did not select.
cudaError_t launch_ffn_decode(Handle* h, const __nv_bfloat16* x, int T, __nv_bfloat16* out, bool publish,
                              int32_t* ids_out, float* gates_out, cudaStream_t s);
cudaError_t launch_ffn_prefill(Handle* h, const __nv_bfloat16* x, int T, __nv_bfloat16* out, cudaStream_t s);
// The prefill router on the tensor cores (E <= 128 and planes present):
// ids, gates and the per-32-token expert counts in h->hist. false = not taken.
bool route_prefill_mma_available(const Handle* h);
cudaError_t launch_route_prefill_mma(Handle* h, const __nv_bfloat16* x, int T, int32_t* ids_out, float* gates_out,
                                     cudaStream_t s);
cudaError_t launch_split_router(Handle* h, cudaStream_t s);
cudaError_t launch_get_permutation(const Handle* h, int T, int32_t* offsets, int32_t* perm, int32_t* inv,
                                   cudaStream_t s);

}  // namespace fw

// ---------------------------------------------------------------- device helpers
namespace fw {
namespace dev {

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every wait in these kernels gives up after this long and reports kStatusTimeout.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same with a suspend-time hint: the thread sleeps in the barrier until the
// phase completes (or the hint runs out) instead of re-polling, so waiting
// warps take no issue slots from the working ones.
constexpr uint32_t kSuspendHintNs = 100000;

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete. false = gave up.
// A short wait polls; past about a microsecond the thread also sleeps between
// polls, so that warps parked on a barrier for long leave the issue slots to
// the working ones. Only the first poll is inlined at each call site (code
// size: these kernels are sensitive to instruction-cache misses).
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity) {
  const long long c0 = clock64();
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (clock64() - c0 > 2048) __nanosleep(64);
    if ((i & 63u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity);
}

// Ordering of tensor-core (tcgen05) operations around thread synchronisation.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// One bulk asynchronous copy global -> shared (16-byte aligned, size % 16 == 0),
// completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bulk prefetch of global memory into L2 (16-byte aligned, size % 16 == 0); no
// completion to wait for.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch as a programmatic dependent of the previous kernel in the stream:
// it may start while that kernel's last CTAs still run. Every kernel launched
// so waits (pdl_wait) before it reads or writes global memory, so it
// completes only after its predecessor has -- a chain of such kernels keeps
// the stream's order for all that came before.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Four offset-binary codes (q + 128) packed in a word -> four exact floats q,
// without a conversion instruction: placing byte b in the low mantissa byte of
// 2^23 gives the float 2^23 + q_b + 128 exactly, and subtracting 2^23 + 128
// leaves q_b.
__device__ __forceinline__ void u8x4_to_f32(uint32_t u, float& a, float& b, float& c, float& d) {
  const float bias = 8388736.0f;  // 2^23 + 128
  a = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - bias;
  b = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - bias;
  c = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - bias;
  d = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - bias;
}

// Two bf16 packed in a word -> two floats (exact).
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

__device__ __forceinline__ float half_bits_to_f32(uint16_t b) { return __half2float(__ushort_as_half(b)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ void report(Meta* m, int bits) { atomicOr(&m->status, bits); }

// Sites of bounded waits, recorded with the first timeout (see Meta::diag).
enum WaitSite {
  kSiteGuX = 1, kSiteGuFull = 2, kSiteGuEmpty = 3, kSiteDnH = 4, kSiteDnFull = 5, kSiteDnEmpty = 6,
  kSiteGemm = 7, kSiteGrid = 8, kSiteRouteX = 9
};

static __device__ __noinline__ void report_wait(Meta* m, int site, int64_t stage, int detail) {
  if (atomicCAS(&m->diag[0], 0, site) == 0) {
    m->diag[1] = blockIdx.x;
    m->diag[2] = (int32_t)stage;
    m->diag[3] = detail;
  }
  atomicOr(&m->status, kStatusTimeout);
}

}  // namespace dev
}  // namespace fw
