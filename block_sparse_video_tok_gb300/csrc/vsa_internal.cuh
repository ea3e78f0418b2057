// vsa_internal.cuh -- definitions shared by the CUDA translation units of libvsa.so: constants,
// the workspace layouts, the scale exponents of the fp16 operand copies, and the
// host-side launch functions of every kernel.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/vsa.h"

namespace vsa {

constexpr int BLOCK = 64;      // tokens per sparse block
constexpr int HEAD_DIM = 128;  // the only supported head dimension
constexpr int KP = 5;          // P is carried as P * 2^KP in fp16 (see operand_exponent)
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr int ORDER_MIN_KV_TILES = 1024;  // the backward sorts its items from here on
constexpr uint64_t DEFAULT_WAIT_LIMIT_NS = 4000000000ull;  // pipeline waits: 4 s
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;          // in-flight copies after an abort: 0.2 s

// The limit of every pipeline wait in kernels launched from now on (vsa_set_wait_limit_ns; the
// default unless a caller changed it).  The drains after an abort keep DRAIN_LIMIT_NS.
uint64_t wait_limit_ns();
// Sets it (0: back to DEFAULT_WAIT_LIMIT_NS); returns the previous limit.
uint64_t set_wait_limit_ns(uint64_t ns);

// ---------------------------------------------------------------------------- workspaces
//
// Every workspace starts with a 256-byte header (the device error word at offset 0) followed
// by per-(b, h) statistics of the operands (HEAD_STATS uint32 float bits per head, see HeadStat),
// then 1024-byte aligned arrays.  The backward also keeps statistics per 64-token kv tile
// (TILE_STATS words per tile of each head, see TileStat).

constexpr int HEAD_STATS = 8;
enum HeadStat : int {
  HS_Q = 0,        // max |Q| of the head
  HS_K = 1,        // max |K|
  HS_V = 2,        // max |V|
  HS_DO = 3,       // max |dO|
  HS_DO_NORM = 4,  // max over rows of the row's L2 norm of dO (backward)
  HS_DELTA = 5     // max over rows of |Delta| (backward)
};
constexpr int TILE_STATS = 4;
enum TileStat : int {
  TS_K = 0,      // max |K| over the tile's 64 rows
  TS_V = 1,      // max |V|
  TS_V_NORM = 2  // max over the tile's rows of the row's L2 norm of V
};

struct BwdLayout {
  size_t err, sched, absmax, tstat, split_row, split_acc, delta, order, vbs64, dqacc, q16, k16,
      v16, do16, total;
};

// The backward's main kernel hands out its last items as `parts` claims each (consecutive
// shares of the item's step list), so that the grid ends on short claims: quarters
// (SPLIT_PARTS), or halves when there are fewer than 8 items per SM (bwd_split_plan).  Each part
// fills a slot of 64 KB ([dV, dK][64][128] fp32); split_slots(W): the workspace's slots for W =
// B * H * S / 64 items, a quarter of W (about 256 bytes per token row) and at most
// SPLIT_MAX_SLOTS.
constexpr int SPLIT_PARTS = 4;
constexpr int SPLIT_CLAIMS = 2;  // split claims per CTA, on average
constexpr int SPLIT_MAX_SLOTS = 512;
inline long split_slots(long W) { return W / 4 < SPLIT_MAX_SLOTS ? W / 4 : SPLIT_MAX_SLOTS; }
struct FwdLayout {
  size_t err, sched, absmax, bitmap, vbs64, v16, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline BwdLayout bwd_layout(long B, long H, long S) {
  BwdLayout L{};
  const size_t bh = static_cast<size_t>(B) * H, rows = bh * S, nb = S / BLOCK;
  size_t off = 0;
  L.err = off;
  L.sched = 128;  // work counter of the main kernel's dynamic scheduler (inside the header)
  off += 256;
  L.absmax = off;
  off = align_up(off + bh * HEAD_STATS * sizeof(uint32_t), 1024);
  L.tstat = off;
  off = align_up(off + bh * nb * TILE_STATS * sizeof(uint32_t), 1024);
  // Split items: the first output row of each (at most one item per slot), and the parts'
  // [dV, dK][64][128] fp32 rows, one slot each.
  const size_t slots = static_cast<size_t>(split_slots(static_cast<long>(bh * nb)));
  L.split_row = off;
  off = align_up(off + slots * sizeof(int32_t), 1024);
  L.split_acc = off;
  off = align_up(off + slots * 2 * BLOCK * HEAD_DIM * sizeof(float), 1024);
  L.delta = off;
  off = align_up(off + rows * sizeof(float), 1024);
  L.order = off;
  off = align_up(off + bh * nb * sizeof(int32_t), 1024);
  L.vbs64 = off;
  off = align_up(off + nb * sizeof(int32_t), 1024);
  L.dqacc = off;
  off = align_up(off + rows * HEAD_DIM * sizeof(float), 1024);
  L.q16 = off;
  off = align_up(off + rows * HEAD_DIM * sizeof(__half), 1024);
  L.k16 = off;
  off = align_up(off + rows * HEAD_DIM * sizeof(__half), 1024);
  L.v16 = off;
  off = align_up(off + rows * HEAD_DIM * sizeof(__half), 1024);
  L.do16 = off;
  off = align_up(off + rows * HEAD_DIM * sizeof(__half), 1024);
  L.total = off;
  return L;
}

inline FwdLayout fwd_layout(long B, long H, long S) {
  FwdLayout L{};
  const size_t bh = static_cast<size_t>(B) * H, rows = bh * S, nb = S / BLOCK;
  const size_t words = (nb + 31) / 32;
  size_t off = 0;
  L.err = off;
  L.sched = 128;  // work counter of the main kernel's dynamic scheduler (inside the header)
  off += 256;
  L.absmax = off;
  off = align_up(off + bh * HEAD_STATS * sizeof(uint32_t), 1024);
  L.bitmap = off;
  off = align_up(off + bh * nb * words * sizeof(uint32_t), 1024);
  L.vbs64 = off;
  off = align_up(off + nb * sizeof(int32_t), 1024);
  L.v16 = off;
  off = align_up(off + rows * HEAD_DIM * sizeof(__half), 1024);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------- operand scales
//
// The tensor-core operands are fp16 copies X' = X * 2^-e of the bf16 inputs, with e the binary
// exponent of max|X| over a group of values, so |X'| < 2: Q and dO per (b, h) head, K and V of
// the backward per 64-token kv tile (so that an outlier only moves the scale of its own tile), V
// of the forward per head.  A value converts exactly unless it lies 17 or more binades below its
// group's maximum (fp16 subnormals: absolute error <= 2^(e-25)).  P is carried as P * 2^KP
// (P <= 1).  dS of kv tile j is carried as 2^kappa_j P (dP' - Delta'), with kappa_j from a bound
// of |dP' - Delta'| (ds_exponent): a fixed scale would have to allow for the worst case, and an
// outlier in dO or V would then push the dS values of every other row into fp16's subnormal
// range.  The exponents are clamped to [-40, 40]; NaN or Inf maxima give 0 (non-finite inputs
// then propagate).

__host__ __device__ inline int operand_exponent(uint32_t absmax_bits) {
  const uint32_t bits = absmax_bits & 0x7FFFFFFFu;
  const int field = static_cast<int>((bits >> 23) & 0xFFu);
  if (bits == 0u || field == 0xFF) return 0;
  int e = field - 127;  // subnormal maxima give -127 and clamp to -40
  return e < -40 ? -40 : (e > 40 ? 40 : e);
}

// 2^n as a float, exactly, for |n| <= 126.
__host__ __device__ inline float exp2i(int n) {
  union {
    uint32_t u;
    float f;
  } x;
  x.u = static_cast<uint32_t>(n + 127) << 23;
  return x.f;
}

__host__ __device__ inline float bits_float(uint32_t u) {
  union {
    uint32_t u;
    float f;
  } x;
  x.u = u;
  return x.f;
}

__host__ __device__ inline int clamp_exponent(int n, int lim) {
  return n < -lim ? -lim : (n > lim ? lim : n);
}

// kappa_j, the exponent of the dS operand of kv tile j: dS' = fp16(2^kappa P (dP' - Delta')) with
// dP' = dO'.V' = 2^-(eo + ev) dO.V (dO' scaled per head by 2^-eo, V' per tile by 2^-ev) and Delta'
// = 2^-(eo + ev) Delta.  By Cauchy-Schwarz |dO_r . V_t| <= |dO_r| |V_t| (row L2 norms), so with
// P <= 1, |dS'| <= 2^kappa 2^-(eo + ev) (max_r |dO_r| max_t|V_t| + max_r |Delta_r|) = 2^kappa b.
// kappa = 13 - floor(log2 b) keeps |dS'| below 2^14, a factor of 4 under the fp16 maximum for the
// rounding of the operands and of the fp32 sums.  Clamped to [-60, 60]; 0 if b is 0 or not finite.
__host__ __device__ inline int ds_exponent(float do_norm, float v_norm, float delta_max, int eo,
                                           int ev) {
  const float a = exp2i(-eo), c = exp2i(-ev);
  const float b = (do_norm * a) * (v_norm * c) + (delta_max * a) * c;
  if (!(b > 0.f && b <= 3.4028235e38f)) return 0;
  union {
    float f;
    uint32_t u;
  } x;
  x.f = b;
  const int f = static_cast<int>((x.u >> 23) & 0xFFu) - 127;  // floor(log2 b); -127 if subnormal
  return clamp_exponent(13 - f, 60);
}

// Programmatic dependent launch: wait until the previous grid on the stream has completed and its
// memory operations are visible (a no-op when the kernel was launched without the attribute).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------- launches
// `kernel` launched so that it may start before the previous kernel on `stream` has finished
// (programmatic dependent launch); it calls grid_dependency_wait() before it touches global
// memory that the previous kernels write or read.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Each returns cudaSuccess or the launch error.  `stream` is the caller's stream.

// Zeroes `bytes` (a multiple of 16) from `p` (16-byte aligned) on.
cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t stream);

cudaError_t launch_invert(const int32_t* q2k_idx, const int32_t* q2k_num, int topk, int BH,
                          int nb, int32_t* k2q_idx, int32_t* k2q_num, uint32_t* err,
                          cudaStream_t stream);

// Per-head absolute maxima of the operands; with `o`/`dout` non-null also Delta = rowsum(O*dO)
// and zeroing of the fp32 dQ accumulator.
// A job too small for a launch of its own, done by the absmax_delta grid: the valid size of
// every 64-token kv tile, vbs64[t] = clamp(vbs[t / tiles] - 64 (t % tiles), 0, 64) (an entry
// outside [0, 64 tiles] raises VSA_DEVERR_VBS in *err).
// With `tstat` non-null (the backward), the grid also writes the statistics of every 64-token kv
// tile of K and V (TILE_STATS words each) and the per-head dO row-norm and |Delta| maxima, and,
// since each CTA holds one whole tile of K and V, their fp16 copies scaled by the tile's own
// exponent (k16, v16: row-major [BH * S, 128]).  With `order` non-null it also writes the work
// order of the nsel k2q rows of every head (launch_order's permutation; counts k2q_num clamped
// to [0, max_q]).
struct PreExtras {
  const int32_t* vbs;
  int nb, tiles;
  int32_t* vbs64;
  uint32_t* err;
  uint32_t* tstat;
  __half* k16;
  __half* v16;
  const int32_t* k2q_num;
  int32_t* order;
  int nsel, max_q;
};
cudaError_t launch_absmax_delta(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                const __nv_bfloat16* v, const __nv_bfloat16* dout,
                                const __nv_bfloat16* o, int BH, int S, uint32_t* absmax,
                                float* delta, float* dqacc, const PreExtras& x,
                                cudaStream_t stream);

// fp16 copies X' = X * 2^-e of up to four [BH, S, 128] bf16 tensors (null entries skipped), slot
// t of the per-head statistics giving e; with `tstat` non-null, tensors 1 (K) and 2 (V) take e
// per 64-token tile from the tile statistics instead.
cudaError_t launch_convert(const __nv_bfloat16* const* src, __half* const* dst, int count, int BH,
                           int S, const uint32_t* absmax, const uint32_t* tstat,
                           cudaStream_t stream);
// Q and dO of the backward as tile-transposed fp16: tile i of head bh is stored at
// ((bh * S/64 + i) * 128 + d) * 64 + r for row r of the tile and head dim d, scaled like
// launch_convert (operand slots 0 and 3 of the per-head maxima).
cudaError_t launch_convert_t(const __nv_bfloat16* q, const __nv_bfloat16* dout, __half* q16t,
                             __half* do16t, int BH, int S, const uint32_t* absmax,
                             cudaStream_t stream);

cudaError_t launch_order(const int32_t* k2q_num, int BH, int nb, int max_q, int32_t* order,
                         cudaStream_t stream);

// dQ = bf16(dqacc * scale); then the bf16 dV, dK rows of the main kernel's split items
// (bwd_split_plan): the sum of the `parts` fp32 parts of each, added in part order.
cudaError_t launch_postprocess(const float* dqacc, const uint32_t* absmax, int BH, int S,
                               float sm_scale, __nv_bfloat16* dq, const float* split_acc,
                               const int32_t* split_row, int nsplit, int parts, __nv_bfloat16* dk,
                               __nv_bfloat16* dv, cudaStream_t stream);

struct BwdMainArgs {
  const __half *q16, *k16, *v16, *do16;
  const int32_t* k2q_idx;
  const int32_t* k2q_num;
  const int32_t* order;  // the work order (vsa_work_order's permutation), or null: item order
  const int32_t* vbs;
  const float* lse;
  const float* delta;
  const uint32_t* absmax;
  const uint32_t* tstat;
  float* dqacc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  uint32_t* err;
  int32_t* sched;  // zeroed work counter
  float* split_acc;    // split_slots(B * H * nb) slots of [2][64][128]
  int32_t* split_row;  // [split_slots]: the first output row of each split item
  int B, H, S;
  int nb;     // 64-token tiles per sequence (kv items per head = nb)
  int nsel;   // sparse blocks per sequence (rows of k2q per head); nb = nsel * tiles
  int tiles;  // 64-token tiles per sparse block: 1, or 2 for 128-token blocks
  int max_q;
  float sm_scale;
  uint64_t wait_ns;  // limit of each pipeline wait
};
cudaError_t launch_bwd_main(const BwdMainArgs& a, cudaStream_t stream);
// How the main kernel splits its last items for `items` work items on this device: `nsplit`
// items, `parts` claims each.
struct SplitPlan {
  int parts, nsplit;
};
SplitPlan bwd_split_plan(int items);

// Selection bitmap of the forward at 64-token granularity: [BH, nb * tiles, ceil(nb * tiles / 32)]
// bits from q2k rows that count blocks of `tiles` 64-token tiles (1 or 2).
cudaError_t launch_fwd_bitmap(const int32_t* q2k_idx, const int32_t* q2k_num, int topk, int BH,
                              int nb, int tiles, uint32_t* bitmap, uint32_t* err,
                              cudaStream_t stream);


struct FwdMainArgs {
  const __nv_bfloat16 *q, *k;  // the caller's bf16 Q and K (the S = Q K^T operands)
  const __half* v16;           // V in fp16, scaled by 2^-e_v (the B operand of P.V)
  const uint32_t* bitmap;  // [BH, nb, words] selection bits
  const int32_t* vbs;
  const uint32_t* absmax;
  __nv_bfloat16* o;
  float* lse;
  uint32_t* err;
  int32_t* sched;  // zeroed work counter
  int B, H, S, nb;
  float sm_scale;
  uint64_t wait_ns;  // limit of each pipeline wait
};
cudaError_t launch_fwd_main(const FwdMainArgs& a, cudaStream_t stream);

// Tensor maps (tmap.cu).
// [rows, 128] fp32 (the dQ accumulator), box 32 columns x 64 rows, no swizzle.
cudaError_t make_tmap_rows128_f32(CUtensorMap* map, const void* base, long rows);
// Tile-transposed fp16 operand (launch_convert_t): `rows` token rows give rows * 2 rows of 64
// halves; box 64 columns x 128 * `tiles` rows, 128-byte swizzle.
cudaError_t make_tmap_tiles_t(CUtensorMap* map, const void* base, long rows, int tiles);
// Tensor map of a [rows, 128] fp16 (bf16 with `bf16`) matrix, box 64 columns x 64 rows,
// 128-byte swizzle.
cudaError_t make_tmap_rows128_f16(CUtensorMap* map, const void* base, long rows,
                                  bool bf16 = false);
// The same matrix seen as [2 column halves][rows][64 columns] (coordinates: column within the
// half, row, half), box 64 columns x `box_rows` rows x both halves, 128-byte swizzle.  One copy
// lands both 64-column halves of `box_rows` consecutive rows in shared memory half after half,
// the layout two 2-D boxes per half would give, in one request instead of two or four.
cudaError_t make_tmap_rows128_f16_halves(CUtensorMap* map, const void* base, long rows,
                                         int box_rows, bool bf16 = false);

int device_sm_count();

// Whether vsa_bwd takes its work items in the sorted order (vsa_work_order) on this device:
// from ORDER_MIN_KV_TILES 64-token kv tiles per sequence on, or with fewer than 8 items per SM.
bool use_work_order(int BH, int S);

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current device, once per
// device: the attribute belongs to each device's context, so a process that drives several GPUs
// sets it on each.  `done` keeps one bit per device id below 64 (ids from 64 on set it on every
// call); concurrent first calls may both set it, which is harmless.
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel* kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Records `e` as this thread's last CUDA error (vsa_last_cuda_error) and returns VSA_ERR_CUDA.
vsa_status record_cuda_failure(cudaError_t e);

}  // namespace vsa
