// vsa_internal.cuh -- definitions shared by the CUDA translation units of libvsa.so: constants,
// the workspace layouts, the per-head scale exponents of the fp16 operand copies, and the
// host-side launch functions of every kernel.
#pragma once

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
constexpr int ORDER_MIN_KV_BLOCKS = 1024;  // sort work items by list length from here on
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;   // pipeline waits: 4 s
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;   // in-flight copies after an abort: 0.2 s

// ---------------------------------------------------------------------------- workspaces
//
// Every workspace starts with a 256-byte header (the device error word at offset 0) followed
// by the per-(b, h) absolute maxima of the operands (4 x uint32 float bits per head: Q, K, V,
// dO), then 1024-byte aligned arrays.

struct BwdLayout {
  size_t err, sched, absmax, split_row, split_acc, delta, order, vbs64, dqacc, q16, k16, v16, do16,
      total;
};

// The backward's main kernel hands out its last items as SPLIT_PARTS claims each (shares of the
// item's step list), so that the grid ends on short claims.  split_capacity(W): how many of the
// W = B * H * S / 64 items the workspace has room to split, SPLIT_PARTS slots of 64 KB each,
// at most a quarter of W slots in all (about 256 bytes per token row) and SPLIT_MAX_SLOTS.
#ifndef VSA_SPLIT_PARTS
#define VSA_SPLIT_PARTS 4
#endif
constexpr int SPLIT_PARTS = VSA_SPLIT_PARTS;
#ifndef VSA_SPLIT_CLAIMS
#define VSA_SPLIT_CLAIMS 2
#endif
constexpr int SPLIT_CLAIMS = VSA_SPLIT_CLAIMS;  // split claims per CTA, on average
constexpr int SPLIT_MAX_SLOTS = 512;
inline int split_capacity(long W) {
  const long slots = W / 4 < SPLIT_MAX_SLOTS ? W / 4 : SPLIT_MAX_SLOTS;
  return static_cast<int>(slots / SPLIT_PARTS);
}
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
  off = align_up(off + bh * 4 * sizeof(uint32_t), 1024);
  // Split items: the first output row, and [parts][dV, dK][64][128] fp32 rows each.
  const size_t nsplit = static_cast<size_t>(split_capacity(static_cast<long>(bh * nb)));
  L.split_row = off;
  off = align_up(off + nsplit * sizeof(int32_t), 1024);
  L.split_acc = off;
  off = align_up(off + nsplit * SPLIT_PARTS * 2 * BLOCK * HEAD_DIM * sizeof(float), 1024);
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
  off = align_up(off + bh * 4 * sizeof(uint32_t), 1024);
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
// The tensor-core operands are fp16 copies X' = X * 2^-e of the bf16 inputs, with e the
// binary exponent of max|X| over one (b, h) head, so |X'| < 2.  bf16 -> fp16 of such values is
// exact except below 2^-17 (absolute error <= 2^-25).  P and dS are rounded to fp16 as well;
// with |Q'|,|K'|,|V'|,|dO'| < 2 and head_dim 128, |dO'.V'| and |Delta'| stay below 512, so
// dS' = P * 2^KP * (dP' - Delta') stays below 2^5 * 1026 < 65504.  The exponents are clamped to
// [-40, 40]; NaN or Inf maxima give 0 (non-finite inputs then propagate).

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

// ---------------------------------------------------------------------------- launches
// Each returns cudaSuccess or the launch error.  `stream` is the caller's stream.

cudaError_t launch_invert(const int32_t* q2k_idx, const int32_t* q2k_num, int topk, int BH,
                          int nb, int32_t* k2q_idx, int32_t* k2q_num, uint32_t* err,
                          cudaStream_t stream);

// Per-head absolute maxima of the operands; with `o`/`dout` non-null also Delta = rowsum(O*dO)
// and zeroing of the fp32 dQ accumulator.
// A job too small for a launch of its own, done by the absmax_delta grid: the valid size of
// every 64-token kv tile, vbs64[t] = clamp(vbs[t / tiles] - 64 (t % tiles), 0, 64) (an entry
// outside [0, 64 tiles] raises VSA_DEVERR_VBS in *err).
struct PreExtras {
  const int32_t* vbs;
  int nb, tiles;
  int32_t* vbs64;
  uint32_t* err;
};
cudaError_t launch_absmax_delta(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                const __nv_bfloat16* v, const __nv_bfloat16* dout,
                                const __nv_bfloat16* o, int BH, int S, uint32_t* absmax,
                                float* delta, float* dqacc, const PreExtras& x,
                                cudaStream_t stream);

// fp16 copies X' = X * 2^-e(head) of up to four [BH, S, 128] bf16 tensors (null entries skipped).
cudaError_t launch_convert(const __nv_bfloat16* const* src, __half* const* dst, int count, int BH,
                           int S, const uint32_t* absmax, cudaStream_t stream);
// Q and dO of the backward as tile-transposed fp16: tile i of head bh is stored at
// ((bh * S/64 + i) * 128 + d) * 64 + r for row r of the tile and head dim d, scaled like
// launch_convert (operand slots 0 and 3 of the per-head maxima).
cudaError_t launch_convert_t(const __nv_bfloat16* q, const __nv_bfloat16* dout, __half* q16t,
                             __half* do16t, int BH, int S, const uint32_t* absmax,
                             cudaStream_t stream);

cudaError_t launch_order(const int32_t* k2q_num, int BH, int nb, int max_q, int32_t* order,
                         cudaStream_t stream);

// dQ = bf16(dqacc * scale); then the bf16 dV, dK rows of the main kernel's `nsplit` split items:
// the sum of their SPLIT_PARTS fp32 parts, added in part order.
cudaError_t launch_postprocess(const float* dqacc, const uint32_t* absmax, int BH, int S,
                               float sm_scale, __nv_bfloat16* dq, const float* split_acc,
                               const int32_t* split_row, int nsplit, __nv_bfloat16* dk,
                               __nv_bfloat16* dv, cudaStream_t stream);

struct BwdMainArgs {
  const __half *q16, *k16, *v16, *do16;
  const int32_t* k2q_idx;
  const int32_t* k2q_num;
  const int32_t* order;  // null: identity order
  const int32_t* vbs;
  const float* lse;
  const float* delta;
  const uint32_t* absmax;
  float* dqacc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  uint32_t* err;
  int32_t* sched;  // zeroed work counter
  float* split_acc;    // split_capacity(B * H * nb) x SPLIT_PARTS slots of [2][64][128]
  int32_t* split_row;  // [split_capacity]
  int B, H, S;
  int nb;     // 64-token tiles per sequence (kv items per head = nb)
  int nsel;   // sparse blocks per sequence (rows of k2q per head); nb = nsel * tiles
  int tiles;  // 64-token tiles per sparse block: 1, or 2 for 128-token blocks
  int max_q;
  float sm_scale;
};
cudaError_t launch_bwd_main(const BwdMainArgs& a, cudaStream_t stream);
// Items the main kernel splits in two for `items` work items on this device.
int bwd_split_items(int items);

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

// Records `e` as this thread's last CUDA error (vsa_last_cuda_error) and returns VSA_ERR_CUDA.
vsa_status record_cuda_failure(cudaError_t e);

}  // namespace vsa
