// prepost.cu -- the memory-bound kernels around the tensor-core kernels:
//   absmax_delta  per-head max|X| of the operands (per 64-token kv tile for K and V of the
//                 backward, with the row-norm bounds the dS scale needs); Delta =
//                 rowsum(bf16(O) * dO) in fp32, from
//                 the O the backward receives (FastVideo compare main...vsa_bwd_fix,
//                 block_sparse_bwd_launch_sm100a.cuh, BlockSparseVsaBwdArgs: the preprocess
//                 writes Delta); zeroing of the fp32 dQ accumulator, which the main kernel
//                 reduces into and the postprocess reads (same struct); the valid size of every
//                 64-token kv tile.
//   convert       scaled fp16 copies of the bf16 operands for the tensor cores.
//   convert_t     the same for Q and dO of the backward, each 64-row tile stored transposed
//                 ([128 head dims][64 rows]), so one 16 KB copy brings a whole tile.
//   order         work order: (b, h) segments, items sorted by descending k2q list length,
//                 stable (the commit message: sorted on the device, from 1024 kv blocks per
//                 sequence on; here at every size, computed by the statistics pass).
//   postprocess   dQ = bf16(dqacc * sm_scale * 2^scale) (the commit message's postprocess step
//                 applies sm_scale to dQ); the dV, dK rows of the main kernel's split items.
//   fwd_bitmap    per-q-block selection bitmaps for the forward.
// All are HBM-bound; each thread moves 16-byte vectors, grids cover the data once.
#include "vsa_internal.cuh"

namespace vsa {

namespace {

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t absmax_bits8(uint4 x) {
  uint32_t m = 0;
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = max(m, (w[i] << 16) & 0x7FFFFFFFu);
    m = max(m, w[i] & 0x7FFF0000u);
  }
  return m;
}

__device__ __forceinline__ uint32_t warp_max(uint32_t v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

// 8 bf16 values times s, rounded to fp16 (round to nearest even).
__device__ __forceinline__ uint4 to_half8(uint4 x, float s) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __floats2half2_rn(bf16lo(w[i]) * s, bf16hi(w[i]) * s);
    out[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Sum of squares of the 8 bf16 values of a 16-byte chunk.
__device__ __forceinline__ float sumsq8(uint4 x) {
  float s = bf16lo(x.x) * bf16lo(x.x) + bf16hi(x.x) * bf16hi(x.x);
  s += bf16lo(x.y) * bf16lo(x.y) + bf16hi(x.y) * bf16hi(x.y);
  s += bf16lo(x.z) * bf16lo(x.z) + bf16hi(x.z) * bf16hi(x.z);
  s += bf16lo(x.w) * bf16lo(x.w) + bf16hi(x.w) * bf16hi(x.w);
  return s;
}

// Sum over the 16 lanes that hold one 128-element row.
__device__ __forceinline__ float row_sum16(float s) {
#pragma unroll
  for (int d = 8; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
  return s;
}

// Position of k2q row x of one head in the work order: the rows whose count (clamped to
// [0, max_q]) is larger, plus the rows with an equal count and a smaller index -- a stable sort
// by descending count.  Executed by a whole CTA of 256 threads, which all get the result;
// `scratch` is 8 shared ints, free again on return.
__device__ __forceinline__ int order_position(const int32_t* __restrict__ counts, int n,
                                              int max_q, int x, int* scratch) {
  auto clamped = [max_q](int c) { return c < 0 ? 0 : (c > max_q ? max_q : c); };
  const int cx = clamped(counts[x]);
  int pos = 0;
  for (int y = threadIdx.x; y < n; y += blockDim.x) {
    const int cy = clamped(__ldg(counts + y));
    pos += (cy > cx) || (cy == cx && y < x);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) pos += __shfl_xor_sync(0xffffffffu, pos, d);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = pos;
  __syncthreads();
  int total = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) total += scratch[w];
  __syncthreads();
  return total;
}

// Grid (S / 64, BH), 256 threads: 16 lanes per 128-element row (8 bf16 = 16 B per lane), two
// rows per warp per iteration, 64 rows per CTA.
constexpr int PRE_THREADS = 256;

// Zeroes n 16-byte words from p on (the workspace's header, statistics and split rows, which the
// next kernels accumulate into), as a kernel so that a step's launches chain as programmatic
// dependent launches; the previous call's postprocess may still be reading them, hence the wait.
__global__ void __launch_bounds__(256) zero_kernel(uint4* __restrict__ p, size_t n) {
  grid_dependency_wait();
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    p[i] = z;
}

__global__ void __launch_bounds__(PRE_THREADS, 4) absmax_delta_kernel(
    const uint4* __restrict__ q, const uint4* __restrict__ k, const uint4* __restrict__ v,
    const uint4* __restrict__ dout, const uint4* __restrict__ o, int S, uint32_t* absmax,
    float* __restrict__ delta, float4* __restrict__ dqacc, PreExtras x) {
  grid_dependency_wait();
  // A small job spread over the whole grid: the clamped valid size of every 64-token kv tile
  // (64-token tile t of block t / tiles).
  {
    const size_t gt =
        (static_cast<size_t>(blockIdx.y) * gridDim.x + blockIdx.x) * PRE_THREADS + threadIdx.x;
    const size_t gn = static_cast<size_t>(gridDim.x) * gridDim.y * PRE_THREADS;
    const int lim = BLOCK * x.tiles;
    uint32_t badv = 0;
    for (size_t t = gt; t < static_cast<size_t>(x.nb) * x.tiles; t += gn) {
      const int vv = x.vbs[t / x.tiles];
      if (vv < 0 || vv > lim) badv |= VSA_DEVERR_VBS;
      const int w = (vv < 0 ? 0 : (vv > lim ? lim : vv)) - BLOCK * static_cast<int>(t % x.tiles);
      x.vbs64[t] = w < 0 ? 0 : (w > BLOCK ? BLOCK : w);
    }
    if (badv && x.err) atomicOr(x.err, badv);
  }
  const int bh = blockIdx.y;
  const int half = threadIdx.x >> 4;  // which of the 16 rows-in-flight
  const int sub = threadIdx.x & 15;   // 16-byte chunk of the row
  const bool bwd = (dout != nullptr);
  const bool stats = (x.tstat != nullptr);
  constexpr int ROWS = BLOCK / (PRE_THREADS / 16);  // rows of the tile per thread
  // Maxima as float bits (non-negative floats order like their bits): |Q|, |K|, |V|, |dO|, then
  // the squared row norms of dO and V and |Delta|.
  uint32_t mq = 0, mk = 0, mv = 0, mdo = 0, ndo2 = 0, nv2 = 0, mdl = 0;
  uint4 kt[ROWS], vt[ROWS];  // this thread's chunks of the K and V tile, converted at the end
#pragma unroll
  for (int u = 0; u < ROWS; ++u) {
    const int rr = half + u * (PRE_THREADS / 16);
    const size_t row = static_cast<size_t>(bh) * S + static_cast<size_t>(blockIdx.x) * BLOCK + rr;
    const size_t at = row * 16 + sub;
    if (q) mq = max(mq, absmax_bits8(q[at]));  // a null operand is not scanned (its max stays 0)
    if (k) {
      kt[u] = k[at];
      mk = max(mk, absmax_bits8(kt[u]));
    }
    if (v) {
      vt[u] = v[at];
      mv = max(mv, absmax_bits8(vt[u]));
      if (stats) nv2 = max(nv2, __float_as_uint(row_sum16(sumsq8(vt[u]))));
    }
    if (bwd) {
      const uint4 a = dout[at], b = o[at];
      mdo = max(mdo, absmax_bits8(a));
      float s = bf16lo(a.x) * bf16lo(b.x) + bf16hi(a.x) * bf16hi(b.x);
      s += bf16lo(a.y) * bf16lo(b.y) + bf16hi(a.y) * bf16hi(b.y);
      s += bf16lo(a.z) * bf16lo(b.z) + bf16hi(a.z) * bf16hi(b.z);
      s += bf16lo(a.w) * bf16lo(b.w) + bf16hi(a.w) * bf16hi(b.w);
      s = row_sum16(s);
      if (sub == 0) delta[row] = s;
      if (stats) {
        mdl = max(mdl, __float_as_uint(fabsf(s)));
        ndo2 = max(ndo2, __float_as_uint(row_sum16(sumsq8(a))));
      }
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      float4* dst = dqacc + row * 32 + sub * 2;
      dst[0] = z;
      dst[1] = z;
    }
  }
  constexpr int NRED = 7;
  __shared__ uint32_t red[NRED][PRE_THREADS / 32];
  __shared__ int scratch[PRE_THREADS / 32];
  // A side job of the backward's grid: CTA (tile, head) places k2q row `tile` of its head in the
  // work order (one CTA per row; the rows are blocks of x.tiles 64-token tiles).
  if (x.order != nullptr && static_cast<int>(blockIdx.x) < x.nsel) {
    const int r = blockIdx.x;
    const size_t seg = static_cast<size_t>(bh) * x.nsel;
    const int pos = order_position(x.k2q_num + seg, x.nsel, x.max_q, r, scratch);
    if (threadIdx.x == 0) x.order[seg + pos] = static_cast<int32_t>(seg) + r;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t mine[NRED] = {mq, mk, mv, mdo, ndo2, nv2, mdl};
#pragma unroll
  for (int i = 0; i < NRED; ++i) {
    const uint32_t m = warp_max(mine[i]);
    if (lane == 0) red[i][warp] = m;
  }
  __syncthreads();
  if (threadIdx.x < NRED) {
    uint32_t m = 0;
    for (int w = 0; w < PRE_THREADS / 32; ++w) m = max(m, red[threadIdx.x][w]);
    uint32_t* hs = absmax + bh * HEAD_STATS;
    uint32_t* ts = stats ? x.tstat + (static_cast<size_t>(bh) * gridDim.x + blockIdx.x) * TILE_STATS
                         : nullptr;
    const int i = threadIdx.x;
    if (i < 4) {
      if (m) atomicMax(hs + i, m);  // HS_Q, HS_K, HS_V, HS_DO
      if (stats && i == 1) ts[TS_K] = m;  // one CTA per tile: plain stores
      if (stats && i == 2) ts[TS_V] = m;
    } else if (stats) {
      // Squared norms become norms here (sqrt is monotonic, so the maximum is kept).
      const uint32_t val = (i == 6) ? m : __float_as_uint(sqrtf(__uint_as_float(m)));
      if (i == 4) {
        if (val) atomicMax(hs + HS_DO_NORM, val);
      } else if (i == 5) {
        ts[TS_V_NORM] = val;
      } else {
        if (val) atomicMax(hs + HS_DELTA, val);
      }
    }
  }
  if (x.k16 != nullptr) {
    // The tile's K and V maxima are in red[1], red[2]: convert the chunks held in registers.
    uint32_t tk = 0, tv = 0;
#pragma unroll
    for (int w = 0; w < PRE_THREADS / 32; ++w) {
      tk = max(tk, red[1][w]);
      tv = max(tv, red[2][w]);
    }
    const float sk = exp2i(-operand_exponent(tk)), sv = exp2i(-operand_exponent(tv));
    uint4* k16 = reinterpret_cast<uint4*>(x.k16);
    uint4* v16 = reinterpret_cast<uint4*>(x.v16);
#pragma unroll
    for (int u = 0; u < ROWS; ++u) {
      const int rr = half + u * (PRE_THREADS / 16);
      const size_t at =
          (static_cast<size_t>(bh) * S + static_cast<size_t>(blockIdx.x) * BLOCK + rr) * 16 + sub;
      k16[at] = to_half8(kt[u], sk);
      v16[at] = to_half8(vt[u], sv);
    }
  }
}

// One thread per 8 elements; up to four tensors in one launch (blockIdx.y).
struct ConvertPack {
  const uint4* src[4];
  uint4* dst[4];
  const uint32_t* tstat;  // non-null: K (1) and V (2) take their exponent per 64-token tile
};

__global__ void __launch_bounds__(256) convert_kernel(ConvertPack pk, size_t chunks_per_head,
                                                      size_t total_chunks,
                                                      const uint32_t* __restrict__ absmax) {
  grid_dependency_wait();
  const int t = blockIdx.y;
  const uint4* __restrict__ src = t == 0 ? pk.src[0] : t == 1 ? pk.src[1] : t == 2 ? pk.src[2] : pk.src[3];
  uint4* __restrict__ dst = t == 0 ? pk.dst[0] : t == 1 ? pk.dst[1] : t == 2 ? pk.dst[2] : pk.dst[3];
  if (src == nullptr) return;
  const bool per_tile = pk.tstat != nullptr && (t == 1 || t == 2);
  for (size_t c = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; c < total_chunks;
       c += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int bh = static_cast<int>(c / chunks_per_head);
    // 16 chunks per row, 64 rows per tile: chunk c lies in tile c / 1024 (heads hold whole
    // tiles).
    const uint32_t bits = per_tile ? pk.tstat[(c >> 10) * TILE_STATS + (t == 1 ? TS_K : TS_V)]
                                   : absmax[bh * HEAD_STATS + t];
    dst[c] = to_half8(src[c], exp2i(-operand_exponent(bits)));
  }
}

// Grid (S / 64, BH, count): one 64-row tile of one tensor per CTA, read as rows of 128 bf16,
// scaled, and written as 128 rows (head dims) of 64 fp16 (the tile's rows).  The shared tile has
// rows of 130 halves (65 words), so the column gathers of the write phase hit distinct banks.
struct ConvertTPack {
  const uint4* src[2];
  __half* dst[2];
  int slot[2];  // operand index in the per-head maxima (Q 0, dO 3)
};

__global__ void __launch_bounds__(256) convert_t_kernel(ConvertTPack pk, int S,
                                                        const uint32_t* __restrict__ absmax) {
  grid_dependency_wait();
  constexpr int LD = 130;
  __shared__ __half tl[BLOCK * LD];
  const int t = blockIdx.z, bh = blockIdx.y, tile = blockIdx.x, nt = gridDim.x;
  const uint4* __restrict__ src = t == 0 ? pk.src[0] : pk.src[1];
  __half* __restrict__ dst = t == 0 ? pk.dst[0] : pk.dst[1];
  const float sc =
      exp2i(-operand_exponent(absmax[bh * HEAD_STATS + (t == 0 ? pk.slot[0] : pk.slot[1])]));
  const size_t row0 = static_cast<size_t>(bh) * S + static_cast<size_t>(tile) * BLOCK;
  // The tile's 1024 16-byte chunks, four per thread, all loads in flight before any is used.
  constexpr int PER = BLOCK * 16 / 256;
  uint4 xs[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int c = threadIdx.x + u * 256;
    xs[u] = src[(row0 + (c >> 4)) * 16 + (c & 15)];
  }
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int c = threadIdx.x + u * 256, r = c >> 4, ch = c & 15;
    const uint32_t w[4] = {xs[u].x, xs[u].y, xs[u].z, xs[u].w};
    __half2* d2 = reinterpret_cast<__half2*>(tl + r * LD + ch * 8);
#pragma unroll
    for (int i = 0; i < 4; ++i) d2[i] = __floats2half2_rn(bf16lo(w[i]) * sc, bf16hi(w[i]) * sc);
  }
  __syncthreads();
  uint4* out = reinterpret_cast<uint4*>(dst + (static_cast<size_t>(bh) * nt + tile) * HEAD_DIM *
                                                  BLOCK);
  for (int c = threadIdx.x; c < HEAD_DIM * 8; c += blockDim.x) {
    const int d = c >> 3, rc = c & 7;
    uint32_t v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __halves2half2(tl[(rc * 8 + 2 * i) * LD + d], tl[(rc * 8 + 2 * i + 1) * LD + d]);
      v[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    out[d * 8 + rc] = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

// One CTA per item (grid-stride over the B * H * n items): item x of head bh goes to position
// order_position(x) of its head's segment.  The same function places the items in the backward's
// statistics pass, so this launch (vsa_work_order) shows the order the backward uses.
__global__ void __launch_bounds__(256) order_kernel(const int32_t* __restrict__ k2q_num, int n,
                                                    long items, int max_q,
                                                    int32_t* __restrict__ order) {
  __shared__ int scratch[8];
  for (long i = blockIdx.x; i < items; i += gridDim.x) {
    const long bh = i / n;
    const int x = static_cast<int>(i - bh * n);
    const int pos = order_position(k2q_num + bh * n, n, max_q, x, scratch);
    if (threadIdx.x == 0) order[bh * n + pos] = static_cast<int32_t>(bh * n + x);
  }
}

template <int PARTS>
__global__ void __launch_bounds__(256) postprocess_kernel(
    const float4* __restrict__ dqacc, const uint32_t* __restrict__ absmax, size_t chunks_per_head,
    size_t total_chunks, float sm_scale, uint4* __restrict__ dq,
    const float4* __restrict__ split_acc, const int32_t* __restrict__ split_row, int split_chunks,
    uint4* __restrict__ dk, uint4* __restrict__ dv) {
  grid_dependency_wait();
  for (size_t c = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; c < total_chunks;
       c += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int bh = static_cast<int>(c / chunks_per_head);
    // The main kernel leaves dQ / (sm_scale 2^e) in the accumulator, e the exponent of the
    // head's max |dO| (every other scale is undone per item before the reduction).
    const float s = sm_scale * exp2i(operand_exponent(absmax[bh * HEAD_STATS + HS_DO]));
    const float4 a = dqacc[2 * c], b = dqacc[2 * c + 1];
    const __nv_bfloat162 r0 = __floats2bfloat162_rn(a.x * s, a.y * s);
    const __nv_bfloat162 r1 = __floats2bfloat162_rn(a.z * s, a.w * s);
    const __nv_bfloat162 r2 = __floats2bfloat162_rn(b.x * s, b.y * s);
    const __nv_bfloat162 r3 = __floats2bfloat162_rn(b.z * s, b.w * s);
    dq[c] = make_uint4(*reinterpret_cast<const uint32_t*>(&r0),
                       *reinterpret_cast<const uint32_t*>(&r1),
                       *reinterpret_cast<const uint32_t*>(&r2),
                       *reinterpret_cast<const uint32_t*>(&r3));
  }
  // Split items of the main kernel: part x of split item s holds [dV, dK][64 kv rows][128] fp32
  // in slot s * PARTS + x, already scaled (rows past the block's valid size hold zeros); 16
  // chunks of 8 per row.  The parts are added in order, so the sums do not depend on which part
  // finished first.
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < split_chunks;
       c += gridDim.x * blockDim.x) {
    const int slot = c / (2 * BLOCK * 16), rem = c % (2 * BLOCK * 16);
    const bool is_dk = rem >= BLOCK * 16;
    const int t = (rem / 16) % BLOCK, d8 = rem % 16;
    const float4* part =
        split_acc + (static_cast<size_t>(slot) * PARTS * 2 * BLOCK * 16 + rem) * 2;
    float4 a = part[0], b = part[1];
#pragma unroll
    for (int x = 1; x < PARTS; ++x) {
      const float4 a2 = part[x * 2 * BLOCK * 16 * 2], b2 = part[x * 2 * BLOCK * 16 * 2 + 1];
      a = make_float4(a.x + a2.x, a.y + a2.y, a.z + a2.z, a.w + a2.w);
      b = make_float4(b.x + b2.x, b.y + b2.y, b.z + b2.z, b.w + b2.w);
    }
    const __nv_bfloat162 r0 = __floats2bfloat162_rn(a.x, a.y);
    const __nv_bfloat162 r1 = __floats2bfloat162_rn(a.z, a.w);
    const __nv_bfloat162 r2 = __floats2bfloat162_rn(b.x, b.y);
    const __nv_bfloat162 r3 = __floats2bfloat162_rn(b.z, b.w);
    const size_t at = (static_cast<size_t>(split_row[slot]) + t) * 16 + d8;
    (is_dk ? dk : dv)[at] = make_uint4(*reinterpret_cast<const uint32_t*>(&r0),
                                       *reinterpret_cast<const uint32_t*>(&r1),
                                       *reinterpret_cast<const uint32_t*>(&r2),
                                       *reinterpret_cast<const uint32_t*>(&r3));
  }
}

// One thread per q2k entry: set bit j of q block i's row of the selection bitmap.
// q2k rows count blocks of `tiles` 64-token tiles; the bitmap has one row of nb * tiles bits per
// 64-token query tile, so a selected (I, J) sets the tiles x tiles bits of that block pair.
__global__ void __launch_bounds__(256) fwd_bitmap_kernel(const int32_t* __restrict__ q2k_idx,
                                                         const int32_t* __restrict__ q2k_num,
                                                         int topk, int nb, int tiles,
                                                         size_t entries,
                                                         uint32_t* __restrict__ bitmap,
                                                         uint32_t* err) {
  grid_dependency_wait();
  const int nt = nb * tiles;
  const int words = (nt + 31) >> 5;
  uint32_t bad = 0;
  for (size_t e = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; e < entries;
       e += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t r = e / topk;  // bh * nb + I
    const int s = static_cast<int>(e - r * topk);
    const int c = q2k_num[r];
    const int cnt = c < 0 ? 0 : (c > topk ? topk : c);
    if (s == 0 && cnt != c) bad |= VSA_DEVERR_Q2K_COUNT;
    if (s >= cnt) continue;
    const int j = q2k_idx[e];
    if (j < 0 || j >= nb) {
      bad |= VSA_DEVERR_Q2K_ID;
      continue;
    }
    const size_t bh = r / nb;
    const size_t row0 = bh * nt + (r - bh * nb) * tiles;
    for (int a = 0; a < tiles; ++a)
      for (int b = 0; b < tiles; ++b) {
        const int t = j * tiles + b;
        atomicOr(bitmap + (row0 + a) * words + (t >> 5), 1u << (t & 31));
      }
  }
  if (bad && err) atomicOr(err, bad);
}

int grid_for(size_t work, int threads, int per_sm) {
  const size_t want = (work + threads - 1) / threads;
  const size_t cap = static_cast<size_t>(device_sm_count()) * per_sm;
  return static_cast<int>(want < cap ? (want < 1 ? 1 : want) : cap);
}

}  // namespace

cudaError_t launch_absmax_delta(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                const __nv_bfloat16* v, const __nv_bfloat16* dout,
                                const __nv_bfloat16* o, int BH, int S, uint32_t* absmax,
                                float* delta, float* dqacc, const PreExtras& x,
                                cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(S / BLOCK), static_cast<unsigned>(BH));
  return launch_dependent(
      absmax_delta_kernel, grid, dim3(PRE_THREADS), 0, stream, reinterpret_cast<const uint4*>(q),
      reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v),
      reinterpret_cast<const uint4*>(dout), reinterpret_cast<const uint4*>(o), S, absmax, delta,
      reinterpret_cast<float4*>(dqacc), x);
}

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t stream) {
  const size_t n = bytes / 16;
  if (n == 0) return cudaSuccess;
  return launch_dependent(zero_kernel, dim3(grid_for(n, 256, 4)), dim3(256), 0, stream,
                          static_cast<uint4*>(p), n);
}

cudaError_t launch_convert(const __nv_bfloat16* const* src, __half* const* dst, int count, int BH,
                           int S, const uint32_t* absmax, const uint32_t* tstat,
                           cudaStream_t stream) {
  ConvertPack pk{};
  pk.tstat = tstat;
  for (int t = 0; t < 4; ++t) {
    pk.src[t] = (t < count && src[t]) ? reinterpret_cast<const uint4*>(src[t]) : nullptr;
    pk.dst[t] = (t < count && src[t]) ? reinterpret_cast<uint4*>(dst[t]) : nullptr;
  }
  const size_t per_head = static_cast<size_t>(S) * HEAD_DIM / 8;
  const size_t total = per_head * BH;
  dim3 grid(static_cast<unsigned>(grid_for(total, 256, 8)), static_cast<unsigned>(count));
  return launch_dependent(convert_kernel, grid, dim3(256), 0, stream, pk, per_head, total, absmax);
}

cudaError_t launch_convert_t(const __nv_bfloat16* q, const __nv_bfloat16* dout, __half* q16t,
                             __half* do16t, int BH, int S, const uint32_t* absmax,
                             cudaStream_t stream) {
  ConvertTPack pk{};
  pk.src[0] = reinterpret_cast<const uint4*>(q);
  pk.src[1] = reinterpret_cast<const uint4*>(dout);
  pk.dst[0] = q16t;
  pk.dst[1] = do16t;
  pk.slot[0] = 0;
  pk.slot[1] = 3;
  dim3 grid(static_cast<unsigned>(S / BLOCK), static_cast<unsigned>(BH), 2u);
  return launch_dependent(convert_t_kernel, grid, dim3(256), 0, stream, pk, S, absmax);
}

cudaError_t launch_order(const int32_t* k2q_num, int BH, int nb, int max_q, int32_t* order,
                         cudaStream_t stream) {
  const long items = static_cast<long>(BH) * nb;
  order_kernel<<<grid_for(static_cast<size_t>(items) * 256, 256, 8), 256, 0, stream>>>(
      k2q_num, nb, items, max_q, order);
  return cudaGetLastError();
}

cudaError_t launch_postprocess(const float* dqacc, const uint32_t* absmax, int BH, int S,
                               float sm_scale, __nv_bfloat16* dq, const float* split_acc,
                               const int32_t* split_row, int nsplit, int parts, __nv_bfloat16* dk,
                               __nv_bfloat16* dv, cudaStream_t stream) {
  const size_t per_head = static_cast<size_t>(S) * HEAD_DIM / 8;
  const size_t total = per_head * BH;
  const int split_chunks = nsplit * 2 * BLOCK * (HEAD_DIM / 8);
  if (parts != 2 && parts != SPLIT_PARTS) return cudaErrorInvalidValue;
  auto kernel = parts == 2 ? postprocess_kernel<2> : postprocess_kernel<SPLIT_PARTS>;
  return launch_dependent(kernel, dim3(grid_for(total, 256, 8)), dim3(256), 0, stream,
      reinterpret_cast<const float4*>(dqacc), absmax, per_head, total, sm_scale,
      reinterpret_cast<uint4*>(dq), reinterpret_cast<const float4*>(split_acc), split_row,
      split_chunks, reinterpret_cast<uint4*>(dk), reinterpret_cast<uint4*>(dv));
}

cudaError_t launch_fwd_bitmap(const int32_t* q2k_idx, const int32_t* q2k_num, int topk, int BH,
                              int nb, int tiles, uint32_t* bitmap, uint32_t* err,
                              cudaStream_t stream) {
  const size_t entries = static_cast<size_t>(BH) * nb * topk;
  return launch_dependent(fwd_bitmap_kernel, dim3(grid_for(entries, 256, 4)), dim3(256), 0, stream,
                          q2k_idx, q2k_num, topk, nb, tiles, entries, bitmap, err);
}

}  // namespace vsa
