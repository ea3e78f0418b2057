// invert.cu -- q2k -> k2q inversion of the block selection (FastVideo block_sparse_attn_bwd_sm100a.py,
// block_sparse_attn_backward_sm100a, which inverts the selection before the backward kernels; the
// row order is ascending as in the compare page's tests, invert_indices_torch).
//
// Two passes over a bitmap of the selection, kept in the output itself:
//   bitmap   one CTA per (group of 32 q rows, head): the CTA ORs bit i % 32 of kv column j into a
//            shared-memory word per column for every active slot j of its rows i (duplicate ids
//            collapse, set semantics for free), then stores the nb words -- word i / 32 of every
//            column, written by this CTA alone, zero or not, so nothing needs clearing first.
//            Word w of column j goes to slot nq - words + w of k2q row j, the tail of the row the
//            compaction will overwrite.  q2k is read once.
//   compact  one warp per (head, kv column): copies the row's tail words to shared memory, then
//            lane l takes word l (and l + 32, ...): a warp prefix sum of the popcounts gives each
//            lane its output offset, and the lane writes its set bits in ascending order, then the
//            zero padding and the count.
// The result is deterministic (no atomics decide positions) and rows come out sorted.  Rows too
// long for a column word per kv block in shared memory (nb above 56K) take the single-kernel
// version below, which rescans a head's q2k once per slice of columns.
#include "vsa_internal.cuh"

namespace vsa {

namespace {

constexpr int INV_MIN_COLS = 32;  // kv blocks per CTA, at least (unless shared memory is short)
constexpr int INV_THREADS = 1024;  // 32 warps: many q2k rows in flight per CTA
constexpr size_t INV_SMEM_CAP = 200 * 1024;

__global__ void __launch_bounds__(INV_THREADS) invert_kernel(const int32_t* __restrict__ q2k_idx,
                                                             const int32_t* __restrict__ q2k_num,
                                                             int topk, int nb, int cols,
                                                             int32_t* __restrict__ k2q_idx,
                                                             int32_t* __restrict__ k2q_num,
                                                             uint32_t* err) {
  extern __shared__ uint32_t bm[];  // [cols][words]
  const int nq = nb;
  const int words = (nq + 31) >> 5;
  const int bh = blockIdx.x;
  const int j0 = blockIdx.y * cols;
  const int ncols = min(cols, nb - j0);

  for (int x = threadIdx.x; x < cols * words; x += blockDim.x) bm[x] = 0u;
  __syncthreads();

  uint32_t bad = 0;
  const int32_t* idx = q2k_idx + static_cast<size_t>(bh) * nq * topk;
  const int32_t* num = q2k_num + static_cast<size_t>(bh) * nq;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  // One warp per q2k row: coalesced loads of the row's active prefix, four in flight per lane.
  for (int i = warp; i < nq; i += nwarps) {
    const int c = num[i];
    const int cnt = c < 0 ? 0 : (c > topk ? topk : c);
    if (cnt != c) bad |= VSA_DEVERR_Q2K_COUNT;
    const int32_t* row = idx + static_cast<size_t>(i) * topk;
    const uint32_t bit = 1u << (i & 31);
    for (int s0 = 0; s0 < cnt; s0 += 4 * 32) {
      int jv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int s = s0 + u * 32 + lane;
        jv[u] = s < cnt ? row[s] : 0;  // unused: lanes past the count skip it below
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (s0 + u * 32 + lane >= cnt) continue;
        const int j = jv[u];
        if (j < 0 || j >= nb) {
          bad |= VSA_DEVERR_Q2K_ID;
          continue;
        }
        const int jj = j - j0;
        if (jj >= 0 && jj < ncols) atomicOr(&bm[jj * words + (i >> 5)], bit);
      }
    }
  }
  // Report invalid entries once per head (the first slice sees all of them).
  if (bad && blockIdx.y == 0 && err) atomicOr(err, bad);
  __syncthreads();

  for (int jj = warp; jj < ncols; jj += nwarps) {
    const int j = j0 + jj;
    int32_t* out = k2q_idx + (static_cast<size_t>(bh) * nb + j) * nq;
    int base = 0;
    for (int w0 = 0; w0 < words; w0 += 32) {
      const int w = w0 + lane;
      uint32_t bits = (w < words) ? bm[jj * words + w] : 0u;
      const int cnt = __popc(bits);
      int incl = cnt;  // inclusive warp prefix sum
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
      }
      int pos = base + incl - cnt;
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        out[pos++] = (w << 5) + b;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    for (int t = base + lane; t < nq; t += 32) out[t] = 0;  // padding: a valid id
    if (lane == 0) k2q_num[static_cast<size_t>(bh) * nb + j] = base;
  }
}

constexpr int BM_THREADS = 256;
constexpr int CP_WARPS = 8;

__global__ void __launch_bounds__(BM_THREADS) invert_bitmap_kernel(
    const int32_t* __restrict__ q2k_idx, const int32_t* __restrict__ q2k_num, int topk, int nb,
    int32_t* __restrict__ k2q_idx, uint32_t* err) {
  extern __shared__ uint32_t col[];  // [nb]: this CTA's word of every kv column
  const int nq = nb, words = (nq + 31) >> 5;
  const int g = blockIdx.x, bh = blockIdx.y;
  for (int j = threadIdx.x; j < nb; j += blockDim.x) col[j] = 0u;
  __syncthreads();
  uint32_t bad = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t* idx = q2k_idx + static_cast<size_t>(bh) * nq * topk;
  const int32_t* num = q2k_num + static_cast<size_t>(bh) * nq;
  // One warp per q2k row, four loads in flight per lane.
  for (int r = warp; r < 32; r += BM_THREADS / 32) {
    const int i = g * 32 + r;
    if (i >= nq) break;
    const int c = num[i];
    const int cnt = c < 0 ? 0 : (c > topk ? topk : c);
    if (cnt != c) bad |= VSA_DEVERR_Q2K_COUNT;
    const int32_t* row = idx + static_cast<size_t>(i) * topk;
    const uint32_t bit = 1u << r;
    for (int s0 = 0; s0 < cnt; s0 += 4 * 32) {
      int jv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int s = s0 + u * 32 + lane;
        jv[u] = s < cnt ? row[s] : 0;  // unused: lanes past the count skip it below
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (s0 + u * 32 + lane >= cnt) continue;
        const int j = jv[u];
        if (j < 0 || j >= nb) {
          bad |= VSA_DEVERR_Q2K_ID;
          continue;
        }
        atomicOr(&col[j], bit);
      }
    }
  }
  if (bad && err) atomicOr(err, bad);
  __syncthreads();
  int32_t* out = k2q_idx + static_cast<size_t>(bh) * nb * nq + (nq - words) + g;
  for (int j = threadIdx.x; j < nb; j += blockDim.x)
    out[static_cast<size_t>(j) * nq] = static_cast<int32_t>(col[j]);
}

__global__ void __launch_bounds__(CP_WARPS * 32) invert_compact_kernel(int nb, long rows,
                                                                       int32_t* __restrict__ k2q_idx,
                                                                       int32_t* __restrict__ k2q_num) {
  grid_dependency_wait();
  extern __shared__ uint32_t tails[];  // [CP_WARPS][words]
  const int nq = nb, words = (nq + 31) >> 5;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* tw = tails + static_cast<size_t>(warp) * words;
  for (long rj = static_cast<long>(blockIdx.x) * CP_WARPS + warp; rj < rows;
       rj += static_cast<long>(gridDim.x) * CP_WARPS) {
    int32_t* out = k2q_idx + rj * nq;
    for (int w = lane; w < words; w += 32) tw[w] = static_cast<uint32_t>(out[nq - words + w]);
    __syncwarp();
    int base = 0;
    for (int w0 = 0; w0 < words; w0 += 32) {
      const int w = w0 + lane;
      uint32_t bits = (w < words) ? tw[w] : 0u;
      const int cnt = __popc(bits);
      int incl = cnt;  // inclusive warp prefix sum
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
      }
      int pos = base + incl - cnt;
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        out[pos++] = (w << 5) + b;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    for (int t = base + lane; t < nq; t += 32) out[t] = 0;  // padding: a valid id
    if (lane == 0) k2q_num[rj] = base;
    __syncwarp();  // the tail copy is read before the next row overwrites it
  }
}

}  // namespace

cudaError_t launch_invert(const int32_t* q2k_idx, const int32_t* q2k_num, int topk, int BH,
                          int nb, int32_t* k2q_idx, int32_t* k2q_num, uint32_t* err,
                          cudaStream_t stream) {
  constexpr size_t SMEM_MAX = 227 * 1024;
  const size_t bm_smem = static_cast<size_t>(nb) * sizeof(uint32_t);
  const size_t words = static_cast<size_t>((nb + 31) / 32);
  const size_t cp_smem = CP_WARPS * words * sizeof(uint32_t);
  if (bm_smem <= SMEM_MAX && cp_smem <= SMEM_MAX) {
    static std::atomic<uint64_t> bm_set{0}, cp_set{0};
    cudaError_t e;
    if (bm_smem > 48 * 1024 &&
        (e = ensure_smem_limit(invert_bitmap_kernel, static_cast<int>(SMEM_MAX), bm_set)) !=
            cudaSuccess)
      return e;
    if (cp_smem > 48 * 1024 &&
        (e = ensure_smem_limit(invert_compact_kernel, static_cast<int>(SMEM_MAX), cp_set)) !=
            cudaSuccess)
      return e;
    invert_bitmap_kernel<<<dim3(static_cast<unsigned>(words), static_cast<unsigned>(BH)),
                           BM_THREADS, bm_smem, stream>>>(q2k_idx, q2k_num, topk, nb, k2q_idx,
                                                          err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long rows = static_cast<long>(BH) * nb;
    const long want = (rows + CP_WARPS - 1) / CP_WARPS;
    const long cap = 16L * device_sm_count();
    return launch_dependent(invert_compact_kernel, dim3(static_cast<unsigned>(want < cap ? want : cap)),
                            dim3(CP_WARPS * 32), cp_smem, stream, nb, rows, k2q_idx, k2q_num);
  }
  const size_t col_bytes = static_cast<size_t>((nb + 31) / 32) * sizeof(uint32_t);
  // Widest slice shared memory holds, but no wider than two waves of CTAs need.
  const long fit = static_cast<long>(INV_SMEM_CAP / col_bytes);
  const long two_waves = (static_cast<long>(BH) * nb + 2L * device_sm_count() - 1) /
                         (2L * device_sm_count());
  long cols = two_waves > INV_MIN_COLS ? two_waves : INV_MIN_COLS;
  if (cols > fit) cols = fit;
  if (cols > nb) cols = nb;
  if (cols < 1) return cudaErrorInvalidValue;  // nb beyond 1.6 M blocks: a column exceeds smem
  const size_t smem = static_cast<size_t>(cols) * col_bytes;
  if (smem > 48 * 1024) {
    static std::atomic<uint64_t> inv_set{0};
    cudaError_t e = ensure_smem_limit(invert_kernel, static_cast<int>(INV_SMEM_CAP), inv_set);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(static_cast<unsigned>(BH), static_cast<unsigned>((nb + cols - 1) / cols));
  invert_kernel<<<grid, INV_THREADS, smem, stream>>>(q2k_idx, q2k_num, topk, nb,
                                                      static_cast<int>(cols), k2q_idx, k2q_num,
                                                      err);
  return cudaGetLastError();
}

}  // namespace vsa
