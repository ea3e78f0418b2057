// invert.cu -- q2k -> k2q inversion of the block selection (FastVideo block_sparse_attn_bwd_sm100a.py,
// block_sparse_attn_backward_sm100a, which inverts the selection before the backward kernels; the
// row order is ascending as in the compare page's tests, invert_indices_torch).
//
// One CTA per (head, slice of kv-block columns).  Phase 1 scans the head's q2k rows and sets
// bit i of column j in a shared-memory bitmap (column-major: one run of nq bits per kv block), so
// duplicate ids collapse and the set semantics come for free.  Every slice rescans the head's q2k,
// so slices are as wide as shared memory allows while the grid still fills about two waves of
// SMs: 32 columns at 32k tokens, about 200 at 524k.  Phase 2 gives each warp whole
// columns: lane l owns 32-bit word l (and l+32, ...) of the column, a warp prefix sum of the
// popcounts gives every lane its output offset, and the lane writes its set bits in ascending
// order.  The result is deterministic (no atomics decide positions) and rows come out sorted.
// Traffic per head: q2k read once per slice (from L2), k2q written once.
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

}  // namespace

cudaError_t launch_invert(const int32_t* q2k_idx, const int32_t* q2k_num, int topk, int BH,
                          int nb, int32_t* k2q_idx, int32_t* k2q_num, uint32_t* err,
                          cudaStream_t stream) {
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
    cudaError_t e = cudaFuncSetAttribute(invert_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  dim3 grid(static_cast<unsigned>(BH), static_cast<unsigned>((nb + cols - 1) / cols));
  invert_kernel<<<grid, INV_THREADS, smem, stream>>>(q2k_idx, q2k_num, topk, nb,
                                                      static_cast<int>(cols), k2q_idx, k2q_num,
                                                      err);
  return cudaGetLastError();
}

}  // namespace vsa
