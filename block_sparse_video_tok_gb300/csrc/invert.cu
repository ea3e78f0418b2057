// invert.cu -- q2k -> k2q inversion of the block selection (FastVideo block_sparse_attn_bwd_sm100a.py,
// block_sparse_attn_backward_sm100a: "k2q_idx, k2q_num = invert_indices(...)"; the row order is
// ascending as in the compare page's tests, invert_indices_torch).
//
// One CTA per (head, 32-column slice of kv blocks).  Phase 1 scans the head's q2k rows and sets
// bit i of column j in a shared-memory bitmap (column-major: one run of nq bits per kv block), so
// duplicate ids collapse and the set semantics come for free.  Phase 2 gives each warp whole
// columns: lane l owns 32-bit word l (and l+32, ...) of the column, a warp prefix sum of the
// popcounts gives every lane its output offset, and the lane writes its set bits in ascending
// order.  The result is deterministic (no atomics decide positions) and rows come out sorted.
// HBM traffic per head: q2k read once per slice (L2-resident), k2q written once.
#include "vsa_internal.cuh"

namespace vsa {

namespace {

constexpr int INV_COLS = 32;     // kv blocks per CTA
constexpr int INV_THREADS = 256;

__global__ void __launch_bounds__(INV_THREADS) invert_kernel(const int32_t* __restrict__ q2k_idx,
                                                             const int32_t* __restrict__ q2k_num,
                                                             int topk, int nb,
                                                             int32_t* __restrict__ k2q_idx,
                                                             int32_t* __restrict__ k2q_num,
                                                             uint32_t* err) {
  extern __shared__ uint32_t bm[];  // [INV_COLS][words]
  const int nq = nb;
  const int words = (nq + 31) >> 5;
  const int bh = blockIdx.x;
  const int j0 = blockIdx.y * INV_COLS;
  const int ncols = min(INV_COLS, nb - j0);

  for (int x = threadIdx.x; x < INV_COLS * words; x += blockDim.x) bm[x] = 0u;
  __syncthreads();

  uint32_t bad = 0;
  const int32_t* idx = q2k_idx + static_cast<size_t>(bh) * nq * topk;
  const int32_t* num = q2k_num + static_cast<size_t>(bh) * nq;
  const int entries = nq * topk;
  // Sixteen independent loads per thread before any is used, so the scan is not bound by one
  // L2 round trip per entry.
  constexpr int U = 16;
  for (int e0 = 0; e0 < entries; e0 += U * INV_THREADS) {
    int jv[U], cv[U], sv[U], iv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * INV_THREADS + static_cast<int>(threadIdx.x);
      const bool in = e < entries;
      const int i = in ? e / topk : 0;
      iv[u] = i;
      sv[u] = in ? e - i * topk : topk;  // topk: never an active slot
      jv[u] = in ? idx[e] : 0;
      cv[u] = in ? num[i] : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = cv[u];
      const int cnt = c < 0 ? 0 : (c > topk ? topk : c);
      if (sv[u] == 0 && cnt != c) bad |= VSA_DEVERR_Q2K_COUNT;
      if (sv[u] >= cnt) continue;
      const int j = jv[u];
      if (j < 0 || j >= nb) {
        bad |= VSA_DEVERR_Q2K_ID;
        continue;
      }
      const int jj = j - j0;
      if (jj >= 0 && jj < ncols) atomicOr(&bm[jj * words + (iv[u] >> 5)], 1u << (iv[u] & 31));
    }
  }
  // Report invalid entries once per head (the first slice sees all of them).
  if (bad && blockIdx.y == 0 && err) atomicOr(err, bad);
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
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
  const int words = (nb + 31) / 32;
  const size_t smem = static_cast<size_t>(INV_COLS) * words * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(invert_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  dim3 grid(static_cast<unsigned>(BH), static_cast<unsigned>((nb + INV_COLS - 1) / INV_COLS));
  invert_kernel<<<grid, INV_THREADS, smem, stream>>>(q2k_idx, q2k_num, topk, nb, k2q_idx,
                                                      k2q_num, err);
  return cudaGetLastError();
}

}  // namespace vsa
