// fwd_main.cu -- forward of block-sparse attention on sm_103a, producing O and the base-2 "M form"
// log-sum-exp that the backward consumes (FastVideo block_sparse_attn_bwd_sm100a.py docstring:
// lse = max(qk * sm_scale * log2e) + log2(l); compare main...vsa_bwd_fix, tests,
// reference(): softmax over the selected blocks with keys past variable_block_sizes masked).
//
// Work unit: one (b, h, q pair) item -- q blocks 2x and 2x+1 -- so the UMMA M dimension is 128
// and row m of every accumulator is TMEM lane m.  The item walks the UNION of the two q blocks'
// selected kv blocks (ascending); for each row, kv blocks its own q block did not select are
// masked.  Two passes over the union:
//   pass 1  S = Q_p K_j^T, per-row running max / sum of exp2 (statistics only),
//   pass 2  S again, P = exp2(S*c - lse) (exactly normalised, fp16 * 2^KP) -> shared memory,
//           O += P V_j   (A = P K-major, B = V_j MN-major; fp32 accumulator in TMEM).
// No rescaling of O is needed, at the price of recomputing S once.
//
// Roles (320 threads): warps 0-7 softmax -- warps w and w+4 share TMEM lane quarter w (query
// rows 32w..32w+31) and split the 64 kv columns of S (and the 128 columns of O) in halves, merging
// their pass-1 row statistics through shared memory; warp 8 TMA producer and TMEM owner; warp 9
// UMMA issuer, which in pass 2 issues S of the next kv block before waiting for P of the current
// one, so the softmax and the tensor pipe overlap.  TMEM (256 columns): S x2 [0,128),
// O [128,256).
#include "ptx.cuh"
#include "vsa_internal.cuh"

namespace vsa {

namespace {

constexpr int NUM_THREADS = 320;
constexpr int SOFTMAX_WARPS = 8;
constexpr int TMA_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int KV_STAGES = 4;

constexpr uint32_t SM_Q = 0;                                // 2 chunks x [128 q x 128 B]
constexpr uint32_t SM_KV = 32768;                           // stages x (K 16 KB, V 16 KB)
constexpr uint32_t SM_P = SM_KV + KV_STAGES * 32768;        // 2 x [128 q x 128 B]
constexpr uint32_t SM_STAT = SM_P + 2 * 16384;              // [2 halves][128 rows] (max, sum)
constexpr uint32_t SM_BAR = SM_STAT + 2 * 128 * 8;

enum Bar : uint32_t {
  Q_FULL = 0,
  Q_EMPTY,
  KV_FULL0,
  KV_EMPTY0 = KV_FULL0 + KV_STAGES,
  S_FULL0 = KV_EMPTY0 + KV_STAGES,
  S_FREE0 = S_FULL0 + 2,
  P_READY0 = S_FREE0 + 2,
  P_FREE0 = P_READY0 + 2,
  O_FULL = P_FREE0 + 2,
  O_EMPTY,
  DRAIN,
  STAT0,  // one per lane quarter: the two column-half warps have published their statistics
  NUM_BARS = STAT0 + 4
};
constexpr uint32_t SM_TMEM_SLOT = SM_BAR + NUM_BARS * 8;
constexpr uint32_t SM_ABORT = SM_TMEM_SLOT + 4;
constexpr uint32_t SMEM_BYTES = SM_ABORT + 4 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t TM_S = 0, TM_O = 128;
constexpr uint32_t IDESC_S = idesc_f16_f32acc(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_f16_f32acc(128, 128, false, true);

struct Params {
  const uint32_t* bitmap;
  const int32_t* vbs;
  const uint32_t* absmax;
  __nv_bfloat16* o;
  float* lse;
  uint32_t* err;
  int S, nb, words, npairs, total;
  float sm_scale;
};

struct Pair {
  int bh, i0, i1;  // i1 < 0: no second q block
  const uint32_t* bm0;
  const uint32_t* bm1;
};

__device__ __forceinline__ Pair decode_pair(const Params& p, int w) {
  Pair q;
  q.bh = w / p.npairs;
  const int x = w - q.bh * p.npairs;
  q.i0 = 2 * x;
  q.i1 = (2 * x + 1 < p.nb) ? 2 * x + 1 : -1;
  q.bm0 = p.bitmap + (static_cast<size_t>(q.bh) * p.nb + q.i0) * p.words;
  q.bm1 = q.i1 >= 0 ? q.bm0 + p.words : nullptr;
  return q;
}

__device__ __forceinline__ uint32_t union_word(const Pair& q, int wi) {
  return q.bm0[wi] | (q.bm1 ? q.bm1[wi] : 0u);
}

__device__ __forceinline__ int union_size(const Params& p, const Pair& q) {
  int n = 0;
  for (int wi = 0; wi < p.words; ++wi) n += __popc(union_word(q, wi));
  return n;
}

// Calls f(j) for every kv block of the pair's union, ascending; stops when f returns false.
template <typename F>
__device__ __forceinline__ bool for_union(const Params& p, const Pair& q, F f) {
  for (int wi = 0; wi < p.words; ++wi) {
    uint32_t u = union_word(q, wi);
    while (u) {
      const int b = __ffs(u) - 1;
      u &= u - 1;
      if (!f(wi * 32 + b)) return false;
    }
  }
  return true;
}

__device__ __forceinline__ int clamp_vbs(int v) { return v < 0 ? 0 : (v > BLOCK ? BLOCK : v); }

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait_bounded(bar, parity, abort, WAIT_LIMIT_NS) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void raise_abort(volatile int* abort, uint32_t* err) {
  *abort = 1;
  atomicOr(err, VSA_DEVERR_TIMEOUT);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    fwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + SM_ABORT);
  const uint32_t* tmem_slot = reinterpret_cast<const uint32_t*>(gbase + SM_TMEM_SLOT);
  auto bar = [&](uint32_t b) { return base + SM_BAR + 8u * b; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S;

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(bar(Q_FULL), 1);
    mbar_init(bar(Q_EMPTY), 1);
    for (int s = 0; s < KV_STAGES; ++s) {
      mbar_init(bar(KV_FULL0 + s), 1);
      mbar_init(bar(KV_EMPTY0 + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(S_FULL0 + s), 1);
      mbar_init(bar(S_FREE0 + s), SOFTMAX_WARPS);
      mbar_init(bar(P_READY0 + s), SOFTMAX_WARPS);
      mbar_init(bar(P_FREE0 + s), 1);
    }
    mbar_init(bar(O_FULL), 1);
    mbar_init(bar(O_EMPTY), SOFTMAX_WARPS);
    mbar_init(bar(DRAIN), 1);
    for (int qq = 0; qq < 4; ++qq) mbar_init(bar(STAT0 + qq), 2);
    fence_barrier_init();
  }
  if (warp == TMA_WARP) {
    tmem_alloc(base + SM_TMEM_SLOT, 256);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == TMA_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t lg = 0, itc = 0, q_loads = 0;
      int64_t last_lg[KV_STAGES];
      for (int s = 0; s < KV_STAGES; ++s) last_lg[s] = -1;
      bool ok = true;
      for (int w = blockIdx.x; w < p.total && ok; w += gridDim.x) {
        const Pair q = decode_pair(p, w);
        if (union_size(p, q) == 0) continue;
        if (!mbar_wait_bounded(bar(Q_EMPTY), (itc & 1u) ^ 1u, abort, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        const int r0 = q.bh * S + q.i0 * BLOCK;
        const int r1 = q.bh * S + (q.i1 >= 0 ? q.i1 : q.i0) * BLOCK;
        mbar_arrive_expect_tx(bar(Q_FULL), 32768);
        tma_load_2d(base + SM_Q, &tm_q, bar(Q_FULL), 0, r0);
        tma_load_2d(base + SM_Q + 8192, &tm_q, bar(Q_FULL), 0, r1);
        tma_load_2d(base + SM_Q + 16384, &tm_q, bar(Q_FULL), 64, r0);
        tma_load_2d(base + SM_Q + 24576, &tm_q, bar(Q_FULL), 64, r1);
        ++q_loads;
        for (int pass = 0; pass < 2 && ok; ++pass) {
          ok = for_union(p, q, [&](int j) {
            const uint32_t st = lg % KV_STAGES;
            if (!mbar_wait_bounded(bar(KV_EMPTY0 + st), ((lg / KV_STAGES) & 1u) ^ 1u, abort,
                                   WAIT_LIMIT_NS))
              return false;
            const int rk = q.bh * S + j * BLOCK;
            const uint32_t kd = base + SM_KV + st * 32768u;
            mbar_arrive_expect_tx(bar(KV_FULL0 + st), pass ? 32768u : 16384u);
            tma_load_2d(kd, &tm_k, bar(KV_FULL0 + st), 0, rk);
            tma_load_2d(kd + 8192, &tm_k, bar(KV_FULL0 + st), 64, rk);
            if (pass) {
              tma_load_2d(kd + 16384, &tm_v, bar(KV_FULL0 + st), 0, rk);
              tma_load_2d(kd + 24576, &tm_v, bar(KV_FULL0 + st), 64, rk);
            }
            last_lg[st] = lg;
            ++lg;
            return true;
          });
        }
        ++itc;
      }
      if (!ok) {
        raise_abort(abort, p.err);
        volatile int never = 0;
        if (q_loads) mbar_wait_bounded(bar(Q_FULL), (q_loads - 1) & 1u, &never, DRAIN_LIMIT_NS);
        for (int s = 0; s < KV_STAGES; ++s)
          if (last_lg[s] >= 0)
            mbar_wait_bounded(bar(KV_FULL0 + s),
                              (static_cast<uint32_t>(last_lg[s]) / KV_STAGES) & 1u, &never,
                              DRAIN_LIMIT_NS);
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      uint32_t lg = 0, sg = 0, pg = 0, itc = 0;
      bool ok = true, issued = false;
      const uint64_t q_kmaj = sdesc_sw128(base + SM_Q, 16, 1024);
      const uint64_t kv_kmaj = sdesc_sw128(base + SM_KV, 16, 1024);    // K of stage 0
      const uint64_t kv_mn = sdesc_sw128(base + SM_KV + 16384u, 8192, 1024);  // V of stage 0
      const uint64_t p_kmaj = sdesc_sw128(base + SM_P, 16, 1024);
      // S = Q_p K_j^T into S buffer sg & 1, K from KV stage lg % KV_STAGES.
      auto issue_s = [&]() -> bool {
        const uint32_t st = lg % KV_STAGES, sb = sg & 1u;
        if (!mbar_wait_bounded(bar(KV_FULL0 + st), (lg / KV_STAGES) & 1u, abort, WAIT_LIMIT_NS))
          return false;
        if (!mbar_wait_bounded(bar(S_FREE0 + sb), ((sg >> 1) & 1u) ^ 1u, abort, WAIT_LIMIT_NS))
          return false;
        tc_fence_after_sync();
        const uint64_t kd = sdesc_advance(kv_kmaj, st * 32768u);
        const uint32_t ts = tmem + TM_S + sb * 64u;
        umma_f16_c<false>(ts, q_kmaj, kd, IDESC_S);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk) {
          const uint32_t off = (kk & 3) * 32u;
          umma_f16_c<true>(ts, sdesc_advance(q_kmaj, (kk >> 2) * 16384u + off),
                           sdesc_advance(kd, (kk >> 2) * 8192u + off), IDESC_S);
        }
        umma_commit(bar(S_FULL0 + sb));
        issued = true;
        ++sg;
        return true;
      };
      // O += P V_j with P buffer pg & 1 and V of KV stage `st`.
      auto issue_pv = [&](uint32_t st, bool first) -> bool {
        const uint32_t pb = pg & 1u;
        if (!mbar_wait_bounded(bar(P_READY0 + pb), (pg >> 1) & 1u, abort, WAIT_LIMIT_NS))
          return false;
        if (first && !mbar_wait_bounded(bar(O_EMPTY), (itc & 1u) ^ 1u, abort, WAIT_LIMIT_NS))
          return false;
        tc_fence_after_sync();
        const uint64_t pa = sdesc_advance(p_kmaj, pb * 16384u);
        const uint64_t vb = sdesc_advance(kv_mn, st * 32768u);
        if (first)
          umma_f16_c<false>(tmem + TM_O, pa, vb, IDESC_PV);
        else
          umma_f16_c<true>(tmem + TM_O, pa, vb, IDESC_PV);
#pragma unroll
        for (int kk = 1; kk < 4; ++kk)
          umma_f16_c<true>(tmem + TM_O, sdesc_advance(pa, kk * 32u), sdesc_advance(vb, kk * 2048u),
                           IDESC_PV);
        umma_commit(bar(P_FREE0 + pb));
        umma_commit(bar(KV_EMPTY0 + st));
        ++pg;
        return true;
      };
      for (int w = blockIdx.x; w < p.total && ok; w += gridDim.x) {
        const Pair q = decode_pair(p, w);
        const int nu = union_size(p, q);
        if (nu == 0) continue;
        if (!mbar_wait_bounded(bar(Q_FULL), itc & 1u, abort, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        // Pass 1: S of every union block; K stages are released as soon as S is done.
        for (int e = 0; e < nu && ok; ++e) {
          const uint32_t st = lg % KV_STAGES;
          if (!issue_s()) {
            ok = false;
            break;
          }
          umma_commit(bar(KV_EMPTY0 + st));
          ++lg;
        }
        if (!ok) break;
        // Pass 2: S(e+1) is issued before P.V(e) waits for the softmax of block e.
        const uint32_t lg0 = lg;
        if (!issue_s()) {
          ok = false;
          break;
        }
        for (int e = 0; e < nu && ok; ++e) {
          if (e + 1 < nu) {
            lg = lg0 + e + 1;
            if (!issue_s()) {
              ok = false;
              break;
            }
          }
          if (!issue_pv((lg0 + e) % KV_STAGES, e == 0)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        lg = lg0 + nu;
        umma_commit(bar(O_FULL));
        umma_commit(bar(Q_EMPTY));
        ++itc;
      }
      if (!ok) raise_abort(abort, p.err);
      if (issued) {
        umma_commit(bar(DRAIN));
        volatile int never = 0;
        mbar_wait_bounded(bar(DRAIN), 0, &never, DRAIN_LIMIT_NS);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-7)
    const int quarter = warp & 3, h = warp >> 2;  // TMEM lane quarter; column half
    const int r = quarter * 32 + lane;            // query row of the pair == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t sw = static_cast<uint32_t>(r & 7);
    float2* stat = reinterpret_cast<float2*>(gbase + SM_STAT);  // [half][row] (max, sum)
    uint32_t sg = 0, pg = 0, itc = 0;
    for (int w = blockIdx.x; w < p.total; w += gridDim.x) {
      const Pair q = decode_pair(p, w);
      const bool valid = (r < 64) || (q.i1 >= 0);
      const uint32_t* own = (r < 64) ? q.bm0 : q.bm1;
      const size_t grow = static_cast<size_t>(q.bh) * S +
                          static_cast<size_t>(r < 64 ? q.i0 : (q.i1 >= 0 ? q.i1 : q.i0)) * BLOCK +
                          (r & 63);
      uint4* orow = reinterpret_cast<uint4*>(p.o + grow * HEAD_DIM) + h * 8;
      if (union_size(p, q) == 0) {
        if (valid) {
          for (int c = 0; c < 8; ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
          if (h == 0) p.lse[grow] = -INFINITY;
        }
        continue;
      }
      const uint32_t* am = p.absmax + q.bh * 4;
      const int eq = operand_exponent(am[0]), ek = operand_exponent(am[1]);
      const int ev = operand_exponent(am[2]);
      const float c1 = p.sm_scale * LOG2E_F * exp2i(eq + ek);
      float m = -INFINITY, l = 0.f, lse = -INFINITY;
      bool ok = true;
      for (int pass = 0; pass < 2 && ok; ++pass) {
        ok = for_union(p, q, [&](int j) {
          const uint32_t sb = sg & 1u;
          if (!warp_wait(bar(S_FULL0 + sb), (sg >> 1) & 1u, abort, lane)) return false;
          tc_fence_after_sync();
          const bool mine = valid && ((own[j >> 5] >> (j & 31)) & 1u);
          const int vb = mine ? clamp_vbs(p.vbs[j]) - h * 32 : 0;  // visible columns in my half
          uint32_t sv[32];
          tmem_ld_32x32b_x32(tmem + lane_off + TM_S + sb * 64u + h * 32u, sv);
          tmem_wait_ld();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(S_FREE0 + sb));
          ++sg;
          if (pass == 0) {
            if (vb > 0) {
              float mloc = -INFINITY;
#pragma unroll
              for (int u = 0; u < 32; ++u)
                if (u < vb) mloc = fmaxf(mloc, __uint_as_float(sv[u]) * c1);
              const float mn = fmaxf(m, mloc);
              float acc = 0.f;
#pragma unroll
              for (int u = 0; u < 32; ++u)
                if (u < vb) acc += ex2(__uint_as_float(sv[u]) * c1 - mn);
              l = l * ex2(m - mn) + acc;
              m = mn;
            }
            return true;
          }
          const float off = static_cast<float>(KP) - lse;
          uint32_t pk[16];
#pragma unroll
          for (int u = 0; u < 32; u += 2) {
            const float p0 = (u < vb) ? ex2(fmaf(__uint_as_float(sv[u]), c1, off)) : 0.f;
            const float p1 = (u + 1 < vb) ? ex2(fmaf(__uint_as_float(sv[u + 1]), c1, off)) : 0.f;
            pk[u >> 1] = pack_half2(p0, p1);
          }
          const uint32_t pb = pg & 1u;
          if (!warp_wait(bar(P_FREE0 + pb), ((pg >> 1) & 1u) ^ 1u, abort, lane)) return false;
          const uint32_t prow = base + SM_P + pb * 16384u + static_cast<uint32_t>(r) * 128u;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint32_t phys = ((static_cast<uint32_t>(h * 4 + ch)) ^ sw) * 16u;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + phys),
                         "r"(pk[4 * ch]), "r"(pk[4 * ch + 1]), "r"(pk[4 * ch + 2]),
                         "r"(pk[4 * ch + 3])
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(P_READY0 + pb));
          ++pg;
          return true;
        });
        if (pass == 0 && ok) {
          // Merge the two column halves' statistics of each row.  The slot is rewritten only in
          // the next item's pass 1, which cannot start before both warps finished this item.
          stat[h * 128 + r] = make_float2(m, l);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(STAT0 + quarter));
          if (!warp_wait(bar(STAT0 + quarter), itc & 1u, abort, lane)) {
            ok = false;
            break;
          }
          const float2 o2 = stat[(1 - h) * 128 + r];
          const float mm = fmaxf(m, o2.x);
          const float ll = (mm == -INFINITY) ? 0.f : l * ex2(m - mm) + o2.y * ex2(o2.x - mm);
          lse = (ll > 0.f) ? mm + log2f(ll) : -INFINITY;
        }
      }
      if (!ok) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      if (!warp_wait(bar(O_FULL), itc & 1u, abort, lane)) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      tc_fence_after_sync();
      const float os = exp2i(ev - KP);
      uint32_t v[64];  // O columns h*64 .. h*64+63 of row r
      tmem_ld_32x32b_x32(tmem + lane_off + TM_O + h * 64u, v);
      tmem_ld_32x32b_x32(tmem + lane_off + TM_O + h * 64u + 32u, v + 32);
      tmem_wait_ld();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(O_EMPTY));
      if (valid) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int u = 8 * c;
          orow[c] = make_uint4(
              pack_bf162(__uint_as_float(v[u]) * os, __uint_as_float(v[u + 1]) * os),
              pack_bf162(__uint_as_float(v[u + 2]) * os, __uint_as_float(v[u + 3]) * os),
              pack_bf162(__uint_as_float(v[u + 4]) * os, __uint_as_float(v[u + 5]) * os),
              pack_bf162(__uint_as_float(v[u + 6]) * os, __uint_as_float(v[u + 7]) * os));
        }
        if (h == 0) p.lse[grow] = lse;
      }
      ++itc;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == TMA_WARP) tmem_dealloc(tmem, 256);
}

}  // namespace

cudaError_t launch_fwd_main(const FwdMainArgs& a, cudaStream_t stream) {
  const long rows = static_cast<long>(a.B) * a.H * a.S;
  CUtensorMap tq, tk, tv;
  cudaError_t e;
  if ((e = make_tmap_rows128_f16(&tq, a.q16, rows)) != cudaSuccess) return e;
  if ((e = make_tmap_rows128_f16(&tk, a.k16, rows)) != cudaSuccess) return e;
  if ((e = make_tmap_rows128_f16(&tv, a.v16, rows)) != cudaSuccess) return e;
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(fwd_main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  Params p{};
  p.bitmap = a.bitmap;
  p.vbs = a.vbs;
  p.absmax = a.absmax;
  p.o = a.o;
  p.lse = a.lse;
  p.err = a.err;
  p.S = a.S;
  p.nb = a.nb;
  p.words = (a.nb + 31) / 32;
  p.npairs = (a.nb + 1) / 2;
  p.total = a.B * a.H * p.npairs;
  p.sm_scale = a.sm_scale;
  const int sms = device_sm_count();
  const int grid = p.total < sms ? p.total : sms;
  fwd_main_kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace vsa
