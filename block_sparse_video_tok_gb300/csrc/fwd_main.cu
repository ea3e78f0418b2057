// fwd_main.cu -- forward of block-sparse attention on sm_103a, producing O and the base-2 "M form"
// log-sum-exp that the backward consumes (FastVideo block_sparse_attn_bwd_sm100a.py docstring:
// lse = max(qk * sm_scale * log2e) + log2(l); compare main...vsa_bwd_fix, tests,
// reference(): softmax over the selected blocks with keys past variable_block_sizes masked).
//
// Work unit: one (b, h, q pair) item -- q blocks 2x and 2x+1 -- so the UMMA M dimension is 128
// and row m of every accumulator is TMEM lane m.  The item walks the UNION of the two q blocks'
// selected kv blocks (ascending); for each row, kv blocks its own q block did not select are
// masked.  One pass with an online softmax per kv block j:
//   S = Q_p K_j^T (both operands in shared memory, fp32 accumulator in TMEM);
//   the row maximum of the block; if it exceeds the row's reference maximum m by more than
//   RESCALE (log2 units), m moves up to it and the O row and the running sum are scaled by
//   2^(m_old - m_new) first (otherwise m stays, so P stays below 2^(RESCALE + KPF));
//   P = 2^(s - m + KPF) in fp16, written to TMEM, where it is the A operand of
//   O += P V_j (B = V_j from shared memory, MN-major).
// At the end O / l and lse = m + log2(l).  P never passes through shared memory, so per kv block
// the tensor pipe reads Q_p, K_j and V_j only.
//
// Roles (320 threads): warps 0-7 softmax -- warps w and w+4 share TMEM lane quarter w (query
// rows 32w..32w+31) and split the 64 kv columns of S (and the 128 columns of O) in halves,
// exchanging their block maxima through shared memory; warp 8 TMA producer, TMEM owner and work
// claimer; warp 9 UMMA issuer, which issues S of the next kv block before P.V of the current one
// so the softmax of one block overlaps the tensor work of its neighbours.
// TMEM (512 columns allocated): O [0,128), S x2 [128,256), P x2 [256,320).
#include "ptx.cuh"
#include "queue.cuh"
#include "vsa_internal.cuh"

namespace vsa {

namespace {

constexpr int NUM_THREADS = 320;
constexpr int SOFTMAX_WARPS = 8;
constexpr int TMA_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int KV_STAGES = 4;
constexpr int KPF = 7;               // P is carried as P * 2^KPF: below 2^(RESCALE + KPF) = 2^15
constexpr float RESCALE = 8.0f;      // log2 units the block maximum may exceed m by before a rescale

constexpr uint32_t SM_Q = 0;                          // 2 stages x 2 chunks x [128 q x 128 B]
constexpr uint32_t SM_KV = 2 * 32768;                 // stages x (K 16 KB, V 16 KB)
constexpr uint32_t SM_XCH = SM_KV + KV_STAGES * 32768;  // [2 parity][2 halves][128 rows] float
constexpr uint32_t SM_BAR = SM_XCH + 2 * 2 * 128 * 4;

enum Bar : uint32_t {
  Q_FULL0 = 0,
  Q_EMPTY0 = Q_FULL0 + 2,
  KV_FULL0 = Q_EMPTY0 + 2,
  KV_EMPTY0 = KV_FULL0 + KV_STAGES,
  S_FULL0 = KV_EMPTY0 + KV_STAGES,
  S_FREE0 = S_FULL0 + 2,
  P_READY0 = S_FREE0 + 2,
  P_FREE0 = P_READY0 + 2,
  PV_DONE = P_FREE0 + 2,  // one phase per P.V, for the rescale of O
  O_FULL,
  O_EMPTY,
  DRAIN,
  XCH0,  // one per lane quarter: both column-half warps have published a value
  ITEM_FULL0 = XCH0 + 4,
  ITEM_EMPTY0 = ITEM_FULL0 + ITEM_SLOTS,
  NUM_BARS = ITEM_EMPTY0 + ITEM_SLOTS
};
constexpr uint32_t ITEM_CONSUMERS = 1 + SOFTMAX_WARPS;  // the UMMA thread and the softmax warps
constexpr uint32_t SM_TMEM_SLOT = SM_BAR + NUM_BARS * 8;
constexpr uint32_t SM_ABORT = SM_TMEM_SLOT + 4;
constexpr uint32_t SM_QUEUE = SM_ABORT + 4;
constexpr uint32_t SMEM_BYTES = SM_QUEUE + 4 * ITEM_SLOTS + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t TM_O = 0, TM_S = 128, TM_P = 256;
constexpr uint32_t IDESC_S = idesc_f16_f32acc(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_f16_f32acc(128, 128, false, true);

struct Params {
  const uint32_t* bitmap;
  const int32_t* vbs;
  const uint32_t* absmax;
  __nv_bfloat16* o;
  float* lse;
  uint32_t* err;
  int32_t* sched;
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
  volatile int* queue = reinterpret_cast<volatile int*>(gbase + SM_QUEUE);
  const uint32_t* tmem_slot = reinterpret_cast<const uint32_t*>(gbase + SM_TMEM_SLOT);
  auto bar = [&](uint32_t b) { return base + SM_BAR + 8u * b; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S;

  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Q_FULL0 + s), 1);
      mbar_init(bar(Q_EMPTY0 + s), 1);
      mbar_init(bar(S_FULL0 + s), 1);
      mbar_init(bar(S_FREE0 + s), SOFTMAX_WARPS);
      mbar_init(bar(P_READY0 + s), SOFTMAX_WARPS);
      mbar_init(bar(P_FREE0 + s), 1);
    }
    for (int s = 0; s < KV_STAGES; ++s) {
      mbar_init(bar(KV_FULL0 + s), 1);
      mbar_init(bar(KV_EMPTY0 + s), 1);
    }
    mbar_init(bar(PV_DONE), 1);
    mbar_init(bar(O_FULL), 1);
    mbar_init(bar(O_EMPTY), SOFTMAX_WARPS);
    mbar_init(bar(DRAIN), 1);
    for (int qq = 0; qq < 4; ++qq) mbar_init(bar(XCH0 + qq), 2);
    for (int s = 0; s < ITEM_SLOTS; ++s) {
      mbar_init(bar(ITEM_FULL0 + s), 1);
      mbar_init(bar(ITEM_EMPTY0 + s), ITEM_CONSUMERS);
    }
    fence_barrier_init();
  }
  if (warp == TMA_WARP) {
    tmem_alloc(base + SM_TMEM_SLOT, 512);
    tmem_relinquish();
  }
  if (warp == TMA_WARP && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == TMA_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t lg = 0, itc = 0;  // kv blocks loaded; items with a non-empty union
      int64_t last_lg[KV_STAGES], last_q[2] = {-1, -1};
      for (int s = 0; s < KV_STAGES; ++s) last_lg[s] = -1;
      bool ok = true;
      for (uint32_t k = 0;; ++k) {
        int w;
        if (!publish_item(bar(ITEM_FULL0), bar(ITEM_EMPTY0), queue, k, p.sched, abort, &w)) {
          ok = false;
          break;
        }
        if (w >= p.total) break;  // the end marker
        const Pair q = decode_pair(p, w);
        if (union_size(p, q) == 0) continue;
        const uint32_t qs = itc & 1u;
        if (!mbar_wait_bounded(bar(Q_EMPTY0 + qs), ((itc >> 1) & 1u) ^ 1u, abort,
                               WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        const int r0 = q.bh * S + q.i0 * BLOCK;
        const int r1 = q.bh * S + (q.i1 >= 0 ? q.i1 : q.i0) * BLOCK;
        const uint32_t qd = base + SM_Q + qs * 32768u;
        mbar_arrive_expect_tx(bar(Q_FULL0 + qs), 32768);
        tma_load_2d(qd, &tm_q, bar(Q_FULL0 + qs), 0, r0);
        tma_load_2d(qd + 8192, &tm_q, bar(Q_FULL0 + qs), 0, r1);
        tma_load_2d(qd + 16384, &tm_q, bar(Q_FULL0 + qs), 64, r0);
        tma_load_2d(qd + 24576, &tm_q, bar(Q_FULL0 + qs), 64, r1);
        last_q[qs] = itc;
        ok = for_union(p, q, [&](int j) {
          const uint32_t st = lg % KV_STAGES;
          if (!mbar_wait_bounded(bar(KV_EMPTY0 + st), ((lg / KV_STAGES) & 1u) ^ 1u, abort,
                                 WAIT_LIMIT_NS))
            return false;
          const int rk = q.bh * S + j * BLOCK;
          const uint32_t kd = base + SM_KV + st * 32768u;
          mbar_arrive_expect_tx(bar(KV_FULL0 + st), 32768u);
          tma_load_2d(kd, &tm_k, bar(KV_FULL0 + st), 0, rk);
          tma_load_2d(kd + 8192, &tm_k, bar(KV_FULL0 + st), 64, rk);
          tma_load_2d(kd + 16384, &tm_v, bar(KV_FULL0 + st), 0, rk);
          tma_load_2d(kd + 24576, &tm_v, bar(KV_FULL0 + st), 64, rk);
          last_lg[st] = lg;
          ++lg;
          return true;
        });
        if (!ok) break;
        ++itc;
      }
      if (!ok) {
        raise_abort(abort, p.err);
        // Let the copies already issued land before the CTA's shared memory goes away.
        volatile int never = 0;
        for (int s = 0; s < 2; ++s)
          if (last_q[s] >= 0)
            mbar_wait_bounded(bar(Q_FULL0 + s), (static_cast<uint32_t>(last_q[s]) >> 1) & 1u,
                              &never, DRAIN_LIMIT_NS);
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
      uint32_t t = 0, itc = 0;  // kv blocks issued (one S and one P.V each); items
      bool ok = true, issued = false;
      const uint64_t q_kmaj = sdesc_sw128(base + SM_Q, 16, 1024);
      const uint64_t k_kmaj = sdesc_sw128(base + SM_KV, 16, 1024);           // K of stage 0
      const uint64_t v_mn = sdesc_sw128(base + SM_KV + 16384u, 8192, 1024);  // V of stage 0
      // S = Q_p K_j^T of kv block tb into S buffer tb & 1; Q from stage qs.
      auto issue_s = [&](uint32_t tb, uint32_t qs) -> bool {
        const uint32_t st = tb % KV_STAGES, sb = tb & 1u;
        if (!mbar_wait_bounded(bar(KV_FULL0 + st), (tb / KV_STAGES) & 1u, abort, WAIT_LIMIT_NS))
          return false;
        if (!mbar_wait_bounded(bar(S_FREE0 + sb), ((tb >> 1) & 1u) ^ 1u, abort, WAIT_LIMIT_NS))
          return false;
        tc_fence_after_sync();
        const uint64_t qa = sdesc_advance(q_kmaj, qs * 32768u);
        const uint64_t kd = sdesc_advance(k_kmaj, st * 32768u);
        const uint32_t ts = tmem + TM_S + sb * 64u;
        umma_f16_c<false>(ts, qa, kd, IDESC_S);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk) {
          const uint32_t off = (kk & 3) * 32u;
          umma_f16_c<true>(ts, sdesc_advance(qa, (kk >> 2) * 16384u + off),
                           sdesc_advance(kd, (kk >> 2) * 8192u + off), IDESC_S);
        }
        umma_commit(bar(S_FULL0 + sb));
        issued = true;
        return true;
      };
      // O += P V_j of kv block tb: A = P buffer tb & 1 in TMEM (8 columns per 16 kv), B = V_j.
      auto issue_pv = [&](uint32_t tb, bool first) -> bool {
        const uint32_t pb = tb & 1u, st = tb % KV_STAGES;
        if (!mbar_wait_bounded(bar(P_READY0 + pb), (tb >> 1) & 1u, abort, WAIT_LIMIT_NS))
          return false;
        if (first && !mbar_wait_bounded(bar(O_EMPTY), (itc & 1u) ^ 1u, abort, WAIT_LIMIT_NS))
          return false;
        tc_fence_after_sync();
        const uint32_t pa = tmem + TM_P + pb * 32u;
        const uint64_t vb = sdesc_advance(v_mn, st * 32768u);
        if (first)
          umma_f16_ta<false>(tmem + TM_O, pa, vb, IDESC_PV);
        else
          umma_f16_ta<true>(tmem + TM_O, pa, vb, IDESC_PV);
#pragma unroll
        for (int kk = 1; kk < 4; ++kk)
          umma_f16_ta<true>(tmem + TM_O, pa + kk * 8u, sdesc_advance(vb, kk * 2048u), IDESC_PV);
        umma_commit(bar(P_FREE0 + pb));
        umma_commit(bar(KV_EMPTY0 + st));
        umma_commit(bar(PV_DONE));
        return true;
      };
      for (uint32_t k = 0;; ++k) {
        int w;
        if (!take_item(bar(ITEM_FULL0), bar(ITEM_EMPTY0), queue, k, abort, &w)) {
          ok = false;
          break;
        }
        if (w >= p.total) break;
        const Pair q = decode_pair(p, w);
        const int nu = union_size(p, q);
        if (nu == 0) continue;
        const uint32_t qs = itc & 1u;
        if (!mbar_wait_bounded(bar(Q_FULL0 + qs), (itc >> 1) & 1u, abort, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        const uint32_t t0 = t;
        if (!issue_s(t0, qs)) {
          ok = false;
          break;
        }
        for (int e = 0; e < nu; ++e) {
          if (e + 1 < nu) {
            if (!issue_s(t0 + e + 1, qs)) {
              ok = false;
              break;
            }
          } else {
            umma_commit(bar(Q_EMPTY0 + qs));  // every S of the item has been issued
          }
          if (!issue_pv(t0 + e, e == 0)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        umma_commit(bar(O_FULL));
        t = t0 + nu;
        ++itc;
      }
      if (!ok) raise_abort(abort, p.err);
      if (issued) {
        // Every UMMA has completed before TMEM is released.
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
    float* xch = reinterpret_cast<float*>(gbase + SM_XCH);
    uint32_t t = 0, itc = 0, xc = 0;  // kv blocks seen; items with a non-empty union; exchanges
    // The partner warp's value of this row (the other column half).  Slots alternate with the
    // exchange count, so a slot is rewritten only after the partner has read it.
    auto exchange = [&](float x, float* y) -> bool {
      float* slot = xch + (xc & 1u) * 256u;
      slot[h * 128 + r] = x;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(XCH0 + quarter));
      if (!warp_wait(bar(XCH0 + quarter), xc & 1u, abort, lane)) return false;
      __syncwarp();
      *y = slot[(1 - h) * 128 + r];
      ++xc;
      return true;
    };
    for (uint32_t k = 0;; ++k) {
      int w;
      if (!warp_take_item(bar(ITEM_FULL0), bar(ITEM_EMPTY0), queue, k, abort, lane, &w)) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      if (w >= p.total) break;
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
      const float c1 = p.sm_scale * LOG2E_F * exp2i(eq + ek);  // S' -> s (log2 units)
      float m = -INFINITY, l = 0.f;  // reference maximum; this half's sum of P * 2^KPF
      bool first = true;
      const bool ok = for_union(p, q, [&](int j) {
        const uint32_t sb = t & 1u;
        if (!warp_wait(bar(S_FULL0 + sb), (t >> 1) & 1u, abort, lane)) return false;
        tc_fence_after_sync();
        const bool mine = valid && ((own[j >> 5] >> (j & 31)) & 1u);
        const int vb = mine ? clamp_vbs(p.vbs[j]) - h * 32 : 0;  // visible columns in my half
        uint32_t sv[32];
        tmem_ld_32x32b_x32(tmem + lane_off + TM_S + sb * 64u + h * 32u, sv);
        tmem_wait_ld();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(S_FREE0 + sb));
        float mloc = -INFINITY;
#pragma unroll
        for (int u = 0; u < 32; ++u)
          if (u < vb) mloc = fmaxf(mloc, __uint_as_float(sv[u]) * c1);
        float mo;
        if (!exchange(mloc, &mo)) return false;
        const float mb = fmaxf(mloc, mo);  // the row's maximum over this kv block
        const bool need = mb > m + RESCALE;
        // P buffer sb is free once P.V of block t-2 has completed; from then on P.V of block
        // t-1 is the only one that can still be accumulating into O.
        if (!warp_wait(bar(P_FREE0 + sb), ((t >> 1) & 1u) ^ 1u, abort, lane)) return false;
        if (__any_sync(0xffffffffu, need)) {
          const float f = need ? ex2(m - mb) : 1.f;  // m = -inf: f = 0 (nothing accumulated)
          if (!first) {
            if (!warp_wait(bar(PV_DONE), (t - 1) & 1u, abort, lane)) return false;
            tc_fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
              uint32_t ov[32];
              const uint32_t ta = tmem + lane_off + TM_O + h * 64u + c * 32u;
              tmem_ld_32x32b_x32(ta, ov);
              tmem_wait_ld();
#pragma unroll
              for (int u = 0; u < 32; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * f);
              tmem_st_32x32b_x32(ta, ov);
            }
            tmem_wait_st();
          }
          l *= f;
          if (need) m = mb;
        }
        const float off = static_cast<float>(KPF) - m;
        uint32_t pk[16];
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          const float p0 = (u < vb) ? ex2(fmaf(__uint_as_float(sv[u]), c1, off)) : 0.f;
          const float p1 = (u + 1 < vb) ? ex2(fmaf(__uint_as_float(sv[u + 1]), c1, off)) : 0.f;
          acc += p0 + p1;
          pk[u >> 1] = pack_half2(p0, p1);
        }
        l += acc;
        tmem_st_32x32b_x16(tmem + lane_off + TM_P + sb * 32u + h * 16u, pk);
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P_READY0 + sb));
        ++t;
        first = false;
        return true;
      });
      float lo = 0.f;
      if (!ok || !exchange(l, &lo)) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      const float lt = l + lo;
      if (!warp_wait(bar(O_FULL), itc & 1u, abort, lane)) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      tc_fence_after_sync();
      uint32_t v[64];  // O columns h*64 .. h*64+63 of row r
      tmem_ld_32x32b_x32(tmem + lane_off + TM_O + h * 64u, v);
      tmem_ld_32x32b_x32(tmem + lane_off + TM_O + h * 64u + 32u, v + 32);
      tmem_wait_ld();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(O_EMPTY));
      if (valid) {
        // O = (sum P 2^KPF V') 2^ev / (sum P 2^KPF); an empty row (lt = 0) gives O = 0 and
        // lse = -inf.
        const float os = lt > 0.f ? exp2i(ev) / lt : 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int u = 8 * c;
          orow[c] = make_uint4(
              pack_bf162(__uint_as_float(v[u]) * os, __uint_as_float(v[u + 1]) * os),
              pack_bf162(__uint_as_float(v[u + 2]) * os, __uint_as_float(v[u + 3]) * os),
              pack_bf162(__uint_as_float(v[u + 4]) * os, __uint_as_float(v[u + 5]) * os),
              pack_bf162(__uint_as_float(v[u + 6]) * os, __uint_as_float(v[u + 7]) * os));
        }
        if (h == 0) p.lse[grow] = lt > 0.f ? m + log2f(lt) - static_cast<float>(KPF) : -INFINITY;
      }
      ++itc;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == TMA_WARP) tmem_dealloc(tmem, 512);
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
  p.sched = a.sched;
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
