// fwd_main.cu -- forward of block-sparse attention on sm_103a, producing O and the base-2 "M form"
// log-sum-exp that the backward consumes (FastVideo block_sparse_attn_bwd_sm100a.py docstring:
// lse = max(qk * sm_scale * log2e) + log2(l); compare main...vsa_bwd_fix, tests,
// reference(): softmax over the selected blocks with keys past variable_block_sizes masked).
//
// Work unit: one (b, h, q pair) item -- 64-token q tiles 2x and 2x+1 (one 128-token q block when
// blocks are 128 tokens) -- so the UMMA M dimension is 128 and row m of every accumulator is TMEM
// lane m.  The item walks the UNION of the two tiles' selected kv tiles (ascending); for each
// row, kv tiles its own q tile did not select are masked.  The union is taken two kv tiles at a
// time: S = Q_p [K_a; K_b]^T is one set of 128x128x16 UMMAs (the caller's bf16 Q and K, both in
// shared memory, fp32 accumulator in TMEM), and softmax group 0 takes tile a, group 1 tile b.
// Per group and kv tile, an online softmax:
//   the row maximum of the tile; if it exceeds the row's reference maximum m by more than
//   RESCALE (log2 units), m moves up to it and the group's O row and running sum are scaled by
//   2^(m_old - m_new) first (otherwise m stays, so P stays below 2^(RESCALE + KPF));
//   P = 2^(s - m + KPF) in fp16, written to TMEM, where it is the A operand of
//   O_g += P V_j (B = V_j from shared memory, MN-major; kind::f16 takes one type for A and B,
//   so V comes from the preprocess's fp16 copy, scaled by 2^-e_v).
// P never passes through shared memory, so per kv tile the tensor pipe reads Q_p, K_j and V_j
// only.
//
// Each group has its own online-softmax state (m, l) and its own O accumulator, the split of
// the kv range that flash-decoding uses, so the two groups work independently.  At the end of
// the item the two partial results merge:
//   M = max(m_0, m_1),  w_g = 2^(m_g - M),  O = (w_0 O_0 + w_1 O_1) / (w_0 l_0 + w_1 l_1),
//   lse = M + log2(w_0 l_0 + w_1 l_1).
//
// Roles (352 threads): warps 0-3 softmax group 0 and warps 4-7 group 1 -- warp w owns TMEM lane
// quarter w % 4 (query rows 32(w%4) .. +31), one full row of S per thread; warp 8 work claimer,
// TMEM owner and TMA producer of Q and K pairs; warp 9 UMMA issuer; warp 10 TMA producer of V.
// S is double-buffered in TMEM: pair p uses buffer p & 1, and each group writes its P (fp16
// pairs, 32 columns) over the first half of its own 64 S columns once it holds them in
// registers, so P.V reads its A operand from there.  The tensor pipe runs
//   S(p+1)  P.V(p) (group 0, then group 1)  S(p+2)  P.V(p+1) ...
// S(p+2) waits until both P.V of pair p have completed (the buffer is free again), so while the
// softmax works on pair p+1 the tensor pipe already has S(p+2) to do.  K and V have rings of
// their own: a K stage is free once S has been computed, before P.V frees the V stages of the
// same tiles, so the K loads run further ahead.
// Every softmax warp takes part in every pair (a group without a tile in a pair only signals
// that it has none), so no barrier can complete two phases while a waiter looks at it.
// TMEM (512 columns allocated): O x2 [0,256), S x2 [256,512).
#include "ptx.cuh"
#include "queue.cuh"
#include "vsa_internal.cuh"

namespace vsa {

namespace {

constexpr int NUM_THREADS = 352;
constexpr int SOFTMAX_WARPS = 8;
constexpr int TMA_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int V_WARP = 10;
constexpr int K_STAGES = 2;  // stages of a PAIR of kv blocks (32 KB each), one per S buffer
constexpr int V_STAGES = 5;
constexpr int KPF = 7;               // P is carried as P * 2^KPF: below 2^(RESCALE + KPF) = 2^15
constexpr float RESCALE = 8.0f;      // log2 units the block maximum may exceed m by before a rescale

constexpr uint32_t SM_Q = 0;                         // 2 stages x 2 chunks x [128 q x 128 B]
constexpr uint32_t SM_K = 2 * 32768;                 // K pair stages x 2 chunks x [128 kv x 128 B]
constexpr uint32_t SM_V = SM_K + K_STAGES * 32768;   // V stages x 2 chunks x [64 kv x 128 B]
constexpr uint32_t SM_XCH = SM_V + V_STAGES * 16384;  // [2 parity][2 groups][128 rows] (m, l)
constexpr uint32_t SM_BAR = SM_XCH + 2 * 2 * 128 * 8;

enum Bar : uint32_t {
  Q_FULL0 = 0,
  Q_EMPTY0 = Q_FULL0 + 2,
  K_FULL0 = Q_EMPTY0 + 2,
  V_FULL0 = K_FULL0 + K_STAGES,
  V_EMPTY0 = V_FULL0 + V_STAGES,
  S_FULL0 = V_EMPTY0 + V_STAGES,  // S(p) is in TMEM buffer p & 1 (and K stage p & 1 is free)
  BUF_FREE0 = S_FULL0 + 2,        // both P.V of pair p have completed: buffer p & 1 is free
  // Per group and pair parity: P of the pair is in TMEM (or the group has none).  Alternating
  // barriers keep a warp that runs ahead to pair p + 1 from arriving in pair p's phase.
  P_READY0 = BUF_FREE0 + 2,
  O_FULL = P_READY0 + 4,
  O_EMPTY,
  DRAIN,
  XCH0,  // one per lane quarter: both groups' warps have published (m, l) of the item
  ITEM_FULL0 = XCH0 + 4,
  ITEM_EMPTY0 = ITEM_FULL0 + ITEM_SLOTS,
  NUM_BARS = ITEM_EMPTY0 + ITEM_SLOTS
};
// The UMMA thread, the softmax warps and the V producer.
constexpr uint32_t ITEM_CONSUMERS = 1 + SOFTMAX_WARPS + 1;
constexpr uint32_t GROUP_WARPS = SOFTMAX_WARPS / 2;
constexpr uint32_t SM_TMEM_SLOT = SM_BAR + NUM_BARS * 8;
constexpr uint32_t SM_ABORT = SM_TMEM_SLOT + 4;
constexpr uint32_t SM_QUEUE = SM_ABORT + 4;
constexpr uint32_t SMEM_BYTES = SM_QUEUE + 4 * ITEM_SLOTS + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

static_assert(K_STAGES == 2, "K stages pair up with the two S buffers");
constexpr uint32_t TM_O = 0, TM_S = 256;  // O_g at TM_O + 128 g; S buffer b at TM_S + 128 b
constexpr uint32_t IDESC_S = idesc_f16_f32acc(128, 128, false, false, true);  // bf16 Q, K
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
  uint64_t wait_ns;  // limit of each pipeline wait
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
                                          uint64_t limit_ns, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait_bounded(bar, parity, abort, limit_ns) ? 1 : 0;
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

// Packed fp32 pairs (sm_100 family): one instruction operates on both halves of a 64-bit
// register pair, each half rounded as the scalar instruction would.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Maximum / minimum of 64 raw fp32 scores, four independent chains of 3-input instructions.
__device__ __forceinline__ float row_max64(const uint32_t* sv) {
  float m[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) m[k] = fmaxf(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1]));
#pragma unroll
  for (int u = 8; u < 64; u += 2)
    m[(u >> 1) & 3] = max3(m[(u >> 1) & 3], __uint_as_float(sv[u]), __uint_as_float(sv[u + 1]));
  return max3(fmaxf(m[0], m[1]), m[2], m[3]);
}
__device__ __forceinline__ float row_min64(const uint32_t* sv) {
  float m[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) m[k] = fminf(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1]));
#pragma unroll
  for (int u = 8; u < 64; u += 2)
    m[(u >> 1) & 3] = min3(m[(u >> 1) & 3], __uint_as_float(sv[u]), __uint_as_float(sv[u + 1]));
  return min3(fminf(m[0], m[1]), m[2], m[3]);
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
    fwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q2,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_k2,
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
      mbar_init(bar(BUF_FREE0 + s), 1);
      mbar_init(bar(P_READY0 + 2 * s), GROUP_WARPS);
      mbar_init(bar(P_READY0 + 2 * s + 1), GROUP_WARPS);
    }
    for (int s = 0; s < K_STAGES; ++s) mbar_init(bar(K_FULL0 + s), 1);
    for (int s = 0; s < V_STAGES; ++s) {
      mbar_init(bar(V_FULL0 + s), 1);
      mbar_init(bar(V_EMPTY0 + s), 1);
    }
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
    tma_prefetch_desc(&tm_q2);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_k2);
    tma_prefetch_desc(&tm_v);
  }
  grid_dependency_wait();  // the V copy and the bitmap (programmatic dependent launch)
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == TMA_WARP) {
    // ------------------------------------------------------------------ TMA producer: Q, K
    // Warp-wide: lane 0 claims items and registers the expected bytes; each tile goes out from
    // a lane of its own (a thread's bulk copies are processed one after another).
    uint32_t lg = 0, itc = 0;  // kv blocks loaded; items with a non-empty union
    int64_t last_lg[K_STAGES], last_q[2] = {-1, -1};
    for (int s = 0; s < K_STAGES; ++s) last_lg[s] = -1;
    bool ok = true;
    for (uint32_t k = 0;; ++k) {
      int w = 0, okp = 1;
      if (lane == 0)
        okp = publish_item(bar(ITEM_FULL0), bar(ITEM_EMPTY0), queue, k, p.sched, abort, p.wait_ns,
                           &w)
                  ? 1
                  : 0;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!__shfl_sync(0xffffffffu, okp, 0)) {
        ok = false;
        break;
      }
      if (w >= p.total) break;  // the end marker
      const Pair q = decode_pair(p, w);
      if (union_size(p, q) == 0) continue;
      const uint32_t qs = itc & 1u;
      if (!mbar_wait_warp(bar(Q_EMPTY0 + qs), ((itc >> 1) & 1u) ^ 1u, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      const int r0 = q.bh * S + q.i0 * BLOCK;
      const int r1 = q.bh * S + (q.i1 >= 0 ? q.i1 : q.i0) * BLOCK;
      if (lane == 0) mbar_arrive_expect_tx(bar(Q_FULL0 + qs), 32768);
      __syncwarp();
      if (q.i1 >= 0) {  // the two q tiles are adjacent: both column halves of 128 rows, one copy
        if (lane == 0) tma_load_3d(base + SM_Q + qs * 32768u, &tm_q2, bar(Q_FULL0 + qs), 0, r0, 0);
      } else if (lane < 4) {  // tile t = lane at byte t * 8192: (cols 0-63, i0), (0-63, i1), ...
        tma_load_2d(base + SM_Q + qs * 32768u + static_cast<uint32_t>(lane) * 8192u, &tm_q,
                    bar(Q_FULL0 + qs), (lane & 2) ? 64 : 0, (lane & 1) ? r1 : r0);
      }
      last_q[qs] = itc;
      // K of the union's kv blocks two at a time: block 2p in rows 0-63 of pair stage p, block
      // 2p+1 (if any) in rows 64-127, each as (cols 0-63) and (cols 64-127) chunks of 16 KB.
      int ja = -1, e = 0;
      auto load_pair = [&](int j0, int j1) -> bool {
        const uint32_t st = lg % K_STAGES;
        if (!mbar_wait_warp(bar(S_FULL0 + st), ((lg / K_STAGES) & 1u) ^ 1u, abort,
                            p.wait_ns))
          return false;
        if (lane == 0) mbar_arrive_expect_tx(bar(K_FULL0 + st), j1 >= 0 ? 32768u : 16384u);
        __syncwarp();
        if (j1 == j0 + 1) {  // adjacent kv tiles: 128 rows, both column halves, one copy
          if (lane == 0)
            tma_load_3d(base + SM_K + st * 32768u, &tm_k2, bar(K_FULL0 + st), 0,
                        q.bh * S + j0 * BLOCK, 0);
        } else if (lane < 4 && (lane < 2 || j1 >= 0)) {  // lane: (block lane >> 1, chunk lane & 1)
          tma_load_2d(base + SM_K + st * 32768u + static_cast<uint32_t>(lane & 1) * 16384u +
                          static_cast<uint32_t>(lane >> 1) * 8192u,
                      &tm_k, bar(K_FULL0 + st), (lane & 1) * 64,
                      q.bh * S + ((lane >> 1) ? j1 : j0) * BLOCK);
        }
        last_lg[st] = lg;
        ++lg;
        return true;
      };
      ok = for_union(p, q, [&](int j) {
        if ((e++ & 1) == 0) {
          ja = j;
          return true;
        }
        return load_pair(ja, j);
      });
      if (ok && (e & 1)) ok = load_pair(ja, -1);
      if (!ok) break;
      ++itc;
    }
    if (!ok && lane == 0) {
      raise_abort(abort, p.err);
      // Let the copies already issued land before the CTA's shared memory goes away.
      volatile int never = 0;
      for (int s = 0; s < 2; ++s)
        if (last_q[s] >= 0)
          mbar_wait_bounded(bar(Q_FULL0 + s), (static_cast<uint32_t>(last_q[s]) >> 1) & 1u,
                            &never, DRAIN_LIMIT_NS);
      for (int s = 0; s < K_STAGES; ++s)
        if (last_lg[s] >= 0)
          mbar_wait_bounded(bar(K_FULL0 + s), (static_cast<uint32_t>(last_lg[s]) / K_STAGES) & 1u,
                            &never, DRAIN_LIMIT_NS);
    }
    __syncwarp();
  } else if (warp == V_WARP) {
    // ------------------------------------------------------------------ TMA producer: V
    uint32_t lg = 0;
    int64_t last_lg[V_STAGES];
    for (int s = 0; s < V_STAGES; ++s) last_lg[s] = -1;
    bool ok = true;
    for (uint32_t k = 0;; ++k) {
      int w;
      if (!warp_take_item(bar(ITEM_FULL0), bar(ITEM_EMPTY0), queue, k, abort, p.wait_ns, lane, &w)) {
        ok = false;
        break;
      }
      if (w >= p.total) break;
      const Pair q = decode_pair(p, w);
      ok = for_union(p, q, [&](int j) {
        const uint32_t st = lg % V_STAGES;
        if (!mbar_wait_warp(bar(V_EMPTY0 + st), ((lg / V_STAGES) & 1u) ^ 1u, abort,
                            p.wait_ns))
          return false;
        if (lane == 0) mbar_arrive_expect_tx(bar(V_FULL0 + st), 16384u);
        __syncwarp();
        if (lane == 0)  // both column halves of the tile in one copy
          tma_load_3d(base + SM_V + st * 16384u, &tm_v, bar(V_FULL0 + st), 0, q.bh * S + j * BLOCK,
                      0);
        last_lg[st] = lg;
        ++lg;
        return true;
      });
      if (!ok) break;
    }
    if (!ok && lane == 0) {
      raise_abort(abort, p.err);
      volatile int never = 0;
      for (int s = 0; s < V_STAGES; ++s)
        if (last_lg[s] >= 0)
          mbar_wait_bounded(bar(V_FULL0 + s), (static_cast<uint32_t>(last_lg[s]) / V_STAGES) & 1u,
                            &never, DRAIN_LIMIT_NS);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ UMMA issuer
    // The whole warp runs this role in lockstep; every lane polls the barriers and one elected
    // lane issues each UMMA and commit.
    uint32_t pc = 0, vc = 0, itc = 0;  // kv-tile pairs (S), kv tiles (P.V), items
    bool ok = true, issued = false;
    const uint64_t q_kmaj = sdesc_sw128(base + SM_Q, 16, 1024);
    const uint64_t k_kmaj = sdesc_sw128(base + SM_K, 16, 1024);   // K pair of stage 0
    const uint64_t v_mn = sdesc_sw128(base + SM_V, 8192, 1024);   // V of stage 0
    // S(pb) = Q_p [K_a; K_b]^T (N = 128: columns 0-63 tile a, 64-127 tile b) into TMEM buffer
    // pb & 1, once K stage pb & 1 is loaded and both P.V of pair pb - 2 (which read their P from
    // that buffer) have completed.  Q from stage qs.
    auto issue_s = [&](uint32_t pb, uint32_t qs) -> bool {
      const uint32_t b = pb & 1u;
      if (!mbar_wait2_warp(bar(K_FULL0 + b), (pb >> 1) & 1u, bar(BUF_FREE0 + b),
                           ((pb >> 1) & 1u) ^ 1u, abort, p.wait_ns))
        return false;
      tc_fence_after_sync();
      const uint64_t qa = sdesc_advance(q_kmaj, qs * 32768u);
      const uint64_t kd = sdesc_advance(k_kmaj, b * 32768u);
      const uint32_t ts = tmem + TM_S + b * 128u;
      umma_ss_elect<false>(ts, qa, kd, IDESC_S);
#pragma unroll
      for (int kk = 1; kk < 8; ++kk) {
        const uint32_t off = (kk & 3) * 32u;
        umma_ss_elect<true>(ts, sdesc_advance(qa, (kk >> 2) * 16384u + off),
                            sdesc_advance(kd, (kk >> 2) * 16384u + off), IDESC_S);
      }
      // One commit: it tells the softmax that S is ready and the K producer that the stage is
      // free (a commit issued behind a pending one holds this warp until the first completes).
      umma_commit_elect(bar(S_FULL0 + b));
      issued = true;
      return true;
    };
    // O_g += P_g V_j for group g's kv tile of pair pb (V stage from the global tile count): A =
    // P_g in TMEM (columns 64 g .. 64 g + 31 of buffer pb & 1, 8 columns per 16 kv), B = V_j.
    // `fresh`: the group's first tile of the item overwrites O_g.  The caller has waited for V
    // and for the group's P.
    auto issue_pv = [&](uint32_t pb, uint32_t g, bool fresh) {
      const uint32_t st = vc % V_STAGES;
      const uint32_t pa = tmem + TM_S + (pb & 1u) * 128u + g * 64u, to = tmem + TM_O + g * 128u;
      const uint64_t vb = sdesc_advance(v_mn, st * 16384u);
      if (fresh)
        umma_ts_elect<false>(to, pa, vb, IDESC_PV);
      else
        umma_ts_elect<true>(to, pa, vb, IDESC_PV);
#pragma unroll
      for (int kk = 1; kk < 4; ++kk)
        umma_ts_elect<true>(to, pa + kk * 8u, sdesc_advance(vb, kk * 2048u), IDESC_PV);
      umma_commit_elect(bar(V_EMPTY0 + st));
      ++vc;
    };
    for (uint32_t k = 0;; ++k) {
      int w;
      if (!warp_take_item(bar(ITEM_FULL0), bar(ITEM_EMPTY0), queue, k, abort, p.wait_ns, lane, &w)) {
        ok = false;
        break;
      }
      if (w >= p.total) break;
      const Pair q = decode_pair(p, w);
      const int nu = union_size(p, q);
      if (nu == 0) continue;
      const int npr = (nu + 1) >> 1;
      const uint32_t qs = itc & 1u;
      if (!mbar_wait_warp(bar(Q_FULL0 + qs), (itc >> 1) & 1u, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      const uint32_t p0 = pc;
      ok = issue_s(p0, qs);
      for (int pr = 0; pr < npr && ok; ++pr) {
        const uint32_t pb = p0 + pr;
        if (pr + 1 < npr) {
          if (!issue_s(pb + 1, qs)) {
            ok = false;
            break;
          }
        } else {
          umma_commit_elect(bar(Q_EMPTY0 + qs));  // every S of the item has been issued
        }
        // Group 0 always has a tile; group 1 signals every pair, also when the union's odd last
        // tile leaves it none.  One wait covers both groups' P and both V tiles (each wait costs
        // this warp a few hundred cycles while the softmax warps share its scheduler); the
        // item's first P.V also waits until the previous item's O buffers have been read.
        const bool two = 2 * pr + 1 < nu;
        const uint32_t v1 = two ? vc + 1 : vc;
        const uint32_t wb[4] = {bar(V_FULL0 + vc % V_STAGES), bar(V_FULL0 + v1 % V_STAGES),
                                bar(P_READY0 + (pb & 1u)), bar(P_READY0 + 2 + (pb & 1u))};
        const uint32_t wp[4] = {(vc / V_STAGES) & 1u, (v1 / V_STAGES) & 1u, (pb >> 1) & 1u,
                                (pb >> 1) & 1u};
        ok = (pr != 0 || mbar_wait_warp(bar(O_EMPTY), (itc & 1u) ^ 1u, abort, p.wait_ns)) &&
             mbar_waitn_warp(wb, wp, abort, p.wait_ns);
        if (!ok) break;
        tc_fence_after_sync();
        issue_pv(pb, 0, pr == 0);
        if (two) issue_pv(pb, 1, pr == 0);
        umma_commit_elect(bar(BUF_FREE0 + (pb & 1u)));
      }
      if (!ok) break;
      umma_commit_elect(bar(O_FULL));
      pc = p0 + npr;
      ++itc;
    }
    if (!ok && lane == 0) raise_abort(abort, p.err);
    if (issued) {
      // Every UMMA has completed before TMEM is released.
      umma_commit_elect(bar(DRAIN));
      volatile int never = 0;
      if (lane == 0) mbar_wait_bounded(bar(DRAIN), 0, &never, DRAIN_LIMIT_NS);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-7)
    const int quarter = warp & 3, grp = warp >> 2;  // TMEM lane quarter; softmax group
    const int r = quarter * 32 + lane;              // query row of the pair == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_o = tmem + lane_off + TM_O + grp * 128u;
    float2* xch = reinterpret_cast<float2*>(gbase + SM_XCH);  // [item parity][group][row] (m, l)
    uint32_t pc = 0, itc = 0;  // kv-tile pairs; items
    for (uint32_t k = 0;; ++k) {
      int w;
      if (!warp_take_item(bar(ITEM_FULL0), bar(ITEM_EMPTY0), queue, k, abort, p.wait_ns, lane, &w)) {
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
      uint4* orow = reinterpret_cast<uint4*>(p.o + grow * HEAD_DIM) + grp * 8;
      const int nu = union_size(p, q);
      if (nu == 0) {
        if (valid) {
          for (int c = 0; c < 8; ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
          if (grp == 0) p.lse[grow] = -INFINITY;
        }
        continue;
      }
      const int ev = operand_exponent(p.absmax[q.bh * HEAD_STATS + HS_V]);
      const float c1 = p.sm_scale * LOG2E_F;  // S -> s (log2 units); Q and K are unscaled bf16
      float m = -INFINITY, l = 0.f;  // this group's reference maximum and sum of P * 2^KPF
      bool first = true;             // no block of this group in the item yet
      // The union's kv tiles in pairs (tile 2p for group 0, 2p+1 for group 1); j < 0: the
      // group has no tile in this pair (the union's odd last tile goes to group 0).
      auto do_pair = [&](int j) -> bool {
        const uint32_t pb = pc++;
        const uint32_t b = pb & 1u;
        if (!warp_wait(bar(S_FULL0 + b), (pb >> 1) & 1u, abort, p.wait_ns, lane)) return false;
        tc_fence_after_sync();
        // S of this group's tile, then its P over the first 32 of those columns.
        const uint32_t t_s = tmem + lane_off + TM_S + b * 128u + grp * 64u;
        // Both P.V of the previous pair have completed: O_grp holds every tile so far (needed
        // before a rescale only).  The barrier cannot be a phase behind (S(pb) was issued after
        // the UMMA warp had seen pair pb - 3 complete) nor a phase ahead (pair pb + 1 needs this
        // warp's P), so skipping the wait when nothing is rescaled is safe.
        auto wait_prev = [&]() -> bool {
          return pb == 0 ||
                 warp_wait(bar(BUF_FREE0 + ((pb - 1) & 1u)), ((pb - 1) >> 1) & 1u, abort,
                           p.wait_ns, lane);
        };
        auto ready = [&]() {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(P_READY0 + 2 * grp + b));
        };
        if (j < 0) {
          ready();
          return true;
        }
        // Warp-uniform: the warp's 32 rows belong to one q tile.
        const bool mine = valid && ((own[j >> 5] >> (j & 31)) & 1u);
        const int vb = mine ? clamp_vbs(p.vbs[j]) : 0;  // visible columns of the row
        uint32_t pk[32];
        if (vb == 0) {
          // Nothing of this kv tile is visible to the warp's rows (the other q tile of the pair
          // selected it, or the tile is empty): S is not read, m and l stay, and P is zero.
#pragma unroll
          for (int u = 0; u < 32; ++u) pk[u] = 0u;
          tmem_st_32x32b_x32(t_s, pk);
          tmem_wait_st();
          ready();
          first = false;
          return true;
        }
        uint32_t sv[64];
        tmem_ld_32x32b_x32(t_s, sv);
        tmem_ld_32x32b_x32(t_s + 32u, sv + 32);
        tmem_wait_ld();
        // Columns past the tile's valid count are masked by setting their raw score to the
        // value that scales to -inf (so they neither win the maximum nor contribute to P); with
        // c1 = 0 that does not work and the per-column path below masks instead.
        const bool fast = c1 != 0.f;
        if (fast && vb < BLOCK) {
          const uint32_t pad = c1 > 0.f ? 0xff800000u : 0x7f800000u;  // -inf : +inf
#pragma unroll
          for (int u = 0; u < 64; ++u)
            if (u >= vb) sv[u] = pad;
        }
        // The row's maximum of s over this kv tile: the extremum of the raw scores, scaled once
        // (c1 > 0: max; c1 < 0: min), in 3-input max/min instructions.  Few ALU instructions per
        // element keep this warp from crowding out the UMMA and TMA warps that share its
        // scheduler.
        float mb;
        if (fast) {
          mb = c1 * (c1 > 0.f ? row_max64(sv) : row_min64(sv));
        } else {
          mb = -INFINITY;
#pragma unroll
          for (int u = 0; u < 64; ++u)
            if (u < vb) mb = fmaxf(mb, __uint_as_float(sv[u]) * c1);
        }
        const bool need = mb > m + RESCALE;
        const bool any_need = __any_sync(0xffffffffu, need);
        float f = 1.f;  // factor for O_grp and l (m = -inf: f = 0, nothing accumulated yet)
        if (any_need) {
          f = need ? ex2(m - mb) : 1.f;
          l *= f;
          if (need) m = mb;
        }
        const float off = static_cast<float>(KPF) - m;
        if (fast) {
          // Two columns per packed fp32x2 FMA and add.
          const uint64_t c2 = f2_pack(c1, c1), o2 = f2_pack(off, off);
          uint64_t acc2 = f2_pack(0.f, 0.f);
#pragma unroll
          for (int u = 0; u < 64; u += 2) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[u]), __uint_as_float(sv[u + 1])), c2, o2),
                      a0, a1);
            const float p0 = ex2(a0), p1 = ex2(a1);
            acc2 = f2_add(acc2, f2_pack(p0, p1));
            pk[u >> 1] = pack_half2(p0, p1);
          }
          float s0, s1;
          f2_unpack(acc2, s0, s1);
          l += s0 + s1;
        } else {
          float acc = 0.f;
#pragma unroll
          for (int u = 0; u < 64; u += 2) {
            const float p0 = (u < vb) ? ex2(fmaf(__uint_as_float(sv[u]), c1, off)) : 0.f;
            const float p1 = (u + 1 < vb) ? ex2(fmaf(__uint_as_float(sv[u + 1]), c1, off)) : 0.f;
            acc += p0 + p1;
            pk[u >> 1] = pack_half2(p0, p1);
          }
          l += acc;
        }
        if (any_need && !first) {
          if (!wait_prev()) return false;
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            tmem_ld_32x32b_x32(t_o + c * 32u, ov);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * f);
            tmem_st_32x32b_x32(t_o + c * 32u, ov);
          }
        }
        tmem_st_32x32b_x32(t_s, pk);
        tmem_wait_st();
        ready();
        first = false;
        return true;
      };
      int e = 0, jprev = -1;
      bool ok = for_union(p, q, [&](int j) {
        const bool odd = (e++ & 1) != 0;
        if (!odd) {
          jprev = j;
          return true;
        }
        return do_pair(grp == 0 ? jprev : j);
      });
      if (ok && (e & 1)) ok = do_pair(grp == 0 ? jprev : -1);
      if (!ok) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      // Merge the two groups' partial results of each row.  Slots alternate with the item, so a
      // slot is rewritten only after the partner warp passed the next exchange, i.e. read it.
      float2* slot = xch + (itc & 1u) * 256u;
      slot[grp * 128 + r] = make_float2(m, l);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(XCH0 + quarter));
      if (!warp_wait(bar(XCH0 + quarter), itc & 1u, abort, p.wait_ns, lane)) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      __syncwarp();
      const float2 mo = slot[(1 - grp) * 128 + r];
      if (!warp_wait(bar(O_FULL), itc & 1u, abort, p.wait_ns, lane)) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      tc_fence_after_sync();
      const float m0 = grp == 0 ? m : mo.x, l0 = grp == 0 ? l : mo.y;
      const float m1 = grp == 0 ? mo.x : m, l1 = grp == 0 ? mo.y : l;
      const float mm = fmaxf(m0, m1);
      // A group without any visible column (l = 0; also one without blocks: its O buffer
      // holds stale data) gets weight 0 and its O is not read.
      const float w0 = l0 > 0.f ? ex2(m0 - mm) : 0.f, w1 = l1 > 0.f ? ex2(m1 - mm) : 0.f;
      const float lt = w0 * l0 + w1 * l1;
      const float os = lt > 0.f ? exp2i(ev) / lt : 0.f;
      const float a0 = w0 * os, a1 = w1 * os;
      // This warp writes O columns grp*64 .. grp*64+63 of row r, from both groups' buffers.
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t v0[32], v1[32];
        const uint32_t col = TM_O + grp * 64u + c * 32u;
        tmem_ld_32x32b_x32(tmem + lane_off + col, v0);
        tmem_ld_32x32b_x32(tmem + lane_off + col + 128u, v1);
        tmem_wait_ld();
        if (c == 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(O_EMPTY));
        }
        if (valid) {
#pragma unroll
          for (int u = 0; u < 32; u += 8) {
            float o8[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const float f0 = a0 != 0.f ? __uint_as_float(v0[u + x]) * a0 : 0.f;
              const float f1 = a1 != 0.f ? __uint_as_float(v1[u + x]) * a1 : 0.f;
              o8[x] = f0 + f1;
            }
            orow[c * 4 + u / 8] = make_uint4(pack_bf162(o8[0], o8[1]), pack_bf162(o8[2], o8[3]),
                                             pack_bf162(o8[4], o8[5]), pack_bf162(o8[6], o8[7]));
          }
        }
      }
      if (valid && grp == 0)
        p.lse[grow] = lt > 0.f ? mm + log2f(lt) - static_cast<float>(KPF) : -INFINITY;
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
  // 64-row boxes per column half for tiles anywhere, two-half boxes for adjacent tile pairs
  // (128 rows) and single V tiles (64 rows).
  CUtensorMap tq, tq2, tk, tk2, tv;
  cudaError_t e;
  if ((e = make_tmap_rows128_f16(&tq, a.q, rows, true)) != cudaSuccess) return e;
  if ((e = make_tmap_rows128_f16(&tk, a.k, rows, true)) != cudaSuccess) return e;
  if ((e = make_tmap_rows128_f16_halves(&tv, a.v16, rows, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_rows128_f16_halves(&tq2, a.q, rows, 128, true)) != cudaSuccess) return e;
  if ((e = make_tmap_rows128_f16_halves(&tk2, a.k, rows, 128, true)) != cudaSuccess) return e;
  static std::atomic<uint64_t> smem_set{0};
  if ((e = ensure_smem_limit(fwd_main_kernel, static_cast<int>(SMEM_BYTES), smem_set)) !=
      cudaSuccess)
    return e;
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
  p.wait_ns = a.wait_ns;
  const int sms = device_sm_count();
  const int grid = p.total < sms ? p.total : sms;
  return launch_dependent(fwd_main_kernel, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, stream, tq,
                          tq2, tk, tk2, tv, p);
}

}  // namespace vsa
