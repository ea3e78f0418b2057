// bwd_main.cu -- the main kernel of the block-sparse attention backward on sm_103a.
//
// Work unit: one (b, h, kv block j) item, as in FastVideo's sm_100a backward (its commit message:
// one warp-specialized tcgen05 kernel whose work item is a (batch, head, 64-token kv block) and
// which produces dK, dV and the dQ partials).  The item's k2q list of q blocks is walked two q
// blocks at a time, so every UMMA has M = 128 (the q pair, or the 128 head-dim rows) and the
// fp32 accumulator maps row m to TMEM lane m.  Per q pair (p = the pair's 128 query rows, all
// operands fp16 with power-of-two scales -- per head for Q and dO, per kv tile for K, V and dS,
// see ItemScales -- and fp32 accumulation):
//   S   [128 q  x  64 kv] = Q_p  K_j^T      A = Q_p    (MN-major), B = K_j (K-major)
//   dP  [128 q  x  64 kv] = dO_p V_j^T      A = dO_p   (MN-major), B = V_j (K-major)
//   P   = exp2(S * c - lse), masked (kv row >= vbs[j], missing second q block, or a k2q id
//         outside [0, nb), which is skipped)                                       -> fp16 smem
//   dS  = P * (dP - Delta)                                                          -> fp16 smem
//   dV^T [128 hd x 64 kv] += dO_p^T P         A = dO_p^T (K-major),  B = P  (MN-major)
//   dK^T [128 hd x 64 kv] += Q_p^T  dS        A = Q_p^T  (K-major),  B = dS (MN-major)
//   dQ^T [128 hd x 128 q] =  K_j^T  dS^T      A = K_j    (MN-major), B = dS (K-major)
// Q and dO come from the preprocess tile-transposed (each 64-token tile as [128 head dims][64
// rows], one 16 KB copy), K and V row-major; each shared-memory tile (128-byte swizzle, 8-row
// groups 1024 B apart) serves as a K-major operand of one GEMM and an MN-major operand of
// another.  dQ^T leaves TMEM with head-dim on the lanes, so each warp's fp32 reduction into the
// dQ accumulator covers 128 contiguous bytes of one query row.
//
// Work items are claimed dynamically (queue.cuh).  With 128-token blocks an item is one of the
// two 64-token kv tiles of a block, and each k2q entry supplies a whole q tile pair.  The last
// items of the claim order (one per two CTAs) are handed out as four claims each, one per
// quarter of their step lists (halves when there are fewer than 8 items per SM: the kernel's
// PARTS), so the grid ends on short claims; a part stores its fp32 dK, dV rows in a workspace
// slot of its own, and the postprocess adds the parts and writes bf16.
//
// Roles (448 threads):
//   warps 0-7  softmax: warps w and w+4 share TMEM lane quarter w (query rows 32w..32w+31 of the
//              pair) and split the 64 kv columns in halves.  Two phases per step: P from S as
//              soon as S is in TMEM (fp16, swizzled, into shared memory), then dS from dP.
//   warps 8-11 dQ drain + epilogue: thread d owns head-dim row d; stages dQ^T of each q tile in
//              an 8 KB per-warp box ([64 query rows x 32 head dims] fp32) and adds it into the
//              fp32 accumulator with one TMA bulk tensor reduction.  dK^T and dV^T are read out
//              of TMEM as soon as the item's last dK^T is done (before its last dQ^T is
//              drained) and written as bf16 dK, dV (zeros for padded rows; whole zero blocks
//              for unselected kv tiles), or, for a part of a split item, as fp32 rows.
//   warp 12    TMA producer and work claimer (K_j, V_j once per item, one copy each; Q and dO of
//              each pair into a 2-stage ring: one 16 KB copy per transposed q tile, one 32 KB
//              copy when the pair's tiles are adjacent); also allocates TMEM.
//   warp 13    UMMA issuer, warp-wide (all lanes poll, one elected lane issues).  Per step g the
//              tensor pipe runs dV^T(g), S(g+1), dK^T(g), dP(g+1), dQ^T(g): dV^T waits for P,
//              dK^T for dS, so the softmax of step g+1 overlaps dK^T, dP and dQ^T of step g, and
//              the drain of dQ^T(g) overlaps step g+1 in a second TMEM buffer.
// TMEM (512 columns): S [0,64), dP [64,128), dV^T [128,192), dK^T [192,256),
// dQ^T x2 [256,512).  Shared memory: K_j, V_j; a 2-stage Q/dO ring; P and dS (one buffer each:
// the tensor pipe runs in issue order, so S(g) completing means dV^T(g-1) has read P(g-1), and
// the softmax writes dS(g) only after dQ^T(g-1) has read dS(g-1), a barrier it waits on); dQ
// staging.

#include "ptx.cuh"
#include "queue.cuh"
#include "vsa_internal.cuh"

namespace vsa {

namespace {

constexpr int NUM_THREADS = 448;
constexpr int SOFTMAX_WARPS = 8;  // warps 0-7: lane quarter w % 4, column half w / 4
constexpr int DRAIN_WARP0 = 8;    // warps 8-11: dQ drain + epilogue
constexpr int TMA_WARP = 12;
constexpr int MMA_WARP = 13;

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr uint32_t SM_K = 0;                    // K_j: 2 chunks x [64 kv x 128 B]
constexpr uint32_t SM_V = 16384;                // V_j
constexpr uint32_t SM_Q = 32768;                // 2 stages x 2 chunks x [128 q x 128 B]
constexpr uint32_t SM_DO = SM_Q + 2 * 32768;    // 2 stages, same layout
constexpr uint32_t SM_P = SM_DO + 2 * 32768;    // [128 q x 128 B]
constexpr uint32_t SM_DS = SM_P + 16384;        // [128 q x 128 B]
constexpr uint32_t SM_STG = SM_DS + 16384;      // dQ staging: 4 warps x [64 q x 32 fp32]
constexpr uint32_t SM_BAR = SM_STG + 4 * 8192;  // mbarriers

enum Bar : uint32_t {
  KV_FULL = 0,
  KV_EMPTY,
  QDO_FULL0,
  QDO_FULL1,
  QDO_EMPTY0,
  QDO_EMPTY1,
  S_FULL,    // S of the step is in TMEM
  DP_FULL,   // dP of the step is in TMEM
  P_READY,   // the softmax warps have stored P of the step
  DS_READY,  // ... and dS
  DS_FREE,   // dQ^T of the previous step has read dS
  DQ_FULL0,
  DQ_FULL1,
  DQ_FREE0,
  DQ_FREE1,
  ACC_FULL,
  ACC_EMPTY,
  DRAIN,
  ITEM_FULL0,  // the work-item queue (queue.cuh)
  ITEM_EMPTY0 = ITEM_FULL0 + ITEM_SLOTS,
  NUM_BARS = ITEM_EMPTY0 + ITEM_SLOTS
};
// Every role takes every item from the queue: the UMMA thread, 8 softmax warps, 4 drain warps.
constexpr uint32_t ITEM_CONSUMERS = 1 + SOFTMAX_WARPS + 4;
constexpr uint32_t SM_TMEM_SLOT = SM_BAR + NUM_BARS * 8;
constexpr uint32_t SM_ABORT = SM_TMEM_SLOT + 4;
constexpr uint32_t SM_QUEUE = SM_ABORT + 4;  // int[ITEM_SLOTS]: work-item ids
constexpr uint32_t SM_USED = SM_QUEUE + 4 * ITEM_SLOTS;
constexpr uint32_t SMEM_BYTES = SM_USED + 1024;  // + alignment slack

static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t TM_S = 0, TM_DP = 64, TM_DVT = 128, TM_DKT = 192, TM_DQT = 256;  // dQ^T x2

constexpr uint32_t IDESC_SDP = idesc_f16_f32acc(128, 64, true, false);  // A = Q_p / dO_p, MN-major
constexpr uint32_t IDESC_DVK = idesc_f16_f32acc(128, 64, false, true);  // A = Q_p^T / dO_p^T
constexpr uint32_t IDESC_DQ = idesc_f16_f32acc(128, 128, true, false);

struct Params {
  const int32_t* k2q_idx;
  const int32_t* k2q_num;
  const int32_t* order;
  const int32_t* vbs;
  const float* lse;
  const float* delta;
  const uint32_t* absmax;  // per-head statistics (HeadStat)
  const uint32_t* tstat;   // per-kv-tile statistics (TileStat), [B * H * nb]
  float* dqacc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  uint32_t* err;
  int32_t* sched;  // work counter, zero at launch
  int S;
  int nb;     // 64-token tiles per sequence; work items are (b, h, kv tile)
  int nsel;   // sparse blocks per sequence (k2q rows per head)
  int tiles;  // 64-token tiles per sparse block: 1, or 2 for 128-token blocks
  int max_q;
  // The last `nsplit` items (claim positions split0 ..) are each taken as PARTS claims, one
  // per consecutive share of the item's step list, so that the grid's last claims are short.
  // Part x of split item s stores its dK, dV rows (fp32, scaled; zeros for masked rows and for a
  // part without steps) in slot s * PARTS + x of split_acc ([dV, dK][64 kv rows][128]), and the
  // item's first output row in split_row[s]; the postprocess adds the parts in a fixed order and
  // writes the bf16 rows.
  int split0, nsplit;
  float* split_acc;
  int32_t* split_row;
  int total;  // claim positions: split0 + PARTS * nsplit
  float sm_scale;
  uint64_t wait_ns;  // limit of each pipeline wait
};

// A work item: kv tile j of head bh.  Its k2q row `sel` lists selecting q blocks; each step
// processes a pair of 64-token q tiles: two consecutive list entries (64-token blocks; an odd
// tail repeats the last one), or the two tiles of one 128-token entry.
struct Item {
  int bh, j, sel, n;
  int first, np;  // this claim's steps: first .. first + np - 1 of the item's list
  int slot, part;  // split item and part, or -1 for a whole item
  const int32_t* list;
};

// PARTS: claims per split item (the kernel's template argument, bwd_split_plan).
template <int PARTS>
__device__ __forceinline__ Item decode_item(const Params& p, int u) {
  int w = u, part = -1, slot = -1;
  if (u >= p.split0) {  // one part of a split item
    slot = (u - p.split0) / PARTS;
    part = (u - p.split0) % PARTS;
    w = p.split0 + slot;
  }
  int half = 0, ws = w;
  if (p.tiles == 2) {
    half = w & 1;
    ws = w >> 1;
  }
  const int sel = p.order ? p.order[ws] : ws;
  Item it;
  it.bh = sel / p.nsel;
  it.j = (sel - it.bh * p.nsel) * p.tiles + half;
  it.sel = sel;
  const int n = p.k2q_num[sel];
  it.n = n < 0 ? 0 : (n > p.max_q ? p.max_q : n);
  const int np = p.tiles == 2 ? it.n : (it.n + 1) >> 1;
  // Part x of P takes steps [np x / P, np (x + 1) / P): shares differ by at most one, and a part
  // may have none when the list is short.
  it.first = part < 0 ? 0 : np * part / PARTS;
  it.np = part < 0 ? np : np * (part + 1) / PARTS - it.first;
  it.slot = slot;
  it.part = part;
  it.list = p.k2q_idx + static_cast<size_t>(sel) * p.max_q;
  return it;
}

// Entry x of the item's k2q list, or -1 for an id outside [0, nq): such a slot is skipped (its
// rows are masked and its dQ partial is not written), as an invalid q2k slot is.
__device__ __forceinline__ int q_block(const Item& it, int x, int nq) {
  const int i = it.list[x];
  return (i < 0 || i >= nq) ? -1 : i;
}

// The two 64-token q tiles of a step.  i0, i1 are always tiles of the head (loaded); v0, v1 say
// whether the rows of each take part: not for the repeat of the first tile at the odd tail of a
// 64-token list, nor for a skipped slot (its tile is loaded as tile 0 or as a repeat).
struct StepTiles {
  int i0, i1;
  bool v0, v1;
};

__device__ __forceinline__ StepTiles step_tiles(const Params& p, const Item& it, int pp) {
  const int ps = it.first + pp;
  StepTiles t;
  if (p.tiles == 2) {  // one 128-token entry: both tiles of its block, or neither
    const int i = q_block(it, ps, p.nsel);
    t.v0 = t.v1 = i >= 0;
    t.i0 = i >= 0 ? 2 * i : 0;
    t.i1 = t.i0 + 1;
    return t;
  }
  const int a = q_block(it, 2 * ps, p.nsel);
  const int b = 2 * ps + 1 < it.n ? q_block(it, 2 * ps + 1, p.nsel) : -1;
  t.v0 = a >= 0;
  t.v1 = b >= 0;
  t.i0 = a >= 0 ? a : 0;
  t.i1 = b >= 0 ? b : t.i0;
  return t;
}

__device__ __forceinline__ int clamp_vbs(int v) { return v < 0 ? 0 : (v > BLOCK ? BLOCK : v); }

// Scale exponents of an item: Q' = 2^-eq Q and dO' = 2^-eo dO (per head), K' = 2^-ek K and
// V' = 2^-ev V (per kv tile), dS' = 2^kap P (dP' - Delta') (per kv tile, ds_exponent).  Then
//   S'   = Q' K'^T   = 2^-(eq+ek) S            dP' = dO' V'^T = 2^-(eo+ev) dP
//   dV^T accumulates dO'^T (2^KP P)  = 2^(KP-eo) dV^T
//   dK^T accumulates Q'^T dS'        = 2^(kap-eq-eo-ev) dK^T / sm_scale
//   dQ^T partial     K'^T dS'^T      = 2^(kap-ek-eo-ev) dQ^T / sm_scale
// and the drain brings every dQ partial to 2^-eo dQ / sm_scale before adding it.
struct ItemScales {
  int eq, eo, ek, ev, kap;
};

__device__ __forceinline__ ItemScales item_scales(const Params& p, const Item& it) {
  const uint32_t* hs = p.absmax + it.bh * HEAD_STATS;
  const uint32_t* ts = p.tstat + (static_cast<size_t>(it.bh) * p.nb + it.j) * TILE_STATS;
  ItemScales e;
  e.eq = operand_exponent(hs[HS_Q]);
  e.eo = operand_exponent(hs[HS_DO]);
  e.ek = operand_exponent(ts[TS_K]);
  e.ev = operand_exponent(ts[TS_V]);
  e.kap = ds_exponent(bits_float(hs[HS_DO_NORM]), bits_float(ts[TS_V_NORM]),
                      bits_float(hs[HS_DELTA]), e.eo, e.ev);
  return e;
}

// One elected lane waits; the result is broadcast so the warp stays converged.
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

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int PARTS>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q2,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_do2,
                    const __grid_constant__ CUtensorMap tm_dq, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + SM_ABORT);
  volatile int* queue = reinterpret_cast<volatile int*>(gbase + SM_QUEUE);
  const uint32_t* tmem_slot = reinterpret_cast<const uint32_t*>(gbase + SM_TMEM_SLOT);
  auto bar = [&](uint32_t b) { return base + SM_BAR + 8u * b; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S, nq = p.nsel;

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(bar(KV_FULL), 1);
    mbar_init(bar(KV_EMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(QDO_FULL0 + s), 1);
      mbar_init(bar(QDO_EMPTY0 + s), 1);
      mbar_init(bar(DQ_FULL0 + s), 1);
      mbar_init(bar(DQ_FREE0 + s), 4);
    }
    mbar_init(bar(S_FULL), 1);
    mbar_init(bar(DP_FULL), 1);
    mbar_init(bar(P_READY), SOFTMAX_WARPS);
    mbar_init(bar(DS_READY), SOFTMAX_WARPS);
    mbar_init(bar(ACC_FULL), 1);
    mbar_init(bar(ACC_EMPTY), 4);
    mbar_init(bar(DRAIN), 1);
    mbar_init(bar(DS_FREE), 1);
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
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_do2);
    tma_prefetch_desc(&tm_dq);
  }
  grid_dependency_wait();  // the preprocess's outputs (programmatic dependent launch)
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == TMA_WARP) {
    // ------------------------------------------------------------------ TMA producer
    // The whole warp runs this role; lane 0 claims items and registers the expected bytes, and
    // each tile of a load goes out from a lane of its own (a thread's bulk copies are processed
    // one after another, so spreading them over lanes keeps them in flight together).
    uint32_t g = 0;      // global pair-step counter
    uint32_t itc = 0;    // items with a non-empty list
    uint32_t kv_loads = 0;
    int64_t last_g[2] = {-1, -1};
    bool ok = true;
    // Items are handed out dynamically: the next one is claimed from the global counter once
    // the loads of the current one are issued, so the CTAs that finish early take more.
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
      const Item it = decode_item<PARTS>(p, w);
      uint32_t bad = 0;
      if (lane == 0 && p.k2q_num[it.sel] != it.n) bad |= VSA_DEVERR_K2Q_COUNT;
      for (int x = lane; x < it.n; x += 32) {
        const int i = it.list[x];
        if (i < 0 || i >= nq) bad |= VSA_DEVERR_K2Q_ID;
      }
      bad = __reduce_or_sync(0xffffffffu, bad);
      if (bad && lane == 0) atomicOr(p.err, bad);
      if (it.np == 0) continue;  // nothing to compute (an unselected block, or an empty part)
      if (!mbar_wait_warp(bar(KV_EMPTY), (itc & 1u) ^ 1u, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      const int row_kv = it.bh * S + it.j * BLOCK;
      if (lane == 0) mbar_arrive_expect_tx(bar(KV_FULL), 32768);
      __syncwarp();
      if (lane < 2)  // lane 0: K, lane 1: V, both column halves of the tile in one copy each
        tma_load_3d(base + (lane == 0 ? SM_K : SM_V), lane == 0 ? &tm_k : &tm_v, bar(KV_FULL),
                    0, row_kv, 0);
      ++kv_loads;
      const int np = it.np;
      for (int pp = 0; pp < np; ++pp, ++g) {
        const uint32_t s = g & 1u;
        if (!mbar_wait_warp(bar(QDO_EMPTY0 + s), ((g >> 1) & 1u) ^ 1u, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        const StepTiles st = step_tiles(p, it, pp);
        const int i0 = st.i0, i1 = st.i1;
        if (lane == 0) mbar_arrive_expect_tx(bar(QDO_FULL0 + s), 65536);
        __syncwarp();
        // Q and dO are stored tile-transposed: 64-token tile i of the head is 128 rows (head
        // dims) of 64 queries from row (bh * S / 64 + i) * 128 on, 16 KB.  Stage layout: tile i0
        // at byte 0, tile i1 at 16384, for Q and for dO.
        const int tile0 = it.bh * (S / BLOCK);
        const int t0 = (tile0 + i0) * HEAD_DIM, t1 = (tile0 + i1) * HEAD_DIM;
        if (i1 == i0 + 1) {  // adjacent q tiles (always with 128-token blocks): one 32 KB copy
          if (lane < 2)
            tma_load_2d(base + (lane == 0 ? SM_Q : SM_DO) + s * 32768u,
                        lane == 0 ? &tm_q2 : &tm_do2, bar(QDO_FULL0 + s), 0, t0);
        } else if (lane < 4) {  // lanes 0, 1: Q tiles i0, i1; lanes 2, 3: dO tiles
          tma_load_2d(base + ((lane < 2) ? SM_Q : SM_DO) + s * 32768u + (lane & 1) * 16384u,
                      (lane < 2) ? &tm_q : &tm_do, bar(QDO_FULL0 + s), 0, (lane & 1) ? t1 : t0);
        }
        last_g[s] = g;
      }
      if (!ok) break;
      ++itc;
    }
    if (!ok && lane == 0) {
      raise_abort(abort, p.err);
      // Let the copies already issued land before the CTA's shared memory goes away.
      volatile int never = 0;
      if (kv_loads > 0)
        mbar_wait_bounded(bar(KV_FULL), (kv_loads - 1) & 1u, &never, DRAIN_LIMIT_NS);
      for (int s = 0; s < 2; ++s)
        if (last_g[s] >= 0)
          mbar_wait_bounded(bar(QDO_FULL0 + s), (static_cast<uint32_t>(last_g[s]) >> 1) & 1u,
                            &never, DRAIN_LIMIT_NS);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ UMMA issuer
    // The whole warp runs this role in lockstep; every lane polls the barriers and one elected
    // lane issues each UMMA and commit.
    uint32_t g = 0, itc = 0;
    bool ok = true, issued = false;
    // Operand descriptors, built once; each UMMA only adds a constant byte offset to them.
    //   K-major: 32 B per k-step inside a 128-B row, 64-element chunks (K/V column halves, or
    //   the two transposed q tiles of Q_p^T / dO_p^T) 8 or 16 KB apart.
    //   MN-major: 2048 B (16 rows) per k-step; Q_p and dO_p as A of S and dP take their two
    //   64-query chunks from the two transposed tiles (LBO 16 KB).
    const uint64_t k_kmaj = sdesc_sw128(base + SM_K, 16, 1024);
    const uint64_t v_kmaj = sdesc_sw128(base + SM_V, 16, 1024);
    const uint64_t k_mn = sdesc_sw128(base + SM_K, 8192, 1024);
    const uint64_t p_mn = sdesc_sw128(base + SM_P, 16384, 1024);
    const uint64_t q_kmaj = sdesc_sw128(base + SM_Q, 16, 1024);
    const uint64_t do_kmaj = sdesc_sw128(base + SM_DO, 16, 1024);
    const uint64_t q_mn = sdesc_sw128(base + SM_Q, 16384, 1024);
    const uint64_t do_mn = sdesc_sw128(base + SM_DO, 16384, 1024);
    const uint64_t ds_mn = sdesc_sw128(base + SM_DS, 16384, 1024);
    const uint64_t ds_kmaj = sdesc_sw128(base + SM_DS, 16, 1024);
    const uint32_t t_s = tmem + TM_S, t_dp = tmem + TM_DP, t_dv = tmem + TM_DVT,
                   t_dk = tmem + TM_DKT;
    // S = Q_p K_j^T of step gs (stage gs & 1).  A = Q_p read MN-major from the two transposed
    // q tiles (64 queries per 128-byte row, one tile per 64-query chunk), 16 head dims (rows)
    // per k-step.
    auto issue_s = [&](uint32_t gs) {
      const uint64_t qa = sdesc_advance(q_mn, (gs & 1u) * 32768u);
      umma_ss_elect<false>(t_s, qa, k_kmaj, IDESC_SDP);
#pragma unroll
      for (int kk = 1; kk < 8; ++kk)
        umma_ss_elect<true>(t_s, sdesc_advance(qa, kk * 2048u),
                            sdesc_advance(k_kmaj, (kk >> 2) * 8192u + (kk & 3) * 32u), IDESC_SDP);
      umma_commit_elect(bar(S_FULL));
    };
    // dP = dO_p V_j^T of step gs.
    auto issue_dp = [&](uint32_t gs) {
      const uint64_t da = sdesc_advance(do_mn, (gs & 1u) * 32768u);
      umma_ss_elect<false>(t_dp, da, v_kmaj, IDESC_SDP);
#pragma unroll
      for (int kk = 1; kk < 8; ++kk)
        umma_ss_elect<true>(t_dp, sdesc_advance(da, kk * 2048u),
                            sdesc_advance(v_kmaj, (kk >> 2) * 8192u + (kk & 3) * 32u), IDESC_SDP);
      umma_commit_elect(bar(DP_FULL));
    };
    // dQ^T = K_j^T dS^T of step gs into TMEM buffer gs & 1; then the dS buffer is free.
    auto issue_dq = [&](uint32_t gs) -> bool {
      const uint32_t b = gs & 1u;
      if (!mbar_wait_warp(bar(DQ_FREE0 + b), ((gs >> 1) & 1u) ^ 1u, abort, p.wait_ns))
        return false;
      tc_fence_after_sync();
      const uint64_t dsb = ds_kmaj;
      const uint32_t t_dq = tmem + TM_DQT + b * 128u;
      umma_ss_elect<false>(t_dq, k_mn, dsb, IDESC_DQ);
#pragma unroll
      for (int kk = 1; kk < 4; ++kk)
        umma_ss_elect<true>(t_dq, sdesc_advance(k_mn, kk * 2048u), sdesc_advance(dsb, kk * 32u),
                         IDESC_DQ);
      umma_commit_elect(bar(DQ_FULL0 + b));
      umma_commit_elect(bar(DS_FREE));
      return true;
    };
    // dV^T += dO_p^T P of step gs; the first step of an item overwrites.  A = dO_p^T read K-major
    // from the transposed tiles: 128 head-dim rows, 16 queries per k-step (tile kk >> 2).
    auto issue_dv = [&](uint32_t gs, bool first) {
      const uint64_t da = sdesc_advance(do_kmaj, (gs & 1u) * 32768u);
      if (first)
        umma_ss_elect<false>(t_dv, da, p_mn, IDESC_DVK);
      else
        umma_ss_elect<true>(t_dv, da, p_mn, IDESC_DVK);
#pragma unroll
      for (int kk = 1; kk < 8; ++kk)
        umma_ss_elect<true>(t_dv, sdesc_advance(da, (kk >> 2) * 16384u + (kk & 3) * 32u),
                            sdesc_advance(p_mn, kk * 2048u), IDESC_DVK);
    };
    // dK^T += Q_p^T dS of step gs; the first step of an item overwrites.
    auto issue_dk = [&](uint32_t gs, bool first) {
      const uint64_t qa = sdesc_advance(q_kmaj, (gs & 1u) * 32768u);
      const uint64_t dsb = ds_mn;
      if (first)
        umma_ss_elect<false>(t_dk, qa, dsb, IDESC_DVK);
      else
        umma_ss_elect<true>(t_dk, qa, dsb, IDESC_DVK);
#pragma unroll
      for (int kk = 1; kk < 8; ++kk)
        umma_ss_elect<true>(t_dk, sdesc_advance(qa, (kk >> 2) * 16384u + (kk & 3) * 32u),
                            sdesc_advance(dsb, kk * 2048u), IDESC_DVK);
    };
    for (uint32_t k = 0;; ++k) {
      int w;
      if (!warp_take_item(bar(ITEM_FULL0), bar(ITEM_EMPTY0), queue, k, abort, p.wait_ns, lane, &w)) {
        ok = false;
        break;
      }
      if (w >= p.total) break;
      const Item it = decode_item<PARTS>(p, w);
      if (it.np == 0) continue;  // nothing to compute (an unselected block, or an empty part)
      const int np = it.np;
      if (!mbar_wait_warp(bar(KV_FULL), itc & 1u, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      // The tensor pipe runs, per step g of the item:  dV^T(g)  S(g+1)  dK^T(g)  dP(g+1)  dQ^T(g),
      // so the softmax of step g+1 (which needs S(g+1), then dP(g+1)) overlaps dK^T, dP and
      // dQ^T of step g.  S and dP of the item's first step go in up front.
      const uint32_t g0 = g;
      if (!mbar_wait_warp(bar(QDO_FULL0 + (g0 & 1u)), (g0 >> 1) & 1u, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      issue_s(g0);
      issue_dp(g0);
      issued = true;
      for (int pp = 0; pp < np; ++pp, ++g) {
        const bool more = pp + 1 < np;
        // The softmax read S(g) before P_READY(g); P(g) is in shared memory.
        if (!mbar_wait_warp(bar(P_READY), g & 1u, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        if (pp == 0 &&
            !mbar_wait_warp(bar(ACC_EMPTY), (itc & 1u) ^ 1u, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_dv(g, pp == 0);
        if (more) {
          // S(g+1) overwrites S(g), already read.  P(g+1) is written by the softmax only once
          // S(g+1) is done, which in the tensor pipe follows dV^T(g).
          if (!mbar_wait_warp(bar(QDO_FULL0 + ((g + 1) & 1u)), ((g + 1) >> 1) & 1u, abort,
                              p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_s(g + 1);
        }
        // The softmax read dP(g) before DS_READY(g); dS(g) is in shared memory.
        if (!mbar_wait_warp(bar(DS_READY), g & 1u, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_dk(g, pp == 0);
        if (more) {
          umma_commit_elect(bar(QDO_EMPTY0 + (g & 1u)));  // Q_p, dO_p of step g are no longer read
          issue_dp(g + 1);
        } else {
          // dV^T and dK^T of the item are complete with dK^T(g): the drain warps read them out
          // while dQ^T(g) runs, and the next item's dV^T can start that much earlier.
          umma_commit_elect(bar(ACC_FULL));
        }
        if (!issue_dq(g)) {
          ok = false;
          break;
        }
        if (!more) umma_commit_elect(bar(QDO_EMPTY0 + (g & 1u)));
      }
      if (!ok) break;
      umma_commit_elect(bar(KV_EMPTY));
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
  } else if (warp < SOFTMAX_WARPS) {
    // ------------------------------------------------------------------ softmax / dS
    const int quarter = warp & 3, h = warp >> 2;  // TMEM lane quarter; S/dP column half
    const int r = quarter * 32 + lane;            // query row of the pair == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t g = 0;
    const uint32_t sw = static_cast<uint32_t>(r & 7);
    for (uint32_t k = 0;; ++k) {
      int w;
      if (!warp_take_item(bar(ITEM_FULL0), bar(ITEM_EMPTY0), queue, k, abort, p.wait_ns, lane, &w)) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      if (w >= p.total) break;
      const Item it = decode_item<PARTS>(p, w);
      if (it.np == 0) continue;  // nothing to compute (an unselected block, or an empty part)
      const int vb = clamp_vbs(p.vbs[it.j]);
      const ItemScales es = item_scales(p, it);
      const float c1 = p.sm_scale * LOG2E_F * exp2i(es.eq + es.ek);
      // dS' = P 2^KP (dP' m - Delta' m) with m = 2^(kap - KP): Delta' in the units of dP'.
      const float dsm = exp2i(es.kap - KP);
      const float dscale = exp2i(-(es.eo + es.ev)) * dsm;
      const int np = it.np;
      bool ok = true;
      for (int pp = 0; pp < np; ++pp, ++g) {
        const StepTiles st = step_tiles(p, it, pp);
        const bool valid = (r < 64) ? st.v0 : st.v1;
        const int qb = (r >= 64) ? st.i1 : st.i0;
        const size_t grow = static_cast<size_t>(it.bh) * S + static_cast<size_t>(qb) * BLOCK + (r & 63);
        const float nlse = static_cast<float>(KP) - p.lse[grow];
        const float dl = p.delta[grow] * dscale;  // Delta' m
        const bool full = valid && (vb == BLOCK);
        // Phase 1: P from S, as soon as S is in TMEM (dP and dQ^T(g-1) are still running).
        if (!warp_wait(bar(S_FULL), g & 1u, abort, p.wait_ns, lane)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t prow = base + SM_P + static_cast<uint32_t>(r) * 128u;
        const uint32_t dsrow = base + SM_DS + static_cast<uint32_t>(r) * 128u;
        float pv[32];  // P of this warp's 32 columns (0 where masked), kept for dS
        {
          uint32_t sv[32];
          tmem_ld_32x32b_x32(tmem + lane_off + TM_S + h * 32u, sv);
          tmem_wait_ld();
          uint32_t pk[16];
          if (full) {  // every column visible: no masking
#pragma unroll
            for (int c = 0; c < 32; ++c) pv[c] = ex2(fmaf(__uint_as_float(sv[c]), c1, nlse));
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              pv[c] = (valid && h * 32 + c < vb) ? ex2(fmaf(__uint_as_float(sv[c]), c1, nlse)) : 0.f;
          }
#pragma unroll
          for (int c = 0; c < 32; c += 2) pk[c >> 1] = pack_half2(pv[c], pv[c + 1]);
          // P's buffer was last read by dV^T(g-1), which precedes S(g) in the tensor pipe.
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint32_t phys = ((static_cast<uint32_t>(h * 4 + ch)) ^ sw) * 16u;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + phys),
                         "r"(pk[4 * ch]), "r"(pk[4 * ch + 1]), "r"(pk[4 * ch + 2]),
                         "r"(pk[4 * ch + 3])
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P_READY));
        // Phase 2: dS = P (dP - Delta) while dV^T(g) runs.
        if (!warp_wait(bar(DP_FULL), g & 1u, abort, p.wait_ns, lane)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        {
          uint32_t dpv[32];
          tmem_ld_32x32b_x32(tmem + lane_off + TM_DP + h * 32u, dpv);
          tmem_wait_ld();
          uint32_t dk[16];  // dS', fp16 pairs (masked columns have P = 0, so dS' = 0 exactly)
#pragma unroll
          for (int c = 0; c < 32; c += 2)
            dk[c >> 1] = pack_half2(pv[c] * fmaf(__uint_as_float(dpv[c]), dsm, -dl),
                                    pv[c + 1] * fmaf(__uint_as_float(dpv[c + 1]), dsm, -dl));
          // The buffer's previous contents (step g-1) must have been consumed by dQ^T(g-1).
          if (!warp_wait(bar(DS_FREE), (g & 1u) ^ 1u, abort, p.wait_ns, lane)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint32_t phys = ((static_cast<uint32_t>(h * 4 + ch)) ^ sw) * 16u;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dsrow + phys),
                         "r"(dk[4 * ch]), "r"(dk[4 * ch + 1]), "r"(dk[4 * ch + 2]),
                         "r"(dk[4 * ch + 3])
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(DS_READY));
      }
      if (!ok) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
    }
  } else {
    // ------------------------------------------------------------------ dQ drain + epilogue
    const int wq = warp - DRAIN_WARP0;  // lane quarter (DRAIN_WARP0 % 4 == 0)
    const int d = wq * 32 + lane;  // head-dim row == TMEM lane (dK/dV epilogue column)
    const uint32_t stg = base + SM_STG + static_cast<uint32_t>(wq) * 8192u;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    uint32_t g = 0, itc = 0;
    for (uint32_t k = 0;; ++k) {
      int w;
      if (!warp_take_item(bar(ITEM_FULL0), bar(ITEM_EMPTY0), queue, k, abort, p.wait_ns, lane, &w)) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      if (w >= p.total) break;
      const Item it = decode_item<PARTS>(p, w);
      const size_t row_kv = static_cast<size_t>(it.bh) * S + static_cast<size_t>(it.j) * BLOCK;
      __nv_bfloat16* dk_out = p.dk + row_kv * HEAD_DIM + d;
      __nv_bfloat16* dv_out = p.dv + row_kv * HEAD_DIM + d;
      if (it.slot < 0 && it.n == 0) {
        // No q block selects this kv block: exact-zero dK/dV rows.
        const __nv_bfloat16 z = __float2bfloat16_rn(0.f);
        for (int t = 0; t < BLOCK; ++t) {
          dk_out[t * HEAD_DIM] = z;
          dv_out[t * HEAD_DIM] = z;
        }
        continue;
      }
      const ItemScales es = item_scales(p, it);
      const float sv_scale = exp2i(es.eo - KP);
      const float sk_scale =
          p.sm_scale * exp2i(es.eq + es.eo) * exp2i(clamp_exponent(es.ev - es.kap, 126));
      // dQ^T partial -> 2^-eo dQ^T / sm_scale, the accumulator's scale for every item.
      const float dq_scale = exp2i(clamp_exponent(es.ek + es.ev - es.kap, 126));
      const int vb = clamp_vbs(p.vbs[it.j]);
      const int np = it.np;
      bool ok = true;
      // A split part's rows of this warp's 32 head dims: [dV, dK][64 kv rows][128] fp32.
      float* acc = nullptr;
      if (it.slot >= 0)
        acc = p.split_acc +
              static_cast<size_t>(it.slot * PARTS + it.part) * (2 * BLOCK * HEAD_DIM) + d;
      // The item's dV^T and dK^T, complete once its last dK^T is (before its last dQ^T): read
      // out before the last step's dQ^T is drained, so that the next item's dV^T can start.
      auto read_acc = [&]() -> bool {
        if (!warp_wait(bar(ACC_FULL), itc & 1u, abort, p.wait_ns, lane)) return false;
        tc_fence_after_sync();
        // dV^T and dK^T rows (head dim d, kv rows 0..63) in 32-column chunks; masked kv rows get
        // an explicit +0.0.  A split part stores its scaled fp32 rows in its own slot instead.
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const bool is_dk = c >= 2;
          const uint32_t col = (is_dk ? TM_DKT : TM_DVT) + (c & 1) * 32u;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + lane_off + col, v);
          tmem_wait_ld();
          if (c == 3) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(ACC_EMPTY));
          }
          const float sc = is_dk ? sk_scale : sv_scale;
          if (acc) {
            float* a = acc + ((is_dk ? BLOCK : 0) + (c & 1) * 32) * HEAD_DIM;
#pragma unroll
            for (int t = 0; t < 32; ++t)
              a[t * HEAD_DIM] = (c & 1) * 32 + t < vb ? __uint_as_float(v[t]) * sc : 0.f;
          } else {
            __nv_bfloat16* out = (is_dk ? dk_out : dv_out) + (c & 1) * 32 * HEAD_DIM;
#pragma unroll
            for (int t = 0; t < 32; ++t)
              out[t * HEAD_DIM] =
                  __float2bfloat16_rn((c & 1) * 32 + t < vb ? __uint_as_float(v[t]) * sc : 0.f);
          }
        }
        ++itc;
        return true;
      };
      for (int pp = 0; pp < np; ++pp, ++g) {
        if (pp == np - 1 && !read_acc()) {
          ok = false;
          break;
        }
        const StepTiles st = step_tiles(p, it, pp);
        const uint32_t buf = g & 1u;
        if (!warp_wait(bar(DQ_FULL0 + buf), (g >> 1) & 1u, abort, p.wait_ns, lane)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        // Four 32-column chunks of dQ^T: chunks 0, 1 are rows 0-31, 32-63 of q block i0,
        // chunks 2, 3 those of i1.  Each goes TMEM -> registers -> this warp's staging box
        // (row q: 32 fp32 of head dims 32*wq .. 32*wq+31, so the 32 lanes' stores of one row
        // are 128 contiguous bytes).  A q block's two chunks fill the box (64 rows, 8 KB), which
        // one TMA reduce adds into the accumulator: a thread's bulk requests are processed one
        // after another, so few large requests move more than many small ones.  The load of
        // chunk c+1 is in flight while chunk c is staged.
        // A tile whose rows do not take part (odd tail, skipped slot) has no partial to add.
        auto stage = [&](const uint32_t* v, int c) {
          if (!(c < 2 ? st.v0 : st.v1)) return;
          const uint32_t rows = stg + static_cast<uint32_t>(c & 1) * 4096u;
          if ((c & 1) == 0) {
            if (lane == 0) bulk_wait_read<0>();  // the previous reduce has read the box
            __syncwarp();
          }
#pragma unroll
          for (int q = 0; q < 32; ++q)
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(rows + static_cast<uint32_t>(q) * 128u +
                                                          static_cast<uint32_t>(lane) * 4u),
                         "f"(__uint_as_float(v[q]) * dq_scale)
                         : "memory");
          if (c & 1) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&tm_dq, stg, wq * 32,
                                it.bh * S + ((c < 2) ? st.i0 : st.i1) * BLOCK);
              bulk_commit_group();
            }
          }
        };
        const uint32_t tq = tmem + lane_off + TM_DQT + buf * 128u;
        uint32_t va[32], vb[32];
        tmem_ld_32x32b_x32(tq, va);
        tmem_wait_ld_regs(va);
        tmem_ld_32x32b_x32(tq + 32u, vb);
        stage(va, 0);
        tmem_wait_ld_regs(vb);
        tmem_ld_32x32b_x32(tq + 64u, va);
        stage(vb, 1);
        tmem_wait_ld_regs(va);
        tmem_ld_32x32b_x32(tq + 96u, vb);
        stage(va, 2);
        tmem_wait_ld_regs(vb);
        // The TMEM buffer is free once all four chunks are in registers.
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(DQ_FREE0 + buf));
        stage(vb, 3);
      }
      if (!ok) {
        if (lane == 0) raise_abort(abort, p.err);
        break;
      }
      if (acc && np == 0) {  // a part without steps contributes zeros
        for (int t = 0; t < 2 * BLOCK; ++t) acc[t * HEAD_DIM] = 0.f;
      }
      if (acc && wq == 0 && lane == 0) p.split_row[it.slot] = static_cast<int32_t>(row_kv);
    }
    // Every reduction this warp issued has landed before the CTA retires.
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == TMA_WARP) tmem_dealloc(tmem, 512);
}

}  // namespace

SplitPlan bwd_split_plan(int items) {
  // SPLIT_CLAIMS split claims per CTA on average: enough short claims at the end of the grid
  // for the CTAs that finish their whole items early to even out the finishing times, as far as
  // the workspace's slots go.  With fewer than 8 items per SM (about 8 steps each at 4k tokens,
  // 25 %) a quarter of an item costs about as much in its item boundary as it computes, and
  // halves measured faster (71.7 against 75.8 µs at 4k; at 32k halves were 0.5 % slower).
  const int sms = device_sm_count();
  const int grid = items < sms ? items : sms;
  SplitPlan sp;
  sp.parts = static_cast<long>(items) < 8L * sms ? 2 : SPLIT_PARTS;
  const int want = SPLIT_CLAIMS * grid / sp.parts > 0 ? SPLIT_CLAIMS * grid / sp.parts : 1;
  const int cap = static_cast<int>(split_slots(items) / sp.parts);
  sp.nsplit = want < cap ? want : cap;
  return sp;
}

cudaError_t launch_bwd_main(const BwdMainArgs& a, cudaStream_t stream) {
  const long rows = static_cast<long>(a.B) * a.H * a.S;
  // Q and dO (tile-transposed): one tile (128 rows of 64) or two adjacent tiles per box; K and
  // V: one 64-row two-half box per tile.
  CUtensorMap tq, tq2, tk, tv, tdo, tdo2, tdq;
  cudaError_t e;
  if ((e = make_tmap_rows128_f32(&tdq, a.dqacc, rows)) != cudaSuccess) return e;
  if ((e = make_tmap_tiles_t(&tq, a.q16, rows, 1)) != cudaSuccess) return e;
  if ((e = make_tmap_tiles_t(&tdo, a.do16, rows, 1)) != cudaSuccess) return e;
  if ((e = make_tmap_tiles_t(&tq2, a.q16, rows, 2)) != cudaSuccess) return e;
  if ((e = make_tmap_tiles_t(&tdo2, a.do16, rows, 2)) != cudaSuccess) return e;
  if ((e = make_tmap_rows128_f16_halves(&tk, a.k16, rows, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_rows128_f16_halves(&tv, a.v16, rows, 64)) != cudaSuccess) return e;
  const int items = a.B * a.H * a.nb;
  const SplitPlan sp = bwd_split_plan(items);
  auto kernel = sp.parts == 2 ? bwd_main_kernel<2> : bwd_main_kernel<SPLIT_PARTS>;
  static std::atomic<uint64_t> smem_set2{0}, smem_set4{0};
  if ((e = ensure_smem_limit(kernel, static_cast<int>(SMEM_BYTES),
                             sp.parts == 2 ? smem_set2 : smem_set4)) != cudaSuccess)
    return e;
  Params p{};
  p.k2q_idx = a.k2q_idx;
  p.k2q_num = a.k2q_num;
  p.order = a.order;
  p.vbs = a.vbs;
  p.lse = a.lse;
  p.delta = a.delta;
  p.absmax = a.absmax;
  p.tstat = a.tstat;
  p.dqacc = a.dqacc;
  p.dk = a.dk;
  p.dv = a.dv;
  p.err = a.err;
  p.sched = a.sched;
  p.S = a.S;
  p.nb = a.nb;
  p.nsel = a.nsel;
  p.tiles = a.tiles;
  p.max_q = a.max_q;
  p.sm_scale = a.sm_scale;
  p.wait_ns = a.wait_ns;
  const int sms = device_sm_count();
  const int grid = items < sms ? items : sms;
  p.nsplit = sp.nsplit;
  p.split0 = items - p.nsplit;
  p.total = items + (sp.parts - 1) * p.nsplit;
  p.split_acc = a.split_acc;
  p.split_row = a.split_row;
  return launch_dependent(kernel, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, stream, tq, tq2, tk,
                          tv, tdo, tdo2, tdq, p);
}

}  // namespace vsa
