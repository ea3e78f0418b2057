// api.cu -- the extern "C" entry points declared in include/vsa.h: argument checks, workspace
// carving and the stream-ordered launch sequence of each operation.  Follows the host surface of
// FastVideo's backward (compare main...vsa_bwd_fix, block_sparse_bwd_launch_sm100a.cuh:
// block_sparse_bwd_supported returns an error for bad configurations; the launch chains
// preprocess -> order -> main -> postprocess on one stream without a host sync; here the order
// is computed inside the preprocess) and the caller-
// workspace contract of cudnn-frontend PR #926's follow-up (no allocation on the hot path).
#include <climits>
#include <cmath>

#include "vsa_internal.cuh"

namespace vsa {

namespace {
std::atomic<uint64_t> g_wait_limit_ns{DEFAULT_WAIT_LIMIT_NS};
}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

uint64_t set_wait_limit_ns(uint64_t ns) {
  return g_wait_limit_ns.exchange(ns == 0 ? DEFAULT_WAIT_LIMIT_NS : ns);
}

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int sms = 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 1;
  if (dev >= 0 && dev < 64) cached[dev] = sms;
  return sms;
}

bool use_work_order(int BH, int S) {
  const long tiles = S / BLOCK;
  return tiles >= ORDER_MIN_KV_TILES || BH * tiles < 8L * device_sm_count();
}

}  // namespace vsa

namespace {

thread_local int g_last_cuda_error = 0;

vsa_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return VSA_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape rules: B, H >= 1; head_dim 128; block 64 or 128 (0 read as 64); S a positive multiple of
// the block; B*H*S rows addressable with 32-bit TMA coordinates.  *nb counts sparse blocks of
// *blk tokens.  The kernels work on 64-token tiles: a 128-token block is two of them with the
// same selection.
vsa_status check_shape(const vsa_shape& s, int* nb, int* blk = nullptr) {
  if (s.batch < 1 || s.heads < 1 || s.seqlen < 1) return VSA_ERR_INVALID_ARG;
  if (s.head_dim != vsa::HEAD_DIM) return VSA_ERR_UNSUPPORTED;
  const int b = s.block == 0 ? vsa::BLOCK : s.block;
  if (b != vsa::BLOCK && b != 2 * vsa::BLOCK) return VSA_ERR_UNSUPPORTED;
  if (s.seqlen % b != 0) return VSA_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(s.batch) * s.heads * s.seqlen;
  if (rows > INT_MAX / 2) return VSA_ERR_UNSUPPORTED;
  // Some grids put B * H on their second dimension (at most 65535 blocks).
  if (static_cast<long long>(s.batch) * s.heads > 65535) return VSA_ERR_UNSUPPORTED;
  *nb = s.seqlen / b;
  if (blk) *blk = b;
  return VSA_OK;
}

// The kernels are built for sm_103a only.
vsa_status check_device() {
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return cuda_fail(e);
  return (major == 10 && minor == 3) ? VSA_OK : VSA_ERR_UNSUPPORTED;
}

cudaError_t record(void* event, cudaStream_t s) {
  return event ? cudaEventRecord(static_cast<cudaEvent_t>(event), s) : cudaSuccess;
}

template <typename T>
T* ws_at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

}  // namespace

namespace vsa {

vsa_status record_cuda_failure(cudaError_t e) { return cuda_fail(e); }

}  // namespace vsa

extern "C" {

const char* vsa_status_string(vsa_status status) {
  switch (status) {
    case VSA_OK:
      return "VSA_OK";
    case VSA_ERR_INVALID_ARG:
      return "VSA_ERR_INVALID_ARG";
    case VSA_ERR_UNSUPPORTED:
      return "VSA_ERR_UNSUPPORTED";
    case VSA_ERR_WORKSPACE:
      return "VSA_ERR_WORKSPACE";
    case VSA_ERR_CUDA:
      return "VSA_ERR_CUDA";
  }
  return "VSA_ERR_UNKNOWN";
}

int vsa_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t vsa_set_wait_limit_ns(uint64_t limit_ns) { return vsa::set_wait_limit_ns(limit_ns); }

vsa_status vsa_invert_indices(const int32_t* q2k_idx, const int32_t* q2k_num, int32_t topk,
                              vsa_shape shape, int32_t* k2q_idx, int32_t* k2q_num,
                              uint32_t* dev_err, void* stream) {
  int nb = 0;
  vsa_status st = check_shape(shape, &nb);
  if (st != VSA_OK) return st;
  if (topk < 1 || !q2k_idx || !q2k_num || !k2q_idx || !k2q_num) return VSA_ERR_INVALID_ARG;
  if (!aligned(q2k_idx, 4) || !aligned(q2k_num, 4) || !aligned(k2q_idx, 4) || !aligned(k2q_num, 4) ||
      !aligned(dev_err, 4))
    return VSA_ERR_INVALID_ARG;
  if ((st = check_device()) != VSA_OK) return st;
  const cudaError_t e =
      vsa::launch_invert(q2k_idx, q2k_num, topk, shape.batch * shape.heads, nb, k2q_idx, k2q_num,
                         dev_err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VSA_OK : cuda_fail(e);
}

size_t vsa_fwd_workspace_bytes(vsa_shape shape) {
  int nb = 0;
  if (check_shape(shape, &nb) != VSA_OK) return 0;
  return vsa::fwd_layout(shape.batch, shape.heads, shape.seqlen).total;
}

size_t vsa_bwd_workspace_bytes(vsa_shape shape) {
  int nb = 0;
  if (check_shape(shape, &nb) != VSA_OK) return 0;
  return vsa::bwd_layout(shape.batch, shape.heads, shape.seqlen).total;
}

vsa_status vsa_fwd(const void* q, const void* k, const void* v, const int32_t* q2k_idx,
                   const int32_t* q2k_num, int32_t topk, const int32_t* vbs, float sm_scale,
                   vsa_shape shape, void* o, float* lse, void* workspace, size_t workspace_bytes,
                   void* stream) {
  int nb = 0, blk = 0;
  vsa_status st = check_shape(shape, &nb, &blk);
  if (st != VSA_OK) return st;
  if (!q || !k || !v || !q2k_idx || !q2k_num || !vbs || !o || !lse) return VSA_ERR_INVALID_ARG;
  if (topk < 1 || !std::isfinite(sm_scale)) return VSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(q2k_idx, 4) || !aligned(q2k_num, 4) || !aligned(vbs, 4))
    return VSA_ERR_INVALID_ARG;
  const vsa::FwdLayout L = vsa::fwd_layout(shape.batch, shape.heads, shape.seqlen);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return VSA_ERR_WORKSPACE;
  if ((st = check_device()) != VSA_OK) return st;

  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = shape.batch * shape.heads, S = shape.seqlen;
  uint32_t* err = ws_at<uint32_t>(workspace, L.err);
  uint32_t* absmax = ws_at<uint32_t>(workspace, L.absmax);
  uint32_t* bitmap = ws_at<uint32_t>(workspace, L.bitmap);
  int32_t* vbs64 = ws_at<int32_t>(workspace, L.vbs64);
  __half* v16 = ws_at<__half>(workspace, L.v16);
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);

  cudaError_t e = vsa::launch_zero(workspace, L.v16, s);  // header, maxima, bitmap
  if (e != cudaSuccess) return cuda_fail(e);
  // S = Q K^T takes the bf16 Q and K as given; only V needs the scaled fp16 copy that P.V (fp16
  // P) takes, so only V's maximum is scanned.
  vsa::PreExtras x{};
  x.vbs = vbs;
  x.nb = nb;
  x.tiles = blk / vsa::BLOCK;
  x.vbs64 = vbs64;
  x.err = err;
  x.tstat = nullptr;
  x.k16 = x.v16 = nullptr;
  x.k2q_num = nullptr;
  x.order = nullptr;
  if ((e = vsa::launch_absmax_delta(nullptr, nullptr, vb, nullptr, nullptr, BH, S, absmax, nullptr,
                                    nullptr, x, s)) != cudaSuccess)
    return cuda_fail(e);
  // V of the forward is scaled per head: P.V accumulates over the kv tiles in one accumulator.
  const __nv_bfloat16* src[3] = {nullptr, nullptr, vb};
  __half* dst[3] = {nullptr, nullptr, v16};
  if ((e = vsa::launch_convert(src, dst, 3, BH, S, absmax, nullptr, s)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = vsa::launch_fwd_bitmap(q2k_idx, q2k_num, topk, BH, nb, blk / vsa::BLOCK, bitmap, err,
                                  s)) != cudaSuccess)
    return cuda_fail(e);
  vsa::FwdMainArgs a{};
  a.q = qb;
  a.k = kb;
  a.v16 = v16;
  a.bitmap = bitmap;
  a.vbs = vbs64;
  a.absmax = absmax;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.err = err;
  a.sched = ws_at<int32_t>(workspace, L.sched);
  a.B = shape.batch;
  a.H = shape.heads;
  a.S = S;
  a.nb = S / vsa::BLOCK;
  a.sm_scale = sm_scale;
  a.wait_ns = vsa::wait_limit_ns();
  if ((e = vsa::launch_fwd_main(a, s)) != cudaSuccess) return cuda_fail(e);
  return VSA_OK;
}

vsa_status vsa_bwd(const void* dout, const void* q, const void* k, const void* v, const void* o,
                   const float* lse, const int32_t* k2q_idx, const int32_t* k2q_num,
                   int32_t max_q_blocks, const int32_t* vbs, float sm_scale, vsa_shape shape,
                   void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                   void* stream) {
  return vsa_bwd_timed(dout, q, k, v, o, lse, k2q_idx, k2q_num, max_q_blocks, vbs, sm_scale, shape,
                       dq, dk, dv, workspace, workspace_bytes, nullptr, stream);
}

vsa_status vsa_bwd_timed(const void* dout, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const int32_t* k2q_idx,
                         const int32_t* k2q_num, int32_t max_q_blocks, const int32_t* vbs,
                         float sm_scale, vsa_shape shape, void* dq, void* dk, void* dv,
                         void* workspace, size_t workspace_bytes, const vsa_bwd_events* events,
                         void* stream) {
  int nb = 0, blk = 0;
  vsa_status st = check_shape(shape, &nb, &blk);
  if (st != VSA_OK) return st;
  if (!dout || !q || !k || !v || !o || !lse || !k2q_idx || !k2q_num || !vbs || !dq || !dk || !dv)
    return VSA_ERR_INVALID_ARG;
  if (max_q_blocks < 1 || !std::isfinite(sm_scale)) return VSA_ERR_INVALID_ARG;
  if (!aligned(dout, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(o, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(k2q_idx, 4) || !aligned(k2q_num, 4) || !aligned(vbs, 4))
    return VSA_ERR_INVALID_ARG;
  const vsa::BwdLayout L = vsa::bwd_layout(shape.batch, shape.heads, shape.seqlen);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return VSA_ERR_WORKSPACE;
  if ((st = check_device()) != VSA_OK) return st;

  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = shape.batch * shape.heads, S = shape.seqlen;
  uint32_t* err = ws_at<uint32_t>(workspace, L.err);
  uint32_t* absmax = ws_at<uint32_t>(workspace, L.absmax);
  uint32_t* tstat = ws_at<uint32_t>(workspace, L.tstat);
  float* delta = ws_at<float>(workspace, L.delta);
  int32_t* order = ws_at<int32_t>(workspace, L.order);
  int32_t* vbs64 = ws_at<int32_t>(workspace, L.vbs64);
  float* dqacc = ws_at<float>(workspace, L.dqacc);
  __half* q16 = ws_at<__half>(workspace, L.q16);
  __half* k16 = ws_at<__half>(workspace, L.k16);
  __half* v16 = ws_at<__half>(workspace, L.v16);
  __half* do16 = ws_at<__half>(workspace, L.do16);
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  const auto* dob = static_cast<const __nv_bfloat16*>(dout);
  const auto* ob = static_cast<const __nv_bfloat16*>(o);

  cudaError_t e = record(events ? events->start : nullptr, s);
  if (e != cudaSuccess) return cuda_fail(e);
  // Header, work counter, head and tile statistics and the split items' rows.
  if ((e = vsa::launch_zero(workspace, L.split_acc, s)) != cudaSuccess) return cuda_fail(e);
  vsa::PreExtras x{};
  x.vbs = vbs;
  x.nb = nb;
  x.tiles = blk / vsa::BLOCK;
  x.vbs64 = vbs64;
  x.err = err;
  x.tstat = tstat;
  // K and V are scaled per 64-token tile, so the statistics pass converts them as it goes
  // (row-major); Q and dO are scaled per head and converted once the head's maxima are known,
  // tile-transposed (one 16 KB copy per 64-row tile in the main kernel, whatever the distance
  // between the two q tiles of a step).
  x.k16 = k16;
  x.v16 = v16;
  // The work order (items by descending list length, stable, per head), a side job of the same
  // grid, is used from 1024 kv tiles on (the pages' rule) and when there are fewer than 8 items
  // per SM (the longest items first then even out the CTAs' few items: 3 % off the main kernel
  // at 4k tokens); in between, the item order is as fast and the side job would cost a few µs.
  const bool sorted = vsa::use_work_order(BH, S);
  x.k2q_num = k2q_num;
  x.order = sorted ? order : nullptr;
  x.nsel = nb;
  x.max_q = max_q_blocks;
  if ((e = vsa::launch_absmax_delta(qb, kb, vb, dob, ob, BH, S, absmax, delta, dqacc, x, s)) !=
      cudaSuccess)
    return cuda_fail(e);
  if ((e = vsa::launch_convert_t(qb, dob, q16, do16, BH, S, absmax, s)) != cudaSuccess)
    return cuda_fail(e);
  vsa::BwdMainArgs a{};
  a.q16 = q16;
  a.k16 = k16;
  a.v16 = v16;
  a.do16 = do16;
  a.k2q_idx = k2q_idx;
  a.k2q_num = k2q_num;
  a.order = sorted ? order : nullptr;
  a.vbs = vbs64;
  a.lse = lse;
  a.delta = delta;
  a.absmax = absmax;
  a.tstat = tstat;
  a.dqacc = dqacc;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.err = err;
  a.sched = ws_at<int32_t>(workspace, L.sched);
  a.split_acc = ws_at<float>(workspace, L.split_acc);
  a.split_row = ws_at<int32_t>(workspace, L.split_row);
  a.B = shape.batch;
  a.H = shape.heads;
  a.S = S;
  a.nb = S / vsa::BLOCK;
  a.nsel = nb;
  a.tiles = blk / vsa::BLOCK;
  a.max_q = max_q_blocks;
  a.sm_scale = sm_scale;
  a.wait_ns = vsa::wait_limit_ns();
  if ((e = record(events ? events->before_main : nullptr, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = vsa::launch_bwd_main(a, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = record(events ? events->after_main : nullptr, s)) != cudaSuccess) return cuda_fail(e);
  const vsa::SplitPlan sp = vsa::bwd_split_plan(BH * a.nb);  // as launch_bwd_main splits
  if ((e = vsa::launch_postprocess(dqacc, absmax, BH, S, sm_scale,
                                   static_cast<__nv_bfloat16*>(dq), a.split_acc, a.split_row,
                                   sp.nsplit, sp.parts, a.dk, a.dv, s)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = record(events ? events->end : nullptr, s)) != cudaSuccess) return cuda_fail(e);
  return VSA_OK;
}

vsa_status vsa_work_order(const int32_t* k2q_num, int32_t max_q_blocks, vsa_shape shape,
                          int32_t* order, void* stream) {
  int nb = 0;
  vsa_status st = check_shape(shape, &nb);
  if (st != VSA_OK) return st;
  if (!k2q_num || !order || max_q_blocks < 1) return VSA_ERR_INVALID_ARG;
  if (!aligned(k2q_num, 4) || !aligned(order, 4)) return VSA_ERR_INVALID_ARG;
  if ((st = check_device()) != VSA_OK) return st;
  const cudaError_t e = vsa::launch_order(k2q_num, shape.batch * shape.heads, nb, max_q_blocks,
                                          order, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VSA_OK : cuda_fail(e);
}

vsa_status vsa_read_device_error(const void* workspace, uint32_t* bits, void* stream) {
  if (!workspace || !bits || !aligned(workspace, 256)) return VSA_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemcpy(bits, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? VSA_OK : cuda_fail(e);
}

}  // extern "C"
