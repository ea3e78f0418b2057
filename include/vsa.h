/*
 * vsa.h -- C ABI of the GB300 (sm_103a) block-sparse video attention library (libvsa.so).
 *
 * Block-sparse attention with 64- or 128-token blocks ("VSA"): query block i attends only to
 * the kv blocks its q2k row selects, and inside kv block j only to the first
 * variable_block_sizes[j] keys.  The library computes
 *   - the inversion of the block selection (q2k -> k2q),
 *   - the forward (O and the base-2 "M form" log-sum-exp the backward consumes),
 *   - the backward (dQ, dK, dV).
 * Sources (web pages; cited by title and section):
 *   [FV-bwd]  FastVideo commit 749a9c5 "[kernel] sm_100a CUDA backward for VSA block-sparse
 *             attention (64-token blocks)": commit message (Semantics) and the module
 *             fastvideo_kernel/block_sparse_attn_bwd_sm100a.py (docstrings).
 *   [FV-diff] FastVideo, compare main...vsa_bwd_fix: block_sparse_bwd_launch_sm100a.cuh
 *             (BlockSparseVsaBwdArgs, block_sparse_bwd_supported, the launch sequence),
 *             block_sparse_bwd_sm100a.cu (argument checks), tests/test_block_sparse_bwd_sm100a.py
 *             (reference(), invert_indices_torch()).
 *   [cuDNN]   NVIDIA cudnn-frontend PR #926, Summary (slot validity and clamping) and the
 *             follow-up commit on the no-allocation plan + caller workspace contract.
 *   [FV-fwd]  FastVideo fastvideo_kernel, the sm_100a/sm_103a forward's description: two
 *             instantiations, for 64- and 128-token sparse blocks, the block size inferred from
 *             the metadata.
 *
 * Conventions shared by every entry point:
 *   - Layout: activations are contiguous [B, H, S, 128] bf16 (B batch, H heads, S tokens,
 *     head_dim 128), S = block * nb with nb the number of sparse blocks of `block` tokens (64 or
 *     128, vsa_shape.block; [FV-diff] BlockSparseVsaBwdArgs with VSA_BHSD; the torch binding
 *     expects sequences already padded to whole blocks; [FV-fwd]).  Any nb >= 1 is accepted (no
 *     even-nb rule).  Block ids, q2k/k2q rows and variable_block_sizes all count blocks of
 *     `block` tokens.
 *   - Pointers: every buffer is device memory owned and allocated by the caller; activation
 *     and workspace pointers must be 16-byte (activations) / 256-byte (workspace) aligned.
 *     The library never allocates, keeps no per-call state between calls (the wait limit of
 *     vsa_set_wait_limit_ns is a process-wide setting) and never synchronises the stream except
 *     in vsa_read_device_error and vsa_bwd_no_alloc_device_error.  `stream` is a cudaStream_t
 *     (NULL = legacy default stream).  Work is enqueued on it in order (kernels only; all but
 *     the first of vsa_invert_indices and the one of vsa_work_order are programmatic dependent
 *     launches, each of which waits, before it touches memory, until the previous work on the
 *     stream has completed, so the caller's own work before and after keeps its order); the
 *     call returns before the GPU finishes and may be captured in a CUDA graph.
 *   - Errors: problems visible on the host (null pointer, bad size, misalignment, too small a
 *     workspace, non-finite sm_scale, wrong device) return a status before anything is
 *     enqueued (an unsupported configuration is an error, never a silently wrong result:
 *     [FV-diff] block_sparse_bwd_sm100a.cu).  Problems only visible on the
 *     device never trap: an out-of-range block id is skipped, a count is clamped to its row
 *     width, a block size is clamped to [0, block] ([cuDNN] Summary: a slot participates only
 *     inside the bounded active prefix with its index in [0, nb)), and a bit is set in the
 *     device error word (VSA_DEVERR_*).  Every pipeline wait inside a kernel has a time limit;
 *     a wait that runs out sets VSA_DEVERR_TIMEOUT and the kernel exits (outputs invalid).
 */
#ifndef VSA_H
#define VSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vsa_status {
  VSA_OK = 0,
  VSA_ERR_INVALID_ARG = 1, /* null pointer, bad size or stride, misalignment, bad sm_scale */
  VSA_ERR_UNSUPPORTED = 2, /* head_dim != 128, block not 64/128, S not a multiple of block,
                              B * H above 65535, or not an sm_103 device */
  VSA_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or smaller than required */
  VSA_ERR_CUDA = 4         /* a CUDA runtime or driver call failed (see vsa_last_cuda_error) */
} vsa_status;

/* Bits of the device error word. */
#define VSA_DEVERR_Q2K_ID 0x01u    /* a q2k block id outside [0, nb) was skipped */
#define VSA_DEVERR_Q2K_COUNT 0x02u /* a q2k count outside [0, topk] was clamped */
#define VSA_DEVERR_K2Q_ID 0x04u    /* a k2q block id outside [0, nb) was skipped */
#define VSA_DEVERR_K2Q_COUNT 0x08u /* a k2q count outside [0, max_q_blocks] was clamped */
#define VSA_DEVERR_VBS 0x10u       /* a variable_block_sizes entry outside [0, block] was clamped */
#define VSA_DEVERR_TIMEOUT 0x20u   /* a pipeline wait ran past its limit; outputs are invalid */

typedef struct vsa_shape {
  int32_t batch;    /* B >= 1 */
  int32_t heads;    /* H >= 1 */
  int32_t seqlen;   /* S = block * nb, nb >= 1 */
  int32_t head_dim; /* must be 128 */
  int32_t block;    /* tokens per sparse block: 64 or 128 (0 is read as 64) */
} vsa_shape;

/* Human-readable name of a status code (static storage; never NULL). */
const char* vsa_status_string(vsa_status status);

/* The last CUDA error code seen by this thread's calls (0 if none); for VSA_ERR_CUDA. */
int vsa_last_cuda_error(void);

/*
 * vsa_set_wait_limit_ns -- the time limit of every pipeline wait inside the kernels that this
 * process launches from now on, on any device (the default is 4 s; 0 restores it).  Returns the
 * previous limit.  The pages have no counterpart: it is the watchdog of the bounded waits that
 * the error contract above describes.  A wait that runs past the limit sets VSA_DEVERR_TIMEOUT,
 * the kernel lets the copies it has in flight land, frees its tensor memory and exits, and the
 * outputs of that call are invalid; the device stays usable and later calls are unaffected.  A
 * limit far below a kernel's normal waits (microseconds) makes every call time out, which is how
 * a caller can check its handling of that error.  Thread-safe; launches already enqueued keep
 * the limit they were given.
 */
uint64_t vsa_set_wait_limit_ns(uint64_t limit_ns);

/*
 * vsa_invert_indices -- k2q from q2k.
 * Defined by [FV-bwd] block_sparse_attn_backward_sm100a (the backward first inverts the
 * selection into per-kv-block lists) and [FV-diff] invert_indices_torch: for every
 * (b, h, kv block j), the q blocks i whose active q2k slots contain j, each once, in ASCENDING
 * order of i, and their count.
 *   q2k_idx  [B, H, nb, topk] int32: kv block ids selected by each q block (read: the first
 *            q2k_num entries of each row; duplicates count once; ids outside [0, nb) skipped).
 *   q2k_num  [B, H, nb] int32: active slots per row (clamped to [0, topk]).
 *   topk     row width of q2k_idx, >= 1.
 *   k2q_idx  [B, H, nb, nb] int32 (written): row j lists the selecting q blocks ascending;
 *            entries past the count are written as 0.
 *   k2q_num  [B, H, nb] int32 (written): count per kv block (0 allowed).
 *   dev_err  optional device uint32 (NULL allowed): VSA_DEVERR_Q2K_* bits are OR-ed in; the
 *            library never clears it.
 * Deterministic: the output is a pure function of the input.
 */
vsa_status vsa_invert_indices(const int32_t* q2k_idx, const int32_t* q2k_num, int32_t topk,
                              vsa_shape shape, int32_t* k2q_idx, int32_t* k2q_num,
                              uint32_t* dev_err, void* stream);

/* Bytes of device workspace vsa_fwd needs for `shape` (0 for an invalid shape). */
size_t vsa_fwd_workspace_bytes(vsa_shape shape);

/*
 * vsa_fwd -- forward of block-sparse attention, producing the operands of the backward.
 * Defined by [FV-diff] tests reference() (softmax over the selected blocks, keys at or past
 * variable_block_sizes[j] masked to -inf) and [FV-bwd] module docstring (lse in the "M form"
 * max(qk * sm_scale * log2e) + log2(l)):
 *   O[r]   = sum_t softmax_t(q_r . k_t * sm_scale) v_t over the visible keys t of row r,
 *   lse[r] = max_t(q_r . k_t * sm_scale * log2e) + log2(sum_t exp2(q_r . k_t * sm_scale * log2e
 *            - max)).
 * A row with no visible key gets O = 0 and lse = -inf.
 *   q, k, v   [B, H, S, 128] bf16 (read).
 *   q2k_idx, q2k_num, topk: the block selection, as for vsa_invert_indices.
 *   vbs       [nb] int32: valid kv tokens per block (clamped to [0, block]); shared by all (b, h).
 *   sm_scale  finite softmax scale.
 *   o         [B, H, S, 128] bf16 (written, round-to-nearest-even).
 *   lse       [B, H, S] fp32 (written).
 *   workspace device buffer of at least vsa_fwd_workspace_bytes(shape) bytes, 256-B aligned.
 */
vsa_status vsa_fwd(const void* q, const void* k, const void* v, const int32_t* q2k_idx,
                   const int32_t* q2k_num, int32_t topk, const int32_t* vbs, float sm_scale,
                   vsa_shape shape, void* o, float* lse, void* workspace, size_t workspace_bytes,
                   void* stream);

/* Bytes of device workspace vsa_bwd needs for `shape` (0 for an invalid shape). */
size_t vsa_bwd_workspace_bytes(vsa_shape shape);

/*
 * vsa_bwd -- backward of block-sparse attention.
 * Defined by [FV-diff] BlockSparseVsaBwdArgs / launch_block_sparse_bwd_sm100a and [FV-bwd]
 * (Semantics; module docstring): with P recomputed from lse (M form),
 *   Delta_r = sum_d O_rd dO_rd      (O as given, bf16)
 *   P_rt    = exp2(q_r . k_t * sm_scale * log2e - lse_r) on visible (r, t), else 0
 *   dS_rt   = P_rt (dO_r . v_t - Delta_r)
 *   dV_t = sum_r P_rt dO_r,   dK_t = sm_scale sum_r dS_rt q_r,   dQ_r = sm_scale sum_t dS_rt k_t.
 * kv blocks no q block selects and kv rows at or past vbs[j] get exact-zero (+0.0) dK/dV rows.
 *   dout, q, k, v, o  [B, H, S, 128] bf16 (read).
 *   lse          [B, H, S] fp32, M form, as written by vsa_fwd (read).
 *   k2q_idx      [B, H, nb, max_q_blocks] int32: per kv block the selecting q blocks (any
 *                order; entries past the count unread), e.g. from vsa_invert_indices with
 *                max_q_blocks = nb.  An id outside [0, nb) is skipped (VSA_DEVERR_K2Q_ID).  A
 *                row must not repeat an id (vsa_invert_indices never does): a repeated id is
 *                counted as often as it appears.
 *   k2q_num      [B, H, nb] int32 (clamped to [0, max_q_blocks]).
 *   max_q_blocks row stride of k2q_idx, >= 1.
 *   vbs, sm_scale: as for vsa_fwd.
 *   dq, dk, dv   [B, H, S, 128] bf16 (written, every element; round-to-nearest-even).
 *   workspace    device buffer of at least vsa_bwd_workspace_bytes(shape) bytes, 256-B
 *                aligned; its contents need no initialisation and are scratch after the call.
 * The dQ partial sums are added in fp32 in an order that varies from run to run, so two runs
 * can differ in the last bits of dQ; dK, dV and the zero rows are run-to-run identical.
 */
vsa_status vsa_bwd(const void* dout, const void* q, const void* k, const void* v, const void* o,
                   const float* lse, const int32_t* k2q_idx, const int32_t* k2q_num,
                   int32_t max_q_blocks, const int32_t* vbs, float sm_scale, vsa_shape shape,
                   void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * vsa_work_order -- the order in which vsa_bwd's main kernel takes its work items.  Defined by
 * [FV-bwd] commit message (Semantics: from 1024 kv blocks on, the items are sorted on the device
 * by the length of their k2q lists) and [FV-diff] ORDER_MIN_KV_BLOCKS: within each (b, h)
 * segment, in head order, the kv blocks sorted by DESCENDING count, stable (equal counts keep
 * ascending block order).  vsa_bwd computes this order inside its preprocess, with the same
 * device code as this call, and takes its items in it from 1024 kv tiles of 64 tokens on (as the
 * pages do) and when there are fewer than 8 items (kv tiles of all heads) per SM, where the
 * longest items first even out the CTAs' few items; otherwise it takes them in item order.
 *   k2q_num       [B, H, nb] int32 (read; each count clamped to [0, max_q_blocks] before
 *                 sorting).
 *   max_q_blocks  >= 1.
 *   order         [B * H * nb] int32 (written): position x of segment bh holds the flat item id
 *                 bh * nb + j of the kv block that comes x-th.
 */
vsa_status vsa_work_order(const int32_t* k2q_num, int32_t max_q_blocks, vsa_shape shape,
                          int32_t* order, void* stream);

/*
 * vsa_bwd_timed -- vsa_bwd, plus CUDA events recorded on `stream` around its stages, for callers
 * that time the kernels (a benchmark's roofline).  `events` may be NULL (then it is vsa_bwd);
 * any NULL member is skipped.  Members are cudaEvent_t handles created by the caller:
 *   start        before the preprocess,        before_main  before the main kernel,
 *   after_main   after the main kernel,         end          after the dQ postprocess.
 * The events do not change what is computed.
 */
typedef struct vsa_bwd_events {
  void* start;
  void* before_main;
  void* after_main;
  void* end;
} vsa_bwd_events;

vsa_status vsa_bwd_timed(const void* dout, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const int32_t* k2q_idx,
                         const int32_t* k2q_num, int32_t max_q_blocks, const int32_t* vbs,
                         float sm_scale, vsa_shape shape, void* dq, void* dk, void* dv,
                         void* workspace, size_t workspace_bytes, const vsa_bwd_events* events,
                         void* stream);

/* Largest workspace vsa_bwd_no_alloc can serve (32 MiB): the size of the static scratch array
 * that every GPU loading this library holds until the process exits.  A shape needs
 * vsa_bwd_workspace_bytes(shape) of it, about 1800 bytes per (batch, head, token) row on such
 * small shapes (1540 plus the fp32 parts of the main kernel's split items) and a small header: for
 * example B = 1, H = 4, S = 4096 fits, H = 8 at S = 4096 does not. */
#define VSA_BWD_NO_ALLOC_MAX_WORKSPACE_BYTES (32u * 1024u * 1024u)

/*
 * vsa_bwd_no_alloc -- the backward (same arguments, same results as vsa_bwd) without a workspace
 * argument, for callers that cannot allocate device memory.  The pages have no counterpart of
 * this entry point; it exists for this library's users.
 *
 * Who needs it: code that runs inside a host framework which owns all device memory and does not
 * let a plugin allocate (cudaMalloc synchronises the device, can fail under fragmentation and
 * escapes the framework's accounting), or a service with a fixed device-memory budget that has
 * no room to hand over a workspace per call.  Such callers still pass every input and output
 * buffer; only the scratch moves into the library.
 *
 * How: the scratch is a static device array of VSA_BWD_NO_ALLOC_MAX_WORKSPACE_BYTES inside
 * libvsa.so.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that first call before
 * any stream capture.  No call allocates anything.
 *
 * Limits and sharing: a shape needing more than VSA_BWD_NO_ALLOC_MAX_WORKSPACE_BYTES of scratch
 * is rejected with VSA_ERR_WORKSPACE before anything is enqueued.  Every call uses the same
 * array, which keeps the previous call's contents (each call clears what must start at zero).
 * Calls whose GPU work overlaps -- on different streams, or from host threads that are not
 * ordered -- race on the array; order them (one stream, or events).  The device error word of
 * the last call sits at the start of the array: read it with vsa_bwd_no_alloc_device_error (not
 * vsa_read_device_error, which takes a workspace pointer).
 */
vsa_status vsa_bwd_no_alloc(const void* dout, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const int32_t* k2q_idx,
                            const int32_t* k2q_num, int32_t max_q_blocks, const int32_t* vbs,
                            float sm_scale, vsa_shape shape, void* dq, void* dk, void* dv,
                            void* stream);

/*
 * vsa_bwd_no_alloc_device_error -- synchronise `stream`, then copy to *bits the device error word
 * that the last vsa_bwd_no_alloc call on the current device left in the static scratch array
 * (VSA_DEVERR_* bits; 0 if no call has run on this device yet).  Like the entry point it serves,
 * it allocates nothing.  Another call's GPU work that overlaps the read races with it.
 */
vsa_status vsa_bwd_no_alloc_device_error(uint32_t* bits, void* stream);

/*
 * vsa_read_device_error -- synchronise `stream`, then copy the device error word of a
 * vsa_fwd / vsa_bwd workspace (the bits raised by the last call that used it) to *bits.
 */
vsa_status vsa_read_device_error(const void* workspace, uint32_t* bits, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VSA_H */
