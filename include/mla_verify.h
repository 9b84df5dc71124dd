/*
 * mla_verify.h -- C ABI of the GB300 (sm_103a) MLA speculative-verify attention library.
 *
 * The operation ("The Occupancy Epiphany: How a CUDA Kernel Designer Discovered
 * That GPU Utilization Trumps Memory Bandwidth", section "Context: The Problem
 * and the Stakes"; "The Occupancy Probe", section "The Scene: What Came Before"):
 * for every stream b, draft t < q_len and head h,
 *
 *     n = seq_lens[b], p = n - q_len                  (the drafts are the last q_len keys)
 *     key j (0 <= j < n) is visible to draft t iff j < p, or mask[b,t,j-p] != 0
 *     s_j   = scale * sum_{d<576} q[b,t,h,d] * kv[slot_table[b,j], d]
 *     lse   = ln sum_{visible j} exp(s_j)
 *     out[d] = sum_{visible j} exp(s_j - lse) * kv[slot_table[b,j], d]      (d < 512)
 *
 * i.e. masked softmax(Q K^T * scale) V of Multi-head Latent Attention in absorbed
 * form: a 576-d query (512 latent + 64 rope) against 576-d latent KV rows whose
 * first 512 dims double as V, over a page_size=1 paged cache.  The draft mask
 * carries a causal chain or a draft tree ("The Occupancy Epiphany: How One
 * Environment Variable Unlocked 3x Throughput ...", section "The Broader
 * Context").  A draft that sees no key gets out = 0 and lse = -inf.
 *
 * The work is split along the keys (KV split, "flash decode"): split s writes a
 * normalised partial output and its log-sum-exp, and a combine merges them
 * ("The Occupancy Epiphany: How One Environment Variable ...", sections "The
 * Occupancy Revelation" and "Output Knowledge Created").
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller; the library keeps
 *    none of them after the call returns and allocates no device memory.
 *  - Work is enqueued on `stream` (NULL = the legacy default stream).  No entry
 *    point synchronises except mla_verify_status(), which says so.  The attention
 *    kernels are launched as programmatic dependents of the kernel before them on the
 *    stream and wait for its completion (and the visibility of its writes) before
 *    reading any input, so stream order is kept; the KV-append kernels let the
 *    attention kernel that follows them become resident early.
 *  - Return value: MLA_OK (0) or a negative mla_status.  Argument errors are
 *    detected on the host before anything is enqueued.  Errors that only the
 *    device can see (a slot index outside [0, n_pool), a seq_len outside
 *    [q_len, slot_stride], a bounded wait that expired) set bits of a per-device
 *    status word, read with mla_verify_status(); the kernel never reads outside
 *    its buffers because of them (it substitutes pool row 0 for a bad slot and
 *    writes out = 0, lse = NaN for a stream with a bad length).
 *  - Layouts are dense row-major C arrays with the shapes given below; bf16 is
 *    IEEE bfloat16 bit patterns (uint16).
 */
#ifndef MLA_VERIFY_H
#define MLA_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* mla_stream_t;

typedef enum {
    MLA_OK = 0,
    MLA_ERR_NULL = -1,       /* a required pointer is NULL */
    MLA_ERR_SHAPE = -2,      /* a size is outside the supported range */
    MLA_ERR_ALIGN = -3,      /* a pointer is not aligned as required */
    MLA_ERR_WORKSPACE = -4,  /* workspace NULL or smaller than mla_verify_workspace_bytes() */
    MLA_ERR_NSPLIT = -5,     /* nsplit outside [0, MLA_MAX_NSPLIT] */
    MLA_ERR_LAUNCH = -6,     /* the CUDA launch failed (cudaGetLastError) */
    MLA_ERR_DEVICE = -7,     /* no usable sm_103 device / CUDA runtime error */
    MLA_ERR_ARG = -8         /* any other invalid argument (e.g. non-finite scale) */
} mla_status;

/* Device status word bits (mla_verify_status). */
#define MLA_DEV_BAD_SLOT 0x1u  /* a slot index outside [0, n_pool); pool row 0 was read instead */
#define MLA_DEV_BAD_LEN 0x2u   /* a seq_len outside [q_len, slot_stride]; that stream was skipped */
#define MLA_DEV_TIMEOUT 0x4u   /* a bounded device-side wait expired (or the pipeline could not start); the CTA gave up */

/* Supported ranges. */
#define MLA_D_QK 576           /* query / key width: 512 latent + 64 rope */
#define MLA_D_V 512            /* value / output width */
#define MLA_MAX_Q_LEN 64        /* drafts per stream: a draft tree of up to 64 nodes */
#define MLA_MAX_HEADS 128
#define MLA_MAX_NSPLIT 1024

/*
 * Bytes of workspace that mla_verify_attn() needs for `nsplit` key splits
 * (nsplit >= 1; 0 when nsplit == 1, which needs none).  Layout, 256-byte
 * aligned sections: partial outputs fp32 [B, q_len, H, nsplit, 512], then
 * partial log-sum-exps fp32 [B, q_len, H, nsplit].  Pure host function.
 */
size_t mla_verify_workspace_bytes(int B, int q_len, int H, int nsplit);

/*
 * The split count that mla_verify_attn() uses when called with nsplit = 0:
 * deterministic in (B, q_len, H, max_seq = slot_stride, num_sms, ws_bytes),
 * chosen so that the launch fills the SMs ("The Occupancy Epiphany: How One
 * Environment Variable ...", section "The Occupancy Revelation": grid =
 * streams x q_len x heads x NSPLIT blocks, and too few waves starve the GPU)
 * while keeping every split at least a few key tiles long, and never more
 * splits than the workspace holds.  Pure host function.
 */
int mla_verify_auto_nsplit(int B, int q_len, int H, int max_seq, int num_sms, size_t ws_bytes);

/*
 * Verify attention (definition above).
 *   q          bf16 [B, q_len, H, 576], 16-byte aligned
 *   kv_cache   bf16 [n_pool, 576] latent KV pool, 16-byte aligned; row = 512 latent | 64 rope
 *   slot_table int32 [B, slot_stride]: pool row of key j of stream b; the drafts are
 *              keys seq_lens[b]-q_len .. seq_lens[b]-1, in draft order
 *   seq_lens   int32 [B], keys per stream (prefix + q_len); q_len <= seq_lens[b] <= slot_stride
 *   draft_mask uint8 [B, q_len, q_len] (mask[b,t,i] != 0: draft t sees draft i) or NULL
 *              for a causal chain (draft t sees drafts 0..t)
 *   scale      multiplies every score (e.g. 1/sqrt(192))
 *   out        fp32 [B, q_len, H, 512], 16-byte aligned
 *   lse        fp32 [B, q_len, H], natural log of sum exp(scaled scores)
 *   nsplit     0 = automatic (mla_verify_auto_nsplit), else 1..MLA_MAX_NSPLIT key splits
 *   workspace  device scratch of ws_bytes >= mla_verify_workspace_bytes(B,q_len,H,nsplit_used),
 *              256-byte aligned; may be NULL when the split count used is 1
 * Limits: 1 <= q_len <= 64, 1 <= H <= 128, 0 <= B <= 65535 (B == 0 is a no-op),
 *         1 <= n_pool <= 2^31 - 1, B * q_len * H <= 2^31 - 1.
 */
int mla_verify_attn(const void* q, const void* kv_cache, int64_t n_pool,
                    const int32_t* slot_table, int slot_stride, const int32_t* seq_lens,
                    const uint8_t* draft_mask, int B, int q_len, int H, float scale,
                    float* out, float* lse, int nsplit, void* workspace, size_t ws_bytes,
                    mla_stream_t stream);

/*
 * mla_verify_attn() with the draft mask bit-packed, for draft trees of up to 64
 * nodes ("The Occupancy Epiphany: How One Environment Variable Unlocked 3x
 * Throughput ...", sections "The Broader Context" and "Input Knowledge Required":
 * DDTree draft trees verified in one pass).
 *   draft_mask_bits uint64 [B, q_len], 8-byte aligned: bit i of word (b, t) set means
 *                   draft t sees draft i (bits i >= q_len are ignored); NULL = causal chain
 * Every other argument, limit and error is that of mla_verify_attn().
 */
int mla_verify_attn_packed(const void* q, const void* kv_cache, int64_t n_pool,
                           const int32_t* slot_table, int slot_stride, const int32_t* seq_lens,
                           const uint64_t* draft_mask_bits, int B, int q_len, int H, float scale,
                           float* out, float* lse, int nsplit, void* workspace, size_t ws_bytes,
                           mla_stream_t stream);

/*
 * KV append, the step before a verify call: the q_len new draft rows of every
 * stream enter the paged latent cache.  Row i of stream b, new_kv[b, i, 0:576],
 * is written to pool row slot_table[b, seq_lens[b] - q_len + i] (the drafts are
 * the last q_len keys of the stream, as mla_verify_attn() reads them; the
 * allocator's slots may be scattered: "The Occupancy Epiphany: How One
 * Environment Variable ...", section "The Broader Context").
 *   kv_cache   bf16 [n_pool, 576], 16-byte aligned, written in place
 *   slot_table int32 [B, slot_stride]; seq_lens int32 [B] (as for mla_verify_attn)
 *   new_kv     bf16 [B, q_len, 576], 16-byte aligned, read only
 * The draft slots of one call must be distinct (otherwise which row lands in a
 * shared slot is unspecified).  A stream whose seq_len is outside
 * [q_len, slot_stride] is skipped and sets MLA_DEV_BAD_LEN; a slot outside
 * [0, n_pool) skips that row and sets MLA_DEV_BAD_SLOT.
 * Limits: 1 <= q_len <= 64, 0 <= B <= 65535, 1 <= n_pool <= 2^31 - 1.
 */
int mla_kv_append(void* kv_cache, int64_t n_pool, const int32_t* slot_table, int slot_stride,
                  const int32_t* seq_lens, const void* new_kv, int B, int q_len, mla_stream_t stream);

/*
 * KV append for the fp8 cache of mla_sparse_fp8_decode(): row i of the new arrays
 * goes to pool row slots[i] of each cache array.  The rows arrive quantised (e4m3
 * codes and their per-token scale, as the cache holds them; the pages fix no
 * quantisation rule), so this is a plain scatter.
 *   kv_lat uint8 [n_pool, 512], kv_scale fp32 [n_pool], kv_rope bf16 [n_pool, 64]: written
 *   slots int32 [n_rows]; new_lat uint8 [n_rows, 512]; new_scale fp32 [n_rows];
 *   new_rope bf16 [n_rows, 64]; lat / rope arrays 16-byte aligned
 * Slots of one call must be distinct.  A slot outside [0, n_pool) skips that row and
 * sets MLA_DEV_BAD_SLOT.  n_rows == 0 is a no-op.
 */
int mla_kv_append_fp8(uint8_t* kv_lat, float* kv_scale, void* kv_rope, int64_t n_pool, const int32_t* slots,
                      const uint8_t* new_lat, const float* new_scale, const void* new_rope, int n_rows,
                      mla_stream_t stream);

/*
 * The split stage of mla_verify_attn() alone: with nsplit >= 2 it writes the
 * partial outputs and log-sum-exps into `workspace` (layout of
 * mla_verify_workspace_bytes) and enqueues nothing else; nsplit must be given
 * explicitly (>= 1); with nsplit == 1 it writes out/lse directly, like
 * mla_verify_attn.  Split s of a stream with n keys covers keys
 * [s*c, (s+1)*c) intersected with [0, n), where c = ceil(n / nsplit) rounded up
 * to a multiple of 32; trailing splits may be empty (lse = -inf, out = 0).
 * mla_verify_partials() followed by mla_verify_combine() on the workspace
 * sections is exactly mla_verify_attn() with the same nsplit.
 * nsplit == 0 runs the split stage exactly as mla_verify_attn() with nsplit = 0
 * would, including the balanced split it picks for 2..64 streams (all streams'
 * keys cut into equal chunks over one wave of CTAs, chosen on the device from
 * seq_lens); the partials' layout is then internal: use it to time the split stage
 * of an automatic call, not as input to mla_verify_combine().
 */
int mla_verify_partials(const void* q, const void* kv_cache, int64_t n_pool,
                        const int32_t* slot_table, int slot_stride, const int32_t* seq_lens,
                        const uint8_t* draft_mask, int B, int q_len, int H, float scale,
                        float* out, float* lse, int nsplit, void* workspace, size_t ws_bytes,
                        mla_stream_t stream);

/*
 * Log-sum-exp merge of KV-split partials for n_rows = B*q_len*H rows:
 *   part_out fp32 [n_rows, S, 512] (each split's normalised output), 16-byte aligned
 *   part_lse fp32 [n_rows, S] (each split's log-sum-exp; -inf for an empty split)
 *   lse = ln sum_s exp(part_lse[s]);  out = sum_s exp(part_lse[s] - lse) * part_out[s]
 * A row whose splits are all empty gets out = 0, lse = -inf.  1 <= S <= MLA_MAX_NSPLIT.
 */
int mla_verify_combine(const float* part_out, const float* part_lse, int B, int q_len, int H,
                       int S, float* out, float* lse, mla_stream_t stream);

/*
 * fp8 sparse decode ("The Occupancy Probe", section "The Scene: What Came Before":
 * DeepSeek-V4's decode attention over scattered fp8 KV cache gathers with per-token
 * scales and top-k token lists): q_len = 1, every head of stream b attends to the
 * topk keys listed in topk_slots[b], with no mask:
 *     k_j = [ decode_e4m3(kv_lat[s_j, 0:512]) * kv_scale[s_j] | kv_rope[s_j, 0:64] ]
 *     v_j = decode_e4m3(kv_lat[s_j, 0:512]) * kv_scale[s_j]
 *     out[b,h] = softmax_j(scale * q[b,h] . k_j) v_j,  lse[b,h] = ln sum_j exp(...)
 * decode_e4m3 is the OCP FP8 E4M3 ("fn") value of the byte.  The kernel dequantises
 * each latent value once, as the fp32 product decode_e4m3(code) * kv_scale rounded to
 * bf16 (one rounding, relative error at most 2^-8), and uses the rope dims as stored.
 *   q          bf16 [B, H, 576] (= [B, 1, H, 576]), 16-byte aligned
 *   kv_lat     uint8 [n_pool, 512] e4m3 codes, 16-byte aligned
 *   kv_scale   fp32 [n_pool]
 *   kv_rope    bf16 [n_pool, 64], 16-byte aligned
 *   topk_slots int32 [B, topk], pool rows (any order; duplicates count twice)
 *   out fp32 [B, H, 512], lse fp32 [B, H]; nsplit / workspace as for mla_verify_attn
 *   (mla_verify_workspace_bytes(B, 1, H, nsplit)).  nsplit = 0: every stream has the
 *   same topk keys, so the automatic count fills one wave of CTAs, min(SMs / (B x row
 *   tiles), ceil(topk / 128)) splits per stream (a workspace sized for
 *   mla_verify_auto_nsplit(B, 1, H, topk, SMs, ...) always holds it).
 * Limits: 1 <= H <= 128, 0 <= B <= 65535, topk >= 1, 1 <= n_pool <= 2^31 - 1.
 * An index outside [0, n_pool) sets MLA_DEV_BAD_SLOT and reads pool row 0.
 */
int mla_sparse_fp8_decode(const void* q, const uint8_t* kv_lat_e4m3, const float* kv_scale, const void* kv_rope,
                          int64_t n_pool, const int32_t* topk_slots, int topk, int B, int H, float scale,
                          float* out, float* lse, int nsplit, void* workspace, size_t ws_bytes,
                          mla_stream_t stream);

/* The split stage of mla_sparse_fp8_decode() alone (nsplit >= 1 explicit), like
 * mla_verify_partials(); partials then merge with mla_verify_combine(..., q_len = 1, ...). */
int mla_sparse_fp8_partials(const void* q, const uint8_t* kv_lat_e4m3, const float* kv_scale, const void* kv_rope,
                            int64_t n_pool, const int32_t* topk_slots, int topk, int B, int H, float scale,
                            float* out, float* lse, int nsplit, void* workspace, size_t ws_bytes,
                            mla_stream_t stream);

/*
 * Verify attention without a caller-provided workspace, for callers that cannot
 * allocate device memory: plugins hosted by a runtime that owns all device
 * memory (a serving engine's caching allocator or a fixed arena that must not
 * be bypassed) and latency-critical loops where cudaMalloc/cudaFree, which can
 * synchronise the device or fail under memory pressure, are not allowed.  The
 * pages have no counterpart of this entry point.
 *
 * Same arguments and result as mla_verify_attn() minus the workspace.  The
 * KV-split partials go to a file-scope device array of MLA_STATIC_SCRATCH_BYTES.
 * A device holds that array from the moment the library's device code is loaded
 * there until the process exits: under CUDA's default lazy module loading at the
 * latest from the first static-scratch call on that device, and on every device
 * from its context's creation when CUDA_MODULE_LOADING=EAGER.  Nothing is
 * allocated per call (no cudaMalloc, no cudaFree, no allocating library
 * routine).  With nsplit = 0 the split count is chosen to fit the array; an
 * explicit nsplit whose partials need more than MLA_STATIC_SCRATCH_BYTES
 * (mla_verify_workspace_bytes) returns MLA_ERR_WORKSPACE.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current.  The address is cached per
 * device ordinal for the device's primary context (the CUDA runtime's context):
 * the entry point supports that context only, and must not be used again after
 * cudaDeviceReset.  All calls on a device share the one array and it keeps the
 * last call's contents (every call overwrites what it reads, so nothing needs
 * clearing); calls whose GPU work overlaps -- on different streams, or from
 * different host threads -- race on it and must be serialised by the caller.
 */
#define MLA_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
int mla_verify_attn_static_scratch(const void* q, const void* kv_cache, int64_t n_pool,
                                   const int32_t* slot_table, int slot_stride, const int32_t* seq_lens,
                                   const uint8_t* draft_mask, int B, int q_len, int H, float scale,
                                   float* out, float* lse, int nsplit, mla_stream_t stream);

/*
 * Reads (and with clear != 0 resets) the calling device's status word of
 * MLA_DEV_* bits.  SYNCHRONISES `stream`.  Returns MLA_OK or MLA_ERR_DEVICE.
 */
int mla_verify_status(mla_stream_t stream, uint32_t* device_status, int clear);

/* Static string for an mla_status value. */
const char* mla_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int mla_verify_version(void);

/*
 * Test hook for the failure-detection path: the next split-kernel launch (any entry
 * point, any device) has its gather warps withhold their arrival on the first key
 * tile, so the pipeline's bounded waits expire after about a second: the kernel sets
 * MLA_DEV_TIMEOUT, writes zeros, releases its tensor memory and exits; no trap, no
 * hang, and the context stays usable.  One-shot; returns MLA_OK.
 */
int mla_debug_stall_next_launch(void);

/*
 * Test counter of the online softmax's lazy rescale.  The kernels keep a running
 * row maximum and rescale the resident output accumulator only when a later key
 * tile raises some row's maximum by more than 2^8 (about 5.5 in natural-log units);
 * every (CTA, key tile) on which that happens adds one to a per-device counter.
 * This reads it (with clear != 0 also resets it to zero) so that a test can show
 * that its inputs really drove the rescale path.  SYNCHRONISES `stream`.  Returns
 * MLA_OK, MLA_ERR_NULL (count is NULL) or MLA_ERR_DEVICE.  No counterpart in the
 * pages: the online softmax with a running maximum is theirs, the counter is a
 * test aid.
 */
int mla_debug_rescale_count(mla_stream_t stream, uint64_t* count, int clear);

#ifdef __cplusplus
}
#endif

#endif /* MLA_VERIFY_H */
