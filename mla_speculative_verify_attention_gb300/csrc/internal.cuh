// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

constexpr int D_QK = 576;     // 512 latent + 64 rope
constexpr int D_V = 512;

// Status word bits (same values as MLA_DEV_* in include/mla_verify.h).
constexpr unsigned DEV_BAD_SLOT = 0x1u;
constexpr unsigned DEV_BAD_LEN = 0x2u;
constexpr unsigned DEV_TIMEOUT = 0x4u;

// One verify launch.  Row r of stream b is (t, h) with r = t * H + h, the
// natural order of q [B, q_len, H, 576] and out [B, q_len, H, 512].
struct VerifyArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* kv;
    int64_t n_pool;
    const int32_t* slot;
    int slot_stride;
    const int32_t* seq_lens;
    const uint8_t* mask;          // [B, q_len, q_len] or nullptr = causal chain
    const uint64_t* mask_bits;    // [B, q_len] bit-packed mask (bit i: sees draft i); overrides mask
    int B, q_len, H;
    float scale;
    float* out;                   // [B, q_len, H, 512], used when nsplit == 1
    float* lse;                   // [B, q_len, H]
    float* part_out;              // [B, q_len, H, nsplit, 512], used when nsplit > 1
    float* part_lse;              // [B, q_len, H, nsplit]
    int nsplit;
    unsigned* status;             // device status word
    // fp8 sparse decode (kv_fp8 != 0): keys come from per-stream index lists
    // (slot = topk_slots [B, slot_stride = topk], seq_lens unused, q_len = 1) and
    // each key row is an e4m3 latent [512] with a per-token fp32 scale plus a bf16
    // rope [64]; kv is unused.
    int kv_fp8;
    const uint8_t* kv_lat;
    const float* kv_scale;
    const __nv_bfloat16* kv_rope;
};

// Key range [begin, end) of split s of a stream with n keys: S contiguous
// chunks of ceil(n / S) keys each, rounded up to whole key tiles of `tile`
// keys; trailing chunks may be empty.
__host__ __device__ inline void split_range(int n, int S, int s, int tile, int* begin, int* end) {
    int chunk = (n + S - 1) / S;
    chunk = (chunk + tile - 1) / tile * tile;
    long long b = (long long)s * chunk;
    long long e = b + chunk;
    *begin = (int)(b < n ? b : n);
    *end = (int)(e < n ? e : n);
}

// Launchers (each returns the cudaError_t of the launch).
cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream);
// Row tiling of the tensor-core split kernel: n_tiles CTAs of R_step rows over
// q_len * H rows, each padded to R (multiple of 16) MMA columns.
void tc_tiling(int rows, int max_r, int* n_tiles, int* R_step, int* R);
constexpr int TC_MAX_ROWS = 96;
cudaError_t launch_kv_append(__nv_bfloat16* kv, const int32_t* slot, int slot_stride, const int32_t* seq_lens,
                             const __nv_bfloat16* new_kv, int B, int q_len, int64_t n_pool, unsigned* status,
                             cudaStream_t stream);
cudaError_t launch_combine(const float* part_out, const float* part_lse, long long n_rows, int S,
                           float* out, float* lse, cudaStream_t stream);

}  // namespace mla
