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
    int nsplit;                   // uniform splits per stream, or (balanced) split slots
    unsigned* status;             // device status word
    unsigned long long* rescales; // test counter: tiles on which a CTA rescaled its O^T accumulator
    // balanced split (several streams of unequal length, see balanced_plan): grid.x =
    // nsplit slots shared by all streams; partials are slot-major,
    // part_out [nsplit][q_len * H][512], part_lse [nsplit][q_len * H]
    int balanced;
    int bal_G;
    // test hook (mla_debug_stall_next_launch): the gather warps withhold their arrival on
    // key tile 0, so the pipeline's bounded waits expire and report DEV_TIMEOUT
    int debug_stall;
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

// Balanced key split of one launch over B <= 64 streams of unequal length, decided on
// the device (the host does not know the lengths): with T the sum of the valid lengths,
// the keys are cut into chunks of chunk = max(128, ceil(T / G) rounded up to 32) keys;
// stream b gets ns_b = ceil(n_b / chunk) consecutive split slots (one for a stream whose
// length is invalid, which then writes NaN), slots numbered stream after stream, at
// most G + B of them.  Every warp evaluates it alike (lane i holds streams i and
// i + 32), so no barrier or shared memory is needed.
struct BalancedPlan {
    int chunk;
    int n[2];       // lengths of streams lane and lane + 32 (0 past B)
    int ns[2];      // split slots of streams lane and lane + 32
    int incl[2];    // inclusive prefix sums of the slot counts at those streams
};

__device__ inline BalancedPlan balanced_plan(const int32_t* seq_lens, int B, int q_len, int slot_stride, int G) {
    const int lane = threadIdx.x & 31;
    BalancedPlan P;
    int* n = P.n;
    bool ok[2];
    long long t = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        n[h] = i < B ? seq_lens[i] : 0;
        ok[h] = i < B && n[h] >= q_len && n[h] <= slot_stride;
        if (ok[h]) t += n[h];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    // 32-bit divisions whenever the total fits (warp-uniform branch)
    long long c = t < (1ll << 30) ? (long long)(((unsigned)t + (unsigned)G - 1u) / (unsigned)G) : (t + G - 1) / G;
    c = (c + 31) / 32 * 32;
    if (c < 128) c = 128;
    if (c > (1 << 30)) c = 1 << 30;
    P.chunk = (int)c;
    int run = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        P.ns[h] = i < B ? (ok[h] ? (int)(((unsigned)n[h] + (unsigned)c - 1u) / (unsigned)c) : 1) : 0;
        int v = P.ns[h];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        P.incl[h] = v + run;
        run += __shfl_sync(0xffffffffu, v, 31);
    }
    return P;
}

// Stream and split of slot x (b = -1: slot unused).  Whole warp.
__device__ inline void balanced_slot(const BalancedPlan& P, int x, int* b, int* s) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const unsigned m = __ballot_sync(0xffffffffu, x < P.incl[h]);
        if (m) {
            const int L = __ffs(m) - 1;
            const int incl = __shfl_sync(0xffffffffu, P.incl[h], L);
            const int ns = __shfl_sync(0xffffffffu, P.ns[h], L);
            *b = L + 32 * h;
            *s = x - (incl - ns);
            return;
        }
    }
    *b = -1;
    *s = 0;
}

// First slot and slot count of stream b (0 <= b < B <= 64).  Whole warp.
__device__ inline void balanced_stream(const BalancedPlan& P, int b, int* first, int* count) {
    const int h = b >> 5, L = b & 31;
    const int incl = __shfl_sync(0xffffffffu, h ? P.incl[1] : P.incl[0], L);
    const int ns = __shfl_sync(0xffffffffu, h ? P.ns[1] : P.ns[0], L);
    *first = incl - ns;
    *count = ns;
}

constexpr int BALANCED_MAX_STREAMS = 64;

// One-shot test hook, consumed by the next split-kernel launch on any device.
bool take_debug_stall();

// Launchers (each returns the cudaError_t of the launch).
cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream);
// Row tiling of the tensor-core split kernel: n_tiles CTAs of R_step rows over
// q_len * H rows, each padded to R (multiple of 16) MMA columns.
void tc_tiling(int rows, int max_r, int* n_tiles, int* R_step, int* R);
constexpr int TC_MAX_ROWS = 96;
cudaError_t launch_kv_append(__nv_bfloat16* kv, const int32_t* slot, int slot_stride, const int32_t* seq_lens,
                             const __nv_bfloat16* new_kv, int B, int q_len, int64_t n_pool, unsigned* status,
                             cudaStream_t stream);
cudaError_t launch_kv_append_fp8(uint8_t* kv_lat, float* kv_scale, __nv_bfloat16* kv_rope, int64_t n_pool,
                                 const int32_t* slots, const uint8_t* new_lat, const float* new_scale,
                                 const __nv_bfloat16* new_rope, int n_rows, unsigned* status, cudaStream_t stream);
cudaError_t launch_combine(const float* part_out, const float* part_lse, long long n_rows, int S,
                           float* out, float* lse, cudaStream_t stream);
// Combine of a balanced split (slot-major partials of VerifyArgs::balanced).
cudaError_t launch_combine_balanced(const VerifyArgs& a, cudaStream_t stream);

}  // namespace mla
