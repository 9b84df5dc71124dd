// mla_verify_attn_static_scratch(): verify attention for callers that cannot
// allocate device memory.  Some callers are not allowed to call cudaMalloc or to
// allocate through any other allocator: plugins hosted by a runtime that owns
// every byte of device memory (a serving engine's caching allocator or fixed
// arena that must not be bypassed), and latency-critical loops where an
// allocation, which can implicitly synchronise the device or fail under memory
// pressure, is not permitted.  This entry point needs no workspace from them:
// the KV-split partials live in a file-scope device array that is part of the
// library's device code.
//
// The array holds MLA_STATIC_SCRATCH_BYTES (64 MiB).  A device holds it from the
// moment this translation unit's device code is loaded there until the process
// exits: with CUDA's default lazy module loading that is at the latest the first
// static-scratch call on that device, with CUDA_MODULE_LOADING=EAGER it is the
// creation of the device's context.
#include <atomic>

#include "../../include/mla_verify.h"
#include "internal.cuh"

namespace {

constexpr size_t kScratchBytes = MLA_STATIC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte sections");

// Shared by every call on a device; it keeps the last call's contents.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
// Device address of g_scratch per device ordinal, looked up once per device.  Host
// threads may make their first call on a device at the same time: they look up and
// store the same value, so relaxed atomics suffice.  The address belongs to the
// device's primary context (the one the CUDA runtime uses); it is not valid in
// another context on that device nor after cudaDeviceReset.
std::atomic<void*> g_scratch_ptr[kMaxDevices];

}  // namespace

extern "C" int mla_verify_attn_static_scratch(const void* q, const void* kv_cache, int64_t n_pool,
                                              const int32_t* slot_table, int slot_stride,
                                              const int32_t* seq_lens, const uint8_t* draft_mask, int B,
                                              int q_len, int H, float scale, float* out, float* lse,
                                              int nsplit, mla_stream_t stream) {
    if (B < 0 || q_len < 1 || H < 1) return MLA_ERR_SHAPE;
    if (nsplit < 0 || nsplit > MLA_MAX_NSPLIT) return MLA_ERR_NSPLIT;
    // An explicit split count whose partials do not fit the static array is refused.
    if (nsplit > 1 && mla_verify_workspace_bytes(B, q_len, H, nsplit) > kScratchBytes) return MLA_ERR_WORKSPACE;
    if (B == 0) return mla_verify_attn(q, kv_cache, n_pool, slot_table, slot_stride, seq_lens, draft_mask, B,
                                       q_len, H, scale, out, lse, nsplit, nullptr, 0, stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_DEVICE;
    void* scratch = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (scratch == nullptr) {
        // One-time set-up on this device (the device is current): in host code the
        // array's name is only a host-side stand-in, so take its device address.
        if (cudaGetSymbolAddress(&scratch, g_scratch) != cudaSuccess || scratch == nullptr) return MLA_ERR_DEVICE;
        g_scratch_ptr[dev].store(scratch, std::memory_order_relaxed);
    }
    // The split stage writes every partial (empty splits included) before the
    // combine reads it, so nothing in the array needs clearing between calls.
    return mla_verify_attn(q, kv_cache, n_pool, slot_table, slot_stride, seq_lens, draft_mask, B, q_len, H, scale,
                           out, lse, nsplit, scratch, kScratchBytes, stream);
}
