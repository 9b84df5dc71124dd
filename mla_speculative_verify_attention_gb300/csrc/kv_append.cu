// KV append: the q_len draft rows of every stream are written into their slots of
// the paged latent cache just before the verify call reads them.  One warp per
// row copies 1152 bytes as 72 16-byte vectors (a plain scatter: bandwidth-bound,
// no reuse, nothing to stage).  Slots come from the stream's slot list: draft i of
// stream b goes to slot_table[b, seq_lens[b] - q_len + i], the drafts being the
// last q_len keys of the stream ("The Occupancy Epiphany: How One Environment
// Variable Unlocked 3x Throughput ...", section "The Broader Context": KV slots
// handed out by a paged allocator, possibly scattered).
#include "internal.cuh"

namespace mla {
namespace {

constexpr int APPEND_THREADS = 256;

__global__ void __launch_bounds__(APPEND_THREADS)
    kv_append_kernel(__nv_bfloat16* __restrict__ kv, const int32_t* __restrict__ slot, int slot_stride,
                     const int32_t* __restrict__ seq_lens, const __nv_bfloat16* __restrict__ new_kv, int B,
                     int q_len, int64_t n_pool, unsigned* status) {
    // the verify kernel that usually follows may become resident now; its
    // griddepcontrol.wait still holds it until this grid's writes are visible
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long warp = ((long long)blockIdx.x * APPEND_THREADS + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= (long long)B * q_len) return;
    const int b = (int)(warp / q_len), i = (int)(warp % q_len);
    const int n = seq_lens[b];
    if (n < q_len || n > slot_stride) {                  // bad length: write nothing for this stream
        if (lane == 0 && i == 0) atomicOr(status, DEV_BAD_LEN);
        return;
    }
    const int s = slot[(int64_t)b * slot_stride + (n - q_len + i)];
    if (s < 0 || (int64_t)s >= n_pool) {                 // bad slot: skip the row
        if (lane == 0) atomicOr(status, DEV_BAD_SLOT);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(new_kv + ((int64_t)b * q_len + i) * D_QK);
    uint4* dst = reinterpret_cast<uint4*>(kv + (int64_t)s * D_QK);
    for (int k = lane; k < D_QK / 8; k += 32) dst[k] = __ldg(src + k);
}

// fp8 cache: one warp per appended row; lanes 0-31 copy the 512 code bytes, lanes 0-7
// the 128 rope bytes, lane 0 the scale.  The rows arrive quantised.
__global__ void __launch_bounds__(APPEND_THREADS)
    kv_append_fp8_kernel(uint8_t* __restrict__ kv_lat, float* __restrict__ kv_scale,
                         __nv_bfloat16* __restrict__ kv_rope, int64_t n_pool, const int32_t* __restrict__ slots,
                         const uint8_t* __restrict__ new_lat, const float* __restrict__ new_scale,
                         const __nv_bfloat16* __restrict__ new_rope, int n_rows, unsigned* status) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // as in kv_append_kernel
    const long long i = ((long long)blockIdx.x * APPEND_THREADS + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (i >= n_rows) return;
    const int s = slots[i];
    if (s < 0 || (int64_t)s >= n_pool) {
        if (lane == 0) atomicOr(status, DEV_BAD_SLOT);
        return;
    }
    reinterpret_cast<uint4*>(kv_lat + (int64_t)s * D_V)[lane] =
        __ldg(reinterpret_cast<const uint4*>(new_lat + i * D_V) + lane);
    if (lane < 8)
        reinterpret_cast<uint4*>(kv_rope + (int64_t)s * 64)[lane] =
            __ldg(reinterpret_cast<const uint4*>(new_rope + i * 64) + lane);
    if (lane == 0) kv_scale[s] = __ldg(new_scale + i);
}

}  // namespace

cudaError_t launch_kv_append_fp8(uint8_t* kv_lat, float* kv_scale, __nv_bfloat16* kv_rope, int64_t n_pool,
                                 const int32_t* slots, const uint8_t* new_lat, const float* new_scale,
                                 const __nv_bfloat16* new_rope, int n_rows, unsigned* status, cudaStream_t stream) {
    const long long threads = (long long)n_rows * 32;
    const unsigned blocks = (unsigned)((threads + APPEND_THREADS - 1) / APPEND_THREADS);
    kv_append_fp8_kernel<<<blocks, APPEND_THREADS, 0, stream>>>(kv_lat, kv_scale, kv_rope, n_pool, slots, new_lat,
                                                                 new_scale, new_rope, n_rows, status);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(__nv_bfloat16* kv, const int32_t* slot, int slot_stride, const int32_t* seq_lens,
                             const __nv_bfloat16* new_kv, int B, int q_len, int64_t n_pool, unsigned* status,
                             cudaStream_t stream) {
    const long long threads = (long long)B * q_len * 32;
    const unsigned blocks = (unsigned)((threads + APPEND_THREADS - 1) / APPEND_THREADS);
    kv_append_kernel<<<blocks, APPEND_THREADS, 0, stream>>>(kv, slot, slot_stride, seq_lens, new_kv, B, q_len,
                                                             n_pool, status);
    return cudaGetLastError();
}

}  // namespace mla
