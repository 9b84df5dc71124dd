// KV-split verify attention on the CUDA cores (FP32 FMA): the first, simple
// split stage of the library.  One CTA handles 16 query rows of one stream over
// one key split.  Key tiles of 32 rows are gathered through the slot table with
// 16-byte cp.async copies into shared memory (double buffered); each warp owns
// two query rows, computes one key's 576-d dot product per lane (the warp-per-key
// idea of "The Occupancy Epiphany: How a CUDA Kernel Designer Discovered ...",
// section "The Warp-Per-Key Dot Product", turned so that the warp spans keys),
// keeps a running max / sum per row with warp-shuffle reductions (online
// softmax) and accumulates P V in registers, 16 output dims per lane per row.
#include "internal.cuh"

namespace mla {
namespace {

constexpr int NTHREADS = 256;
constexpr int KROW = D_QK + 8;                                   // bf16 per smem key row (1168 B, bank-spread)
constexpr int SMEM_Q = SIMT_ROWS * D_QK * 4;                     // fp32 queries
constexpr int SMEM_KV = 2 * SIMT_NK * KROW * 2;                  // two bf16 key tiles
constexpr int SMEM_TOTAL = SMEM_Q + SMEM_KV;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Gather key tile [k0, k0 + 32) of stream b (keys >= k_end repeat key k_end-1,
// which keeps the smem rows finite; they are masked out of the softmax).
__device__ __forceinline__ void load_tile(const VerifyArgs& a, int b, int k0, int k_end,
                                          __nv_bfloat16* dst, bool& bad_slot) {
    const int tid = threadIdx.x;
    // 32 keys x 72 pieces of 16 bytes; consecutive threads copy consecutive pieces of a key row
    for (int idx = tid; idx < SIMT_NK * (D_QK / 8); idx += NTHREADS) {
        int kk = idx / (D_QK / 8);
        int c = idx % (D_QK / 8);
        int j = min(k0 + kk, k_end - 1);
        int64_t slot = a.slot[(int64_t)b * a.slot_stride + j];
        if (slot < 0 || slot >= a.n_pool) { bad_slot = true; slot = 0; }
        cp_async16(dst + kk * KROW + c * 8, a.kv + slot * D_QK + c * 8);
    }
}

__global__ void __launch_bounds__(NTHREADS, 2) verify_simt_kernel(const VerifyArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    float* qs = reinterpret_cast<float*>(smem);
    __nv_bfloat16* kvs = reinterpret_cast<__nv_bfloat16*>(smem + SMEM_Q);

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows = a.q_len * a.H;
    const int n = a.seq_lens[b];
    const bool bad_len = n < a.q_len || n > a.slot_stride;
    int k_begin = 0, k_end = 0;
    if (!bad_len) split_range(n, a.nsplit, s, SIMT_NK, &k_begin, &k_end);
    const int p = n - a.q_len;

    // queries of this CTA's 16 rows, as fp32
    for (int idx = tid; idx < SIMT_ROWS * (D_QK / 8); idx += NTHREADS) {
        int rr = idx / (D_QK / 8), c = idx % (D_QK / 8);
        int r = g * SIMT_ROWS + rr;
        float f[8];
        if (r < rows) {
            uint4 u = *reinterpret_cast<const uint4*>(a.q + ((int64_t)b * rows + r) * D_QK + c * 8);
            bf16x8_to_f32(u, f);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) qs[rr * D_QK + c * 8 + i] = f[i];
    }

    // per-warp rows and their draft visibility bits
    int rloc[2], rglob[2];
    unsigned vis[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        rloc[i] = warp * 2 + i;
        rglob[i] = g * SIMT_ROWS + rloc[i];
        int t = min(rglob[i], rows - 1) / a.H;
        unsigned v = 0;
        for (int d = 0; d < a.q_len; ++d) {
            bool seen = a.mask ? a.mask[((int64_t)b * a.q_len + t) * a.q_len + d] != 0 : d <= t;
            v |= (seen ? 1u : 0u) << d;
        }
        vis[i] = v;
    }

    const float c2 = a.scale * LOG2E;          // scores in log2 units
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[2][16];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int d = 0; d < 16; ++d) o[i][d] = 0.f;

    bool bad_slot = false;
    const int ntiles = (k_end - k_begin + SIMT_NK - 1) / SIMT_NK;
    if (ntiles > 0) load_tile(a, b, k_begin, k_end, kvs, bad_slot);
    cp_async_commit();

    for (int it = 0; it < ntiles; ++it) {
        const int k0 = k_begin + it * SIMT_NK;
        __nv_bfloat16* cur = kvs + (it & 1) * SIMT_NK * KROW;
        if (it + 1 < ntiles) load_tile(a, b, k0 + SIMT_NK, k_end, kvs + ((it + 1) & 1) * SIMT_NK * KROW, bad_slot);
        cp_async_commit();
        cp_async_wait1();
        __syncthreads();

        // scores: lane = key, two rows per warp
        const uint4* krow = reinterpret_cast<const uint4*>(cur + lane * KROW);
        const float4* q0 = reinterpret_cast<const float4*>(qs + rloc[0] * D_QK);
        const float4* q1 = reinterpret_cast<const float4*>(qs + rloc[1] * D_QK);
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
        for (int c = 0; c < D_QK / 8; ++c) {
            float kf[8];
            bf16x8_to_f32(krow[c], kf);
            float4 a0 = q0[2 * c], a1 = q0[2 * c + 1], b0 = q1[2 * c], b1 = q1[2 * c + 1];
            acc0 += a0.x * kf[0] + a0.y * kf[1] + a0.z * kf[2] + a0.w * kf[3] +
                    a1.x * kf[4] + a1.y * kf[5] + a1.z * kf[6] + a1.w * kf[7];
            acc1 += b0.x * kf[0] + b0.y * kf[1] + b0.z * kf[2] + b0.w * kf[3] +
                    b1.x * kf[4] + b1.y * kf[5] + b1.z * kf[6] + b1.w * kf[7];
        }
        const int j = k0 + lane;
        float pj[2];
        float accs[2] = {acc0, acc1};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            bool ok = j < k_end && rglob[i] < rows && (j < p || ((vis[i] >> (j - p)) & 1u));
            float sc = ok ? accs[i] * c2 : -INFINITY;
            float mt = warp_max(sc);
            float mn = fmaxf(m[i], mt);
            float mu = mn == -INFINITY ? 0.f : mn;
            float alpha = exp2f(m[i] - mu);
            pj[i] = exp2f(sc - mu);
            l[i] = l[i] * alpha + warp_sum(pj[i]);
            m[i] = mn;
#pragma unroll
            for (int d = 0; d < 16; ++d) o[i][d] *= alpha;
        }
        // P V: lane owns dims 4 lane + 128 q (q = 0..3)
#pragma unroll 4
        for (int kk = 0; kk < SIMT_NK; ++kk) {
            float p0 = __shfl_sync(0xffffffffu, pj[0], kk);
            float p1 = __shfl_sync(0xffffffffu, pj[1], kk);
            const __nv_bfloat16* vrow = cur + kk * KROW;
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                uint2 u = *reinterpret_cast<const uint2*>(vrow + qd * 128 + lane * 4);
                float v0 = __uint_as_float(u.x << 16), v1 = __uint_as_float(u.x & 0xffff0000u);
                float v2 = __uint_as_float(u.y << 16), v3 = __uint_as_float(u.y & 0xffff0000u);
                o[0][qd * 4 + 0] += p0 * v0; o[0][qd * 4 + 1] += p0 * v1;
                o[0][qd * 4 + 2] += p0 * v2; o[0][qd * 4 + 3] += p0 * v3;
                o[1][qd * 4 + 0] += p1 * v0; o[1][qd * 4 + 1] += p1 * v1;
                o[1][qd * 4 + 2] += p1 * v2; o[1][qd * 4 + 3] += p1 * v3;
            }
        }
        __syncthreads();
    }
    cp_async_wait0();

    if (bad_slot) atomicOr(a.status, DEV_BAD_SLOT);
    if (bad_len && tid == 0) atomicOr(a.status, DEV_BAD_LEN);

#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = rglob[i];
        if (r >= rows) continue;
        float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
        float lse_v = l[i] > 0.f ? (m[i] + log2f(l[i])) * LN2 : -INFINITY;
        if (bad_len) { inv = 0.f; lse_v = __int_as_float(0x7fc00000); }
        float* dst;
        const int64_t row = (int64_t)b * rows + r;
        if (a.nsplit == 1) {
            dst = a.out + row * D_V;
            if (lane == 0) a.lse[row] = lse_v;
        } else {
            dst = a.part_out + (row * a.nsplit + s) * D_V;
            if (lane == 0) a.part_lse[row * a.nsplit + s] = lse_v;
        }
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
            float4 v = make_float4(o[i][qd * 4] * inv, o[i][qd * 4 + 1] * inv, o[i][qd * 4 + 2] * inv,
                                   o[i][qd * 4 + 3] * inv);
            *reinterpret_cast<float4*>(dst + qd * 128 + lane * 4) = v;
        }
    }
}

}  // namespace

cudaError_t launch_verify_simt(const VerifyArgs& a, cudaStream_t stream) {
    static bool attr_set[64];           // the attribute is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(verify_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int rows = a.q_len * a.H;
    dim3 grid(a.nsplit, (rows + SIMT_ROWS - 1) / SIMT_ROWS, a.B);
    verify_simt_kernel<<<grid, NTHREADS, SMEM_TOTAL, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace mla
