// Test-only probe of the tensor-core building blocks the verify kernel uses:
// D[128 x N] = A[128 x K] * B[N x K]^T with bf16 operands staged into the
// canonical no-swizzle shared-memory layouts (A K-major or M-major, B K-major),
// accumulated by tcgen05.mma in TMEM and read back with tcgen05.ld.
// For the M-major A the two stride fields can be passed swapped, so one run
// shows which descriptor field strides along M and which along K.  Every
// variant reads only inside its own 64 KB shared-memory region.
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../mla_speculative_verify_attention_gb300/csrc/tc_ptx.cuh"

using namespace mla::tc;

namespace {

constexpr int M = 128;
constexpr int A_BYTES = 64 * 1024;
constexpr int B_BYTES = 32 * 1024;

__global__ void __launch_bounds__(128) probe_kernel(const uint16_t* A, const uint16_t* B, float* D, int N, int K,
                                                    int a_mode, int swap, int* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sa = smem;
    uint8_t* sb = smem + A_BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + A_BYTES + B_BYTES);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + A_BYTES + B_BYTES + 64);
    __shared__ int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int i = tid; i < (A_BYTES + B_BYTES) / 4; i += 128) reinterpret_cast<uint32_t*>(smem)[i] = 0;
    __syncthreads();
    // A: element (m, k).  K-major: core (m/8, k/8) at (k/8)*2048 + (m/8)*128, row m%8 at 16 B, k%8 at 2 B.
    //    M-major: core (m/8, k/8) at (k/8)*2048 + (m/8)*128, row k%8 at 16 B, m%8 at 2 B.
    for (int i = tid; i < M * K; i += 128) {
        int m = i / K, k = i % K;
        uint32_t off = (k / 8) * 2048 + (m / 8) * 128;
        off += a_mode == 0 ? (m % 8) * 16 + (k % 8) * 2 : (k % 8) * 16 + (m % 8) * 2;
        *reinterpret_cast<uint16_t*>(sa + off) = A[i];
    }
    // B: element (n, k), K-major: core (n/8, k/8) at (k/8)*(N*16) + (n/8)*128.
    for (int i = tid; i < N * K; i += 128) {
        int n = i / K, k = i % K;
        uint32_t off = (k / 8) * (N * 16) + (n / 8) * 128 + (n % 8) * 16 + (k % 8) * 2;
        *reinterpret_cast<uint16_t*>(sb + off) = B[i];
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (tid == 0) {
        uint32_t a_lbo = 2048, a_sbo = 128;                  // along K, along M
        if (a_mode == 1 && swap) { a_lbo = 128; a_sbo = 2048; }
        const uint32_t idesc = idesc_bf16(M, N, a_mode == 1, false);
        for (int ks = 0; ks < K / 16; ++ks) {
            uint64_t ad = smem_desc(smem_u32(sa) + ks * 2 * 2048, a_lbo, a_sbo);
            uint64_t bd = smem_desc(smem_u32(sb) + ks * 2 * (N * 16), N * 16, 128);
            mma_bf16(tmem, ad, bd, idesc, ks > 0);
        }
        mma_commit(bar);
    }
    __syncwarp();
    bool ok = mbar_wait(bar, 0, &abort_flag);
    tc_fence_after();
    if (!ok) {
        if (lane == 0) atomicOr(status, 4);
    } else {
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + c0, r);
            tmem_ld_wait();
            int row = 32 * warp + lane;
            for (int j = 0; j < 16; ++j) D[row * N + c0 + j] = __uint_as_float(r[j]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

extern "C" int umma_probe(const uint16_t* A, const uint16_t* B, float* D, int N, int K, int a_mode, int swap,
                          int* status, cudaStream_t stream) {
    if (N < 16 || N > 256 || N % 16 || K < 16 || K > 64 || K % 16) return -2;
    const int smem = A_BYTES + B_BYTES + 128;
    cudaError_t e = cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return -7;
    probe_kernel<<<1, 128, smem, stream>>>(A, B, D, N, K, a_mode, swap, status);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}
