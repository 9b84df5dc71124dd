// Test-only probes of the tensor-core and TMA building blocks of the verify kernel.
//
// umma_probe: D[128 x N] = A[128 x K] * B[N x K]^T with bf16 operands staged by
//   hand into canonical shared-memory layouts -- A K-major or M-major, each without
//   swizzle or with the 128-byte swizzle; B K-major without or with swizzle --
//   multiplied by tcgen05.mma into TMEM and read back with tcgen05.ld.  For the
//   M-major A the two stride fields can be passed swapped, so one run shows which
//   field strides along M and which along K.  a_mode 2 puts A in TMEM instead (lane =
//   row, two consecutive K elements per 32-bit column, written with tcgen05.st), the
//   form used when the query tile stays in tensor memory.  Every variant reads only
//   inside its own shared-memory region and its own TMEM columns.
// tma_tile_probe: rows [row0, row0 + R) of a [n, 576] bf16 matrix loaded with nine
//   2-D tile copies (box 64 columns x R rows, 128-byte swizzle) into nine regions of
//   R x 128 B; the raw shared-memory bytes are copied out.
// fp8_decode_probe: the fp8 key path's e4m3 -> bf16 decoder applied to n codes (n a
//   multiple of 16), sixteen per thread, bf16 bit patterns out; with scales, the scaled
//   decoder of the widening warps, group i of sixteen codes times scales[i].
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../mla_speculative_verify_attention_gb300/csrc/fp8_decode.cuh"

#include "../../mla_speculative_verify_attention_gb300/csrc/tc_ptx.cuh"
#include "../../mla_speculative_verify_attention_gb300/csrc/tmap.h"

using namespace mla::tc;

namespace {

constexpr int M = 128;
constexpr int A_BYTES = 64 * 1024;
constexpr int B_BYTES = 32 * 1024;

// byte offset of element (row, col) of a K-major operand whose K extent is split into
// 64-element swizzled regions of `rows` rows each (rows a multiple of 8)
__device__ uint32_t off_sw128_kmajor(int row, int col, int rows) {
    int region = col / 64, c = (col % 64) / 8;
    return region * rows * 128 + (row / 8) * 1024 + (row % 8) * 128 + ((c ^ (row % 8)) * 16) + (col % 8) * 2;
}

__global__ void __launch_bounds__(128) probe_kernel(const uint16_t* A, const uint16_t* B, float* D, int N, int K,
                                                    int a_mode, int a_sw, int b_sw, int swap, int* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sa = smem;
    uint8_t* sb = smem + A_BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + A_BYTES + B_BYTES);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + A_BYTES + B_BYTES + 64);
    int& abort_flag = *reinterpret_cast<int*>(smem + A_BYTES + B_BYTES + 96);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (smem_u32(smem) & 1023u) {            // the swizzled layouts below assume a 1024-byte aligned base
        if (tid == 0) atomicOr(status, 8);
        return;
    }

    for (int i = tid; i < (A_BYTES + B_BYTES) / 4; i += 128) reinterpret_cast<uint32_t*>(smem)[i] = 0;
    __syncthreads();
    for (int i = tid; i < M * K && a_mode != 2; i += 128) {
        int m = i / K, k = i % K;
        uint32_t off;
        if (a_mode == 0 && a_sw == 0) off = (k / 8) * 2048 + (m / 8) * 128 + (m % 8) * 16 + (k % 8) * 2;
        else if (a_mode == 1 && a_sw == 0) off = (k / 8) * 2048 + (m / 8) * 128 + (k % 8) * 16 + (m % 8) * 2;
        else if (a_mode == 0) off = off_sw128_kmajor(m, k, M);
        else off = off_sw128_kmajor(k, m, K);      // M-major: rows are K, the 64-wide regions run along M
        *reinterpret_cast<uint16_t*>(sa + off) = A[i];
    }
    for (int i = tid; i < N * K; i += 128) {
        int n = i / K, k = i % K;
        uint32_t off = b_sw ? off_sw128_kmajor(n, k, N)
                            : (k / 8) * (N * 16) + (n / 8) * 128 + (n % 8) * 16 + (k % 8) * 2;
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
    constexpr uint32_t A_COL = 256;                  // A in TMEM: columns 256 .. 256 + K / 2
    if (a_mode == 2) {
        // thread = row m = TMEM lane (warp w reaches lanes 32 w .. 32 w + 31)
        const int m = tid;
        for (int c0 = 0; c0 < K / 2; c0 += 16) {
            uint32_t r[16];
            for (int j = 0; j < 16; ++j) {
                const int k = 2 * (c0 + j);
                r[j] = (uint32_t)A[m * K + k] | ((uint32_t)A[m * K + k + 1] << 16);
            }
            tmem_st16(tmem + ((uint32_t)(32 * warp) << 16) + A_COL + c0, r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    if (tid == 0) {
        const uint32_t idesc = idesc_bf16(M, N, a_mode == 1, false);
        const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
        for (int ks = 0; ks < K / 16; ++ks) {
            uint64_t ad, bd;
            if (a_sw == 0) {
                uint32_t a_lbo = 2048, a_sbo = 128;                  // along K, along M
                if (a_mode == 1 && swap) { a_lbo = 128; a_sbo = 2048; }
                ad = smem_desc(a0 + ks * 2 * 2048, a_lbo, a_sbo);
            } else if (a_mode == 0) {
                ad = smem_desc_sw128(a0 + (ks / 4) * M * 128 + (ks % 4) * 32, 16, 1024);
            } else {
                uint32_t lbo = K * 128, sbo = 1024;                 // between 64-wide M chunks, between 8-row K groups
                if (swap) { lbo = 1024; sbo = K * 128; }
                ad = smem_desc_sw128(a0 + ks * 2048, lbo, sbo);
            }
            if (b_sw == 0) bd = smem_desc(b0 + ks * 2 * (N * 16), N * 16, 128);
            else bd = smem_desc_sw128(b0 + (ks / 4) * N * 128 + (ks % 4) * 32, 16, 1024);
            if (a_mode == 2) mma_bf16_ta(tmem, tmem + A_COL + ks * 8, bd, idesc, ks > 0);
            else mma_bf16(tmem, ad, bd, idesc, ks > 0);
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

__global__ void __launch_bounds__(128) tma_probe_kernel(const __grid_constant__ CUtensorMap map, int row0, int R,
                                                        uint8_t* out, int* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int DATA = 9 * 128 * 128;
    uint64_t& bar = *reinterpret_cast<uint64_t*>(smem + DATA);
    int& abort_flag = *reinterpret_cast<int*>(smem + DATA + 8);
    const int tid = threadIdx.x;
    const uint32_t bytes = 9 * R * 128;
    if (smem_u32(smem) & 1023u) {            // TMA destinations and the swizzle phase need an aligned base
        if (tid == 0) atomicOr(status, 8);
        return;
    }
    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar, bytes);
        const uint32_t s0 = smem_u32(smem);
        for (int c = 0; c < 9; ++c) tma_load_2d(s0 + c * R * 128, &map, c * 64, row0, &bar);
    }
    bool ok = mbar_wait(&bar, 0, &abort_flag);
    if (!ok && tid == 0) atomicOr(status, 4);
    for (uint32_t i = tid; i < bytes / 16; i += 128)
        reinterpret_cast<uint4*>(out)[i] = ok ? reinterpret_cast<const uint4*>(smem)[i] : make_uint4(0, 0, 0, 0);
}

__global__ void fp8_decode_kernel(const uint4* codes, uint4* out, int groups) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= groups) return;
    uint4 lo, hi;
    mla::e4m3x16_to_bf16(codes[i], lo, hi);
    out[2 * i] = lo;
    out[2 * i + 1] = hi;
}

__global__ void fp8_decode_scaled_kernel(const uint4* codes, const float* scales, uint4* out, int groups) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= groups) return;
    uint4 lo, hi;
    mla::e4m3x16_to_bf16_scaled(codes[i], scales[i], lo, hi);
    out[2 * i] = lo;
    out[2 * i + 1] = hi;
}

}  // namespace

// codes: n e4m3 bytes, out: n bf16 bit patterns; both device pointers, 16-byte aligned
extern "C" int fp8_decode_probe(const uint8_t* codes, uint16_t* out, int n, cudaStream_t stream) {
    if (n <= 0 || n % 16 || ((uintptr_t)codes | (uintptr_t)out) % 16) return -2;
    const int groups = n / 16;
    fp8_decode_kernel<<<(groups + 127) / 128, 128, 0, stream>>>(reinterpret_cast<const uint4*>(codes),
                                                               reinterpret_cast<uint4*>(out), groups);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}

// as fp8_decode_probe, codes of group i (sixteen codes) times scales[i] (n / 16 floats)
extern "C" int fp8_decode_scaled_probe(const uint8_t* codes, const float* scales, uint16_t* out, int n,
                                       cudaStream_t stream) {
    if (n <= 0 || n % 16 || ((uintptr_t)codes | (uintptr_t)out) % 16 || (uintptr_t)scales % 4) return -2;
    const int groups = n / 16;
    fp8_decode_scaled_kernel<<<(groups + 127) / 128, 128, 0, stream>>>(
        reinterpret_cast<const uint4*>(codes), scales, reinterpret_cast<uint4*>(out), groups);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}

extern "C" int umma_probe(const uint16_t* A, const uint16_t* B, float* D, int N, int K, int a_mode, int a_sw,
                          int b_sw, int swap, int* status, cudaStream_t stream) {
    if (N < 16 || N > 256 || N % 16 || K < 16 || K > 64 || K % 16) return -2;
    if (a_sw && a_mode == 0 && K != 64) return -2;
    if (a_mode < 0 || a_mode > 2 || (a_mode == 2 && (K % 32 || a_sw))) return -2;
    if (b_sw && K != 64) return -2;
    const int smem = A_BYTES + B_BYTES + 128;
    cudaError_t e = cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return -7;
    probe_kernel<<<1, 128, smem, stream>>>(A, B, D, N, K, a_mode, a_sw, b_sw, swap, status);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}

// rows [row0, row0 + R) of src [n, 576] bf16 (R a multiple of 8, <= 128, row0 + R <= n)
extern "C" int tma_tile_probe(const void* src, long long n, int row0, int R, uint8_t* out, int* status,
                              cudaStream_t stream) {
    if (R < 8 || R > 128 || R % 8 || row0 < 0 || row0 + R > n) return -2;
    CUtensorMap map;
    if (!mla::encode_bf16_2d_sw128(&map, src, 576, (uint64_t)n, 1152, 64, R, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
        return -7;
    const int smem = 9 * 128 * 128 + 64;
    cudaError_t e = cudaFuncSetAttribute(tma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return -7;
    tma_probe_kernel<<<1, 128, smem, stream>>>(map, row0, R, out, status);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}
