// KV-split verify attention on the 5th-generation tensor cores (tcgen05, TMEM).
//
// One CTA handles up to 96 query rows (r = t * H + h of one stream) over one key
// split.  Per tile of 32 keys:
//   S   = Q K^T        tcgen05.mma M=128 (query rows) x N=32 (keys) x K=576, fp32 in TMEM
//   P   = softmax(S)   one thread per query row reads its S row from TMEM, applies
//                      the draft mask, keeps a running max / sum (online softmax)
//                      and writes P (bf16) to shared memory
//   O^T += V^T P^T     tcgen05.mma M=128 (value dims) x N=rows x K=32 (keys), four
//                      128-dim chunks, fp32 accumulators resident in TMEM
// Computing P V transposed keeps O^T in 4 x rows <= 384 TMEM columns, so the
// two S buffers (64 columns) fit beside it in the 512-column TMEM and Q K^T is
// computed once per tile.  The same shared-memory key tile is the K-major B
// operand of Q K^T and the M-major A operand of V^T P^T (V = first 512 dims).
//
// Warp roles (256 threads):
//   warp 0      TMEM allocation; lane 0 issues every MMA and commit
//   warps 1-3   slot-table gather of key tiles into a 3-stage ring (warp w owns
//               stage w-1), 16-byte cp.async through the page_size=1 slot table
//   warps 4-7   softmax (thread = query row = TMEM lane) and the epilogue
//               (thread = value dim = TMEM lane of O^T)
// The head-tile amortisation, warp-per-key dot products and NSPLIT tuning of
// "The Occupancy Epiphany" pages are replaced here by packing heads x drafts as
// MMA rows and by the split-count policy of the host code.
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int NK = 32;                               // keys per tile
constexpr int STAGES = 3;                            // key-tile ring
constexpr int MAX_R = 96;                            // query rows per CTA
constexpr int NTHREADS = 256;
constexpr int DB = D_QK / 8;                         // 72 blocks of 8 dims
constexpr int KB_BYTES = DB * 128;                   // one 8-key block of a tile: 9216 B
constexpr int STAGE_BYTES = (NK / 8) * KB_BYTES;     // 36864 B
constexpr uint32_t TMEM_COLS = 512;
constexpr int O_COL0 = 2 * NK;                       // O^T columns start after two S buffers
constexpr float TAU = 8.0f;                          // lazy rescale threshold (log2 units)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// barrier indices
enum { B_KV_FULL = 0, B_KV_EMPTY = 3, B_S_FULL = 6, B_S_FREE = 8, B_P_FULL = 10, B_Q_FULL = 11, N_BARS = 12 };

struct Layout {
    int q_off, kv_off, p_off, misc_off, total;
};

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline Layout layout_for(int R) {
    Layout L;
    L.q_off = 0;
    const int q_bytes = DB * R * 16 + (128 - R) * 16;      // rows R..127 read past the end: a zero tail
    L.kv_off = align_up(q_bytes, 1024);
    L.p_off = L.kv_off + STAGES * STAGE_BYTES;
    L.misc_off = align_up(L.p_off + R * NK * 2, 128);
    L.total = L.misc_off + 128 + 128 + 512 + 512;         // barriers, tmem slot / flags, alpha[], 1/l[]
    return L;
}

struct Misc {
    uint64_t* bars;
    uint32_t* tmem_slot;
    volatile int* abort;
    float* alpha;
    float* rinv;
};

__device__ __forceinline__ Misc misc_at(uint8_t* smem, const Layout& L) {
    Misc m;
    m.bars = reinterpret_cast<uint64_t*>(smem + L.misc_off);
    m.tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc_off + 128);
    m.abort = reinterpret_cast<volatile int*>(smem + L.misc_off + 132);
    m.alpha = reinterpret_cast<float*>(smem + L.misc_off + 256);
    m.rinv = reinterpret_cast<float*>(smem + L.misc_off + 768);
    return m;
}

__device__ __forceinline__ void give_up(const Misc& m, unsigned* status) {
    if (atomicExch(const_cast<int*>(m.abort), 1) == 0) atomicOr(status, DEV_TIMEOUT);
}

__global__ void __launch_bounds__(NTHREADS, 1) verify_tc_kernel(const VerifyArgs a, int R, int R_step) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const Layout L = layout_for(R);
    const Misc M = misc_at(smem, L);
    uint8_t* q_s = smem + L.q_off;
    uint8_t* p_s = smem + L.p_off;
    const uint32_t q_addr = smem_u32(q_s), kv_addr = smem_u32(smem + L.kv_off), p_addr = smem_u32(p_s);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int rows = a.q_len * a.H;
    const int row0 = g * R_step;
    const int nrows = min(R_step, rows - row0);
    const int n = a.seq_lens[b];
    const bool bad_len = n < a.q_len || n > a.slot_stride;
    int k_begin = 0, k_end = 0;
    if (!bad_len) split_range(n, a.nsplit, s, NK, &k_begin, &k_end);
    const int T = (k_end - k_begin + NK - 1) / NK;
    const int p = n - a.q_len;

    // ---- set-up: TMEM, barriers
    if (warp == 0) {
        tmem_alloc(M.tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int i = 0; i < 3; ++i) {
            mbar_init(&M.bars[B_KV_FULL + i], 32);
            mbar_init(&M.bars[B_KV_EMPTY + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&M.bars[B_S_FULL + i], 1);
            mbar_init(&M.bars[B_S_FREE + i], 128);
        }
        mbar_init(&M.bars[B_P_FULL], 128);
        mbar_init(&M.bars[B_Q_FULL], 160);
        *M.abort = 0;
        mbar_init_fence();
        if (bad_len) atomicOr(a.status, DEV_BAD_LEN);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *M.tmem_slot;

    // ---- queries of this CTA's rows -> Q tile (A operand, K-major, no swizzle):
    //      row r, dims 8 db .. 8 db + 7 at db * (R * 16) + r * 16; rows >= nrows and
    //      the tail read by MMA rows R..127 are zero.
    if (warp == 0 || warp >= 4) {
        const int qt = warp == 0 ? lane : tid - 96;          // 0..159
        const __nv_bfloat16* qsrc = a.q + ((int64_t)b * rows + row0) * D_QK;
        for (int idx = qt; idx < DB * R; idx += 160) {
            const int db = idx / R, r = idx % R;
            const uint32_t dst = q_addr + db * (R * 16) + r * 16;
            if (r < nrows) cp_async16(dst, qsrc + (int64_t)r * D_QK + db * 8);
            else *reinterpret_cast<uint4*>(q_s + db * (R * 16) + r * 16) = make_uint4(0, 0, 0, 0);
        }
        for (int i = qt; i < 128 - R; i += 160)
            *reinterpret_cast<uint4*>(q_s + DB * R * 16 + i * 16) = make_uint4(0, 0, 0, 0);
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&M.bars[B_Q_FULL]);
    }

    if (warp == 0) {
        // ================= MMA issuer =================
        if (lane == 0 && T > 0) {
            const uint32_t id_qk = idesc_bf16(128, NK, false, false);
            const uint32_t id_pv = idesc_bf16(128, R, true, false);
            bool ok = mbar_wait(&M.bars[B_Q_FULL], 0, M.abort);
            auto issue_pv = [&](int j) {
                ok = ok && mbar_wait(&M.bars[B_P_FULL], j & 1, M.abort);
                if (!ok) return;
                tc_fence_after();
                const uint32_t st = kv_addr + (j % STAGES) * STAGE_BYTES;
#pragma unroll
                for (int ci = 0; ci < 4; ++ci)
#pragma unroll
                    for (int kk = 0; kk < NK / 16; ++kk) {
                        // A = V^T (M = 128 dims, K = 16 keys), M-major: dim blocks 128 B apart, key blocks KB_BYTES apart
                        const uint64_t ad = smem_desc(st + ci * 16 * 128 + kk * 2 * KB_BYTES, KB_BYTES, 128);
                        // B = P (N = R rows, K = 16 keys), K-major: key blocks R*16 apart, row blocks 128 B apart
                        const uint64_t bd = smem_desc(p_addr + kk * 2 * (R * 16), R * 16, 128);
                        mma_bf16(tmem + O_COL0 + ci * R, ad, bd, id_pv, j > 0 || kk > 0);
                    }
                mma_commit(&M.bars[B_KV_EMPTY + j % STAGES]);
            };
            for (int i = 0; i < T && ok; ++i) {
                const int st = i % STAGES;
                ok = mbar_wait(&M.bars[B_KV_FULL + st], (i / STAGES) & 1, M.abort);
                if (ok && i >= 2) ok = mbar_wait(&M.bars[B_S_FREE + (i & 1)], ((i - 2) >> 1) & 1, M.abort);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kv_st = kv_addr + st * STAGE_BYTES;
#pragma unroll 4
                for (int ks = 0; ks < D_QK / 16; ++ks) {
                    // A = Q (M = 128 rows, K = 16 dims): dim blocks R*16 apart, row blocks 128 B apart
                    const uint64_t ad = smem_desc(q_addr + ks * 2 * (R * 16), R * 16, 128);
                    // B = K tile (N = 32 keys, K = 16 dims): dim blocks 128 B apart, key blocks KB_BYTES apart
                    const uint64_t bd = smem_desc(kv_st + ks * 2 * 128, 128, KB_BYTES);
                    mma_bf16(tmem + (i & 1) * NK, ad, bd, id_qk, ks > 0);
                }
                mma_commit(&M.bars[B_S_FULL + (i & 1)]);
                if (i >= 1) issue_pv(i - 1);
            }
            if (ok) issue_pv(T - 1);
            if (!ok) give_up(M, a.status);
        }
        __syncwarp();
    } else if (warp <= 3) {
        // ================= key-tile gather =================
        const int st = warp - 1;
        bool bad_slot = false;
        const uint32_t dst0 = kv_addr + st * STAGE_BYTES + (lane & 7) * 16;
        for (int i = st; i < T; i += STAGES) {
            if (i >= STAGES && !mbar_wait(&M.bars[B_KV_EMPTY + st], ((i - STAGES) / STAGES) & 1, M.abort)) {
                give_up(M, a.status);
                break;
            }
            const int k0 = k_begin + i * NK;
            int64_t slot[NK / 8];
#pragma unroll
            for (int gk = 0; gk < NK / 8; ++gk) {
                const int j = min(k0 + gk * 8 + (lane & 7), k_end - 1);   // past the split: repeat a valid key
                int64_t sl = a.slot[(int64_t)b * a.slot_stride + j];
                if (sl < 0 || sl >= a.n_pool) { bad_slot = true; sl = 0; }
                slot[gk] = sl;
            }
#pragma unroll
            for (int gk = 0; gk < NK / 8; ++gk) {
                const __nv_bfloat16* src = a.kv + slot[gk] * D_QK;
#pragma unroll 6
                for (int it = 0; it < DB / 4; ++it) {
                    const int pc = it * 4 + (lane >> 3);           // 16-byte piece = dim block
                    cp_async16(dst0 + gk * KB_BYTES + pc * 128, src + pc * 8);
                }
            }
            cp_async_wait_all();
            fence_proxy_async_smem();
            mbar_arrive(&M.bars[B_KV_FULL + st]);
        }
        if (bad_slot) atomicOr(a.status, DEV_BAD_SLOT);
    } else {
        // ================= softmax + epilogue =================
        const int sw = warp - 4;                       // TMEM lane quadrant
        const int r = sw * 32 + lane;                  // query row of this thread (S lane)
        const uint32_t lane_base = (uint32_t)(sw * 32) << 16;
        const bool row_ok = r < nrows;
        const int t = row_ok ? (row0 + r) / a.H : 0;
        unsigned vis = 0;
        if (row_ok)
            for (int d = 0; d < a.q_len; ++d) {
                const bool seen = a.mask ? a.mask[((int64_t)b * a.q_len + t) * a.q_len + d] != 0 : d <= t;
                vis |= (seen ? 1u : 0u) << d;
            }
        const float c2 = a.scale * LOG2E;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < T; ++i) {
            ok = mbar_wait(&M.bars[B_S_FULL + (i & 1)], (i >> 1) & 1, M.abort);
            if (bar_red_or(1, 128, !ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t sv[NK];
            tmem_ld32(tmem + lane_base + (i & 1) * NK, sv);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&M.bars[B_S_FREE + (i & 1)]);

            const int k0 = k_begin + i * NK;
            float x[NK];
            float mt = -INFINITY;
#pragma unroll
            for (int k = 0; k < NK; ++k) {
                const int j = k0 + k;
                const bool vk = row_ok && j < k_end && (j < p || ((vis >> (j - p)) & 1u));
                x[k] = vk ? __uint_as_float(sv[k]) * c2 : -INFINITY;
                mt = fmaxf(mt, x[k]);
            }
            const bool need = mt > m + TAU;
            float alpha = 1.f;
            if (need) {
                alpha = exp2f(m - mt);
                l *= alpha;
                m = mt;
            }
            const bool any = bar_red_or(1, 128, need);
            if (i >= 1) ok = mbar_wait(&M.bars[B_KV_EMPTY + (i - 1) % STAGES], ((i - 1) / STAGES) & 1, M.abort);
            if (bar_red_or(1, 128, !ok)) { ok = false; break; }
            if (any && i >= 1) {
                // O^T column r (query row r) *= alpha_r; thread = TMEM lane = value dim
                M.alpha[r] = alpha;
                bar_sync(2, 128);
                tc_fence_after();
                for (int ci = 0; ci < 4; ++ci)
                    for (int c0 = 0; c0 < R; c0 += 16) {
                        uint32_t v[16];
                        const uint32_t ta = tmem + lane_base + O_COL0 + ci * R + c0;
                        tmem_ld16(ta, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) v[jj] = __float_as_uint(__uint_as_float(v[jj]) * M.alpha[c0 + jj]);
                        tmem_st16(ta, v);
                    }
                tmem_st_wait();
            }
            const float mu = m == -INFINITY ? 0.f : m;
            uint32_t pk[NK / 2];
            float ladd = 0.f;
#pragma unroll
            for (int k = 0; k < NK; k += 2) {
                const float p0 = exp2f(x[k] - mu), p1 = exp2f(x[k + 1] - mu);
                ladd += p0 + p1;                        // the row sum keeps fp32 probabilities
                __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                pk[k / 2] = *reinterpret_cast<uint32_t*>(&h);
            }
            l += ladd;
            if (r < R) {
                // P (B operand, K-major): keys 8 kb .. 8 kb + 7 of row r at kb * (R * 16) + r * 16
#pragma unroll
                for (int kb = 0; kb < NK / 8; ++kb)
                    *reinterpret_cast<uint4*>(p_s + kb * (R * 16) + r * 16) =
                        make_uint4(pk[4 * kb], pk[4 * kb + 1], pk[4 * kb + 2], pk[4 * kb + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&M.bars[B_P_FULL]);
        }
        if (ok && T > 0) ok = mbar_wait(&M.bars[B_KV_EMPTY + (T - 1) % STAGES], ((T - 1) / STAGES) & 1, M.abort);
        const bool failed = bar_red_or(1, 128, !ok);
        if (failed) give_up(M, a.status);
        tc_fence_after();

        float inv, lse_v;
        if (bad_len) { inv = 0.f; lse_v = __int_as_float(0x7fc00000); }
        else if (l > 0.f) { inv = 1.f / l; lse_v = (m + log2f(l)) * LN2; }
        else { inv = 0.f; lse_v = -INFINITY; }
        M.rinv[r] = inv;
        const int64_t grow = (int64_t)b * rows + row0 + r;
        if (row_ok) {
            if (a.nsplit == 1) a.lse[grow] = lse_v;
            else a.part_lse[grow * a.nsplit + s] = lse_v;
        }
        bar_sync(2, 128);
        const bool have_o = T > 0 && !failed;
        const int64_t grow0 = (int64_t)b * rows + row0;
        for (int ci = 0; ci < 4; ++ci) {
            const int dim = ci * 128 + sw * 32 + lane;
            for (int c0 = 0; c0 < nrows; c0 += 16) {
                uint32_t v[16];
                if (have_o) {
                    tmem_ld16(tmem + lane_base + O_COL0 + ci * R + c0, v);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) v[jj] = 0u;
                }
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int rr = c0 + jj;
                    if (rr < nrows) {
                        float* dst = a.nsplit == 1 ? a.out + (grow0 + rr) * D_V
                                                   : a.part_out + ((grow0 + rr) * a.nsplit + s) * D_V;
                        dst[dim] = __uint_as_float(v[jj]) * M.rinv[rr];
                    }
                }
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

void tc_tiling(int rows, int* n_tiles, int* R_step, int* R) {
    *n_tiles = (rows + MAX_R - 1) / MAX_R;
    *R_step = (rows + *n_tiles - 1) / *n_tiles;
    *R = (*R_step + 15) / 16 * 16;
}

cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream) {
    static bool attr_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 layout_for(MAX_R).total);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    int n_tiles, R_step, R;
    tc_tiling(a.q_len * a.H, &n_tiles, &R_step, &R);
    dim3 grid(a.nsplit, n_tiles, a.B);
    verify_tc_kernel<<<grid, NTHREADS, layout_for(R).total, stream>>>(a, R, R_step);
    return cudaGetLastError();
}

int tc_smem_bytes(int R) { return layout_for(R).total; }

}  // namespace mla
