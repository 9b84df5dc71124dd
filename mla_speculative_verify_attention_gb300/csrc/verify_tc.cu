// KV-split verify attention on the 5th-generation tensor cores (tcgen05, TMEM).
//
// One CTA handles up to 96 query rows (r = t * H + h of one stream) over one key
// split.  Per tile of 32 keys:
//   gather   four warps copy the tile's 32 key rows (slot-table indexed, 576 bf16
//            each) with 16-byte cp.async into a 128-byte-swizzled shared-memory
//            stage; arrivals are asynchronous, so a warp moves on to the next tile
//            while its copies are in flight (measured on GB300: random 1152-byte
//            rows gather about twice as fast this way as with TMA tile::gather4,
//            whose per-instruction cost caps a 512-byte gather).  fp8 keys: two more
//            warps copy the raw rows (e4m3 latent, bf16 rope, fp32 scale) by cp.async
//            into a ring of raw slots up to a few tiles ahead, and the four gather
//            warps widen them into the same bf16 stage layout, each latent value
//            multiplied by its key's scale (bf16(scale_t * code), relative error at
//            most 2^-8; the rope dims are bf16 already), so from there on both paths
//            are the same
//   S        = Q K^T: tcgen05.mma M=128 (query rows) x N=32 (keys) x K=576, fp32 in TMEM;
//            the first 64-dim chunks of Q sit in TMEM (A operand read from tensor
//            memory, no shared-memory traffic), the rest in shared memory
//   P        = softmax(S): one thread per query row reads its S row from TMEM, applies
//            the draft mask, keeps a running max / sum (online softmax) and writes
//            P (bf16) to a shared-memory buffer; it waits for P V of the previous tile
//            only when the running max moved enough to rescale O^T or when P has one
//            buffer, so softmax of tile i otherwise overlaps P V of tile i - 1
//   O^T     += V^T P^T: tcgen05.mma M=128 (value dims) x N=rows x K=32 (keys), four
//            128-dim chunks, fp32 accumulators resident in TMEM
// Computing P V transposed keeps O^T in 4 x rows <= 384 TMEM columns, so the S
// buffers (one or two of 32 columns) fit beside it in the 512-column TMEM and Q K^T
// runs once per tile; the columns left over hold as many 32-column Q chunks as fit
// (bf16: 5 up to 80 rows with one S buffer, 2 at 96 with two; fp8: 7 up to 64 rows, 5
// at 80).  Measured on GB300, an M=128 x N=32 x K=16 MMA issued from a converged warp
// takes ~17 cycles with A in TMEM and ~40 with A in shared memory (bound by
// shared-memory reads of the 4 KB A tile), so every Q chunk moved to TMEM takes four MMAs
// off the shared-memory port, and the freed shared memory buys key stages: five for up
// to 80 bf16 rows (one P buffer), three at 96 rows and on the fp8 path.  The same
// swizzled key stage is the K-major B operand of Q K^T and the M-major A operand of
// V^T P^T (V = first 512 dims of each key row).
//
// Warp roles (320 threads; 384 on the fp8 path):
//   warp 0      TMEM allocation; Q K^T issue loop run by the whole warp (operands stay
//               warp-uniform), one elected lane issuing each MMA and commit
//   warp 1      TMA copies of the shared-memory part of the Q tile (64-dim boxes of R
//               rows), then the P V issue loop in the same style
//   warps 2-5   Q chunks into TMEM (thread = query row), softmax (thread = query row =
//               TMEM lane) and the epilogue (thread = value dim = TMEM lane of O^T);
//               TMEM lane quadrant = warp % 4
//   warps 6-9   key-tile gather into the stage ring (bf16) or widening of the raw rows
//               (fp8); warp 6 + w handles keys 8w .. 8w+7
//   warps 10-11 fp8 only: raw-row copies, warp 10 + c keys 16c .. 16c+15
// Every role initialises its own mbarriers and starts its first cold reads (Q, slot
// indices, key rows) before the block-wide set-up barrier, which the gather warps only
// arrive at.
// The pages' sm_120 designs (head-tile amortisation, warp-per-key dot products,
// NSPLIT tuning) are replaced by packing heads x drafts as MMA rows, a slot-table
// gather sized to the SM's load path, and the split-count policy of the host code.
#include <cuda_fp8.h>

#include "fp8_decode.cuh"
#include "internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace tc;

constexpr int NK = 32;                               // keys per tile
constexpr int MAX_R = 96;                            // query rows per CTA
constexpr int NTHREADS = 320;                        // bf16 path: ten warps
constexpr int GATHER_WARPS = 4;
// fp8 path: two more warps (10, 11) copy the raw rows, so warps 6-9 only widen.  Twelve
// warps still give a thread the 168 registers of three warps per SM sub-partition.
template <bool FP8> constexpr int block_threads() { return FP8 ? NTHREADS + 64 : NTHREADS; }
constexpr int NCHUNK = D_QK / 64;                    // 9 swizzled 64-dim regions per row
constexpr int REGION = NK * 128;                     // one 64-dim region of a stage: 4096 B
constexpr int STAGE_BYTES = NCHUNK * REGION;         // 36864 B
// fp8 path: raw slot of one key tile as read from memory, before widening to bf16
constexpr int RAW_ROPE = NK * D_V;                   // e4m3 latents [NK][512], then
constexpr int RAW_SCALE = RAW_ROPE + NK * 128;       // bf16 ropes [NK][64], then
constexpr int RAW_SLOT = RAW_SCALE + NK * 4;         // fp32 scales [NK]: 20608 B
constexpr int MAX_RAW_SLOTS = 4;
constexpr uint32_t TMEM_COLS = 512;
// TMEM columns: S buffers first (32 columns each), then O^T, then Q chunks.
// S buffers (SB) and P buffers (PB) per instantiation.  Two S buffers let Q K^T of the
// next tile run ahead of the softmax; two P buffers let the softmax of tile i write P
// while P V of tile i - 1 still reads the other.  One S buffer leaves a Q chunk's worth
// more of TMEM columns.  The five-stage bf16 variant takes one S and one P buffer: the
// TMEM columns and shared memory they free hold a fifth Q chunk in TMEM and a fifth key
// stage.
constexpr float TAU = 8.0f;                          // lazy rescale threshold (log2 units)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// mbarriers: key-stage full / empty per stage, then the fixed ones
template <int STAGES> struct Bars {
    static constexpr int KV_FULL = 0, KV_EMPTY = STAGES, S_FULL = 2 * STAGES, S_FREE = 2 * STAGES + 2,
                         P_FULL = 2 * STAGES + 4, Q_FULL = 2 * STAGES + 6, QT_FULL = 2 * STAGES + 7,
                         RAW_FULL = 2 * STAGES + 8, RAW_EMPTY = 2 * STAGES + 12,   // fp8 raw slots
                         COUNT = 2 * STAGES + 16;   // S_FULL / S_FREE / P_FULL: one per buffer
};
constexpr int BAR_BYTES = 256;
static_assert(Bars<5>::COUNT * 8 <= BAR_BYTES, "barrier area");

struct Layout {
    int q_off, kv_off, p_off, misc_off, total;
};

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Q: the nq_s shared-memory chunks, regions of R rows x 128 B (MMA rows R..127 read on
// into the next region and, past the last one, into the key stages: those rows' scores
// are never used).  Then the key stages, the pb P buffers and the small items: barriers,
// the TMEM address and abort flag, alpha[] and 1/l[].
__host__ __device__ inline Layout layout_for(int R, int nq_s, int stages, int pb) {
    Layout L;
    L.q_off = 0;
    L.kv_off = align_up(nq_s * R * 128, 1024);
    L.p_off = L.kv_off + stages * STAGE_BYTES;
    L.misc_off = align_up(L.p_off + pb * R * NK * 2, 128);
    L.total = L.misc_off + BAR_BYTES + 128 + 512 + 512;
    return L;
}

// TMEM columns left for Q chunks (32 columns each) beside sb S buffers and O^T.
__host__ __device__ inline int q_tmem_chunks(int R, int sb) {
    const int used = sb * NK + 4 * R;
    const int c = ((int)TMEM_COLS - used) / 32;
    return c < 0 ? 0 : (c > NCHUNK ? NCHUNK : c);
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
    m.tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc_off + BAR_BYTES);
    m.abort = reinterpret_cast<volatile int*>(smem + L.misc_off + BAR_BYTES + 4);
    m.alpha = reinterpret_cast<float*>(smem + L.misc_off + BAR_BYTES + 128);
    m.rinv = reinterpret_cast<float*>(smem + L.misc_off + BAR_BYTES + 640);
    return m;
}

__device__ __forceinline__ void give_up(const Misc& m, unsigned* status) {
    if (atomicExch(const_cast<int*>(m.abort), 1) == 0) atomicOr(status, DEV_TIMEOUT);
}


template <bool FP8, int STAGES, int NQT, int SB, int PB>
__global__ void __launch_bounds__(block_threads<FP8>(), 1)
    verify_tc_kernel(const VerifyArgs a, const __grid_constant__ CUtensorMap q_map, int R, int R_step, int raw_n) {
    constexpr int NT = block_threads<FP8>();
    constexpr int SC = NK;                               // TMEM columns of one S buffer
    constexpr int O_COL0 = SB * SC;
    using BR = Bars<STAGES>;
    constexpr int B_KV_FULL = BR::KV_FULL, B_KV_EMPTY = BR::KV_EMPTY, B_S_FULL = BR::S_FULL,
                  B_S_FREE = BR::S_FREE, B_P_FULL = BR::P_FULL, B_Q_FULL = BR::Q_FULL, B_QT_FULL = BR::QT_FULL,
                  B_RAW_FULL = BR::RAW_FULL, B_RAW_EMPTY = BR::RAW_EMPTY;
    constexpr int nq_t = NQT;                            // Q chunks 0 .. NQT-1 live in TMEM,
    constexpr int nq_s = NCHUNK - NQT;                   // chunks NQT .. 8 in shared memory
    // TMEM chunks loaded before the set-up barrier (an odd count leaves pairs for the loop,
    // which keeps the register peak of the five- and seven-chunk variants below the 168 a
    // thread gets)
    constexpr int NQ0 = (nq_t == 5 || nq_t == 7) ? 3 : (nq_t < 4 ? nq_t : 4);
    const int Q_COL0 = O_COL0 + 4 * R;                   // Q chunk c < nq_t: TMEM columns Q_COL0 + 32 c ..
    extern __shared__ __align__(1024) uint8_t smem[];
    // Launched as a programmatic dependent of the previous kernel on the stream (the KV
    // append, typically): the CTAs become resident while it drains, and wait here until
    // it has completed and its writes are visible, before the first global read.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const Layout L = layout_for(R, nq_s, STAGES, PB);
    const Misc M = misc_at(smem, L);
    const int raw_off = align_up(L.total, 128);          // fp8 path: raw_n raw slots from here
    uint8_t* p_s = smem + L.p_off;
    const uint32_t q_addr = smem_u32(smem + L.q_off), kv_addr = smem_u32(smem + L.kv_off), p_addr = smem_u32(p_s);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.y;
    int s = blockIdx.x, b = blockIdx.z;
    const int rows = a.q_len * a.H;
    const int row0 = g * R_step;
    const int nrows = min(R_step, rows - row0);
    // the swizzled layouts need a 1024-byte aligned base: otherwise report and do no work
    const bool misaligned = (smem_u32(smem) & 1023u) != 0;
    const bool balanced = !FP8 && a.balanced;
    // Q-to-TMEM warps: the first NQ0 chunks of Q row r (rows past the tile: zeros)
    uint4 qraw[4 * 8];
    auto load_q0 = [&]() {
        const int r = (warp & 3) * 32 + lane;
        const uint4* qrow = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * rows + row0 + r) * D_QK);
#pragma unroll
        for (int j = 0; j < 8 * NQ0; ++j)
            qraw[j] = r < nrows ? __ldg(qrow + j) : make_uint4(0u, 0u, 0u, 0u);
    };
    // With the stream known from the grid (not balanced), the cold reads that need no length
    // go out before seq_lens[b] is read: the Q-to-TMEM warps' first chunks of Q and, since
    // streams usually fill their table row (n == slot_stride), the gather warps' slot
    // indices of their first two groups of tiles for the split range that length gives
    // (kept when the real range is the same; the indices read stay inside the stream's
    // table row).
    int spec_cur = 0, spec_nxt = 0, spec_gb = -1, spec_ge = -1;
    if (!balanced) {
        if (!FP8 && warp >= 6) {
            split_range(a.slot_stride, a.nsplit, s, NK, &spec_gb, &spec_ge);
            const int Tg = (spec_ge - spec_gb + NK - 1) / NK;
            const int32_t* srow = a.slot + (int64_t)b * a.slot_stride;
            const int key = 8 * (warp - 6) + (lane & 7);
            const int t0 = lane >> 3;
            if (t0 < Tg) spec_cur = __ldg(srow + min(spec_gb + t0 * NK + key, spec_ge - 1));
            if (t0 + 4 < Tg) spec_nxt = __ldg(srow + min(spec_gb + (t0 + 4) * NK + key, spec_ge - 1));
        } else if (warp >= 2 && warp < 6 && !misaligned && nq_t > 0) {
            load_q0();
        }
    }
    int bal_chunk = 0, bal_n = 0;
    if (balanced) {
        // one grid of split slots shared by all streams (every warp finds the same slot)
        const BalancedPlan P = balanced_plan(a.seq_lens, a.B, a.q_len, a.slot_stride, a.bal_G);
        balanced_slot(P, blockIdx.x, &b, &s);
        if (b < 0) return;                               // slot beyond the streams' need: no work
        bal_chunk = P.chunk;
        bal_n = __shfl_sync(0xffffffffu, b < 32 ? P.n[0] : P.n[1], b & 31);   // seq_lens[b], read by the plan
    }
    const int n = FP8 ? a.slot_stride : (balanced ? bal_n : a.seq_lens[b]);
    const bool bad_len = FP8 ? false : (n < a.q_len || n > a.slot_stride);
    int k_begin = 0, k_end = 0;
    if (!bad_len) {
        if (balanced) {
            k_begin = min(n, s * bal_chunk);
            k_end = (int)min((long long)n, (long long)(s + 1) * bal_chunk);
        } else {
            split_range(n, a.nsplit, s, NK, &k_begin, &k_end);
        }
    }
    // partial row of stream row rr: uniform [B * rows][nsplit] or balanced [slot][rows]
    const int64_t part_row0 = balanced ? (int64_t)blockIdx.x * rows + row0
                                       : ((int64_t)b * rows + row0) * a.nsplit + s;
    const int64_t part_row_step = balanced ? 1 : a.nsplit;
    const int T = misaligned ? 0 : (k_end - k_begin + NK - 1) / NK;
    const int p = FP8 ? n : n - a.q_len;                 // first draft key (none on the fp8 path)
    const bool spec_ok = !balanced && spec_gb == k_begin && spec_ge == k_end;

    // ---- set-up.  Each role initialises the barriers it uses and starts its first cold
    // loads before the block-wide barrier, so Q, the slot indices and the first key rows
    // arrive in parallel instead of after it.  The gather warps only arrive at that barrier
    // (they use no TMEM) and start copying as soon as their slot indices are in.
    if (warp == 0) {
        tmem_alloc(M.tmem_slot, TMEM_COLS);
        tmem_relinquish();
    } else if (warp == 1) {
        if (lane == 0) {
            for (int i = 0; i < 2; ++i) {
                mbar_init(&M.bars[B_S_FULL + i], 1);
                mbar_init(&M.bars[B_S_FREE + i], 128);
            }
            mbar_init(&M.bars[B_P_FULL], 128);
            mbar_init(&M.bars[B_P_FULL + 1], 128);
            mbar_init(&M.bars[B_Q_FULL], 1);
            mbar_init(&M.bars[B_QT_FULL], 128);
            mbar_init_fence();
            // Q tile copies.  The bf16 path issues them before its key range is known (it
            // depends on seq_lens); a CTA that turns out to have no keys waits for them
            // before it exits.
            if (!misaligned && (!FP8 || T > 0)) {
                mbar_arrive_expect_tx(&M.bars[B_Q_FULL], (uint32_t)(nq_s * R * 128));
                const int qrow = b * rows + row0;
                for (int c = nq_t; c < NCHUNK; ++c)
                    tma_load_2d(q_addr + (c - nq_t) * R * 128, &q_map, c * 64, qrow, &M.bars[B_Q_FULL]);
            }
        }
        __syncwarp();
    } else if (warp >= 6) {
        if (tid == 32 * 6) {
            for (int i = 0; i < STAGES; ++i) {
                mbar_init(&M.bars[B_KV_FULL + i], 32 * GATHER_WARPS);
                mbar_init(&M.bars[B_KV_EMPTY + i], 1);
            }
            if (FP8)
                for (int i = 0; i < MAX_RAW_SLOTS; ++i) {
                    mbar_init(&M.bars[B_RAW_FULL + i], 64);   // the copy warps' cp.async arrivals
                    mbar_init(&M.bars[B_RAW_EMPTY + i], GATHER_WARPS);
                }
            *M.abort = misaligned ? 1 : 0;
            mbar_init_fence();
        }
        __syncwarp();
        bar_sync(4, NT - 32 * 6);                        // the gather warps see their barriers
        bar_arrive(3, NT);
    } else if (balanced && !misaligned && nq_t > 0) {
        load_q0();                                       // the stream is known only now
    }
    if (warp < 6) {
        tc_fence_before();
        __syncwarp();
        bar_sync(3, NT);
        tc_fence_after();
    }
    const uint32_t tmem = warp < 6 ? *M.tmem_slot : 0u;

    if (warp <= 1) {
        // ================= MMA issue: warp 0 Q K^T, warp 1 P V =================
        // Two issuers: Q K^T of tile i goes out as soon as its keys and S buffer are ready,
        // P V of tile j as soon as its P is written, so a key stage is released right after
        // its P V instead of after the next tile's Q K^T (measured on GB300: c4 -7%,
        // c3-64k -5%; fp8 c5 -1.3 us).  They write different TMEM columns (S buffers /
        // O^T) and only read shared memory; each commit tracks its own thread's MMAs.
        if (T > 0) {
            const uint32_t id_qk = idesc_bf16(128, NK, false, false);
            const uint32_t id_pv = idesc_bf16(128, R, true, false);
            // Q (shared-memory chunks): K-major, 128-byte swizzle, 8-row groups 1024 B apart;
            // a 16-dim step moves 32 B inside the 128-byte rows, a 64-dim step moves to the
            // next region (R * 128 B)
            const uint64_t dq = smem_desc_sw128(q_addr, 16, 1024);
            // key stage: the same layout with 32-row regions (REGION bytes)
            const uint64_t dk = smem_desc_sw128(kv_addr, 16, 1024);
            // V^T: M-major, 64-dim chunks REGION apart, 8-key groups 1024 B apart
            const uint64_t dv = smem_desc_sw128(kv_addr, REGION, 1024);
            // P: K-major, no swizzle, 8-key blocks R * 16 B apart, 8-row blocks 128 B apart
            const uint64_t dp = smem_desc(p_addr, R * 16, 128);
            const uint32_t q_region16 = (uint32_t)(R * 128) >> 4;
            bool ok = true;
            if (warp == 1) {
                for (int j = 0; j < T && ok; ++j) {
                    ok = mbar_wait(&M.bars[B_P_FULL + j % PB], (j / PB) & 1, M.abort);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t st16 = (uint64_t)((j % STAGES) * STAGE_BYTES) >> 4;
                    if (elect_one()) {
#pragma unroll
                    for (int ci = 0; ci < 4; ++ci)
#pragma unroll
                        for (int kk = 0; kk < NK / 16; ++kk)
                            mma_bf16(tmem + O_COL0 + ci * R,
                                     dv + st16 + (uint64_t)((2 * ci * REGION + kk * 2048) >> 4),
                                     dp + (uint64_t)(((j % PB) * R * NK * 2 + kk * 2 * R * 16) >> 4), id_pv,
                                     j > 0 || kk > 0);
                    mma_commit(&M.bars[B_KV_EMPTY + j % STAGES]);
                    }
                    __syncwarp();
                }
            } else {
                ok = mbar_wait(&M.bars[B_Q_FULL], 0, M.abort);
                ok = ok && mbar_wait(&M.bars[B_QT_FULL], 0, M.abort);
                ok = __all_sync(0xffffffffu, ok);
                for (int i = 0; i < T && ok; ++i) {
                    const int st = i % STAGES;
                    ok = mbar_wait(&M.bars[B_KV_FULL + st], (i / STAGES) & 1, M.abort);
                    if (ok && i >= SB) ok = mbar_wait(&M.bars[B_S_FREE + i % SB], ((i - SB) / SB) & 1, M.abort);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    fence_proxy_async_smem();          // cp.async (generic proxy) data -> tensor-core reads
                    tc_fence_after();
                    const uint64_t st16 = (uint64_t)(st * STAGE_BYTES) >> 4;
                    const uint32_t d_s = tmem + (i % SB) * SC;
                    if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < D_QK / 16; ++ks) {
                        const int c = ks >> 2;
                        const uint32_t ko = (uint32_t)((c * REGION + (ks & 3) * 32) >> 4);
                        if (c < nq_t) {
                            mma_bf16_ta(d_s, tmem + Q_COL0 + ks * 8, dk + st16 + ko, id_qk, ks > 0);
                        } else {
                            const uint32_t qo = (uint32_t)(c - nq_t) * q_region16 + (uint32_t)(ks & 3) * 2;
                            mma_bf16(d_s, dq + qo, dk + st16 + ko, id_qk, ks > 0);
                        }
                    }
                    mma_commit(&M.bars[B_S_FULL + i % SB]);
                    }
                    __syncwarp();
                }
            }
            if (!ok && lane == 0) give_up(M, a.status);
        } else if (warp == 1 && !misaligned && !FP8) {
            mbar_wait(&M.bars[B_Q_FULL], 0, M.abort);   // no keys: the Q copies must land before exit
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ================= key-tile gather: keys 8w .. 8w+7 of every tile =================
        const int w = warp - 6;
        bool bad_slot = false;
        const int32_t* slot_row = a.slot + (int64_t)b * a.slot_stride;
        // Slot indices run four tiles ahead: lane l holds the slot of key 8 w + (l & 7) of
        // tile i0 + (l >> 3) for the current group of four tiles (cur) and the next (nxt),
        // so a tile's row copies never wait on its own index load.  Indices are checked
        // when their group becomes current (by then they have arrived).
        auto load_slots = [&](int i0) -> int {
            const int t = i0 + (lane >> 3);
            if (t >= T) return 0;
            const int j = min(k_begin + t * NK + 8 * w + (lane & 7), k_end - 1);   // past the split: repeat a valid key
            return __ldg(slot_row + j);
        };
        int cur = spec_cur, nxt = spec_nxt;
        if (!FP8 && !spec_ok) {
            cur = load_slots(0);
            nxt = load_slots(4);
        }
        // Slot indices of the next tile to copy: groups advance with the copy position.
        auto next_slots = [&](int j) -> int {
            if ((j & 3) == 0) {
                if (j > 0) {
                    cur = nxt;
                    nxt = load_slots(j + 4);
                }
                if (cur < 0 || (int64_t)cur >= a.n_pool) { bad_slot = true; cur = 0; }
            }
            return __shfl_sync(0xffffffffu, cur, ((j & 3) << 3) + (lane & 7));   // key 8 w + (lane & 7)
        };
        if constexpr (!FP8) {
            // lane l copies 16-byte pieces f = l, l + 32, ... of the warp's 8 rows x 72 pieces
            // straight into the stage; consecutive lanes take consecutive pieces of a row
            for (int i = 0; i < T; ++i) {
                const int st = i % STAGES;
                const int sl = next_slots(i);
                if (i >= STAGES && !mbar_wait(&M.bars[B_KV_EMPTY + st], ((i - STAGES) / STAGES) & 1, M.abort)) {
                    give_up(M, a.status);
                    break;
                }
                const uint32_t base = kv_addr + st * STAGE_BYTES;
#pragma unroll
                for (int it = 0; it < 8 * (D_QK / 8) / 32; ++it) {      // 18 pieces per lane
                    const int f = it * 32 + lane;
                    const int rr = f / (D_QK / 8), pc = f % (D_QK / 8);
                    const int key = 8 * w + rr;
                    const int row_slot = __shfl_sync(0xffffffffu, sl, rr);
                    const uint32_t dst = base + (pc >> 3) * REGION + key * 128 + (((pc & 7) ^ (key & 7)) << 4);
                    cp_async16(dst, a.kv + (int64_t)row_slot * D_QK + pc * 8);
                }
                if (!(a.debug_stall && i == 0)) cp_async_arrive_noinc(&M.bars[B_KV_FULL + st]);
            }
        } else if (warp >= 10) {
            // ---- fp8 raw copies: warp 10 + c copies keys 16 c .. 16 c + 15 of every tile (e4m3
            // latent, bf16 rope, fp32 scale) into the ring of raw_n raw slots, up to raw_n tiles
            // ahead of the widening warps; a slot is refilled once all four widening warps have
            // read it.  Arrivals are asynchronous (cp.async.mbarrier.arrive), so this warp
            // moves on while its copies are in flight.
            const int c = warp - 10;
            const uint32_t raw_addr = smem_u32(smem + raw_off);
            // slot indices two tiles per load: lane l holds key 16 c + (l & 15) of tile t0 + (l >> 4)
            auto load2 = [&](int t0) -> int {
                const int t = t0 + (lane >> 4);
                if (t >= T) return 0;
                const int j = min(k_begin + t * NK + 16 * c + (lane & 15), k_end - 1);   // past the split: a valid key
                return __ldg(slot_row + j);
            };
            cur = load2(0);
            nxt = load2(2);
            for (int j = 0; j < T; ++j) {
                if ((j & 1) == 0) {
                    if (j > 0) {
                        cur = nxt;
                        nxt = load2(j + 2);
                    }
                    if (cur < 0 || (int64_t)cur >= a.n_pool) { bad_slot = true; cur = 0; }
                }
                const int sl = __shfl_sync(0xffffffffu, cur, ((j & 1) << 4) + (lane & 15));   // key 16 c + (lane & 15)
                const int rs = j % raw_n;
                if (j >= raw_n && !mbar_wait(&M.bars[B_RAW_EMPTY + rs], ((j - raw_n) / raw_n) & 1, M.abort)) {
                    give_up(M, a.status);
                    break;
                }
                const uint32_t rb = raw_addr + (uint32_t)(rs * RAW_SLOT);
#pragma unroll
                for (int it = 0; it < 16; ++it) {        // latent: one 512-byte row per step
                    const int row_slot = __shfl_sync(0xffffffffu, sl, it);
                    cp_async16(rb + (16 * c + it) * D_V + lane * 16, a.kv_lat + (int64_t)row_slot * D_V + lane * 16);
                }
#pragma unroll
                for (int it = 0; it < 4; ++it) {         // rope: 16 rows x 8 pieces of 16 bytes
                    const int f = it * 32 + lane;
                    const int row_slot = __shfl_sync(0xffffffffu, sl, f >> 3);
                    cp_async16(rb + RAW_ROPE + (16 * c + (f >> 3)) * 128 + (f & 7) * 16,
                               a.kv_rope + (int64_t)row_slot * 64 + (f & 7) * 8);
                }
                if (lane < 16) cp_async4(rb + RAW_SCALE + (16 * c + lane) * 4, a.kv_scale + sl);
                cp_async_arrive_noinc(&M.bars[B_RAW_FULL + rs]);
            }
        } else {
            // ---- fp8 widening: warp 6 + w widens keys 8 w .. 8 w + 7 of every tile from its raw
            // slot into the swizzled bf16 stage layout, latent values times the key's scale
            // (V = scale_t * code, and Q K^T then needs no per-key step).  lane l widens dims
            // 16 l .. 16 l + 15:
            // 16-byte pieces j0, j0 + 1 of region l / 4.  Lanes of odd regions store their second
            // piece first, so each store covers all eight 16-byte bank groups (four lanes each)
            // instead of four.
            const int region = lane >> 2, j0 = (lane & 3) * 2, odd = region & 1;
            for (int i = 0; i < T; ++i) {
                const int st = i % STAGES, rs = i % raw_n;
                if (!mbar_wait(&M.bars[B_RAW_FULL + rs], (i / raw_n) & 1, M.abort) ||
                    (i >= STAGES && !mbar_wait(&M.bars[B_KV_EMPTY + st], ((i - STAGES) / STAGES) & 1, M.abort))) {
                    give_up(M, a.status);
                    break;
                }
                // All reads of the raw slot first: the compiler cannot tell the raw slot from
                // the stage it writes, so reads placed after a store would wait for it.
                const uint8_t* rb = smem + raw_off + rs * RAW_SLOT;
                uint4 raw[8], rope[2];
#pragma unroll
                for (int it = 0; it < 8; ++it)
                    raw[it] = *reinterpret_cast<const uint4*>(rb + (8 * w + it) * D_V + lane * 16);
#pragma unroll
                for (int it = 0; it < 2; ++it) {
                    const int f = it * 32 + lane;
                    rope[it] = *reinterpret_cast<const uint4*>(rb + RAW_ROPE + (8 * w + (f >> 3)) * 128 + (f & 7) * 16);
                }
                const float4 ks0 = *reinterpret_cast<const float4*>(rb + RAW_SCALE + 8 * w * 4);
                const float4 ks1 = *reinterpret_cast<const float4*>(rb + RAW_SCALE + 8 * w * 4 + 16);
                const float ksc[8] = {ks0.x, ks0.y, ks0.z, ks0.w, ks1.x, ks1.y, ks1.z, ks1.w};
                uint8_t* sbase = smem + L.kv_off + st * STAGE_BYTES;
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int key = 8 * w + it;
                    const uint4 r = odd ? make_uint4(raw[it].z, raw[it].w, raw[it].x, raw[it].y) : raw[it];
                    uint4 first, second;
                    e4m3x16_to_bf16_scaled(r, ksc[it], first, second);
                    uint8_t* row = sbase + region * REGION + key * 128;
                    *reinterpret_cast<uint4*>(row + (((j0 + odd) ^ (key & 7)) << 4)) = first;
                    *reinterpret_cast<uint4*>(row + (((j0 + 1 - odd) ^ (key & 7)) << 4)) = second;
                }
#pragma unroll
                for (int it = 0; it < 2; ++it) {
                    const int f = it * 32 + lane;
                    const int key = 8 * w + (f >> 3), cc = f & 7;
                    *reinterpret_cast<uint4*>(sbase + 8 * REGION + key * 128 + ((cc ^ (key & 7)) << 4)) = rope[it];
                }
                fence_proxy_async_smem();                         // generic stores -> tensor-core reads
                if (!(a.debug_stall && i == 0)) mbar_arrive(&M.bars[B_KV_FULL + st]);
                __syncwarp();                                     // raw slot read by the whole warp
                if (lane == 0) mbar_arrive(&M.bars[B_RAW_EMPTY + rs]);
            }
        }
        cp_async_wait_all();
        if (bad_slot) atomicOr(a.status, DEV_BAD_SLOT);
    } else {
        // ================= softmax + epilogue =================
        const int quad = warp & 3;                     // TMEM lane quadrant of this warp
        const int r = quad * 32 + lane;                // query row of this thread (S lane)
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const bool row_ok = r < nrows;
        const int t = row_ok ? (row0 + r) / a.H : 0;
        // drafts this row sees, bit i = draft i (q_len <= 64)
        uint64_t vis = 0;
        if (row_ok) {
            if (a.mask_bits) {
                vis = a.mask_bits[(int64_t)b * a.q_len + t];
            } else {
                for (int d = 0; d < a.q_len; ++d) {
                    const bool seen = a.mask ? a.mask[((int64_t)b * a.q_len + t) * a.q_len + d] != 0 : d <= t;
                    vis |= (uint64_t)(seen ? 1u : 0u) << d;
                }
            }
        }
        if (!misaligned) {
            // Q chunks 0 .. nq_t-1 of row r into TMEM lane r: chunks 0 .. NQ0-1 were loaded
            // during set-up, the rest follow two at a time
            auto store_chunk = [&](int c, int slot) {
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    v[4 * j] = qraw[8 * slot + j].x; v[4 * j + 1] = qraw[8 * slot + j].y;
                    v[4 * j + 2] = qraw[8 * slot + j].z; v[4 * j + 3] = qraw[8 * slot + j].w;
                }
                tmem_st32(tmem + lane_base + Q_COL0 + c * 32, v);
            };
#pragma unroll
            for (int c = 0; c < NQ0; ++c) store_chunk(c, c);
            const uint4* qrow = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * rows + row0 + r) * D_QK);
#pragma unroll
            for (int c0 = NQ0; c0 < nq_t; c0 += 2) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c0 + (j >> 3) < nq_t) qraw[j] = row_ok ? __ldg(qrow + c0 * 8 + j) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (c0 + h < nq_t) store_chunk(c0 + h, h);
            }
            tmem_st_wait();
            tc_fence_before();
        }
        mbar_arrive(&M.bars[B_QT_FULL]);
        const float c2 = a.scale * LOG2E;
        const int plain_end = min(p, k_end);           // keys below this need no mask
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < T; ++i) {
            ok = mbar_wait(&M.bars[B_S_FULL + i % SB], (i / SB) & 1, M.abort);
            if (bar_red_or(1, 128, !ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t sv[NK];
            tmem_ld32(tmem + lane_base + (i % SB) * SC, sv);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&M.bars[B_S_FREE + i % SB]);

            const int k0 = k_begin + i * NK;
            float x[NK];
            float mt = -INFINITY;
            if (k0 + NK <= plain_end) {                // the whole tile is prefix keys of this split
#pragma unroll
                for (int k = 0; k < NK; ++k) {
                    x[k] = row_ok ? __uint_as_float(sv[k]) * c2 : -INFINITY;
                    mt = fmaxf(mt, x[k]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < NK; ++k) {
                    const int j = k0 + k;
                    const bool vk = row_ok && j < k_end && (j < p || ((vis >> (j - p)) & 1ull));
                    x[k] = vk ? __uint_as_float(sv[k]) * c2 : -INFINITY;
                    mt = fmaxf(mt, x[k]);
                }
            }
            const bool need = mt > m + TAU;
            float alpha = 1.f;
            if (need) {
                alpha = exp2f(m - mt);
                l *= alpha;
                m = mt;
            }
            const bool any = bar_red_or(1, 128, need);
            // P buffer i % PB was last read by P V of tile i - PB; a rescale of O^T also needs
            // P V of tile i - 1 complete (without one, P V of tiles i - 1 and i commute)
            if (ok && (any || PB == 1) && i >= 1)
                ok = mbar_wait(&M.bars[B_KV_EMPTY + (i - 1) % STAGES], ((i - 1) / STAGES) & 1, M.abort);
            else if (ok && i >= 2)
                ok = mbar_wait(&M.bars[B_KV_EMPTY + (i - 2) % STAGES], ((i - 2) / STAGES) & 1, M.abort);
            if (bar_red_or(1, 128, !ok)) { ok = false; break; }
            if (any && i >= 1) {
                // O^T column r (query row r) *= alpha_r; thread = TMEM lane = value dim
                if (r == 0) atomicAdd(a.rescales, 1ull);
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
                // P (B operand, K-major, no swizzle): keys 8 kb .. 8 kb + 7 of row r at kb * (R * 16) + r * 16
#pragma unroll
                for (int kb = 0; kb < NK / 8; ++kb)
                    *reinterpret_cast<uint4*>(p_s + (i % PB) * (R * NK * 2) + kb * (R * 16) + r * 16) =
                        make_uint4(pk[4 * kb], pk[4 * kb + 1], pk[4 * kb + 2], pk[4 * kb + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&M.bars[B_P_FULL + i % PB]);
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
        const int64_t grow0 = (int64_t)b * rows + row0;
        if (row_ok) {
            if (a.nsplit == 1) a.lse[grow0 + r] = lse_v;
            else a.part_lse[part_row0 + r * part_row_step] = lse_v;
        }
        bar_sync(2, 128);
        // O^T -> rows: thread = TMEM lane = value dim, each warp store writes 32 consecutive
        // dims (128 B) of one row.  EPI 128-dim chunks of a group of 16 rows are loaded from
        // TMEM together (one wait) and the group's 1 / l read once.  Measured on GB300: all
        // four chunks per wait take 1-1.6 us off the bf16 calls' epilogue (c3-16k 4.6 ->
        // 3.2 us), while the fp8 instantiation ran 1.4 us slower with it (its raw-row copies
        // started later), so it loads one chunk per wait.
        constexpr int EPI = FP8 ? 1 : 4;
        const bool have_o = T > 0 && !failed;
        float* const out_base = a.nsplit == 1 ? a.out + grow0 * D_V : a.part_out + part_row0 * D_V;
        const int64_t row_step = a.nsplit == 1 ? D_V : part_row_step * D_V;
        for (int cg = 0; cg < 4; cg += EPI)
            for (int c0 = 0; c0 < nrows; c0 += 16) {
                uint32_t v[EPI][16];
                if (have_o) {
#pragma unroll
                    for (int e = 0; e < EPI; ++e) tmem_ld16(tmem + lane_base + O_COL0 + (cg + e) * R + c0, v[e]);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int e = 0; e < EPI; ++e)
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) v[e][jj] = 0u;
                }
                float ri[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) ri[jj] = M.rinv[c0 + jj];
#pragma unroll
                for (int e = 0; e < EPI; ++e)
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int rr = c0 + jj;
                        if (rr < nrows)
                            out_base[rr * row_step + (cg + e) * 128 + quad * 32 + lane] = __uint_as_float(v[e][jj]) * ri[jj];
                    }
            }
    }

    // ---- teardown; the combine launched after this kernel may now be scheduled
    tc_fence_before();
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 32) {
        if (bad_len) atomicOr(a.status, DEV_BAD_LEN);
        if (misaligned) atomicOr(a.status, DEV_TIMEOUT);
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

void tc_tiling(int rows, int max_r, int* n_tiles, int* R_step, int* R) {
    *n_tiles = (rows + max_r - 1) / max_r;
    *R_step = (rows + *n_tiles - 1) / *n_tiles;
    *R = (*R_step + 15) / 16 * 16;
}

namespace {
constexpr int MAX_SMEM = 232448;                     // opt-in shared memory per block on sm_103

// Instantiations: (fp8, key stages, Q chunks in TMEM, S buffers, P buffers).  bf16 up to
// 80 rows: five stages with one S and one P buffer and five Q chunks in TMEM; at 96 rows
// three stages, two chunks in TMEM.  fp8 (one S buffer): seven chunks up to 64 rows,
// five at 80, three bf16 stages so that three or four raw slots fit beside them.
template <bool FP8, int STAGES, int NQT, int SB, int PB>
cudaError_t launch_one(bool set_attr, dim3 grid, cudaStream_t stream, const VerifyArgs& a, const CUtensorMap& q_map,
                       int R, int R_step) {
    auto* k = verify_tc_kernel<FP8, STAGES, NQT, SB, PB>;
    if (set_attr) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_SMEM);
        if (e != cudaSuccess) return e;
    }
    if (q_tmem_chunks(R, SB) < NQT) return cudaErrorInvalidConfiguration;
    int smem = layout_for(R, NCHUNK - NQT, STAGES, PB).total;
    int raw_n = 0;
    if (FP8) {                                       // as many raw slots as still fit
        smem = align_up(smem, 128);
        raw_n = (MAX_SMEM - smem) / RAW_SLOT;
        raw_n = raw_n > MAX_RAW_SLOTS ? MAX_RAW_SLOTS : raw_n;
        if (raw_n < 1) return cudaErrorInvalidConfiguration;
        smem += raw_n * RAW_SLOT;
    }
    if (smem > MAX_SMEM) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block_threads<FP8>());
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddepcontrol.wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k, a, q_map, R, R_step, raw_n);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_verify_tc(const VerifyArgs& a_in, cudaStream_t stream) {
    VerifyArgs a = a_in;
    a.debug_stall = take_debug_stall() ? 1 : 0;
    static bool attr_set[64][5];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int n_tiles, R_step, R;
    // fp8: at 96 rows a single raw slot would fit beside the shared-memory Q tile, the
    // key stages and two P buffers, so its tiles stop at 80 rows
    tc_tiling(a.q_len * a.H, a.kv_fp8 ? 80 : MAX_R, &n_tiles, &R_step, &R);
    CUtensorMap q_map;
    const uint64_t q_rows = (uint64_t)a.B * a.q_len * a.H;
    if (!encode_bf16_2d_sw128(&q_map, a.q, D_QK, q_rows, D_QK * 2, 64, (uint32_t)R,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
        return cudaErrorInvalidValue;
    dim3 grid(a.nsplit, n_tiles, a.balanced ? 1 : a.B);
    int which;
    if (!a.kv_fp8) which = R <= 80 ? 0 : 1;
    else which = q_tmem_chunks(R, 1) >= 7 ? 2 : 3;
    const bool set = !attr_set[dev][which];
    switch (which) {
        case 0: e = launch_one<false, 5, 5, 1, 1>(set, grid, stream, a, q_map, R, R_step); break;
        case 1: e = launch_one<false, 3, 2, 2, 2>(set, grid, stream, a, q_map, R, R_step); break;
        case 2: e = launch_one<true, 3, 7, 1, 2>(set, grid, stream, a, q_map, R, R_step); break;
        case 3: e = launch_one<true, 3, 5, 1, 2>(set, grid, stream, a, q_map, R, R_step); break;
        default: e = cudaErrorInvalidConfiguration; break;
    }
    if (e == cudaSuccess) attr_set[dev][which] = true;
    return e;
}

}  // namespace mla
