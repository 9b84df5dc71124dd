// Host side of the C ABI declared in include/mla_verify.h: argument checks,
// the split-count policy, the per-device status word, and the log-sum-exp
// combine kernel that merges KV-split partials.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "../../include/mla_verify.h"
#include "internal.cuh"

namespace mla {

// Per-device status word of MLA_DEV_* bits (sticky until mla_verify_status clears it).
__device__ unsigned g_status;
// Per-device count of O^T rescales of the online softmax (read by tests through
// mla_debug_rescale_count; the kernels only ever add to it).
__device__ unsigned long long g_rescales;

// Test hook: the next split-kernel launch withholds its first key-tile arrival.
static std::atomic<bool> g_debug_stall{false};
bool take_debug_stall() { return g_debug_stall.exchange(false); }

namespace {

constexpr int MAX_DEVICES = 64;
unsigned* g_status_ptr[MAX_DEVICES];
unsigned long long* g_rescales_ptr[MAX_DEVICES];
int g_num_sms[MAX_DEVICES];
int g_arch_ok[MAX_DEVICES];      // 0 unknown, 1 sm_103, -1 other

// Device properties and the status word's device address for the current device.
int device_state(int* dev_out, unsigned** status, int* num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return MLA_ERR_DEVICE;
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MLA_ERR_DEVICE;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return MLA_ERR_DEVICE;
        g_status_ptr[dev] = static_cast<unsigned*>(p);
        if (cudaGetSymbolAddress(&p, g_rescales) != cudaSuccess) return MLA_ERR_DEVICE;
        g_rescales_ptr[dev] = static_cast<unsigned long long*>(p);
        g_num_sms[dev] = sms;
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_arch_ok[dev] != 1) return MLA_ERR_DEVICE;
    if (dev_out) *dev_out = dev;
    if (status) *status = g_status_ptr[dev];
    if (num_sms) *num_sms = g_num_sms[dev];
    return MLA_OK;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------------------
// Combine.  A work item is (row, 128 output dims); Z warps (Z = 1, 2, 4 or 8, more for
// more splits) share an item, and a CTA of 8 warps holds 8 / Z items.  Lane v of warp
// z sums float4 v of the item's dims over the splits s = z, z + Z, ... with weights
// w_s = exp(lse_s - lse), lse = log sum_s exp(lse_s): the first eight partial loads of
// a warp are issued before the weights are known, every warp derives the row's lse
// from the S split values itself (no barrier before the sums), and the Z warp sums
// meet in shared memory.  The launch may overlap the tail of the split kernel before
// it (programmatic dependent launch): a balanced combine first computes its slot plan
// from the lengths (inputs of the split kernel, final by the time any CTA of this grid
// runs, since every split CTA passed its own dependency wait before it let this grid
// launch), then griddepcontrol.wait holds every thread until the split kernel has
// completed and its writes are visible.
// ---------------------------------------------------------------------------
constexpr int CB_THREADS = 256;
constexpr int CB_WARPS = CB_THREADS / 32;
constexpr int CB_DIMS = 128;
constexpr int CB_BATCH = 8;

// Balanced partials (slot-major): the row's splits are slots first .. first + count - 1
// of its stream, recomputed from the lengths exactly as the split kernel chose them.
struct CombineBalanced {
    int on;
    const int32_t* seq_lens;
    int B, q_len, slot_stride, G, rows;
};

template <int Z>
__global__ void __launch_bounds__(CB_THREADS) combine_kernel(const float* __restrict__ part_out,
                                                             const float* __restrict__ part_lse, int S_all,
                                                             long long n_items, float* __restrict__ out,
                                                             float* __restrict__ lse, const CombineBalanced bal) {
    __shared__ float4 red[CB_WARPS][32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, z = warp % Z;
    const long long item = (long long)blockIdx.x * (CB_WARPS / Z) + warp / Z;
    const bool valid = item < n_items;
    const long long row = valid ? item / (D_V / CB_DIMS) : 0;
    const int quarter = (int)(item % (D_V / CB_DIMS));
    // split s of this row: lse at pl[s * lse_step], output at part_out[po + s * out_step]
    int S = S_all;
    long long lse_step = 1, out_step = D_V;
    const float* pl = part_lse + row * S_all;
    long long po = row * (long long)S_all * D_V;
    if (bal.on) {
        const BalancedPlan P = balanced_plan(bal.seq_lens, bal.B, bal.q_len, bal.slot_stride, bal.G);
        const int b = (int)(row / bal.rows), r = (int)(row % bal.rows);
        int first, count;
        balanced_stream(P, b, &first, &count);
        S = count;
        lse_step = bal.rows;
        out_step = (long long)bal.rows * D_V;
        pl = part_lse + (long long)first * bal.rows + r;
        po = ((long long)first * bal.rows + r) * D_V;
    }
    if (!valid) S = 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float* base = part_out + po + quarter * CB_DIMS + lane * 4;

    float4 v[CB_BATCH];
#pragma unroll
    for (int m = 0; m < CB_BATCH; ++m) {
        const int s = z + Z * m;
        if (s < S) v[m] = __ldg(reinterpret_cast<const float4*>(base + (long long)s * out_step));
    }
    float mx = -INFINITY;
    bool bad = false;
    for (int s = lane; s < S; s += 32) {
        const float x = __ldg(pl + s * lse_step);
        bad |= x != x;
        mx = fmaxf(mx, x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    bad = __any_sync(0xffffffffu, bad);
    const bool live = !bad && mx != -INFINITY;
    float zs = 0.f;
    if (live)
        for (int s = lane; s < S; s += 32) zs += expf(__ldg(pl + s * lse_step) - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o);
    const float L = mx + logf(zs);
    float wl = 0.f;

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
        for (int s0 = 0; s0 < S; s0 += CB_BATCH * Z) {
            // weights of this warp's next 32 splits, one per lane, handed out by shuffles
            if ((s0 / (CB_BATCH * Z)) % (32 / CB_BATCH) == 0) {
                const int s = s0 + z + Z * lane;
                wl = s < S ? expf(__ldg(pl + s * lse_step) - L) : 0.f;
            }
            if (s0 > 0) {
#pragma unroll
                for (int m = 0; m < CB_BATCH; ++m) {
                    const int s = s0 + z + Z * m;
                    if (s < S) v[m] = __ldg(reinterpret_cast<const float4*>(base + (long long)s * out_step));
                }
            }
            const int lane0 = ((s0 / (CB_BATCH * Z)) % (32 / CB_BATCH)) * CB_BATCH;
#pragma unroll
            for (int m = 0; m < CB_BATCH; ++m) {
                const int s = s0 + z + Z * m;
                const float w = __shfl_sync(0xffffffffu, wl, lane0 + m);
                if (s < S) {
                    acc.x += w * v[m].x; acc.y += w * v[m].y; acc.z += w * v[m].z; acc.w += w * v[m].w;
                }
            }
        }
    }
    if (Z > 1) {
        red[warp][lane] = acc;
        __syncthreads();
        if (z == 0)
#pragma unroll
            for (int k = 1; k < Z; ++k) {
                const float4 u = red[warp + k][lane];
                acc.x += u.x; acc.y += u.y; acc.z += u.z; acc.w += u.w;
            }
    }
    if (valid && z == 0) {
        reinterpret_cast<float4*>(out + row * D_V + quarter * CB_DIMS)[lane] = acc;
        if (quarter == 0 && lane == 0) lse[row] = bad ? __int_as_float(0x7fc00000) : (live ? L : -INFINITY);
    }
}

template <int Z>
cudaError_t launch_combine_z(const float* part_out, const float* part_lse, long long n_rows, int S, float* out,
                             float* lse, const CombineBalanced& bal, cudaStream_t stream) {
    const long long items = n_rows * (D_V / CB_DIMS);
    const long long per_cta = CB_WARPS / Z;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((items + per_cta - 1) / per_cta));
    cfg.blockDim = dim3(CB_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel<Z>, part_out, part_lse, S, items, out, lse, bal);
}

}  // namespace

// Z: warps per item, from the split count (up to 16 splits per warp, 8 warps at most;
// balanced partials: a stream holds at most all slots, typically a few dozen; two warps
// per item keep the grid near one wave (measured on c4: 4 warps 60.2 us per call, 2 warps
// 58.3, 1 warp 58.1)).
static cudaError_t launch_combine_any(const float* part_out, const float* part_lse, long long n_rows, int S,
                                      float* out, float* lse, const CombineBalanced& bal, cudaStream_t stream) {
    if (n_rows <= 0) return cudaSuccess;
    const int per = bal.on ? 2 * 16 : S;
    if (per <= 16) return launch_combine_z<1>(part_out, part_lse, n_rows, S, out, lse, bal, stream);
    if (per <= 32) return launch_combine_z<2>(part_out, part_lse, n_rows, S, out, lse, bal, stream);
    if (per <= 64) return launch_combine_z<4>(part_out, part_lse, n_rows, S, out, lse, bal, stream);
    return launch_combine_z<8>(part_out, part_lse, n_rows, S, out, lse, bal, stream);
}

cudaError_t launch_combine(const float* part_out, const float* part_lse, long long n_rows, int S,
                           float* out, float* lse, cudaStream_t stream) {
    CombineBalanced off;
    memset(&off, 0, sizeof off);
    return launch_combine_any(part_out, part_lse, n_rows, S, out, lse, off, stream);
}

// S here bounds the slots of one stream (nsplit slots in all): the weights' shared memory.
cudaError_t launch_combine_balanced(const VerifyArgs& a, cudaStream_t stream) {
    CombineBalanced bal;
    bal.on = 1;
    bal.seq_lens = a.seq_lens;
    bal.B = a.B; bal.q_len = a.q_len; bal.slot_stride = a.slot_stride; bal.G = a.bal_G;
    bal.rows = a.q_len * a.H;
    return launch_combine_any(a.part_out, a.part_lse, (long long)a.B * bal.rows, a.nsplit, a.out, a.lse, bal,
                              stream);
}

}  // namespace mla

using namespace mla;

namespace {

// Tiling of the split kernel that the split-count policy plans for.
constexpr int PLAN_ROWS_PER_CTA = TC_MAX_ROWS;
constexpr int PLAN_CTAS_PER_SM = 1;
constexpr int PLAN_MIN_KEYS_PER_SPLIT = 128;

int check_verify_args(const void* q, const void* kv, int64_t n_pool, const int32_t* slot, int slot_stride,
                      const int32_t* seq_lens, int B, int q_len, int H, float scale, const float* out,
                      const float* lse, int nsplit) {
    if (B < 0 || B > 65535 || q_len < 1 || q_len > MLA_MAX_Q_LEN || H < 1 || H > MLA_MAX_HEADS) return MLA_ERR_SHAPE;
    if (nsplit < 0 || nsplit > MLA_MAX_NSPLIT) return MLA_ERR_NSPLIT;
    if (B == 0) return MLA_OK;
    if (!q || !kv || !slot || !seq_lens || !out || !lse) return MLA_ERR_NULL;
    if (n_pool < 1 || n_pool > 0x7fffffffLL || slot_stride < q_len) return MLA_ERR_SHAPE;
    if ((long long)B * q_len * H > 0x7fffffffLL) return MLA_ERR_SHAPE;
    if (!isfinite(scale)) return MLA_ERR_ARG;
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16) || !aligned(slot, 4) ||
        !aligned(seq_lens, 4) || !aligned(lse, 4))
        return MLA_ERR_ALIGN;
    return MLA_OK;
}

int run_verify(bool combine, const void* q, const void* kv, int64_t n_pool, const int32_t* slot,
               int slot_stride, const int32_t* seq_lens, const uint8_t* mask, const uint64_t* mask_bits, int B,
               int q_len, int H, float scale, float* out, float* lse, int nsplit, void* ws, size_t ws_bytes,
               cudaStream_t stream) {
    int rc = check_verify_args(q, kv, n_pool, slot, slot_stride, seq_lens, B, q_len, H, scale, out, lse, nsplit);
    if (rc != MLA_OK) return rc;
    if (B == 0) return MLA_OK;
    unsigned* status = nullptr;
    int num_sms = 0, dev = 0;
    rc = device_state(&dev, &status, &num_sms);
    if (rc != MLA_OK) return rc;
    int ns = nsplit > 0 ? nsplit : mla_verify_auto_nsplit(B, q_len, H, slot_stride, num_sms, ws ? ws_bytes : 0);
    const long long rows = (long long)B * q_len * H;
    VerifyArgs a;
    memset(&a, 0, sizeof a);
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.kv = static_cast<const __nv_bfloat16*>(kv);
    a.n_pool = n_pool;
    a.slot = slot;
    a.slot_stride = slot_stride;
    a.seq_lens = seq_lens;
    a.mask = mask;
    a.mask_bits = mask_bits;
    a.B = B; a.q_len = q_len; a.H = H;
    a.scale = scale;
    a.out = out; a.lse = lse;
    a.nsplit = ns;
    a.status = status;
    a.rescales = g_rescales_ptr[dev];
    // Several streams of unequal length with the automatic split count: cut all their
    // keys into equal chunks over one wave of CTAs (balanced split) when the workspace
    // holds its slot-major partials; the uniform per-stream split otherwise.
    if (nsplit == 0 && B >= 2 && B <= BALANCED_MAX_STREAMS && ws && aligned(ws, 256)) {
        int n_tiles, R_step, R;
        tc_tiling(q_len * H, TC_MAX_ROWS, &n_tiles, &R_step, &R);
        const long long slots = num_sms / n_tiles;
        const long long per_stream = (long long)q_len * H;
        const size_t need = align256((size_t)slots * per_stream * D_V * 4) + align256((size_t)slots * per_stream * 4);
        if (slots - B >= B && need <= ws_bytes) {
            a.balanced = 1;
            a.bal_G = (int)(slots - B);
            a.nsplit = (int)slots;
            a.part_out = static_cast<float*>(ws);
            a.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + align256((size_t)slots * per_stream * D_V * 4));
            if (launch_verify_tc(a, stream) != cudaSuccess) return MLA_ERR_LAUNCH;
            if (combine && launch_combine_balanced(a, stream) != cudaSuccess) return MLA_ERR_LAUNCH;
            return MLA_OK;
        }
    }
    if (ns > 1) {
        size_t need = mla_verify_workspace_bytes(B, q_len, H, ns);
        if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
        if (!aligned(ws, 256)) return MLA_ERR_ALIGN;
        a.part_out = static_cast<float*>(ws);
        a.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + align256((size_t)rows * ns * D_V * 4));
    }
    if (launch_verify_tc(a, stream) != cudaSuccess) return MLA_ERR_LAUNCH;
    if (combine && ns > 1 && launch_combine(a.part_out, a.part_lse, rows, ns, out, lse, stream) != cudaSuccess)
        return MLA_ERR_LAUNCH;
    return MLA_OK;
}

int run_sparse_fp8(bool combine, const void* q, const uint8_t* kv_lat, const float* kv_scale, const void* kv_rope,
                   int64_t n_pool, const int32_t* topk_slots, int topk, int B, int H, float scale, float* out,
                   float* lse, int nsplit, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (B < 0 || B > 65535 || H < 1 || H > MLA_MAX_HEADS) return MLA_ERR_SHAPE;
    if (nsplit < 0 || nsplit > MLA_MAX_NSPLIT) return MLA_ERR_NSPLIT;
    if (B == 0) return MLA_OK;
    if (!q || !kv_lat || !kv_scale || !kv_rope || !topk_slots || !out || !lse) return MLA_ERR_NULL;
    if (topk < 1 || n_pool < 1 || n_pool > 0x7fffffffLL || (long long)B * H > 0x7fffffffLL) return MLA_ERR_SHAPE;
    if (!isfinite(scale)) return MLA_ERR_ARG;
    if (!aligned(q, 16) || !aligned(kv_lat, 16) || !aligned(kv_rope, 16) || !aligned(kv_scale, 4) ||
        !aligned(topk_slots, 4) || !aligned(out, 16) || !aligned(lse, 4))
        return MLA_ERR_ALIGN;
    unsigned* status = nullptr;
    int num_sms = 0, dev = 0;
    int rc = device_state(&dev, &status, &num_sms);
    if (rc != MLA_OK) return rc;
    // automatic split count: every stream has the same topk keys, so one wave of CTAs
    // (no second wave to even out unequal lengths), at least 128 keys per split
    // (measured on c5, 32 streams x 2048 keys: 4 splits per stream in one wave 41.6 us
    // per call, 9 splits in two waves 51.9 us)
    int ns = nsplit;
    if (ns == 0) {
        int n_tiles, R_step, R;
        tc_tiling(H, 80, &n_tiles, &R_step, &R);
        long long per = (long long)num_sms / ((long long)B * n_tiles);
        const long long by_len = (topk + PLAN_MIN_KEYS_PER_SPLIT - 1) / PLAN_MIN_KEYS_PER_SPLIT;
        if (per > by_len) per = by_len;
        if (per > MLA_MAX_NSPLIT) per = MLA_MAX_NSPLIT;
        if (per < 1) per = 1;
        while (per > 1 && mla_verify_workspace_bytes(B, 1, H, (int)per) > (ws ? ws_bytes : 0)) --per;
        ns = (int)per;
    }
    const long long rows = (long long)B * H;
    VerifyArgs a;
    memset(&a, 0, sizeof a);
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.n_pool = n_pool;
    a.slot = topk_slots;
    a.slot_stride = topk;
    a.B = B; a.q_len = 1; a.H = H;
    a.scale = scale;
    a.out = out; a.lse = lse;
    a.nsplit = ns;
    a.status = status;
    a.rescales = g_rescales_ptr[dev];
    a.kv_fp8 = 1;
    a.kv_lat = kv_lat;
    a.kv_scale = kv_scale;
    a.kv_rope = static_cast<const __nv_bfloat16*>(kv_rope);
    if (ns > 1) {
        size_t need = mla_verify_workspace_bytes(B, 1, H, ns);
        if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
        if (!aligned(ws, 256)) return MLA_ERR_ALIGN;
        a.part_out = static_cast<float*>(ws);
        a.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + align256((size_t)rows * ns * D_V * 4));
    }
    if (launch_verify_tc(a, stream) != cudaSuccess) return MLA_ERR_LAUNCH;
    if (combine && ns > 1 && launch_combine(a.part_out, a.part_lse, rows, ns, out, lse, stream) != cudaSuccess)
        return MLA_ERR_LAUNCH;
    return MLA_OK;
}

}  // namespace

extern "C" {

int mla_sparse_fp8_decode(const void* q, const uint8_t* kv_lat_e4m3, const float* kv_scale, const void* kv_rope,
                          int64_t n_pool, const int32_t* topk_slots, int topk, int B, int H, float scale, float* out,
                          float* lse, int nsplit, void* workspace, size_t ws_bytes, mla_stream_t stream) {
    return run_sparse_fp8(true, q, kv_lat_e4m3, kv_scale, kv_rope, n_pool, topk_slots, topk, B, H, scale, out, lse,
                          nsplit, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int mla_sparse_fp8_partials(const void* q, const uint8_t* kv_lat_e4m3, const float* kv_scale, const void* kv_rope,
                            int64_t n_pool, const int32_t* topk_slots, int topk, int B, int H, float scale,
                            float* out, float* lse, int nsplit, void* workspace, size_t ws_bytes,
                            mla_stream_t stream) {
    return run_sparse_fp8(false, q, kv_lat_e4m3, kv_scale, kv_rope, n_pool, topk_slots, topk, B, H, scale, out, lse,
                          nsplit, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t mla_verify_workspace_bytes(int B, int q_len, int H, int nsplit) {
    if (B < 0 || q_len < 1 || H < 1 || nsplit < 1 || nsplit == 1) return 0;
    size_t rows = (size_t)B * q_len * H;
    return align256(rows * nsplit * D_V * 4) + align256(rows * nsplit * 4);
}

int mla_verify_auto_nsplit(int B, int q_len, int H, int max_seq, int num_sms, size_t ws_bytes) {
    if (B <= 0 || q_len < 1 || H < 1 || max_seq < 1 || num_sms < 1) return 1;
    const long long tiles = ((long long)q_len * H + PLAN_ROWS_PER_CTA - 1) / PLAN_ROWS_PER_CTA;
    const long long ctas = (long long)B * tiles;
    // one full wave of CTAs (rounded down, so no CTA spills into a second wave); with
    // several streams of unequal lengths, two waves let the block scheduler even out
    // the per-stream imbalance
    const long long waves = B > 1 ? 2 : 1;
    const long long target = (long long)num_sms * PLAN_CTAS_PER_SM * waves;
    long long ns = target / ctas;
    const long long by_len = (max_seq + PLAN_MIN_KEYS_PER_SPLIT - 1) / PLAN_MIN_KEYS_PER_SPLIT;
    if (ns > by_len) ns = by_len;
    if (ns > MLA_MAX_NSPLIT) ns = MLA_MAX_NSPLIT;
    if (ns < 1) ns = 1;
    while (ns > 1 && mla_verify_workspace_bytes(B, q_len, H, (int)ns) > ws_bytes) --ns;
    return (int)ns;
}

int mla_verify_attn(const void* q, const void* kv_cache, int64_t n_pool, const int32_t* slot_table,
                    int slot_stride, const int32_t* seq_lens, const uint8_t* draft_mask, int B, int q_len,
                    int H, float scale, float* out, float* lse, int nsplit, void* workspace, size_t ws_bytes,
                    mla_stream_t stream) {
    return run_verify(true, q, kv_cache, n_pool, slot_table, slot_stride, seq_lens, draft_mask, nullptr, B, q_len,
                      H, scale, out, lse, nsplit, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int mla_verify_attn_packed(const void* q, const void* kv_cache, int64_t n_pool, const int32_t* slot_table,
                           int slot_stride, const int32_t* seq_lens, const uint64_t* draft_mask_bits, int B,
                           int q_len, int H, float scale, float* out, float* lse, int nsplit, void* workspace,
                           size_t ws_bytes, mla_stream_t stream) {
    if (draft_mask_bits && (reinterpret_cast<uintptr_t>(draft_mask_bits) % 8) != 0) return MLA_ERR_ALIGN;
    return run_verify(true, q, kv_cache, n_pool, slot_table, slot_stride, seq_lens, nullptr, draft_mask_bits, B,
                      q_len, H, scale, out, lse, nsplit, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int mla_kv_append(void* kv_cache, int64_t n_pool, const int32_t* slot_table, int slot_stride,
                  const int32_t* seq_lens, const void* new_kv, int B, int q_len, mla_stream_t stream) {
    if (B < 0 || B > 65535 || q_len < 1 || q_len > MLA_MAX_Q_LEN) return MLA_ERR_SHAPE;
    if (B == 0) return MLA_OK;
    if (!kv_cache || !slot_table || !seq_lens || !new_kv) return MLA_ERR_NULL;
    if (n_pool < 1 || n_pool > 0x7fffffffLL || slot_stride < q_len) return MLA_ERR_SHAPE;
    if (!aligned(kv_cache, 16) || !aligned(new_kv, 16) || !aligned(slot_table, 4) || !aligned(seq_lens, 4))
        return MLA_ERR_ALIGN;
    unsigned* status = nullptr;
    int rc = device_state(nullptr, &status, nullptr);
    if (rc != MLA_OK) return rc;
    if (launch_kv_append(static_cast<__nv_bfloat16*>(kv_cache), slot_table, slot_stride, seq_lens,
                         static_cast<const __nv_bfloat16*>(new_kv), B, q_len, n_pool, status,
                         reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MLA_ERR_LAUNCH;
    return MLA_OK;
}

int mla_verify_partials(const void* q, const void* kv_cache, int64_t n_pool, const int32_t* slot_table,
                        int slot_stride, const int32_t* seq_lens, const uint8_t* draft_mask, int B, int q_len,
                        int H, float scale, float* out, float* lse, int nsplit, void* workspace,
                        size_t ws_bytes, mla_stream_t stream) {
    return run_verify(false, q, kv_cache, n_pool, slot_table, slot_stride, seq_lens, draft_mask, nullptr, B, q_len,
                      H, scale, out, lse, nsplit, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int mla_kv_append_fp8(uint8_t* kv_lat, float* kv_scale, void* kv_rope, int64_t n_pool, const int32_t* slots,
                      const uint8_t* new_lat, const float* new_scale, const void* new_rope, int n_rows,
                      mla_stream_t stream) {
    if (n_rows < 0) return MLA_ERR_SHAPE;
    if (n_rows == 0) return MLA_OK;
    if (!kv_lat || !kv_scale || !kv_rope || !slots || !new_lat || !new_scale || !new_rope) return MLA_ERR_NULL;
    if (n_pool < 1 || n_pool > 0x7fffffffLL) return MLA_ERR_SHAPE;
    if (!aligned(kv_lat, 16) || !aligned(new_lat, 16) || !aligned(kv_rope, 16) || !aligned(new_rope, 16) ||
        !aligned(kv_scale, 4) || !aligned(new_scale, 4) || !aligned(slots, 4))
        return MLA_ERR_ALIGN;
    unsigned* status = nullptr;
    int rc = device_state(nullptr, &status, nullptr);
    if (rc != MLA_OK) return rc;
    if (launch_kv_append_fp8(kv_lat, kv_scale, static_cast<__nv_bfloat16*>(kv_rope), n_pool, slots, new_lat,
                             new_scale, static_cast<const __nv_bfloat16*>(new_rope), n_rows, status,
                             reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MLA_ERR_LAUNCH;
    return MLA_OK;
}

int mla_verify_combine(const float* part_out, const float* part_lse, int B, int q_len, int H, int S, float* out,
                       float* lse, mla_stream_t stream) {
    if (B < 0 || q_len < 1 || H < 1 || (long long)B * q_len * H > 0x7fffffffLL) return MLA_ERR_SHAPE;
    if (S < 1 || S > MLA_MAX_NSPLIT) return MLA_ERR_NSPLIT;
    if (B == 0) return MLA_OK;
    if (!part_out || !part_lse || !out || !lse) return MLA_ERR_NULL;
    if (!aligned(part_out, 16) || !aligned(out, 16) || !aligned(part_lse, 4) || !aligned(lse, 4))
        return MLA_ERR_ALIGN;
    int rc = device_state(nullptr, nullptr, nullptr);
    if (rc != MLA_OK) return rc;
    long long rows = (long long)B * q_len * H;
    if (launch_combine(part_out, part_lse, rows, S, out, lse, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MLA_ERR_LAUNCH;
    return MLA_OK;
}

int mla_verify_status(mla_stream_t stream, uint32_t* device_status, int clear) {
    if (!device_status) return MLA_ERR_NULL;
    unsigned* st = nullptr;
    int rc = device_state(nullptr, &st, nullptr);
    if (rc != MLA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned v = 0;
    if (cudaMemcpyAsync(&v, st, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MLA_ERR_DEVICE;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_DEVICE;
    if (clear) {
        if (cudaMemsetAsync(st, 0, sizeof(unsigned), s) != cudaSuccess) return MLA_ERR_DEVICE;
        if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_DEVICE;
    }
    *device_status = v;
    return MLA_OK;
}

int mla_debug_rescale_count(mla_stream_t stream, uint64_t* count, int clear) {
    if (!count) return MLA_ERR_NULL;
    int dev = 0;
    int rc = device_state(&dev, nullptr, nullptr);
    if (rc != MLA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned long long v = 0;
    if (cudaMemcpyAsync(&v, g_rescales_ptr[dev], sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MLA_ERR_DEVICE;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_DEVICE;
    if (clear) {
        if (cudaMemsetAsync(g_rescales_ptr[dev], 0, sizeof v, s) != cudaSuccess) return MLA_ERR_DEVICE;
        if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_DEVICE;
    }
    *count = (uint64_t)v;
    return MLA_OK;
}

const char* mla_status_string(int status) {
    switch (status) {
        case MLA_OK: return "ok";
        case MLA_ERR_NULL: return "null pointer";
        case MLA_ERR_SHAPE: return "shape out of range";
        case MLA_ERR_ALIGN: return "misaligned pointer";
        case MLA_ERR_WORKSPACE: return "workspace missing or too small";
        case MLA_ERR_NSPLIT: return "nsplit out of range";
        case MLA_ERR_LAUNCH: return "kernel launch failed";
        case MLA_ERR_DEVICE: return "no usable sm_103 device or CUDA runtime error";
        case MLA_ERR_ARG: return "invalid argument";
        default: return "unknown status";
    }
}

int mla_verify_version(void) { return 100; }

int mla_debug_stall_next_launch(void) {
    g_debug_stall.store(true);
    return MLA_OK;
}

}  // extern "C"
