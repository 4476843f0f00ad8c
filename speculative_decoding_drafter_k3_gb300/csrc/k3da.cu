// k3da.cu -- K3 DFlash drafter block attention for sm_103a (GB300).
//
// The operation is the one the page "[None][feat] Share Kimi K3 FP4 modeling
// and add NVFP4 support on SM103" (NVIDIA/TensorRT-LLM PR #20532) defines in
// the commit adding k3_drafter_attn / k3_drafter_attn_qknorm: every draft
// token of a request attends densely (non-causally) to the request's paged
// context (HND pages of 64 tokens) and to its own block's K/V, read from qkv
// and never written to the pool; GQA 6:1; head_dim 64.  The fused variant
// first applies the per-head q/k RMSNorm (eps 1e-5) and NeoX RoPE (base
// 10000) of the drafter's fused_qk_norm_rope cell (commit adding the ops'
// contracts).
//
// Design (one GPU, HBM-bound):
//   * Work unit = (request r, kv head h).  Its items are the block (item 0,
//     the B block keys) and its context pages (items 1..ceil(L/64)).  All
//     units' items are laid end to end and cut into equal contiguous ranges,
//     one per CTA of a grid sized to fill every SM ("stream-K" split), so
//     uneven context lengths never idle an SM.  The split is computed on the
//     device from ctx_lens, so a captured graph replays with new lengths.
//   * A CTA = 3 consumer warps (16 query rows each: 6 q heads x B tokens =
//     48 rows share one kv head) + 1 producer warp.  The producer walks the
//     page table (32 ids per coalesced load, prefetched a batch ahead) and
//     TMA-loads each page's K tile and V tile (64 x 64 bf16, 8 KB each,
//     contiguous in the HND pool) into a ring of shared-memory stages with
//     the 128-byte swizzle, so the ldmatrix reads below are conflict-free.
//   * Consumers: S = Q K^T and O += P V with mma.sync m16n8k16 (bf16 in,
//     fp32 accumulate), online softmax in base 2 with the scale folded in.
//     Q (and, for the unit's first range, the block K/V) are built in shared
//     memory at the start of each range: RMSNorm and RoPE happen on the way
//     in, RoPE angles are reduced in fp64 then turned by an accurate sincosf.
//   * Each (CTA, unit) range writes an unnormalised partial (O, m, l) to the
//     workspace; the combine kernel merges a unit's partials in CTA order
//     (fixed, so reruns are bit-identical) and writes bf16 out.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "k3da.h"

namespace {

constexpr int kD = 64;           // head_dim
constexpr int kP = 64;           // tokens per page
constexpr int kG = 6;            // query heads per kv head
constexpr int kRows = 48;        // kG * max block length
constexpr int kMaxR = 8;
constexpr int kMaxB = 8;
constexpr int kMaxUnits = 32;    // 8 requests x 4 kv heads
constexpr int kConsumerWarps = 3;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kTileBytes = kP * kD * 2;       // 8 KB: one page, one head, K or V
constexpr int kStageBytes = 2 * kTileBytes;   // K + V
constexpr int kStages = 4;
constexpr int kMaxCtasPerSm = 4;
constexpr int kPartialFloats = kRows * kD;    // O of one (CTA, unit) range
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr int kOffStages = 0;
constexpr int kOffQ = kStages * kStageBytes;          // 48 rows x 128 B
constexpr int kOffBlkK = kOffQ + kRows * 128;         // 16 rows x 128 B
constexpr int kOffBlkV = kOffBlkK + 16 * 128;
constexpr int kOffTrig = kOffBlkV + 16 * 128;         // [8][32] float2
constexpr int kOffUnit = kOffTrig + kMaxB * 32 * 8;   // [33] int64
constexpr int kOffLens = kOffUnit + (kMaxUnits + 1) * 8;
constexpr int kOffBar = kOffLens + kMaxR * 4 + 32;    // 2*kStages mbarriers
constexpr int kOffFlag = kOffBar + 2 * kStages * 8;
constexpr int kSmemUsed = kOffFlag + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;          // slack for alignment

struct Params {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *qkv;
    const int32_t *page_table;
    const int32_t *ctx_lens;
    const void *positions;
    const __nv_bfloat16 *q_w;
    const __nv_bfloat16 *k_w;
    float *ws_o;        // [slots][48][64]
    float2 *ws_ml;      // [slots][48]  (m in log2 units, l)
    int32_t *status;
    long long num_pages;
    int page_stride;
    int R, B, Hq, Hkv;
    int pos_i64;
    int grid;           // CTAs of the split pass
    float scale_log2;   // softmax_scale * log2(e)
    float eps;
    double inv_freq[kD / 2];
};

// ------------------------------------------------------------ PTX helpers --

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase.  Gives up when another warp of the CTA
// has given up (abort flag) or after kWaitLimitNs, raising the flag and the
// TIMEOUT status bit; the caller then carries on without the data so every
// warp still reaches every named barrier and the CTA exits.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                            int32_t *status) {
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            if (status) atomicOr(status, K3DA_STATUS_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort_flag, status);
}

__device__ __forceinline__ void tma_load_tile(uint32_t dst, const CUtensorMap *map, int row,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x on the SFU (ex2.approx, flush to zero; 2^-inf = +0).
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Byte offset of (row, dim) in a tile of 128-byte rows stored with the
// 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// --------------------------------------------------------- work partition --
//
// Items of unit u = r*Hkv + h: 1 (the block) + ceil(L_r/64) (pages).  Units
// are laid end to end; ustart[u] is the first item of unit u, ustart[U] = W.
// CTA c of C = min(grid, W) owns items [c*W/C, (c+1)*W/C).

struct Partition {
    long long W;
    int C;
};

// Reads and checks ctx_lens with warp 0; fills lens_s[R] and ustart_s[U+1].
__device__ void build_partition(const Params &p, int *lens_s, long long *ustart_s,
                                bool report) {
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        int L = 0;
        if (lane < p.R) {
            L = __ldg(p.ctx_lens + lane);
            const int cap = p.page_stride * kP;
            bool bad = false;
            if (L < 0) { L = 0; bad = true; }
            if (L > cap) { L = cap; bad = true; }
            if (bad && report && p.status) atomicOr(p.status, K3DA_STATUS_BAD_LENGTH);
            lens_s[lane] = L;
        }
        __syncwarp();
        if (lane == 0) {
            long long acc = 0;
            for (int r = 0; r < p.R; ++r) {
                const long long items = 1 + (lens_s[r] + kP - 1) / kP;
                for (int h = 0; h < p.Hkv; ++h) {
                    ustart_s[r * p.Hkv + h] = acc;
                    acc += items;
                }
            }
            ustart_s[p.R * p.Hkv] = acc;
        }
    }
}

__device__ __forceinline__ long long range_begin(long long c, long long W, long long C) {
    return c * W / C;
}

// The CTA whose range holds item i.
__device__ __forceinline__ int cta_of_item(long long i, long long W, long long C) {
    long long c = i * C / W;
    while (c + 1 < C && range_begin(c + 1, W, C) <= i) ++c;
    while (c > 0 && range_begin(c, W, C) > i) --c;
    return static_cast<int>(c);
}

// ------------------------------------------------------------- consumers --

struct RowState {
    float m[2];   // running max (log2 units) of rows a = lane/4 and b = a + 8
    float l[2];   // running sum (this lane's share)
    float o[8][4];
};

// One tile of NKT*16 keys: K rows and V rows at kbase / vbase (swizzled).
// valid = keys of the tile that are real (the rest are masked out).
template <int NKT>
__device__ __forceinline__ void attend_tile(RowState &st, const uint32_t (&qf)[4][4],
                                            uint32_t kbase, uint32_t vbase, int valid,
                                            float scale_log2, int lane) {
    constexpr int NT = 2 * NKT;  // n-tiles of 8 keys
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    }
    const int mi = lane >> 3, rr = lane & 7;
    // S = Q K^T: B operand = K rows (keys) with dims contiguous.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int kk2 = 0; kk2 < 2; ++kk2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + swz(nt * 8 + rr, kk2 * 4 + mi), b0, b1, b2, b3);
            mma_bf16(s[nt], qf[2 * kk2], b0, b1);
            mma_bf16(s[nt], qf[2 * kk2 + 1], b2, b3);
        }
    }
    const int kq = 2 * (lane & 3);
    if (valid < NKT * 16) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int key = nt * 8 + kq;
            if (key >= valid) { s[nt][0] = -INFINITY; s[nt][2] = -INFINITY; }
            if (key + 1 >= valid) { s[nt][1] = -INFINITY; s[nt][3] = -INFINITY; }
        }
    }
    // Online softmax, base 2, scale folded into the exponent.
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
        mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(kFull, mx[e], 1));
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(kFull, mx[e], 2));
    }
    float mnew[2], alpha[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        mnew[e] = fmaxf(st.m[e], mx[e] * scale_log2);
        alpha[e] = exp2_approx(st.m[e] - mnew[e]);
        st.m[e] = mnew[e];
    }
    float rs[2] = {0.f, 0.f};
    uint32_t pf[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float p0 = exp2_approx(fmaf(s[nt][0], scale_log2, -mnew[0]));
        const float p1 = exp2_approx(fmaf(s[nt][1], scale_log2, -mnew[0]));
        const float p2 = exp2_approx(fmaf(s[nt][2], scale_log2, -mnew[1]));
        const float p3 = exp2_approx(fmaf(s[nt][3], scale_log2, -mnew[1]));
        rs[0] += p0 + p1;
        rs[1] += p2 + p3;
        pf[nt][0] = pack_bf16(p0, p1);
        pf[nt][1] = pack_bf16(p2, p3);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) st.l[e] = st.l[e] * alpha[e] + rs[e];
#pragma unroll
    for (int nd = 0; nd < 8; ++nd) {
        st.o[nd][0] *= alpha[0];
        st.o[nd][1] *= alpha[0];
        st.o[nd][2] *= alpha[1];
        st.o[nd][3] *= alpha[1];
    }
    // O += P V: A operand = P straight from the score registers, B operand =
    // V rows (keys) read transposed.
#pragma unroll
    for (int kk = 0; kk < NKT; ++kk) {
        const uint32_t a[4] = {pf[2 * kk][0], pf[2 * kk][1], pf[2 * kk + 1][0], pf[2 * kk + 1][1]};
#pragma unroll
        for (int ndp = 0; ndp < 4; ++ndp) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vbase + swz(kk * 16 + (mi & 1) * 8 + rr, ndp * 2 + (mi >> 1)), b0, b1, b2, b3);
            if (valid < NKT * 16) {
                // Zero the values of masked keys so that stale non-finite
                // pool contents cannot reach the accumulator (0 * inf).
                const int k0 = kk * 16 + kq;
                const uint32_t lo0 = (k0 < valid) ? 0x0000ffffu : 0u;
                const uint32_t hi0 = (k0 + 1 < valid) ? 0xffff0000u : 0u;
                const uint32_t lo1 = (k0 + 8 < valid) ? 0x0000ffffu : 0u;
                const uint32_t hi1 = (k0 + 9 < valid) ? 0xffff0000u : 0u;
                b0 &= lo0 | hi0;
                b2 &= lo0 | hi0;
                b1 &= lo1 | hi1;
                b3 &= lo1 | hi1;
            }
            mma_bf16(st.o[2 * ndp], a, b0, b1);
            mma_bf16(st.o[2 * ndp + 1], a, b2, b3);
        }
    }
}

// RMSNorm (optional) + NeoX RoPE (optional) of one 64-wide head row held
// as x_lo = dim lane, x_hi = dim lane + 32; stores bf16 into a swizzled tile.
template <bool QKNORM>
__device__ __forceinline__ void prep_row(uint8_t *tile, int row, float x_lo, float x_hi,
                                         const __nv_bfloat16 *w, float eps, float2 cs, int lane) {
    float y_lo = x_lo, y_hi = x_hi;
    if (QKNORM) {
        float ss = x_lo * x_lo + x_hi * x_hi;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
        const float inv = rsqrtf(ss * (1.0f / kD) + eps);
        const float n_lo = x_lo * inv * __bfloat162float(w[lane]);
        const float n_hi = x_hi * inv * __bfloat162float(w[lane + 32]);
        y_lo = n_lo * cs.x - n_hi * cs.y;
        y_hi = n_hi * cs.x + n_lo * cs.y;
    }
    *reinterpret_cast<__nv_bfloat16 *>(tile + swz(row, lane >> 3) + (lane & 7) * 2) =
        __float2bfloat16_rn(y_lo);
    *reinterpret_cast<__nv_bfloat16 *>(tile + swz(row, 4 + (lane >> 3)) + (lane & 7) * 2) =
        __float2bfloat16_rn(y_hi);
}

__device__ __forceinline__ void zero_row(uint8_t *tile, int row, int lane) {
    *reinterpret_cast<__nv_bfloat16 *>(tile + swz(row, lane >> 3) + (lane & 7) * 2) =
        __float2bfloat16_rn(0.f);
    *reinterpret_cast<__nv_bfloat16 *>(tile + swz(row, 4 + (lane >> 3)) + (lane & 7) * 2) =
        __float2bfloat16_rn(0.f);
}

// ------------------------------------------------------------ split pass --

template <bool QKNORM>
__global__ void __launch_bounds__(kThreads, 2)
    k3da_split_kernel(const __grid_constant__ CUtensorMap pool_map, const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    long long *ustart = reinterpret_cast<long long *>(smem + kOffUnit);
    int *lens = reinterpret_cast<int *>(smem + kOffLens);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffFlag);
    const uint32_t bar_full = smem_u32(smem + kOffBar);
    const uint32_t bar_empty = bar_full + kStages * 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    build_partition(p, lens, ustart, blockIdx.x == 0);
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int U = p.R * p.Hkv;
    const long long W = ustart[U];
    const long long C = W < p.grid ? W : p.grid;
    if (blockIdx.x >= C) return;
    const long long beg = range_begin(blockIdx.x, W, C);
    const long long end = range_begin(blockIdx.x + 1, W, C);
    int u0 = 0;
    while (ustart[u0 + 1] <= beg) ++u0;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------ producer warp --
        long long k = 0;  // pages issued by this CTA
        long long i = beg;
        for (int u = u0; i < end; ++u) {
            const long long seg_end = end < ustart[u + 1] ? end : ustart[u + 1];
            const long long a = i - ustart[u], b = seg_end - ustart[u];
            const int r = u / p.Hkv, h = u - r * p.Hkv;
            const long long pa = a == 0 ? 0 : a - 1, pb = b - 1;
            const int n = static_cast<int>(pb - pa);
            const int32_t *row = p.page_table + static_cast<long long>(r) * p.page_stride + pa;
            int next = lane < n ? __ldg(row + lane) : 0;
            for (int base = 0; base < n; base += 32) {
                const int ids = next;
                if (base + 32 < n) next = (base + 32 + lane < n) ? __ldg(row + base + 32 + lane) : 0;
                const int cnt = n - base < 32 ? n - base : 32;
                for (int j = 0; j < cnt; ++j, ++k) {
                    const int page = __shfl_sync(kFull, ids, j);
                    const int s = static_cast<int>(k % kStages);
                    const uint32_t par = static_cast<uint32_t>((k / kStages) & 1);
                    mbar_wait(bar_empty + 8 * s, par ^ 1u, abort_flag, p.status);
                    uint8_t *stage = smem + kOffStages + s * kStageBytes;
                    if (page >= 0 && page < p.num_pages) {
                        if (lane == 0) {
                            mbar_arrive_expect_tx(bar_full + 8 * s, kStageBytes);
                            const int krow = ((page * 2 + 0) * p.Hkv + h) * kP;
                            const int vrow = ((page * 2 + 1) * p.Hkv + h) * kP;
                            tma_load_tile(smem_u32(stage), &pool_map, krow, bar_full + 8 * s);
                            tma_load_tile(smem_u32(stage + kTileBytes), &pool_map, vrow,
                                          bar_full + 8 * s);
                        }
                    } else {
                        // Out-of-range page id: flag it and serve zeros.
                        if (lane == 0 && p.status) atomicOr(p.status, K3DA_STATUS_BAD_PAGE);
                        uint4 *dst = reinterpret_cast<uint4 *>(stage);
                        for (int q = lane; q < kStageBytes / 16; q += 32) dst[q] = make_uint4(0, 0, 0, 0);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_full + 8 * s);
                    }
                    __syncwarp();
                }
            }
            i = seg_end;
        }
        // Drain: every issued load must have landed before the CTA exits
        // (only matters when a wait gave up and the consumers stopped early).
        if (*abort_flag) {
            for (long long j = (k > kStages ? k - kStages : 0); j < k; ++j) {
                const int s = static_cast<int>(j % kStages);
                const uint32_t par = static_cast<uint32_t>((j / kStages) & 1);
                const unsigned long long t0 = global_ns();
                while (!mbar_try_wait(bar_full + 8 * s, par) && global_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        return;
    }

    // ------------------------------------------------------ consumer warps --
    const int ctid = threadIdx.x;  // 0..95
    uint8_t *qtile = smem + kOffQ;
    uint8_t *bk = smem + kOffBlkK;
    uint8_t *bv = smem + kOffBlkV;
    float2 *trig = reinterpret_cast<float2 *>(smem + kOffTrig);
    const int rows = kG * p.B;
    const bool active = warp * 16 < rows;
    const long long row_w = static_cast<long long>(p.Hq + 2 * p.Hkv) * kD;
    const int mi = lane >> 3, rr = lane & 7;
    long long k = 0;
    long long i = beg;
    for (int u = u0; i < end; ++u) {
        const long long seg_end = end < ustart[u + 1] ? end : ustart[u + 1];
        const long long a = i - ustart[u], b = seg_end - ustart[u];
        const int r = u / p.Hkv, h = u - r * p.Hkv;
        const int L = lens[r];

        named_bar_sync(1, 32 * kConsumerWarps);  // previous range is done with the tiles
        if (QKNORM) {
            for (int e = ctid; e < p.B * 32; e += 32 * kConsumerWarps) {
                const int ti = e >> 5, j = e & 31;
                const long long t = static_cast<long long>(r) * p.B + ti;
                const long long pos = p.pos_i64 ? reinterpret_cast<const long long *>(p.positions)[t]
                                                : reinterpret_cast<const int *>(p.positions)[t];
                // Angle in fp64, reduced to [-pi, pi] before the fp32 sincos.
                const double theta = static_cast<double>(pos) * p.inv_freq[j];
                const double turns = rint(theta * 0.15915494309189535);
                double red = fma(-turns, 6.283185307179586, theta);
                red = fma(-turns, 2.4492935982947064e-16, red);
                float sn, cs;
                sincosf(static_cast<float>(red), &sn, &cs);
                trig[ti * 32 + j] = make_float2(cs, sn);
            }
            named_bar_sync(1, 32 * kConsumerWarps);
        }
        // Query rows: row = g*B + i for q head h*6 + g, token i.
        for (int row = warp; row < kRows; row += kConsumerWarps) {
            if (row < rows) {
                const int g = row / p.B, ti = row - g * p.B;
                const long long t = static_cast<long long>(r) * p.B + ti;
                const __nv_bfloat16 *src = p.qkv + t * row_w + static_cast<long long>(h * kG + g) * kD;
                const float x_lo = __bfloat162float(src[lane]);
                const float x_hi = __bfloat162float(src[lane + 32]);
                prep_row<QKNORM>(qtile, row, x_lo, x_hi, p.q_w, p.eps,
                                 QKNORM ? trig[ti * 32 + lane] : make_float2(1.f, 0.f), lane);
            } else {
                zero_row(qtile, row, lane);
            }
        }
        if (a == 0) {
            // The block's own keys (normalised + roped) and values (raw).
            for (int j = warp; j < 16; j += kConsumerWarps) {
                if (j < p.B) {
                    const long long t = static_cast<long long>(r) * p.B + j;
                    const __nv_bfloat16 *ks = p.qkv + t * row_w + static_cast<long long>(p.Hq + h) * kD;
                    const __nv_bfloat16 *vs = p.qkv + t * row_w + static_cast<long long>(p.Hq + p.Hkv + h) * kD;
                    prep_row<QKNORM>(bk, j, __bfloat162float(ks[lane]), __bfloat162float(ks[lane + 32]),
                                     p.k_w, p.eps, QKNORM ? trig[j * 32 + lane] : make_float2(1.f, 0.f),
                                     lane);
                    prep_row<false>(bv, j, __bfloat162float(vs[lane]), __bfloat162float(vs[lane + 32]),
                                    nullptr, 0.f, make_float2(1.f, 0.f), lane);
                } else {
                    zero_row(bk, j, lane);
                    zero_row(bv, j, lane);
                }
            }
        }
        named_bar_sync(1, 32 * kConsumerWarps);

        RowState st;
        st.m[0] = st.m[1] = -INFINITY;
        st.l[0] = st.l[1] = 0.f;
#pragma unroll
        for (int nd = 0; nd < 8; ++nd) st.o[nd][0] = st.o[nd][1] = st.o[nd][2] = st.o[nd][3] = 0.f;
        uint32_t qf[4][4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            ldsm_x4(smem_u32(qtile) + swz(warp * 16 + (mi & 1) * 8 + rr, kk * 2 + (mi >> 1)),
                    qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
        }

        if (a == 0 && active) {
            attend_tile<1>(st, qf, smem_u32(bk), smem_u32(bv), p.B, p.scale_log2, lane);
        }
        const long long pa = a == 0 ? 0 : a - 1, pb = b - 1;
        for (long long pg = pa; pg < pb; ++pg, ++k) {
            const int s = static_cast<int>(k % kStages);
            const uint32_t par = static_cast<uint32_t>((k / kStages) & 1);
            const bool ok = mbar_wait(bar_full + 8 * s, par, abort_flag, p.status);
            if (active && ok) {
                const long long left = static_cast<long long>(L) - pg * kP;
                const int valid = left < kP ? static_cast<int>(left) : kP;
                const uint32_t stage = smem_u32(smem + kOffStages + s * kStageBytes);
                attend_tile<4>(st, qf, stage, stage + kTileBytes, valid, p.scale_log2, lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        }

        // Partial of this (CTA, unit) range.
        if (active) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                st.l[e] += __shfl_xor_sync(kFull, st.l[e], 1);
                st.l[e] += __shfl_xor_sync(kFull, st.l[e], 2);
            }
            const long long slot = static_cast<long long>(blockIdx.x) + u;
            const int ra = warp * 16 + (lane >> 2), rb = ra + 8;
            float *ob = p.ws_o + slot * kPartialFloats;
            const int dq = 2 * (lane & 3);
#pragma unroll
            for (int nd = 0; nd < 8; ++nd) {
                if (ra < rows)
                    *reinterpret_cast<float2 *>(ob + ra * kD + nd * 8 + dq) = make_float2(st.o[nd][0], st.o[nd][1]);
                if (rb < rows)
                    *reinterpret_cast<float2 *>(ob + rb * kD + nd * 8 + dq) = make_float2(st.o[nd][2], st.o[nd][3]);
            }
            if ((lane & 3) == 0) {
                if (ra < rows) p.ws_ml[slot * kRows + ra] = make_float2(st.m[0], st.l[0]);
                if (rb < rows) p.ws_ml[slot * kRows + rb] = make_float2(st.m[1], st.l[1]);
            }
        }
        i = seg_end;
    }
}

// --------------------------------------------------------------- combine --
//
// One CTA per (unit, 16-row chunk); thread = (row, 8 dims).  Merges the
// unit's partials in CTA order and writes the bf16 output row slice.
__global__ void __launch_bounds__(128) k3da_combine_kernel(const __grid_constant__ Params p) {
    __shared__ long long ustart[kMaxUnits + 1];
    __shared__ int lens[kMaxR];
    build_partition(p, lens, ustart, false);
    __syncthreads();
    const int u = blockIdx.x / 3, chunk = blockIdx.x - 3 * (blockIdx.x / 3);
    const int row = chunk * 16 + (threadIdx.x >> 3);
    const int rows = kG * p.B;
    if (row >= rows) return;
    const int d0 = (threadIdx.x & 7) * 8;
    const int U = p.R * p.Hkv;
    const long long W = ustart[U];
    const long long C = W < p.grid ? W : p.grid;
    const int c0 = cta_of_item(ustart[u], W, C);
    const int c1 = cta_of_item(ustart[u + 1] - 1, W, C);
    float M = -INFINITY;
    for (int c = c0; c <= c1; ++c) M = fmaxf(M, p.ws_ml[(static_cast<long long>(c) + u) * kRows + row].x);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float lsum = 0.f;
    for (int c = c0; c <= c1; ++c) {
        const long long slot = static_cast<long long>(c) + u;
        const float2 ml = p.ws_ml[slot * kRows + row];
        const float w = exp2_approx(ml.x - M);
        lsum = fmaf(ml.y, w, lsum);
        const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + slot * kPartialFloats + row * kD + d0);
        const float4 v0 = src[0], v1 = src[1];
        acc[0] = fmaf(v0.x, w, acc[0]);
        acc[1] = fmaf(v0.y, w, acc[1]);
        acc[2] = fmaf(v0.z, w, acc[2]);
        acc[3] = fmaf(v0.w, w, acc[3]);
        acc[4] = fmaf(v1.x, w, acc[4]);
        acc[5] = fmaf(v1.y, w, acc[5]);
        acc[6] = fmaf(v1.z, w, acc[6]);
        acc[7] = fmaf(v1.w, w, acc[7]);
    }
    const float inv = 1.0f / lsum;
    const int r = u / p.Hkv, h = u - r * p.Hkv;
    const int g = row / p.B, ti = row - g * p.B;
    const long long t = static_cast<long long>(r) * p.B + ti;
    uint4 packed;
    packed.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    packed.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    packed.z = pack_bf16(acc[4] * inv, acc[5] * inv);
    packed.w = pack_bf16(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4 *>(p.out + t * (static_cast<long long>(p.Hq) * kD) +
                               static_cast<long long>(h * kG + g) * kD + d0) = packed;
}

// ------------------------------------------------------------------ host --

struct DeviceConfig {
    bool ready;
    int sms;
    int occupancy[2];  // CTAs per SM of the split kernel: [plain, qknorm]
};

std::mutex g_mutex;
thread_local cudaEvent_t g_phase_event = nullptr;
DeviceConfig g_devices[128];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int configure_device(int dev, DeviceConfig *cfg) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (dev < 0 || dev >= 128) return K3DA_EINVAL;
    DeviceConfig &d = g_devices[dev];
    if (!d.ready) {
        int prev = -1;
        if (cudaGetDevice(&prev) != cudaSuccess) return K3DA_ECUDA;
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return K3DA_ECUDA;
        int rc = K3DA_OK;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) rc = K3DA_ECUDA;
        const void *kernels[2] = {reinterpret_cast<const void *>(&k3da_split_kernel<false>),
                                  reinterpret_cast<const void *>(&k3da_split_kernel<true>)};
        int occ[2] = {0, 0};
        for (int v = 0; v < 2 && rc == K3DA_OK; ++v) {
            if (cudaFuncSetAttribute(kernels[v], cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
                cudaSuccess)
                rc = K3DA_ECUDA;
            else if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[v], kernels[v], kThreads, kSmemBytes) !=
                     cudaSuccess)
                rc = K3DA_ECUDA;
        }
        if (rc == K3DA_OK && g_encode == nullptr) {
            cudaDriverEntryPointQueryResult q;
            void *fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                rc = K3DA_ECUDA;
            else
                g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        if (prev != dev) cudaSetDevice(prev);
        if (rc != K3DA_OK) return rc;
        for (int v = 0; v < 2; ++v) {
            if (occ[v] < 1) return K3DA_ECUDA;
            if (occ[v] > kMaxCtasPerSm) occ[v] = kMaxCtasPerSm;
        }
        d.sms = sms;
        d.occupancy[0] = occ[0];
        d.occupancy[1] = occ[1];
        d.ready = true;
    }
    *cfg = d;
    return K3DA_OK;
}

bool supported_heads(int hq, int hkv) { return (hq == 6 && hkv == 1) || (hq == 24 && hkv == 4); }

size_t workspace_for(int sms) {
    const size_t slots = static_cast<size_t>(sms) * kMaxCtasPerSm + kMaxUnits;
    return slots * (kPartialFloats * sizeof(float) + kRows * sizeof(float2));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int launch(void *out, const void *qkv, const void *kv_pool, int64_t num_pages, const int32_t *page_table,
           int page_stride, const int32_t *ctx_lens, int R, int B, int Hq, int Hkv, int head_dim,
           float softmax_scale, bool qknorm, const void *positions, int pos_dtype, const void *q_norm_w,
           const void *k_norm_w, float eps, float rope_base, void *workspace, size_t workspace_bytes,
           int32_t *status, void *stream) {
    if (!out || !qkv || !kv_pool || !page_table || !ctx_lens) return K3DA_EINVAL;
    if (!aligned(out, 16) || !aligned(qkv, 16) || !aligned(kv_pool, 16) || !aligned(page_table, 4) ||
        !aligned(ctx_lens, 4) || (status && !aligned(status, 4)))
        return K3DA_EINVAL;
    if (R < 1 || R > kMaxR || B < 1 || B > kMaxB || page_stride < 1 || num_pages < 1) return K3DA_EINVAL;
    if (head_dim != kD || !supported_heads(Hq, Hkv)) return K3DA_EUNSUPPORTED;
    if (num_pages > ((1LL << 31) - 1) / (2LL * Hkv * kP)) return K3DA_EINVAL;
    if (static_cast<long long>(page_stride) * R > (1LL << 40)) return K3DA_EINVAL;
    if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return K3DA_EINVAL;
    if (qknorm) {
        if (!positions || !q_norm_w || !k_norm_w) return K3DA_EINVAL;
        if (pos_dtype != K3DA_POS_I32 && pos_dtype != K3DA_POS_I64) return K3DA_EINVAL;
        if (!aligned(positions, pos_dtype == K3DA_POS_I64 ? 8 : 4) || !aligned(q_norm_w, 2) ||
            !aligned(k_norm_w, 2))
            return K3DA_EINVAL;
        if (!(eps >= 0.f) || !isfinite(eps) || !(rope_base > 1.f) || !isfinite(rope_base)) return K3DA_EINVAL;
    }
    if (!workspace || !aligned(workspace, 16)) return K3DA_EWORKSPACE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return K3DA_ECUDA;
    DeviceConfig cfg;
    int rc = configure_device(dev, &cfg);
    if (rc != K3DA_OK) return rc;
    if (workspace_bytes < workspace_for(cfg.sms)) return K3DA_EWORKSPACE;

    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD),
                                static_cast<cuuint64_t>(num_pages) * 2 * Hkv * kP};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(kP)};
    const cuuint32_t estrides[2] = {1, 1};
    if (g_encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(kv_pool), dims, strides, box,
                 estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return K3DA_ECUDA;

    Params prm;
    memset(&prm, 0, sizeof prm);
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.qkv = static_cast<const __nv_bfloat16 *>(qkv);
    prm.page_table = page_table;
    prm.ctx_lens = ctx_lens;
    prm.positions = positions;
    prm.q_w = static_cast<const __nv_bfloat16 *>(q_norm_w);
    prm.k_w = static_cast<const __nv_bfloat16 *>(k_norm_w);
    const size_t slots = static_cast<size_t>(cfg.sms) * kMaxCtasPerSm + kMaxUnits;
    prm.ws_o = static_cast<float *>(workspace);
    prm.ws_ml = reinterpret_cast<float2 *>(static_cast<float *>(workspace) + slots * kPartialFloats);
    prm.status = status;
    prm.num_pages = num_pages;
    prm.page_stride = page_stride;
    prm.R = R;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.pos_i64 = pos_dtype == K3DA_POS_I64;
    const int occ = cfg.occupancy[qknorm ? 1 : 0];
    prm.grid = cfg.sms * occ;
    prm.scale_log2 = softmax_scale * 1.4426950408889634f;
    prm.eps = eps;
    for (int j = 0; j < kD / 2; ++j)
        prm.inv_freq[j] = pow(static_cast<double>(rope_base), -2.0 * j / static_cast<double>(kD));

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (qknorm)
        k3da_split_kernel<true><<<prm.grid, kThreads, kSmemBytes, st>>>(map, prm);
    else
        k3da_split_kernel<false><<<prm.grid, kThreads, kSmemBytes, st>>>(map, prm);
    if (cudaGetLastError() != cudaSuccess) return K3DA_ECUDA;
    if (g_phase_event && cudaEventRecord(g_phase_event, st) != cudaSuccess) return K3DA_ECUDA;
    k3da_combine_kernel<<<R * Hkv * 3, 128, 0, st>>>(prm);
    if (cudaGetLastError() != cudaSuccess) return K3DA_ECUDA;
    return K3DA_OK;
}

}  // namespace

extern "C" {

size_t k3da_workspace_bytes(int num_requests, int block_len, int num_q_heads, int num_kv_heads, int device) {
    if (num_requests < 1 || num_requests > kMaxR || block_len < 1 || block_len > kMaxB ||
        !supported_heads(num_q_heads, num_kv_heads))
        return 0;
    int dev = device;
    if (dev < 0 && cudaGetDevice(&dev) != cudaSuccess) return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return workspace_for(sms);
}

int k3da_attn(void *out, const void *qkv, const void *kv_pool, int64_t num_pages, const int32_t *page_table,
              int page_stride, const int32_t *ctx_lens, int num_requests, int block_len, int num_q_heads,
              int num_kv_heads, int head_dim, float softmax_scale, void *workspace, size_t workspace_bytes,
              int32_t *status, void *stream) {
    return launch(out, qkv, kv_pool, num_pages, page_table, page_stride, ctx_lens, num_requests, block_len,
                  num_q_heads, num_kv_heads, head_dim, softmax_scale, false, nullptr, 0, nullptr, nullptr, 0.f,
                  0.f, workspace, workspace_bytes, status, stream);
}

int k3da_attn_qknorm(void *out, const void *qkv, const void *kv_pool, int64_t num_pages,
                     const int32_t *page_table, int page_stride, const int32_t *ctx_lens, int num_requests,
                     int block_len, int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale,
                     const void *positions, int pos_dtype, const void *q_norm_w, const void *k_norm_w, float eps,
                     float rope_base, void *workspace, size_t workspace_bytes, int32_t *status, void *stream) {
    return launch(out, qkv, kv_pool, num_pages, page_table, page_stride, ctx_lens, num_requests, block_len,
                  num_q_heads, num_kv_heads, head_dim, softmax_scale, true, positions, pos_dtype, q_norm_w,
                  k_norm_w, eps, rope_base, workspace, workspace_bytes, status, stream);
}

int k3da_set_phase_event(void *event) {
    g_phase_event = static_cast<cudaEvent_t>(event);
    return K3DA_OK;
}

const char *k3da_error_string(int code) {
    switch (code) {
        case K3DA_OK: return "ok";
        case K3DA_EINVAL: return "invalid argument (NULL or misaligned pointer, size out of range)";
        case K3DA_EUNSUPPORTED: return "unsupported head layout or head_dim";
        case K3DA_ECUDA: return "CUDA runtime call failed";
        case K3DA_EWORKSPACE: return "workspace missing, misaligned or too small";
        case K3DA_STATUS_BAD_LENGTH: return "device: context length out of range (clamped)";
        case K3DA_STATUS_BAD_PAGE: return "device: page id out of range (zeros used)";
        case K3DA_STATUS_TIMEOUT: return "device: an internal wait timed out (output invalid)";
        default: return "several device status bits or an unknown code";
    }
}

int k3da_version(void) { return 100; }

}  // extern "C"
