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
//     the B block keys) and its context pages (items 1..ceil(L/64)).  A unit
//     is cut into chunks of ch(u) items: ceil(items/n) with n = max(16,
//     ceil(304/units)), at least min(ceil(items/16), 4), rounded up to a
//     power of two above 4 and at most kChunkMax (unit_chunking), so chunk
//     boundaries depend on that unit's length and the call's shape alone.
//     All units' items are laid end to end and the line is cut into one
//     slice per CTA of the grid (sized to fill every SM); a CTA takes the
//     chunks that start in its slice.  When every CTA gets several of the
//     largest chunks, the line counts each chunk as its unit's chunk size and
//     is cut into whole-chunk slices of equal size (build_plan).  Long and
//     short contexts thus spread over all SMs, and every chunk's partial
//     result is the same whatever the other requests hold: requests are
//     isolated bit for bit.  The plan is built on the device from ctx_lens,
//     so a captured graph replays with new lengths.
//   * The split pass (k3da_tc_kernel, below) runs on the 5th-generation
//     tensor cores: a producer warp walks the page table (32 ids per
//     coalesced load, a batch ahead) and TMA-loads each page's K and V tiles
//     (64 x 64 bf16, 8 KB each, contiguous in the HND pool, 128-byte
//     swizzle) into a 6-stage ring in shared memory; one warp issues
//     S = Q K^T and another O += P V as M = 64 tcgen05.mma with TMEM
//     accumulators (three S/P buffers, so QK^T runs up to two pages ahead);
//     four row warps run the online softmax (base 2, scale folded in, lazy
//     rescale) and hand P to the P.V product through TMEM.
//   * When a CTA starts on a unit, each row thread loads its q (or block k,
//     v) row's pieces straight from qkv into registers and writes operand tiles:
//     RMSNorm and RoPE happen on the way in.  A RoPE angle is reduced
//     exactly in integer arithmetic (position times a 64-bit fixed-point
//     turn rate, wrapping), then turned by an accurate sincospif.
//   * Each chunk leaves an unnormalised partial (O as bf16, m and l in fp32)
//     in the workspace; the combine kernel folds a unit's chunk partials in
//     a fixed order and writes bf16 out, so reruns are bit-identical.
//   * Inputs and output may be pinned host memory the GPU addresses across
//     the host link.  Then a stage kernel first copies qkv, positions and
//     lengths into the workspace, once, and the split pass (its
//     programmatic dependent) reads the copies.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "k3da.h"
#include "rope_table.h"

namespace {

constexpr int kD = 64;           // head_dim
constexpr int kP = 64;           // tokens per page
constexpr int kG = 6;            // query heads per kv head
constexpr int kRows = 48;        // kG * max block length
constexpr int kMaxR = 8;
constexpr int kMaxB = 8;
constexpr int kMaxUnits = 32;    // 8 requests x 4 kv heads
constexpr int kTileBytes = kP * kD * 2;       // 8 KB: one page, one head, K or V
constexpr int kStageBytes = 2 * kTileBytes;   // K + V
constexpr int kMaxCtasPerSm = 2;
constexpr int kChunkSplits = 16;   // a unit is cut into at most this many chunks ...
constexpr int kChunkTarget = 304;  // ... or, with few units, about this many chunks in all
constexpr int kChunkMax = 32;      // ... of at most this many pages, beyond which it gets more chunks
constexpr int kPartialElems = kRows * kD;     // O of one chunk, bf16
// Workspace: a reserved header, the chunk partials (slot u * slots_per_unit
// + j: bf16 O, then (m, l) fp32 per row), then room to stage host-resident
// inputs (k3da_stage_kernel): qkv sized for the largest call of the head
// layout, so that the workspace never depends on R or B beyond the
// partials, then the positions (at most 64 int64) and the lengths.
constexpr size_t kWsHeaderBytes = 512;  // the partials follow, 16-byte aligned as the workspace is
constexpr size_t kSlotBytes = kPartialElems * 2 + kRows * 8;
__host__ __device__ constexpr size_t staging_qkv_bytes(int Hq, int Hkv) {
    return static_cast<size_t>(kMaxR) * kMaxB * (Hq + 2 * Hkv) * kD * 2;
}
constexpr size_t kStagingPosBytes = kMaxR * kMaxB * 8;
__host__ __device__ constexpr size_t staging_bytes(int Hq, int Hkv) {
    return staging_qkv_bytes(Hq, Hkv) + kStagingPosBytes + 64;
}
constexpr int kMaxPageStride = 0x7fffffff / kP;  // page_stride * 64 stays an int
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

struct Params {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *qkv;
    const int32_t *page_table;
    const int32_t *ctx_lens;
    const void *positions;
    const __nv_bfloat16 *q_w;
    const __nv_bfloat16 *k_w;
    __nv_bfloat16 *ws_o;  // [slots][48][64]: a chunk's unnormalised O, rounded to bf16 once
    float2 *ws_ml;      // [slots][48]  (m in log2 units, l)
    int32_t *status;
    long long num_pages;
    int page_stride;
    int R, B, Hq, Hkv;
    int pos_i64;
    int grid;           // CTAs of the split pass
    int slots_per_unit; // workspace slots of a unit: chunk j of unit u is slot u * slots_per_unit + j
    int splits;         // chunk_splits(R * Hkv)
    float scale_log2;   // softmax_scale * log2(e)
    float eps;
    float rope_mscale;  // multiplier of the rotated q and k (YaRN), 1 for plain RoPE
    unsigned long long turn_rate[kD / 2];  // RoPE frequency of pair j in turns per position, 2^64 = one turn
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
                                            int32_t *status, unsigned long long limit_ns = kWaitLimitNs) {
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > limit_ns) {
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

__device__ __forceinline__ void tma_load_tile(uint32_t dst, const CUtensorMap *map, int row, uint32_t bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 2^x on the SFU (ex2.approx, flush to zero; 2^-inf = +0).
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Pairs of fp32 in one 64-bit register pair (x in the low word) for the
// paired fp32 arithmetic of sm_100-family GPUs (f32x2: each lane rounded
// like its scalar instruction).
__device__ __forceinline__ unsigned long long pack_f32x2(float x, float y) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}

__device__ __forceinline__ float2 unpack_f32x2(unsigned long long v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

__device__ __forceinline__ unsigned long long fma_f32x2(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// max(a, b, c) in one instruction (sm_100 family); NaN operands are dropped
// as by fmaxf.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ unsigned long long add_f32x2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Global stores with an L2 cache-policy hint (the chunk partials: kept in L2
// for the combine while the pool streams through with evict_first).
__device__ __forceinline__ void st_hint_v4(uint4 *p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void st_hint_f2(float2 *p, float2 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(p), "f"(v.x), "f"(v.y), "l"(pol) : "memory");
}

// Byte offset of (row, dim) in a tile of 128-byte rows stored with the
// 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ------------------------------------------------------------ work plan --
//
// Items of unit u = r*Hkv + h: 1 (the block) + ceil(L_r/64) (pages); unit u
// covers items [ustart[u], ustart[u+1]) of the line, W = ustart[U].  Chunk j
// of unit u covers its items [j*ch, min((j+1)*ch, items)) and leaves its
// partial in workspace slot u * slots_per_unit + j.  A CTA takes the chunks
// whose start lies in its slice of the line (build_plan says which line and
// how many slices): one run of consecutive chunks per unit it touches.

struct Plan {
    long long ustart[kMaxUnits + 1];
    int ch[kMaxUnits];
    int nch[kMaxUnits];
    int lens[kMaxR];
    int nrun;
    int run_u[kMaxUnits];
    int run_j0[kMaxUnits];
    int run_j1[kMaxUnits];
    int run_p0[kMaxUnits];          // first page of the run
    int run_pq[kMaxUnits + 1];      // pages of earlier runs (producer sequence)
};
static_assert(sizeof(Plan) <= 1536, "plan fits its shared-memory slot");


// Chunks a unit is cut into (before the kChunkMax cap): 16, or more when
// there are few units so that a single request still spreads over the GPU.
// A function of the call's shape only, never of the lengths, so a chunk's
// partial does not depend on other requests.
__host__ __device__ constexpr int chunk_splits(int units) {
    return (kChunkTarget + units - 1) / units > kChunkSplits ? (kChunkTarget + units - 1) / units : kChunkSplits;
}

// Chunk size and count of a unit of `items` items (the block and its
// pages) in a call of U units (splits = chunk_splits(U)): a function of the
// unit's own length and the call's shape only, so a chunk's partial does
// not depend on other requests.
// Finer chunks for few units, but never below the 16-way split's chunk or 4
// items, whichever is smaller (short units keep the 16-way chunking); chunks
// of 5 or more items take the next power of two (8, 16, 32), so the chunk
// sizes of long units divide one another.
__device__ __forceinline__ void unit_chunking(int items, int splits, int &ch, int &nch) {
    ch = (items + splits - 1) / splits;
    const int ch16 = (items + kChunkSplits - 1) / kChunkSplits;
    const int floor_ch = ch16 < 4 ? ch16 : 4;
    ch = ch > floor_ch ? ch : floor_ch;
    if (ch > 4) ch = 1 << (32 - __clz(ch - 1));
    ch = ch < 1 ? 1 : (ch > kChunkMax ? kChunkMax : ch);
    nch = (ch & (ch - 1)) == 0 ? (items + ch - 1) >> (31 - __clz(ch)) : (items + ch - 1) / ch;
}

// A request's context length, clamped to [0, page_stride * 64] (a length
// outside it is flagged by the split pass).
__device__ __forceinline__ int clamped_length(const Params &p, int L, bool *bad) {
    const int cap = p.page_stride * kP;
    *bad = L < 0 || L > cap;
    return L < 0 ? 0 : (L > cap ? cap : L);
}

// Warp 0 reads and checks ctx_lens and builds the plan, one lane per unit
// with shuffle scans.  The caller syncs.  An item is the block (item 0) or
// one page of the unit; a chunk holds at most kChunkMax items.
__device__ void build_plan(const Params &p, Plan *pl, int cta, int C, bool report) {
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    int L = 0;
    if (lane < p.R) {
        bool bad = false;
        L = clamped_length(p, __ldg(p.ctx_lens + lane), &bad);
        if (bad && report && p.status) atomicOr(p.status, K3DA_STATUS_BAD_LENGTH);
        pl->lens[lane] = L;
    }
    const int U = p.R * p.Hkv;
    const int u = lane;
    const int Lu = __shfl_sync(kFull, L, (u < U ? u / p.Hkv : 0));
    int items = 0, ch = 1, nch = 0;
    if (u < U) {
        items = 1 + (Lu + kP - 1) / kP;
        unit_chunking(items, p.splits, ch, nch);
    }
    // Inclusive scans over units of the items and of the nominal line
    // (nch * ch); 32-bit throughout: items <= 2^25, so W, WN < 2^31.
    const int wn = u < U ? nch * ch : 0;
    int si = items, sw = wn, chmax = u < U ? ch : 1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int ti = __shfl_up_sync(kFull, si, off);
        const int tw = __shfl_up_sync(kFull, sw, off);
        if (lane >= off) { si += ti; sw += tw; }
        chmax = max(chmax, __shfl_xor_sync(kFull, chmax, off == 1 ? 16 : off >> 1));
    }
    const int base = si - items;
    if (u < U) {
        pl->ustart[u] = base;
        pl->ch[u] = ch;
        pl->nch[u] = nch;
    }
    const int W = __shfl_sync(kFull, si, U - 1);
    const int WN = __shfl_sync(kFull, sw, U - 1);
    if (lane == 0) {
        pl->ustart[U] = W;
        pl->run_pq[0] = 0;
        pl->nrun = 0;
    }
    // Which CTA computes which chunk.  With few items per CTA (W < 2 C
    // chmax, chmax the largest chunk), CTA c takes the chunks whose first
    // item lies in the c-th of C equal slices of the item line.  With many
    // (every CTA holds several of the largest chunks), whole chunks would
    // leave some CTAs one chunk more than others and a tail in which only
    // those run; instead each chunk counts as its unit's chunk size ch
    // (the short last chunk too) on a nominal line of WN = sum nch * ch,
    // cut for Ce = ceil(WN / (k chmax)) CTAs with k = ceil(WN / (C chmax)):
    // every CTA then holds k chunks' worth (chunk sizes are powers of two,
    // so the slices hold whole chunks) and all stream to the end together;
    // CTAs c >= Ce take no work.  Either way a function of the lengths that
    // only decides which CTA computes a chunk, never a chunk's boundaries.
    int Ce = C, line_base = base, line_total = W;
    if (W >= 2 * C * chmax) {
        const int k = (WN + C * chmax - 1) / (C * chmax);
        Ce = (WN + k * chmax - 1) / (k * chmax);
        line_base = sw - wn;
        line_total = WN;
    }
    bool has = false;
    int j0 = 0, j1 = 0, p0 = 0, npg = 0;
    if (u < U && cta < Ce) {
        // Slice [ceil(c T / Ce), ceil((c + 1) T / Ce)) of the line, T =
        // line_total, as c q + ceil(c r / Ce) with T = q Ce + r (c <= Ce,
        // so c q <= T: no 64-bit arithmetic).
        const int q = line_total / Ce, rem = line_total - q * Ce;
        const int lo = cta * q + (cta * rem + Ce - 1) / Ce;
        const int hi = (cta + 1) * q + ((cta + 1) * rem + Ce - 1) / Ce;
        int a = lo - line_base <= 0 ? 0 : (lo - line_base + ch - 1) / ch;
        int b = hi - line_base <= 0 ? 0 : (hi - line_base + ch - 1) / ch;
        a = a > nch ? nch : a;
        b = b > nch ? nch : b;
        if (a < b) {
            has = true;
            j0 = a;
            j1 = b;
            const int i0 = j0 * ch;
            const int i1 = j1 * ch < items ? j1 * ch : items;
            p0 = i0 == 0 ? 0 : i0 - 1;
            npg = (i1 - 1) - p0;
        }
    }
    const unsigned mask = __ballot_sync(kFull, has);
    int sp = npg;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(kFull, sp, off);
        if (lane >= off) sp += t;
    }
    if (has) {
        const int idx = __popc(mask & ((1u << lane) - 1u));
        pl->run_u[idx] = u;
        pl->run_j0[idx] = j0;
        pl->run_j1[idx] = j1;
        pl->run_p0[idx] = p0;
        pl->run_pq[idx + 1] = sp;
    }
    if (lane == 0) pl->nrun = __popc(mask);
}

// ---------------------------------------------------- tcgen05 split pass --
//
// The two contractions run on the 5th-generation tensor cores.  An item is
// the block or one page.  Row warp w owns TMEM lane quarter q = w: query row
// rho = 12*q + l (l < 12) is Q-tile row 16*q + l and TMEM lane 32*q + l (the
// M = 64 MMAs put rows 16q..16q+15 in lanes 0-15 of lane quarter q).  Threads
// l and l + 16 of the warp share that lane through the half-split TMEM
// access (shape 16x32bx2): the first handles keys 0..31 of its page, the
// second keys 32..63, so a row's softmax costs two threads half a page each
// and one shuffle to share the row maximum.  The producer warp streams K/V
// pages with TMA; one warp issues the QK^T products and another the P.V
// products (a thread issues one MMA at a time, so two issuers double the
// tensor work a CTA can have in flight):
//   S[b] (64 x 64 fp32, TMEM)  = Q (64 x 64, smem) . K_page^T
//   O    (64 x 64 fp32, TMEM) += P[b] (bf16, TMEM) . V_page
// with three buffers b = item mod 3.  The softmax keeps a per-row exponent
// base m; P = 2^(s*scale*log2e - m) is written as bf16 over the first half
// of the item's own S buffer once the warp has read it (each thread its half
// of the row's keys) and becomes the A operand of the PV MMA, which leaves
// the row's whole O in its lane.  The QK^T of item i+3 reuses the buffer
// once item i's PV has read its P, so the softmax never waits for a PV to
// free a P buffer, and QK^T runs up to two items ahead of it.  O is
// only rescaled when a row's maximum passes m by more than 8 (log2 units;
// P <= 256 is exact enough in bf16 and fp32), so the common path never
// touches O.
namespace tc {
constexpr int kStages = 6;
constexpr int kRowWarps = 4;  // one warp per TMEM lane quarter
constexpr int kRowThreads = 32 * kRowWarps;
constexpr int kRowsPerQuarter = 12;
constexpr int kProducerWarp = kRowWarps;
constexpr int kQkWarp = kRowWarps + 1;  // issues the QK^T products (and owns the TMEM allocation)
constexpr int kPvWarp = kRowWarps + 2;  // issues the P.V products
constexpr int kThreads = 32 * (kRowWarps + 3);
// Tensor memory: S/P buffer b (64 columns; P, 32 columns of bf16 pairs,
// over its first half) at 64*b, O at 192.
constexpr uint32_t kSBufs = 3;
constexpr uint32_t kSCols = 64u;
constexpr uint32_t kColO = kSBufs * kSCols;
constexpr uint32_t kTmemCols = 256u;
static_assert(kColO + 64u <= kTmemCols, "tensor memory columns");
constexpr int kCtasPerSm = 2;  // 2 x 256 of the SM's 512 TMEM columns
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Shared memory (offsets from a 1024-byte aligned base).
constexpr int kOffStages = 0;                        // kStages x (K tile, V tile)
constexpr int kOffQ = kStages * kStageBytes;         // kQRows rows x 128 B, 128B swizzle
constexpr int kBlkRows = 16;                          // block tiles: B <= 8 keys, one 16-row MMA step
constexpr int kQRows = 64;                            // M of the MMAs: rows 16q..16q+15 -> TMEM lanes 32q..32q+15
constexpr int kOffBlkK = kOffQ + kQRows * 128;        // kBlkRows rows x 128 B
constexpr int kOffBlkV = kOffBlkK + kBlkRows * 128;  // kBlkRows rows x 128 B
// RoPE (cos, sin) of pair j and token i at [j][i], kMaxB + 1 entries per
// pair: a warp's rows read one pair for up to 8 tokens at a time.
constexpr int kTrigStride = kMaxB + 1;
constexpr int kOffTrig = kOffBlkV + kBlkRows * 128;
constexpr int kOffNormW = kOffTrig + (kD / 2) * kTrigStride * 8;  // q and k norm weights, [2][64] bf16
constexpr int kOffPlan = kOffNormW + 2 * kD * 2;
constexpr int kNumBars = 2 * kStages + 3 * kSBufs + 2;  // full, empty, s_full[3], p_full[3], o_done[3], q_ready, done
constexpr int kOffBar = kOffPlan + (static_cast<int>(sizeof(Plan)) + 15) / 16 * 16;
constexpr int kOffTaddr = kOffBar + kNumBars * 8;
constexpr int kOffFlag = kOffTaddr + 8;
constexpr int kSmemUsed = kOffFlag + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
// Two CTAs per SM: 228 KB per SM, 1 KB of it reserved per CTA.
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs fit an SM's shared memory");
static_assert(kOffQ % 1024 == 0 && kOffBlkK % 1024 == 0 && kOffBlkV % 1024 == 0, "SW128 tiles need 1 KB alignment");
static_assert(kOffBar % 8 == 0 && kOffPlan % 8 == 0, "mbarrier / int64 alignment");

// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), K-major A and B unless bit 16 makes B
// MN-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t idesc_f16(uint32_t m, uint32_t n, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? 1u << 16 : 0u) | ((n >> 3) << 17) | ((m >> 4) << 24);
}
constexpr uint32_t kIdescQK = idesc_f16(kQRows, 64, false);            // a page's keys
constexpr uint32_t kIdescQKBlock = idesc_f16(kQRows, kBlkRows, false); // the block tile
constexpr uint32_t kIdescPV = idesc_f16(kQRows, 64, true);

// Shared-memory matrix descriptor of a tile stored in 128-byte rows with the
// 128-byte swizzle (8-row, 1 KB atoms): start address >> 4 (bits 0-13),
// leading byte offset 16 B >> 4 (bits 16-29, unused here), stride byte
// offset 1 KB >> 4 between 8-row groups (bits 32-45), descriptor version 1
// (bits 46-47), layout SWIZZLE_128B = 2 (bits 61-63).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t smem_addr) {
    return static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Half-split access (shape 16x32bx2): threads 0-15 reach TMEM lanes
// base+0..15 at columns [c, c+n), threads 16-31 the same lanes at columns
// [c+n, c+2n).  Two threads thus share one lane (one query row), each with
// its own half of the row's columns.
__device__ __forceinline__ void tmem_ld_h32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32], 32;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st_h32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], 32, {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_h16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], 16, {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

}  // namespace tc

// Positions of the call's tokens lane and lane + 32 (row warps 1-3 keep
// them in registers and share them by shuffle).
__device__ __forceinline__ void load_positions(const Params &p, int lane, long long &pos_lo, long long &pos_hi) {
    const int nt = p.R * p.B;
    if (lane < nt)
        pos_lo = p.pos_i64 ? reinterpret_cast<const long long *>(p.positions)[lane]
                           : reinterpret_cast<const int *>(p.positions)[lane];
    if (lane + 32 < nt)
        pos_hi = p.pos_i64 ? reinterpret_cast<const long long *>(p.positions)[lane + 32]
                           : reinterpret_cast<const int *>(p.positions)[lane + 32];
}

// STAGED: qkv and the positions come from the workspace copy that
// k3da_stage_kernel (this grid's programmatic prerequisite) writes; the row
// warps wait for it before their first read of either.
template <bool QKNORM, bool STAGED>
__global__ void __launch_bounds__(tc::kThreads, tc::kCtasPerSm)
    k3da_tc_kernel(const __grid_constant__ CUtensorMap pool_map, const __grid_constant__ Params p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Plan *pl = reinterpret_cast<Plan *>(smem + kOffPlan);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffFlag);
    uint32_t *taddr_slot = reinterpret_cast<uint32_t *>(smem + kOffTaddr);
    const uint32_t bars = smem_u32(smem + kOffBar);
    const uint32_t bar_full = bars, bar_empty = bars + 8 * kStages;
    const uint32_t bar_sfull = bars + 16 * kStages, bar_pfull = bar_sfull + 8 * kSBufs;
    const uint32_t bar_odone = bar_pfull + 8 * kSBufs, bar_qready = bar_odone + 8 * kSBufs, bar_done = bar_qready + 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // The norm weights and the positions of all the call's tokens do not
    // depend on the plan: their loads are issued first and land while the
    // plan is built (the weights go to shared memory once the row warps
    // start; row warps 1-3, which form the RoPE angles, keep the positions
    // in registers and share them by shuffle).
    __nv_bfloat16 w_early = __float2bfloat16_rn(0.f);
    long long pos_lo = 0, pos_hi = 0;  // row warps 1-3: positions of tokens lane and lane + 32
    // A row thread's RoPE pair is j = its lane (every angle it forms): its
    // turn rate, read with constant indices (a lane-dependent index into the
    // kernel parameters would serialize the warp's reads) and early (the
    // first touch of a launch's parameters misses their cache).
    // Only row warps 1-3 form angles, so warp 0 (which builds the plan)
    // never waits for these reads.
    unsigned long long my_rate = 0;
    if (QKNORM && threadIdx.x < kRowThreads) {
        w_early = threadIdx.x < kD ? p.q_w[threadIdx.x] : p.k_w[threadIdx.x - kD];
        if (warp != 0) {
            if (!STAGED) load_positions(p, lane, pos_lo, pos_hi);
#pragma unroll
            for (int j = 0; j < kD / 2; ++j)
                if (lane == j) my_rate = p.turn_rate[j];
        }
    }
    build_plan(p, pl, blockIdx.x, p.grid, blockIdx.x == 0);
    if (STAGED && warp < kRowWarps) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (QKNORM && warp != 0) load_positions(p, lane, pos_lo, pos_hi);
    }
    {
        // Q and block tiles start as zeros: rows without a query row or a
        // block token stay zero for the whole kernel.
        uint4 *z = reinterpret_cast<uint4 *>(smem + kOffQ);
        for (int e = threadIdx.x; e < (kQRows * 128 + 2 * kBlkRows * 128) / 16; e += kThreads) z[e] = make_uint4(0, 0, 0, 0);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < static_cast<int>(kSBufs); ++b) {
            mbar_init(bar_sfull + 8 * b, 1);
            mbar_init(bar_pfull + 8 * b, kRowWarps);
            mbar_init(bar_odone + 8 * b, 1);
        }
        mbar_init(bar_qready, kRowWarps);
        mbar_init(bar_done, 2);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kQkWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(taddr_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *taddr_slot;
    const int nrun = pl->nrun;

    if (warp == kProducerWarp && nrun > 0) {
        // ------------------------------------------------ producer warp --
        // The CTA's pages, run after run, form one sequence; lane l resolves
        // entry base + l of each 32-entry batch (page id -> TMA row of its K
        // tile, -1 if out of range), one batch ahead of the loads it feeds.
        uint64_t policy;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
        const int total = pl->run_pq[nrun];
        auto resolve = [&](int q) -> int {
            if (q >= total) return -1;
            int k = 0;
            while (pl->run_pq[k + 1] <= q) ++k;
            const int u = pl->run_u[k];
            const int r = u / p.Hkv, h = u - r * p.Hkv;
            const int page = __ldg(p.page_table + static_cast<long long>(r) * p.page_stride + pl->run_p0[k] +
                                   (q - pl->run_pq[k]));
            if (page < 0 || page >= p.num_pages) return -1;  // served as zeros, flagged
            return ((page * 2 + 0) * p.Hkv + h) * kP;
        };
        int cur = resolve(lane), nxt = resolve(32 + lane);
        for (int q = 0; q < total; ++q) {
            if (q > 0 && (q & 31) == 0) {
                cur = nxt;
                nxt = resolve(q + 32 + lane);
            }
            const int krow = __shfl_sync(kFull, cur, q & 31);
            const int s = q % kStages;
            const uint32_t par = static_cast<uint32_t>((q / kStages) & 1);
            mbar_wait(bar_empty + 8 * s, par ^ 1u, abort_flag, p.status);
            uint8_t *stage = smem + kOffStages + s * kStageBytes;
            if (krow < 0) {
                // Out-of-range page id: flag it and serve zeros.
                if (lane == 0 && p.status) atomicOr(p.status, K3DA_STATUS_BAD_PAGE);
                uint4 *dz = reinterpret_cast<uint4 *>(stage);
                for (int e = lane; e < kStageBytes / 16; e += 32) dz[e] = make_uint4(0, 0, 0, 0);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            __syncwarp();
            if (lane == 0) {
                if (krow >= 0) {
                    mbar_arrive_expect_tx(bar_full + 8 * s, kStageBytes);
                    tma_load_tile(smem_u32(stage), &pool_map, krow, bar_full + 8 * s, policy);
                    tma_load_tile(smem_u32(stage + kTileBytes), &pool_map, krow + p.Hkv * kP, bar_full + 8 * s,
                                  policy);
                } else {
                    mbar_arrive(bar_full + 8 * s);
                }
            }
            __syncwarp();
        }
        // Drain: every issued load must land before the CTA exits (matters
        // only when a wait gave up and the consumers stopped early).
        if (*abort_flag) {
            for (int j = (total > kStages ? total - kStages : 0); j < total; ++j) {
                const int s = j % kStages;
                const uint32_t par = static_cast<uint32_t>((j / kStages) & 1);
                const unsigned long long t0 = global_ns();
                while (!mbar_try_wait(bar_full + 8 * s, par) && global_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if ((warp == kQkWarp || warp == kPvWarp) && nrun > 0) {
        // ------------------------------------------------- MMA warps --
        // A thread issues one tcgen05.mma at a time, so the two products
        // have an issuing warp each.  The QK^T warp fills buffer b = i mod 3
        // for item i once item i-3's P.V has read the P stored there.  The
        // P.V warp accumulates O once item i's P is in TMEM, then releases
        // the page's stage (the item's QK^T completed before its softmax
        // began).
        const bool is_qk = warp == kQkWarp;
        const uint64_t q_desc = desc_sw128(smem_u32(smem + kOffQ));
        const uint64_t bk_desc = desc_sw128(smem_u32(smem + kOffBlkK));
        const uint64_t bv_desc = desc_sw128(smem_u32(smem + kOffBlkV));
        long long it = 0, kr = 0;
        for (int rn = 0; rn < nrun; ++rn) {
            const int u = pl->run_u[rn];
            const int ch = pl->ch[u];
            const int items = static_cast<int>(pl->ustart[u + 1] - pl->ustart[u]);
            if (is_qk) {
                mbar_wait(bar_qready, static_cast<uint32_t>(rn & 1), abort_flag, p.status);
                fence_after();
            }
            for (int jc = pl->run_j0[rn]; jc < pl->run_j1[rn]; ++jc) {
                const int i0 = jc * ch;
                const int i1 = i0 + ch < items ? i0 + ch : items;
                for (int item = i0; item < i1; ++item, ++it) {
                    const int b = static_cast<int>(static_cast<uint32_t>(it) % kSBufs);
                    const uint32_t ph = (static_cast<uint32_t>(it) / kSBufs) & 1u;
                    const bool is_page = item > 0;
                    const int s = static_cast<int>(kr % kStages);
                    if (is_page) ++kr;
                    if (is_qk) {
                        if (it >= kSBufs) {  // buffer b is free once item it-3's P.V has read its P
                            mbar_wait(bar_odone + 8 * b, ph ^ 1u, abort_flag, p.status);
                            fence_after();
                        }
                        if (is_page) {
                            mbar_wait(bar_full + 8 * s, static_cast<uint32_t>(((kr - 1) / kStages) & 1), abort_flag,
                                      p.status);
                            fence_after();
                        }
                        if (lane == 0) {
                            const uint64_t k_desc =
                                is_page ? desc_sw128(smem_u32(smem + kOffStages + s * kStageBytes)) : bk_desc;
                            const uint32_t idesc = is_page ? kIdescQK : kIdescQKBlock;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ss(tmem + kSCols * b, q_desc + ((kk * 32) >> 4), k_desc + ((kk * 32) >> 4), idesc,
                                       kk > 0 ? 1u : 0u);
                            mma_commit(bar_sfull + 8 * b);
                        }
                        __syncwarp();
                    } else {
                        const bool first = item == i0;
                        mbar_wait(bar_pfull + 8 * b, ph, abort_flag, p.status);
                        fence_after();
                        if (lane == 0) {
                            const uint32_t pcol = tmem + kSCols * b;
                            if (!is_page) {
                                // The block: at most 8 keys, all in the first 16-key step.
                                mma_ts(tmem + kColO, pcol, bv_desc, kIdescPV, first ? 0u : 1u);
                            } else {
                                const uint64_t v_desc =
                                    desc_sw128(smem_u32(smem + kOffStages + s * kStageBytes + kTileBytes));
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_ts(tmem + kColO, pcol + 8u * kk, v_desc + ((kk * 2048) >> 4), kIdescPV,
                                           (kk > 0 || !first) ? 1u : 0u);
                            }
                            mma_commit(bar_odone + 8 * b);  // o_done[it % 3]
                            if (is_page) mma_commit(bar_empty + 8 * s);
                        }
                        __syncwarp();
                    }
                }
            }
        }
        if (lane == 0) mma_commit(bar_done);
        __syncwarp();
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(bar_done, 0) && global_ns() - t0 < kWaitLimitNs) {
        }
    } else if (warp < kRowWarps && nrun > 0) {
        // ------------------------------------------- softmax / row warps --
        const int t = threadIdx.x;
        const int q = warp;
        const int half = lane >> 4;               // key half of this thread
        const int l16 = lane & 15;
        const int rho = l16 < kRowsPerQuarter ? q * kRowsPerQuarter + l16 : 1 << 20;
        const int rows = kG * p.B;
        const bool active = rho < rows;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
        uint8_t *qtile = smem + kOffQ;
        uint8_t *bk = smem + kOffBlkK;
        uint8_t *bv = smem + kOffBlkV;
        float2 *trig = reinterpret_cast<float2 *>(smem + kOffTrig);
        const long long row_w = static_cast<long long>(p.Hq + 2 * p.Hkv) * kD;
        __nv_bfloat16 *normw = reinterpret_cast<__nv_bfloat16 *>(smem + kOffNormW);  // [0..63] q, [64..127] k
        if (QKNORM) {
            normw[t] = w_early;
        }

        // A chunk's partial is written while the next chunk's first item is in
        // flight (its P.V, the last O reader, was confirmed just before), so
        // the wait for the chunk's last P.V hides behind that item's softmax.
        bool epi_pending = false;
        long long epi_slot = 0;
        float epi_m = 0.f, epi_l = 0.f;
        auto write_partial = [&]() {
            // Thread half 0 writes O columns 0-31 of the row's TMEM lane,
            // half 1 columns 32-63.  The row sum adds the two halves' shares.
            const float ltot = epi_l + __shfl_xor_sync(kFull, epi_l, 16);
            uint32_t orr[32];
            tmem_ld_h32(tmem + lane_off + kColO, orr);
            if (active) {
                // The partial's O leaves as bf16: half the bytes for the
                // split pass to write and the combine to read; one rounding
                // (2^-9 relative) of values the combine then averages.  The
                // stores ask L2 to keep the partials (evict_last).
                uint64_t keep;
                asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
                uint4 *dst = reinterpret_cast<uint4 *>(p.ws_o + epi_slot * kPartialElems + rho * kD + 32 * half);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    st_hint_v4(dst + j,
                               make_uint4(pack_bf16(__uint_as_float(orr[8 * j]), __uint_as_float(orr[8 * j + 1])),
                                          pack_bf16(__uint_as_float(orr[8 * j + 2]), __uint_as_float(orr[8 * j + 3])),
                                          pack_bf16(__uint_as_float(orr[8 * j + 4]), __uint_as_float(orr[8 * j + 5])),
                                          pack_bf16(__uint_as_float(orr[8 * j + 6]), __uint_as_float(orr[8 * j + 7]))),
                               keep);
                if (half == 0) st_hint_f2(p.ws_ml + epi_slot * kRows + rho, make_float2(epi_m, ltot), keep);
            }
            epi_pending = false;
        };
        long long it = 0, kr = 0;
        for (int rn = 0; rn < nrun; ++rn) {
            const int u = pl->run_u[rn];
            const int r = u / p.Hkv, h = u - r * p.Hkv;
            const int L = pl->lens[r];
            const int ch = pl->ch[u];
            const int items = static_cast<int>(pl->ustart[u + 1] - pl->ustart[u]);
            const int j0 = pl->run_j0[rn], j1 = pl->run_j1[rn];
            const bool with_block = j0 == 0;

            // ---- stage and build this unit's Q (and block K, V) tiles.
            named_bar_sync(1, kRowThreads);
            const char *qkv_rows = reinterpret_cast<const char *>(p.qkv) + static_cast<long long>(r) * p.B * row_w * 2;
            // Two threads per row: thread t takes row t/2 and the 16 RoPE
            // pairs (j, j+32) with j in [16*(t&1), 16*(t&1)+16).  Rows 0..47
            // are query rows (g*B + i), 48..55 block keys, 56..63 block
            // values.  The row's four 16-byte pieces come straight from qkv
            // into registers, issued now so they land during the angles.
            const int rix = t >> 1, hp = t & 1;
            const char *src = nullptr;
            uint8_t *dst = nullptr;
            int drow = 0, ti = 0;
            bool norm = false;
            const __nv_bfloat16 *w = normw;
            if (rix < kRows) {
                if (rix < rows) {
                    const int g = rix / p.B;
                    ti = rix - g * p.B;
                    src = qkv_rows + ti * row_w * 2 + static_cast<long long>(h * kG + g) * 128;
                    dst = qtile;
                    drow = (rix / kRowsPerQuarter) * 16 + rix % kRowsPerQuarter;
                    norm = QKNORM;
                }
            } else if (rix < kRows + kMaxB) {
                const int j = rix - kRows;
                if (with_block && j < p.B) {
                    ti = j;
                    src = qkv_rows + j * row_w * 2 + static_cast<long long>(p.Hq + h) * 128;
                    dst = bk;
                    drow = j;
                    norm = QKNORM;
                    w = normw + kD;
                }
            } else {
                const int j = rix - kRows - kMaxB;
                if (with_block && j < p.B) {
                    src = qkv_rows + j * row_w * 2 + static_cast<long long>(p.Hq + p.Hkv + h) * 128;
                    dst = bv;
                    drow = j;
                }
            }
            uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0, b0 = a0, b1 = a0;
            if (src != nullptr) {
                const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
                a0 = __ldg(s4 + 2 * hp);
                a1 = __ldg(s4 + 2 * hp + 1);
                b0 = __ldg(s4 + 4 + 2 * hp);
                b1 = __ldg(s4 + 4 + 2 * hp + 1);
            }
            if (QKNORM && warp != 0) {
                // Row warps 1-3 form the B x 32 (token, pair) angles, three
                // each: entry e = (t - 32) + 96 k has pair e % 32 = lane.
#pragma unroll
                for (int k3 = 0; k3 < 3; ++k3) {
                    const int e = (t - 32) + 96 * k3;
                    const int tok = r * p.B + (e >> 5);
                    const long long plo = __shfl_sync(kFull, pos_lo, tok & 31);
                    const long long phi = __shfl_sync(kFull, pos_hi, tok & 31);
                    if (e < p.B * 32) {
                        // The angle's fraction of a turn, exactly (integer
                        // arithmetic wraps whole turns away); its top 32
                        // bits are the signed fraction in [-1/2, 1/2).
                        const unsigned long long turns =
                            static_cast<unsigned long long>(tok < 32 ? plo : phi) * my_rate;
                        const float half_turns = static_cast<float>(static_cast<int>(turns >> 32)) * 0x1p-31f;
                        float sn, cs;
                        sincospif(half_turns, &sn, &cs);
                        trig[(e & 31) * kTrigStride + (e >> 5)] =
                            make_float2(__fmul_rn(cs, p.rope_mscale), __fmul_rn(sn, p.rope_mscale));
                    }
                }
            }
            if (it > 0) {
                // The block tiles are rewritten below: the last P.V (which
                // may have read the previous block's V) must be complete.
                mbar_wait(bar_odone + 8 * (static_cast<uint32_t>(it - 1) % kSBufs),
                          (static_cast<uint32_t>(it - 1) / kSBufs) & 1u, abort_flag, p.status);
                fence_after();
            }
            named_bar_sync(1, kRowThreads);
            {
                float lo[16], hi[16];
                if (src != nullptr) {
                    const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    const uint32_t bv2[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        lo[2 * e] = __uint_as_float(av[e] << 16);
                        lo[2 * e + 1] = __uint_as_float(av[e] & 0xffff0000u);
                        hi[2 * e] = __uint_as_float(bv2[e] << 16);
                        hi[2 * e + 1] = __uint_as_float(bv2[e] & 0xffff0000u);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) lo[e] = hi[e] = 0.f;
                }
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) ss = __fmaf_rn(lo[e], lo[e], __fmaf_rn(hi[e], hi[e], ss));
                ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 1));
                if (norm) {
                    // Rounding pinned operation by operation (the standalone
                    // norm+RoPE call does exactly the same, so it followed by
                    // the plain attention gives this call's bits).
                    const float inv = rsqrtf(__fmaf_rn(ss, 1.0f / kD, p.eps));
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int jp = 16 * hp + e;
                        const float n_lo = __fmul_rn(__fmul_rn(lo[e], inv), __bfloat162float(w[jp]));
                        const float n_hi = __fmul_rn(__fmul_rn(hi[e], inv), __bfloat162float(w[jp + 32]));
                        const float2 cs = trig[jp * kTrigStride + ti];
                        lo[e] = __fmaf_rn(n_lo, cs.x, -__fmul_rn(n_hi, cs.y));
                        hi[e] = __fmaf_rn(n_hi, cs.x, __fmul_rn(n_lo, cs.y));
                    }
                }
                if (dst != nullptr) {
                    uint4 o[4];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        o[c] = make_uint4(pack_bf16(lo[8 * c], lo[8 * c + 1]), pack_bf16(lo[8 * c + 2], lo[8 * c + 3]),
                                          pack_bf16(lo[8 * c + 4], lo[8 * c + 5]), pack_bf16(lo[8 * c + 6], lo[8 * c + 7]));
                        o[2 + c] = make_uint4(pack_bf16(hi[8 * c], hi[8 * c + 1]), pack_bf16(hi[8 * c + 2], hi[8 * c + 3]),
                                              pack_bf16(hi[8 * c + 4], hi[8 * c + 5]), pack_bf16(hi[8 * c + 6], hi[8 * c + 7]));
                    }
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        *reinterpret_cast<uint4 *>(dst + swz(drow, 2 * hp + c)) = o[c];
                        *reinterpret_cast<uint4 *>(dst + swz(drow, 4 + 2 * hp + c)) = o[2 + c];
                    }
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_qready);

            float m_used = 0.f, lsum = 0.f;
            for (int jc = j0; jc < j1; ++jc) {
                const int i0 = jc * ch;
                const int i1 = i0 + ch < items ? i0 + ch : items;
                for (int item = i0; item < i1; ++item) {
                    const int b = static_cast<int>(static_cast<uint32_t>(it) % kSBufs);
                    const bool is_page = item > 0;
                    const int s = static_cast<int>(kr % kStages);
                    int valid = p.B;
                    if (is_page) {
                        const int left = L - (item - 1) * kP;
                        valid = left < kP ? left : kP;
                    }
                    mbar_wait(bar_sfull + 8 * b, (static_cast<uint32_t>(it) / kSBufs) & 1u, abort_flag, p.status);
                    fence_after();
                    // This thread's half of the page's keys.
                    float sv[32];
                    {
                        uint32_t sr[32];
                        tmem_ld_h32(tmem + lane_off + kSCols * b, sr);
#pragma unroll
                        for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(sr[j]);
                    }
                    if (valid < kP) {
                        const int lim = valid - 32 * half;
#pragma unroll
                        for (int j = 0; j < 32; ++j) sv[j] = j < lim ? sv[j] : -INFINITY;
                    }
                    float mx[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) mx[j] = sv[j];
#pragma unroll
                    for (int j = 4; j < 28; j += 8)
#pragma unroll
                        for (int k = 0; k < 4; ++k) mx[k] = fmax3(mx[k], sv[j + k], sv[j + 4 + k]);
                    float rmax = fmax3(fmax3(mx[0], sv[28], sv[29]), fmax3(mx[1], sv[30], sv[31]), fmax3(mx[2], mx[3], mx[3]));
                    rmax = fmaxf(rmax, __shfl_xor_sync(kFull, rmax, 16)) * p.scale_log2;
                    // Exponent base: the row max on a chunk's first item; later,
                    // only when the max passes the base by more than 2^8.
                    const bool first = item == i0;
                    const bool need = !first && rmax > m_used + kRescaleThreshold;
                    const float m_new = (first || need) ? rmax : m_used;
                    const float f = need ? exp2_approx(m_used - m_new) : 1.f;
                    // Keys 2j and 2j + 1 go through the paired fp32 units:
                    // s*scale - m as one f32x2 FMA, the row sum as f32x2 adds.
                    unsigned long long rs2[2] = {0ull, 0ull};
                    {
                        const unsigned long long sl2 = pack_f32x2(p.scale_log2, p.scale_log2);
                        const unsigned long long nm2 = pack_f32x2(-m_new, -m_new);
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float2 x = unpack_f32x2(fma_f32x2(pack_f32x2(sv[2 * j], sv[2 * j + 1]), sl2, nm2));
                            const float p0 = exp2_approx(x.x);
                            const float p1 = exp2_approx(x.y);
                            rs2[j & 1] = add_f32x2(rs2[j & 1], pack_f32x2(p0, p1));
                            pk[j] = pack_bf16(p0, p1);
                        }
                        // The row's P: this thread's half of the keys, 16
                        // columns of bf16 pairs, over the S just read.
                        tmem_st_h16(tmem + lane_off + kSCols * b, pk);
                    }
                    const float2 rsum = unpack_f32x2(add_f32x2(rs2[0], rs2[1]));
                    lsum = (first ? 0.f : lsum * f) + (rsum.x + rsum.y);
                    m_used = m_new;
                    tmem_wait_st();
                    // O is touched (a chunk's partial, a rescale) only once the
                    // previous item's P.V is complete; otherwise P is handed
                    // over at once.  Item i's P.V completes phase i/3 of
                    // o_done[i % 3]; its next phase needs item i+3's P, and
                    // the one before (item i-3's P.V) completed before item
                    // i's QK^T could start, so a wait on it is never a phase
                    // off.
                    const bool touch_o = epi_pending || __any_sync(kFull, need);
                    if (touch_o && it > 0) {
                        mbar_wait(bar_odone + 8 * (static_cast<uint32_t>(it - 1) % kSBufs),
                                  (static_cast<uint32_t>(it - 1) / kSBufs) & 1u, abort_flag, p.status);
                        fence_after();
                    }
                    if (epi_pending) write_partial();  // before this item's P.V overwrites O
                    if (__any_sync(kFull, need)) {
                        // The row's two threads rescale one half of its O each.
                        const uint32_t col = tmem + lane_off + kColO;
                        uint32_t part[32];
                        tmem_ld_h32(col, part);
#pragma unroll
                        for (int j = 0; j < 32; ++j) part[j] = __float_as_uint(__uint_as_float(part[j]) * f);
                        tmem_st_h32(col, part);
                        tmem_wait_st();
                    }
                    if (is_page && valid < kP) {
                        // Stale pool slots past the context may hold
                        // non-finite values: zero them in the page's V tile
                        // before P.V reads them.
                        uint4 *vt = reinterpret_cast<uint4 *>(smem + kOffStages + s * kStageBytes + kTileBytes);
                        for (int e = t; e < (kP - valid) * 8; e += kRowThreads) vt[valid * 8 + e] = make_uint4(0, 0, 0, 0);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_pfull + 8 * b);
                    ++it;
                    if (is_page) ++kr;
                }
                // ---- chunk partial: written during the next item (or below).
                epi_pending = true;
                epi_slot = static_cast<long long>(u) * p.slots_per_unit + jc;
                epi_m = m_used;
                epi_l = lsum;
            }
        }
        if (epi_pending) {
            mbar_wait(bar_odone + 8 * (static_cast<uint32_t>(it - 1) % kSBufs),
                      (static_cast<uint32_t>(it - 1) / kSBufs) & 1u, abort_flag, p.status);
            fence_after();
            write_partial();
        }
        fence_before();
    }

    fence_before();
    __syncthreads();
    fence_after();
    if (warp == kQkWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------------- combine --
//
// One CTA per (unit, 4 query rows), 128 threads: thread = (row, 8 dims,
// chunk lane sg of 4), the 4 chunk lanes of one (row, dims) adjacent in a
// warp.  Lane sg folds the unit's chunk partials sg, sg+4, ... online,
// issuing the loads of kCombineFold of them at once; the lanes then merge by
// a fixed butterfly of shuffles, so the result depends on nothing but the
// unit's own chunks.  (Of 1, 2, 4, 8 and 16 lanes with folds of 1 to 8, 4
// lanes folding 4 at a time measured fastest on every workload.)  Launched
// as a programmatic dependent of the split pass: the unit's chunk count
// comes from its context length (an input, read before griddepcontrol.wait
// while the split pass still runs), its partials sit at fixed slots, and
// griddepcontrol.wait orders every workspace read after the split pass.
constexpr int kCombineRows = 4;
constexpr int kCombineLanes = 4;
constexpr int kCombineThreads = 8 * kCombineLanes * kCombineRows;  // (row, 8 dims, chunk lane) per thread
constexpr int kCombineFold = 4;
static_assert(kRows % kCombineRows == 0 && (kCombineLanes & (kCombineLanes - 1)) == 0 && kCombineLanes <= 32,
              "whole rows per CTA; a row's chunk lanes are adjacent lanes of one warp");

template <bool STAGED>
__global__ void __launch_bounds__(kCombineThreads, 768 / kCombineThreads) k3da_combine_kernel(const __grid_constant__ Params p) {
    const int per_unit = kRows / kCombineRows;
    const int u = blockIdx.x / per_unit;
    const int row = (blockIdx.x - u * per_unit) * kCombineRows + threadIdx.x / (8 * kCombineLanes);
    const int dc = (threadIdx.x / kCombineLanes) & 7, sg = threadIdx.x & (kCombineLanes - 1);
    const int rows = kG * p.B;
    if ((blockIdx.x - u * per_unit) * kCombineRows >= rows) return;  // whole CTA
    const int r = u / p.Hkv, h = u - r * p.Hkv;
    bool bad;
    // The lengths are an input: read before the wait, while the split pass
    // still runs -- unless they were staged (STAGED: the wait then orders the
    // read of the copy after the stage kernel, two grids back).
    int ch = 1, nch = 0;
    if (!STAGED)
        unit_chunking(1 + (clamped_length(p, __ldg(p.ctx_lens + r), &bad) + kP - 1) / kP, p.splits, ch, nch);
    const uint8_t *slots = reinterpret_cast<const uint8_t *>(p.ws_o) +
                           static_cast<long long>(u) * p.slots_per_unit * kPartialElems * 2;
    const float2 *mls = p.ws_ml + static_cast<long long>(u) * p.slots_per_unit * kRows;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (STAGED) {
        // The staged lengths follow the partials, the qkv and the positions.
        const int32_t *lens = reinterpret_cast<const int32_t *>(
            reinterpret_cast<const uint8_t *>(p.ws_o) +
            static_cast<long long>(p.R) * p.Hkv * p.slots_per_unit * kSlotBytes + staging_qkv_bytes(p.Hq, p.Hkv) +
            kStagingPosBytes);
        unit_chunking(1 + (clamped_length(p, lens[r], &bad) + kP - 1) / kP, p.splits, ch, nch);
    }
    float m = -INFINITY, l = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (row < rows) {
        for (int base = 0; base < nch; base += kCombineLanes * kCombineFold) {
            float2 ml[kCombineFold];
            uint4 w[kCombineFold];
#pragma unroll
            for (int f = 0; f < kCombineFold; ++f) {
                const int j = base + sg + f * kCombineLanes;
                if (j < nch) {
                    ml[f] = mls[static_cast<long long>(j) * kRows + row];
                    w[f] = *reinterpret_cast<const uint4 *>(slots + (static_cast<long long>(j) * kPartialElems +
                                                                     row * kD + dc * 8) * 2);
                } else {
                    ml[f] = make_float2(-INFINITY, 0.f);
                    w[f] = make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int f = 0; f < kCombineFold; ++f) {
                const float mm = fmaxf(m, ml[f].x);
                if (mm == -INFINITY) continue;  // nothing folded yet and no chunk here
                const float fo = exp2_approx(m - mm), fn = exp2_approx(ml[f].x - mm);
                m = mm;
                l = l * fo + ml[f].y * fn;
                const uint32_t v[4] = {w[f].x, w[f].y, w[f].z, w[f].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[2 * e] = acc[2 * e] * fo + __uint_as_float(v[e] << 16) * fn;
                    acc[2 * e + 1] = acc[2 * e + 1] * fo + __uint_as_float(v[e] & 0xffff0000u) * fn;
                }
            }
        }
    }
#pragma unroll
    for (int off = kCombineLanes / 2; off >= 1; off >>= 1) {
        const float m2 = __shfl_xor_sync(kFull, m, off);
        const float l2 = __shfl_xor_sync(kFull, l, off);
        const float mm = fmaxf(m, m2);
        const bool none = mm == -INFINITY;  // neither lane holds a chunk
        const float fa = none ? 0.f : exp2_approx(m - mm);
        const float fb = none ? 0.f : exp2_approx(m2 - mm);
        l = l * fa + l2 * fb;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float a2 = __shfl_xor_sync(kFull, acc[j], off);
            acc[j] = acc[j] * fa + a2 * fb;
        }
        m = mm;
    }
    if (sg == 0 && row < rows) {
        const float inv = 1.0f / l;
        const int g = row / p.B, ti = row - g * p.B;
        const long long t = static_cast<long long>(r) * p.B + ti;
        uint4 packed;
        packed.x = pack_bf16(acc[0] * inv, acc[1] * inv);
        packed.y = pack_bf16(acc[2] * inv, acc[3] * inv);
        packed.z = pack_bf16(acc[4] * inv, acc[5] * inv);
        packed.w = pack_bf16(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4 *>(p.out + t * (static_cast<long long>(p.Hq) * kD) +
                                   static_cast<long long>(h * kG + g) * kD + dc * 8) = packed;
    }
}

// ----------------------------------------------------------------- stage --
//
// Host-resident inputs (pinned host memory the GPU addresses directly): the
// split pass reads each unit's q and block rows in every CTA that holds one
// of the unit's chunks, so read across the host link in place they would
// cross it about ten times over.  This kernel copies qkv, the positions and
// the lengths into the workspace once; the split pass is launched as its
// programmatic dependent (its plan and setup overlap the copy, its row warps
// wait for it) and reads the copies.  The page table is read in place: each
// entry is read by one CTA only.
struct StageParams {
    const uint4 *qkv_src;
    uint4 *qkv_dst;
    long long qkv_vecs;  // 16-byte words of qkv
    const int32_t *pos_src;
    int32_t *pos_dst;
    int pos_words;       // 4-byte words of the positions (0 for the plain variant)
    const int32_t *lens_src;
    int32_t *lens_dst;
    int R;
};
constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads) k3da_stage_kernel(const __grid_constant__ StageParams s) {
    // The split pass may start at once: only its row warps wait, in
    // griddepcontrol.wait, for this grid to complete.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long stride = static_cast<long long>(gridDim.x) * kStageThreads;
    const long long t = static_cast<long long>(blockIdx.x) * kStageThreads + threadIdx.x;
    for (long long i = t; i < s.qkv_vecs; i += stride) s.qkv_dst[i] = s.qkv_src[i];
    if (t < s.pos_words) s.pos_dst[t] = s.pos_src[t];
    if (t < s.R) s.lens_dst[t] = s.lens_src[t];
}

// ------------------------------------------------------- wait self-test --
//
// Exercises the bounded wait every kernel of the library uses, on an
// mbarrier that nothing ever completes: warp 0 waits with a short limit and
// must give up, raise the CTA's abort flag and the TIMEOUT status bit; the
// other warps wait on the same barrier with the normal 2 s limit and must
// leave as soon as they see the flag.  A wait that completed would set bit
// 0x100.  No GPU fault is involved: this is how a stuck wait ends.
__global__ void __launch_bounds__(128) k3da_wait_selftest_kernel(int32_t *status, unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    volatile int *flag = &abort_flag;
    if (threadIdx.x == 0) {
        *flag = 0;
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const bool done = threadIdx.x < 32 ? mbar_wait_slow(smem_u32(&bar), 0, flag, status, limit_ns)
                                       : mbar_wait_slow(smem_u32(&bar), 0, flag, status);
    if (done) atomicOr(status, 0x100);
    __syncthreads();
}

constexpr int kSplitThreads = tc::kThreads;
constexpr int kSplitSmem = tc::kSmemBytes;
// Indexed by qknorm + 2 * staged.
const void *const kSplitKernel[4] = {reinterpret_cast<const void *>(&k3da_tc_kernel<false, false>),
                                     reinterpret_cast<const void *>(&k3da_tc_kernel<true, false>),
                                     reinterpret_cast<const void *>(&k3da_tc_kernel<false, true>),
                                     reinterpret_cast<const void *>(&k3da_tc_kernel<true, true>)};

// CTAs of `kernel` that fit on one SM: registers (per-warp allocation in
// units of 256), shared memory (with the per-block reservation), threads,
// and, for the tcgen05 pass, tensor-memory columns (512 per SM).  Computed
// from the kernel's attributes because the runtime's occupancy query counts
// the tcgen05 pass as one CTA per SM.
int occupancy_of(const void *kernel, int threads, int dyn_smem, int dev, int *occ) {
    cudaFuncAttributes fa;
    int smem_sm = 0, smem_rsv = 0, regs_sm = 0, thr_sm = 0, blk_sm = 0;
    if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&blk_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev) != cudaSuccess)
        return K3DA_ECUDA;
    const int warps = (threads + 31) / 32;
    const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
    int n = blk_sm;
    if (regs_warp > 0) n = n < regs_sm / (regs_warp * warps) ? n : regs_sm / (regs_warp * warps);
    const int smem_block = static_cast<int>(fa.sharedSizeBytes) + dyn_smem + smem_rsv;
    n = n < smem_sm / smem_block ? n : smem_sm / smem_block;
    n = n < thr_sm / (warps * 32) ? n : thr_sm / (warps * 32);
    n = n < static_cast<int>(512 / tc::kTmemCols) ? n : static_cast<int>(512 / tc::kTmemCols);
    *occ = n;
    return K3DA_OK;
}

struct DeviceConfig {
    bool ready;
    unsigned long long ctx_id;  // context the kernels were configured in
    int sms;
    int occupancy[2];  // CTAs per SM of the split kernel: [plain, qknorm]
};

std::mutex g_mutex;
thread_local cudaEvent_t g_phase_event = nullptr;
DeviceConfig g_devices[128];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

template <typename Fn>
bool driver_entry(const char *name, int version, Fn *out) {
    if (*out != nullptr) return true;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    *out = reinterpret_cast<Fn>(fn);
    return true;
}

// Process-unique id of the context current on this thread (the device's
// primary context once the runtime has used it).  A device reset makes a new
// context with a new id, so state tied to the old one is set up again.
// Called with g_mutex held.
int current_context_id(int dev, unsigned long long *id) {
    if (!driver_entry("cuCtxGetCurrent", 4000, &g_ctx_current) || !driver_entry("cuCtxGetId", 12000, &g_ctx_id))
        return K3DA_ECUDA;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
        // No context on this thread yet: cudaSetDevice binds the device's
        // primary context.
        if (cudaSetDevice(dev) != cudaSuccess) return K3DA_ECUDA;
        if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return K3DA_ECUDA;
    }
    return g_ctx_id(ctx, id) == CUDA_SUCCESS ? K3DA_OK : K3DA_ECUDA;
}

// Configures the split kernel on `dev` (shared-memory attributes, grid size)
// once per context of that device; later calls return the stored values.
int configure_device(int dev, DeviceConfig *cfg) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (dev < 0 || dev >= 128) return K3DA_EINVAL;
    DeviceConfig &d = g_devices[dev];
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return K3DA_ECUDA;
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return K3DA_ECUDA;
    unsigned long long ctx = 0;
    int rc = current_context_id(dev, &ctx);
    if (rc == K3DA_OK && (!d.ready || d.ctx_id != ctx)) {
        d.ready = false;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) rc = K3DA_ECUDA;
        int occ[4] = {0, 0, 0, 0};
        for (int v = 0; v < 4 && rc == K3DA_OK; ++v) {
            // Ask for the largest shared-memory carveout, then size the grid
            // from the occupancy it allows.
            if (cudaFuncSetAttribute(kSplitKernel[v], cudaFuncAttributeMaxDynamicSharedMemorySize, kSplitSmem) !=
                    cudaSuccess ||
                cudaFuncSetAttribute(kSplitKernel[v], cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared) != cudaSuccess)
                rc = K3DA_ECUDA;
            else
                rc = occupancy_of(kSplitKernel[v], kSplitThreads, kSplitSmem, dev, &occ[v]);
        }
        if (rc == K3DA_OK && !driver_entry("cuTensorMapEncodeTiled", 12000, &g_encode)) rc = K3DA_ECUDA;
        for (int v = 0; v < 4 && rc == K3DA_OK; ++v) {
            if (occ[v] < 1) rc = K3DA_ECUDA;
            if (occ[v] > kMaxCtasPerSm) occ[v] = kMaxCtasPerSm;
        }
        // The staged forms share their plain form's grid.
        if (rc == K3DA_OK && (occ[2] != occ[0] || occ[3] != occ[1])) rc = K3DA_ECUDA;
        if (rc == K3DA_OK) {
            d.sms = sms;
            d.occupancy[0] = occ[0];
            d.occupancy[1] = occ[1];
            d.ctx_id = ctx;
            d.ready = true;
        }
    }
    if (prev != dev) cudaSetDevice(prev);
    if (rc != K3DA_OK) return rc;
    *cfg = d;
    return K3DA_OK;
}

bool supported_heads(int hq, int hkv) { return (hq == 6 && hkv == 1) || (hq == 24 && hkv == 4); }

// Chunks a unit can have: at most chunk_splits(R*Hkv), or ceil(items/ch_max)
// once chunks reach ch_max = kChunkMax items; items <= 1 + page_stride.
constexpr long long slots_per_unit(int R, int Hkv, int page_stride) {
    const long long items = 1 + static_cast<long long>(page_stride);
    const long long by_len = (items + kChunkMax - 1) / kChunkMax;
    const long long splits = chunk_splits(R * Hkv);
    return by_len > splits ? by_len : splits;
}

constexpr size_t workspace_slots(int R, int Hkv, int page_stride) {
    return static_cast<size_t>(R) * Hkv * static_cast<size_t>(slots_per_unit(R, Hkv, page_stride));
}

constexpr size_t workspace_for(int R, int Hkv, int page_stride) {
    return kWsHeaderBytes + workspace_slots(R, Hkv, page_stride) * kSlotBytes;
}

// Pinned host memory (allocated or registered with CUDA) that kernels
// address directly.  Anything else -- device memory, managed memory, a
// pointer CUDA does not know -- is read in place.
bool host_resident(const void *ptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();  // clear the error of an unknown pointer
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Scratch of k3da_attn_qknorm_noalloc: a fixed array in device memory that
// exists on every GPU this library is loaded on, for callers that cannot
// allocate.  8 MiB covers every shape with page_stride <= 1279.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
constexpr int kStaticMaxStride = 1279;
static_assert(workspace_for(kMaxR, 4, kStaticMaxStride) <= kStaticScratchBytes &&
                  workspace_for(kMaxR, 1, kStaticMaxStride) <= kStaticScratchBytes,
              "the no-allocation scratch serves every page_stride up to its stated bound");
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on `dev` (the host-side symbol is only
// a stand-in), looked up with that device current once per context of the
// device: a device reset gives the device a new context, and the address is
// looked up again in it.
int static_scratch_address(int dev, void **out) {
    static void *addr[128] = {nullptr};
    static unsigned long long ctx_of[128] = {0};
    std::lock_guard<std::mutex> lock(g_mutex);
    if (dev < 0 || dev >= 128) return K3DA_EINVAL;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return K3DA_ECUDA;
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return K3DA_ECUDA;
    unsigned long long ctx = 0;
    int rc = current_context_id(dev, &ctx);
    if (rc == K3DA_OK && (addr[dev] == nullptr || ctx_of[dev] != ctx)) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
            rc = K3DA_ECUDA;
        } else {
            addr[dev] = ptr;
            ctx_of[dev] = ctx;
        }
    }
    if (prev != dev) cudaSetDevice(prev);
    if (rc != K3DA_OK) return rc;
    *out = addr[dev];
    return K3DA_OK;
}

int launch(void *out, const void *qkv, const void *kv_pool, int64_t num_pages, const int32_t *page_table,
           int page_stride, const int32_t *ctx_lens, int R, int B, int Hq, int Hkv, int head_dim,
           float softmax_scale, bool qknorm, const void *positions, int pos_dtype, const void *q_norm_w,
           const void *k_norm_w, float eps, float rope_base, const k3da_yarn *yarn, void *workspace,
           size_t workspace_bytes,
           int32_t *status, void *stream, bool staging_optional = false) {
    if (!out || !qkv || !kv_pool || !page_table || !ctx_lens) return K3DA_EINVAL;
    if (!aligned(out, 16) || !aligned(qkv, 16) || !aligned(kv_pool, 16) || !aligned(page_table, 4) ||
        !aligned(ctx_lens, 4) || (status && !aligned(status, 4)))
        return K3DA_EINVAL;
    if (R < 1 || R > kMaxR || B < 1 || B > kMaxB || page_stride < 1 || num_pages < 1) return K3DA_EINVAL;
    if (page_stride > kMaxPageStride) return K3DA_EINVAL;
    if (head_dim != kD || !supported_heads(Hq, Hkv)) return K3DA_EUNSUPPORTED;
    if (num_pages > ((1LL << 31) - 1) / (2LL * Hkv * kP)) return K3DA_EINVAL;
    if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return K3DA_EINVAL;
    if (qknorm) {
        if (!positions || !q_norm_w || !k_norm_w) return K3DA_EINVAL;
        if (pos_dtype != K3DA_POS_I32 && pos_dtype != K3DA_POS_I64) return K3DA_EINVAL;
        if (!aligned(positions, pos_dtype == K3DA_POS_I64 ? 8 : 4) || !aligned(q_norm_w, 2) ||
            !aligned(k_norm_w, 2))
            return K3DA_EINVAL;
        if (!(eps >= 0.f) || !isfinite(eps) || !(rope_base > 1.f) || !isfinite(rope_base)) return K3DA_EINVAL;
        if (yarn != nullptr && !k3da_host::yarn_valid(yarn)) return K3DA_EINVAL;
    }
    if (!workspace || !aligned(workspace, 16)) return K3DA_EWORKSPACE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return K3DA_ECUDA;
    DeviceConfig cfg;
    int rc = configure_device(dev, &cfg);
    if (rc != K3DA_OK) return rc;
    const size_t ws_partials = workspace_for(R, Hkv, page_stride);
    if (workspace_bytes < ws_partials + (staging_optional ? 0 : staging_bytes(Hq, Hkv))) return K3DA_EWORKSPACE;
    // Host-resident qkv, positions or lengths are staged into the workspace
    // by one small kernel first (where it has the room).
    const bool staged = workspace_bytes >= ws_partials + staging_bytes(Hq, Hkv) &&
                        (host_resident(qkv) || host_resident(ctx_lens) || (qknorm && host_resident(positions)));

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
    const size_t slots = workspace_slots(R, Hkv, page_stride);
    prm.slots_per_unit = static_cast<int>(slots_per_unit(R, Hkv, page_stride));
    prm.splits = chunk_splits(R * Hkv);
    prm.ws_o = reinterpret_cast<__nv_bfloat16 *>(static_cast<char *>(workspace) + kWsHeaderBytes);
    prm.ws_ml = reinterpret_cast<float2 *>(prm.ws_o + slots * kPartialElems);
    prm.status = status;
    prm.num_pages = num_pages;
    prm.page_stride = page_stride;
    prm.R = R;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.pos_i64 = pos_dtype == K3DA_POS_I64;
    StageParams sp;
    memset(&sp, 0, sizeof sp);
    if (staged) {
        uint8_t *base = static_cast<uint8_t *>(workspace) + ws_partials;
        const long long qkv_bytes = static_cast<long long>(R) * B * (Hq + 2 * Hkv) * kD * 2;
        sp.qkv_src = static_cast<const uint4 *>(qkv);
        sp.qkv_dst = reinterpret_cast<uint4 *>(base);
        sp.qkv_vecs = qkv_bytes / 16;
        sp.pos_src = static_cast<const int32_t *>(positions);
        sp.pos_dst = reinterpret_cast<int32_t *>(base + staging_qkv_bytes(Hq, Hkv));
        sp.pos_words = qknorm ? R * B * (pos_dtype == K3DA_POS_I64 ? 2 : 1) : 0;
        sp.lens_src = ctx_lens;
        sp.lens_dst = reinterpret_cast<int32_t *>(base + staging_qkv_bytes(Hq, Hkv) + kStagingPosBytes);
        sp.R = R;
        // The split pass reads qkv and the positions from the copies; its
        // plan reads ctx_lens in place (one small read per CTA, before the
        // copy is done) and the combine reads the lengths' copy.
        prm.qkv = reinterpret_cast<const __nv_bfloat16 *>(sp.qkv_dst);
        if (qknorm) prm.positions = sp.pos_dst;
    }
    const int occ = cfg.occupancy[qknorm ? 1 : 0];
    prm.grid = cfg.sms * occ;
    prm.scale_log2 = softmax_scale * 1.4426950408889634f;
    prm.eps = eps;
    {
        double inv_freq[kD / 2];
        k3da_host::rope_frequencies(inv_freq, kD / 2, rope_base, yarn);
        for (int j = 0; j < kD / 2; ++j) prm.turn_rate[j] = k3da_host::turn_rate_fixed64(inv_freq[j]);
    }
    prm.rope_mscale = yarn != nullptr ? k3da_host::yarn_mscale(yarn) : 1.0f;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (staged) {
        // Stage kernel, then the split pass as its programmatic dependent.
        const long long blocks = (sp.qkv_vecs + kStageThreads - 1) / kStageThreads;
        k3da_stage_kernel<<<static_cast<unsigned>(blocks < 1 ? 1 : blocks), kStageThreads, 0, st>>>(sp);
        if (cudaGetLastError() != cudaSuccess) return K3DA_ECUDA;
        cudaLaunchConfig_t sc;
        memset(&sc, 0, sizeof sc);
        sc.gridDim = dim3(static_cast<unsigned>(prm.grid));
        sc.blockDim = dim3(kSplitThreads);
        sc.dynamicSmemBytes = kSplitSmem;
        sc.stream = st;
        cudaLaunchAttribute sa[1];
        sa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        sa[0].val.programmaticStreamSerializationAllowed = 1;
        sc.attrs = sa;
        sc.numAttrs = 1;
        const cudaError_t e = qknorm ? cudaLaunchKernelEx(&sc, k3da_tc_kernel<true, true>, map, prm)
                                     : cudaLaunchKernelEx(&sc, k3da_tc_kernel<false, true>, map, prm);
        if (e != cudaSuccess) return K3DA_ECUDA;
    } else if (qknorm) {
        k3da_tc_kernel<true, false><<<prm.grid, kSplitThreads, kSplitSmem, st>>>(map, prm);
    } else {
        k3da_tc_kernel<false, false><<<prm.grid, kSplitThreads, kSplitSmem, st>>>(map, prm);
    }
    if (cudaGetLastError() != cudaSuccess) return K3DA_ECUDA;
    if (g_phase_event && cudaEventRecord(g_phase_event, st) != cudaSuccess) return K3DA_ECUDA;
    // The combine is a programmatic dependent of the split pass, so its
    // launch and prologue overlap the split pass's tail.
    cudaLaunchConfig_t lc;
    memset(&lc, 0, sizeof lc);
    lc.gridDim = dim3(static_cast<unsigned>(R * Hkv * (kRows / kCombineRows)));
    lc.blockDim = dim3(kCombineThreads);
    lc.dynamicSmemBytes = 0;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (cudaLaunchKernelEx(&lc, staged ? k3da_combine_kernel<true> : k3da_combine_kernel<false>, prm) !=
        cudaSuccess)
        return K3DA_ECUDA;
    if (cudaGetLastError() != cudaSuccess) return K3DA_ECUDA;
    return K3DA_OK;
}

}  // namespace

extern "C" {

size_t k3da_workspace_bytes(int num_requests, int block_len, int num_q_heads, int num_kv_heads,
                            int page_stride) {
    if (num_requests < 1 || num_requests > kMaxR || block_len < 1 || block_len > kMaxB ||
        !supported_heads(num_q_heads, num_kv_heads) || page_stride < 1 || page_stride > kMaxPageStride)
        return 0;
    return workspace_for(num_requests, num_kv_heads, page_stride) + staging_bytes(num_q_heads, num_kv_heads);
}

int k3da_attn(void *out, const void *qkv, const void *kv_pool, int64_t num_pages, const int32_t *page_table,
              int page_stride, const int32_t *ctx_lens, int num_requests, int block_len, int num_q_heads,
              int num_kv_heads, int head_dim, float softmax_scale, void *workspace, size_t workspace_bytes,
              int32_t *status, void *stream) {
    return launch(out, qkv, kv_pool, num_pages, page_table, page_stride, ctx_lens, num_requests, block_len,
                  num_q_heads, num_kv_heads, head_dim, softmax_scale, false, nullptr, 0, nullptr, nullptr, 0.f,
                  0.f, nullptr, workspace, workspace_bytes, status, stream);
}

int k3da_attn_qknorm(void *out, const void *qkv, const void *kv_pool, int64_t num_pages,
                     const int32_t *page_table, int page_stride, const int32_t *ctx_lens, int num_requests,
                     int block_len, int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale,
                     const void *positions, int pos_dtype, const void *q_norm_w, const void *k_norm_w, float eps,
                     float rope_base, void *workspace, size_t workspace_bytes, int32_t *status, void *stream) {
    return launch(out, qkv, kv_pool, num_pages, page_table, page_stride, ctx_lens, num_requests, block_len,
                  num_q_heads, num_kv_heads, head_dim, softmax_scale, true, positions, pos_dtype, q_norm_w,
                  k_norm_w, eps, rope_base, nullptr, workspace, workspace_bytes, status, stream);
}

int k3da_attn_qknorm_yarn(void *out, const void *qkv, const void *kv_pool, int64_t num_pages,
                          const int32_t *page_table, int page_stride, const int32_t *ctx_lens, int num_requests,
                          int block_len, int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale,
                          const void *positions, int pos_dtype, const void *q_norm_w, const void *k_norm_w,
                          float eps, float rope_base, const k3da_yarn *yarn, void *workspace,
                          size_t workspace_bytes, int32_t *status, void *stream) {
    if (!k3da_host::yarn_valid(yarn)) return K3DA_EINVAL;
    return launch(out, qkv, kv_pool, num_pages, page_table, page_stride, ctx_lens, num_requests, block_len,
                  num_q_heads, num_kv_heads, head_dim, softmax_scale, true, positions, pos_dtype, q_norm_w,
                  k_norm_w, eps, rope_base, yarn, workspace, workspace_bytes, status, stream);
}

int k3da_attn_qknorm_noalloc(void *out, const void *qkv, const void *kv_pool, int64_t num_pages,
                             const int32_t *page_table, int page_stride, const int32_t *ctx_lens,
                             int num_requests, int block_len, int num_q_heads, int num_kv_heads, int head_dim,
                             float softmax_scale, const void *positions, int pos_dtype, const void *q_norm_w,
                             const void *k_norm_w, float eps, float rope_base, int32_t *status, void *stream) {
    if (num_requests < 1 || num_requests > kMaxR || num_kv_heads < 1 || page_stride < 1 ||
        page_stride > kMaxPageStride)
        return K3DA_EINVAL;
    if (workspace_for(num_requests, num_kv_heads, page_stride) > kStaticScratchBytes) return K3DA_EWORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return K3DA_ECUDA;
    void *scratch = nullptr;
    const int rc = static_scratch_address(dev, &scratch);
    if (rc != K3DA_OK) return rc;
    return launch(out, qkv, kv_pool, num_pages, page_table, page_stride, ctx_lens, num_requests, block_len,
                  num_q_heads, num_kv_heads, head_dim, softmax_scale, true, positions, pos_dtype, q_norm_w,
                  k_norm_w, eps, rope_base, nullptr, scratch, kStaticScratchBytes, status, stream,
                  /*staging_optional=*/true);
}

size_t k3da_noalloc_scratch_bytes(void) { return kStaticScratchBytes; }

int k3da_split_grid(int device) {
    int dev = device;
    if (dev < 0 && cudaGetDevice(&dev) != cudaSuccess) return 0;
    DeviceConfig cfg;
    if (configure_device(dev, &cfg) != K3DA_OK) return 0;
    return cfg.sms * cfg.occupancy[1];
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

int k3da_selftest_wait_timeout(int32_t *status, unsigned long long limit_ns, void *stream) {
    if (!status || !aligned(status, 4) || limit_ns == 0 || limit_ns > kWaitLimitNs) return K3DA_EINVAL;
    k3da_wait_selftest_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
    return cudaGetLastError() == cudaSuccess ? K3DA_OK : K3DA_ECUDA;
}

}  // extern "C"
