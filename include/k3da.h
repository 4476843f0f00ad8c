/*
 * k3da.h -- C ABI of the K3 DFlash drafter block attention for sm_103a.
 *
 * The operation is the one the page "[None][feat] Share Kimi K3 FP4 modeling
 * and add NVFP4 support on SM103" (NVIDIA/TensorRT-LLM PR #20532) defines in
 * the commit adding the ops k3_drafter_attn and k3_drafter_attn_qknorm, with
 * the parameters fixed by the commit adding their contracts and the
 * drafter's fused_qk_norm_rope cell:
 *
 *   Each of R <= 8 requests brings a draft block of B <= 8 tokens.  Every
 *   block token attends densely (non-causally) to its request's paged
 *   context and to the K/V of its own block.  The block K/V are read from
 *   qkv and never written to the pool.  GQA with 6 query heads per KV head
 *   (head layouts 6/1 and 24/4), head_dim 64, HND pages of 64 tokens.
 *   k3da_attn takes q and k already normalised and roped; k3da_attn_qknorm
 *   applies the per-head q/k RMSNorm and the NeoX RoPE itself.
 *
 * Notation: T = R*B rows, Hq query heads, Hkv KV heads, D = 64, P = 64
 * tokens per page, S = page stride (entries per page-table row), G = Hq/Hkv.
 *
 * Memory.  Every pointer is DEVICE memory owned by the caller, except where
 * a comment says otherwise.  out, qkv, page_table, ctx_lens and positions
 * may instead be pinned HOST memory that the GPU addresses directly (from
 * cudaHostAlloc / cudaMallocHost, or registered with cudaHostRegister, on a
 * system with unified addressing): the kernels then read those inputs and
 * write the output across the host link (NVLink-C2C on a Grace host) with
 * no cudaMemcpy.  When qkv, positions or ctx_lens are host-resident, one
 * small kernel first copies the three into the workspace (qkv is read by
 * every CTA working on a request, so it crosses the link once instead of
 * many times) and the split pass starts as its programmatic dependent; the
 * page table is read in place.  The output is in host memory once the
 * call's work on the stream is complete.  kv_pool, the norm weights,
 * workspace and status are always device memory.  The library allocates nothing, keeps no
 * per-call state, never synchronises and never reads device data on the
 * host: lengths, page table, positions and qkv are read by the kernels, so a
 * call captured in a CUDA graph replays with those buffers rewritten.  The
 * first call on a device (which configures the kernels for it) should come
 * before any stream capture.  The KV pool is only read.
 *
 * Errors.  A host-side check that fails returns a negative k3da_error
 * before anything is launched and nothing is written.  Checks that need
 * device data (lengths, page ids) are made by the kernels: a violation is
 * OR-ed into *status as a K3DA_STATUS_* bit, the offending read is skipped
 * (a clamped length, a page of zeros) and the output stays finite.  The
 * kernels never trap.
 */
#ifndef K3DA_H
#define K3DA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes (host-side). */
typedef enum {
    K3DA_OK = 0,
    K3DA_EINVAL = -1,       /* NULL or misaligned pointer, size out of range */
    K3DA_EUNSUPPORTED = -2, /* head layout, head_dim or page size not served */
    K3DA_ECUDA = -3,        /* a CUDA runtime call failed (launch, attribute) */
    K3DA_EWORKSPACE = -4    /* workspace NULL or smaller than k3da_workspace_bytes */
} k3da_error;

/* Bits OR-ed into the device status word by the kernels. */
enum {
    K3DA_STATUS_BAD_LENGTH = 1, /* ctx_len < 0 or > page_stride*64: clamped */
    K3DA_STATUS_BAD_PAGE = 2,   /* page id outside [0, num_pages): zeros used */
    K3DA_STATUS_TIMEOUT = 4     /* an internal wait ran out: output invalid */
};

/* Integer type of the positions array. */
typedef enum { K3DA_POS_I32 = 0, K3DA_POS_I64 = 1 } k3da_pos_dtype;

/*
 * Bytes of device workspace a call with these sizes needs.  Returns 0 when
 * the sizes are out of contract.  The value does not depend on lengths or on
 * the device, so one buffer serves every call of a captured graph.  It holds
 * the chunk partials and, after them, room to stage host-resident inputs
 * (the qkv of the largest call of this head layout, 64 positions and the
 * lengths).
 */
size_t k3da_workspace_bytes(int num_requests, int block_len, int num_q_heads,
                            int num_kv_heads, int page_stride);

/*
 * k3da_attn -- block attention on already normalised and roped q / k
 * (the op k3_drafter_attn of the commit named above).
 *
 *   out          [T, Hq*64] bf16, written.  16-byte aligned.
 *   qkv          [T, (Hq + 2*Hkv)*64] bf16.  Row r*B + i is token i of
 *                request r: Hq query heads, then Hkv key heads, then Hkv
 *                value heads, 64 dims each.  16-byte aligned.
 *   kv_pool      [num_pages, 2, Hkv, 64, 64] bf16; [page][K=0,V=1][kv head]
 *                [slot][dim].  Read only.  16-byte aligned.
 *   num_pages    pages in the pool, >= 1, num_pages*2*Hkv*64 < 2^31.
 *   page_table   [R, page_stride] int32; context token c of request r is in
 *                page page_table[r*page_stride + c/64], slot c%64.  Entries
 *                past ceil(ctx_len/64) are never read.
 *   page_stride  entries per page-table row, 1 .. 2^25 - 1 (so that
 *                page_stride * 64 fits an int).
 *   ctx_lens     [R] int32 context lengths, 0 <= len <= page_stride*64.
 *   num_requests R in [1, 8];  block_len B in [1, 8].
 *   num_q_heads, num_kv_heads   (6, 1) or (24, 4); query head h reads KV
 *                head h / 6.
 *   head_dim     64.
 *   softmax_scale  multiplier of q.k (1/sqrt(64) for the drafter); finite, > 0.
 *   workspace, workspace_bytes  scratch of at least k3da_workspace_bytes();
 *                contents on entry are irrelevant; 16-byte aligned.
 *   status       int32 device word the kernels OR K3DA_STATUS_* bits into;
 *                may be NULL.  The caller clears it.
 *   stream       cudaStream_t to launch on (NULL = legacy default stream).
 *
 * Returns K3DA_OK once both kernels are enqueued, else a k3da_error.
 * Calls on the same stream are ordered; calls that share a workspace must
 * not overlap on the GPU.
 *
 * Work split and reproducibility.  Each (request, kv head) unit's keys are
 * cut into chunks whose boundaries depend only on that unit's context length
 * and on the call's shape (R, Hkv): at most 32 pages per chunk, and with few
 * units about 304 chunks in all (two per SM of a 152-SM GB300) so that even
 * one request spreads over the GPU.  That count is a constant, not the
 * device's SM count, and the chunk partials are folded in a fixed order: the
 * output is bitwise the same on every run, whatever the other requests hold
 * (requests are isolated bit for bit), and on any device this library runs
 * on, whatever its SM count (which only decides which CTA computes which
 * chunk).
 */
int k3da_attn(void *out, const void *qkv, const void *kv_pool, int64_t num_pages,
              const int32_t *page_table, int page_stride, const int32_t *ctx_lens,
              int num_requests, int block_len, int num_q_heads, int num_kv_heads,
              int head_dim, float softmax_scale, void *workspace, size_t workspace_bytes,
              int32_t *status, void *stream);

/*
 * k3da_attn_qknorm -- as k3da_attn, but q and the block's k are raw: each
 * 64-wide head row x of q (resp. k) becomes
 *     y = x * (mean_j x_j^2 + eps)^(-1/2) * w      (w = q_norm_w, resp. k_norm_w)
 * and then NeoX RoPE at the token's position p: for j < 32,
 *     theta = p * rope_base^(-2j/64),
 *     y'_j = y_j cos(theta) - y_{j+32} sin(theta),
 *     y'_{j+32} = y_{j+32} cos(theta) + y_j sin(theta).
 * Context keys in the pool are used as stored; values are never normalised
 * (the op k3_drafter_attn_qknorm of the commit named above; eps 1e-5 and
 * base 10000 in its fused_qk_norm_rope cell).
 *
 *   positions    [T] int32 or int64 (pos_dtype), 0 <= p < 2^24 for exact
 *                angles; 4- or 8-byte aligned.
 *   q_norm_w, k_norm_w   [64] bf16 RMSNorm weights shared by all heads.
 *   eps          >= 0, finite;  rope_base > 1, finite.
 */
int k3da_attn_qknorm(void *out, const void *qkv, const void *kv_pool, int64_t num_pages,
                     const int32_t *page_table, int page_stride, const int32_t *ctx_lens,
                     int num_requests, int block_len, int num_q_heads, int num_kv_heads,
                     int head_dim, float softmax_scale, const void *positions,
                     int pos_dtype, const void *q_norm_w, const void *k_norm_w, float eps,
                     float rope_base, void *workspace, size_t workspace_bytes,
                     int32_t *status, void *stream);

/*
 * Profiling aid.  When `event` (a cudaEvent_t created by the caller) is not
 * NULL, every later k3da_attn / k3da_attn_qknorm call made from this host
 * thread records it on the call's stream between the split pass and the
 * combine kernel, so the split pass can be timed alone; NULL turns this off.
 * The setting is per host thread.  Returns K3DA_OK.
 */
int k3da_set_phase_event(void *event);

/*
 * k3da_attn_qknorm_noalloc -- k3da_attn_qknorm for callers that cannot
 * allocate device memory: code that runs where cudaMalloc is unavailable or
 * forbidden (a host callback, a real-time path that must not allocate, a
 * plugin whose host framework owns every device allocation) or that has no
 * way to keep a workspace buffer between calls.  An addition of this
 * library with no counterpart in the drafter's own operations: the same
 * computation as k3da_attn_qknorm,
 * with the scratch taken from a fixed array of k3da_noalloc_scratch_bytes()
 * (8 MiB) that the library keeps in the memory of every GPU it is loaded on,
 * for the life of the process.  Arguments are those of k3da_attn_qknorm
 * without workspace / workspace_bytes; the caller still passes every input
 * and output.
 *
 * - Sizes whose chunk partials exceed the array are refused with
 *   K3DA_EWORKSPACE: page_stride <= 1279 always fits.  Host-resident
 *   inputs are staged only where the array also has room for the staging
 *   area of k3da_workspace_bytes; otherwise the kernels read them in place.
 * - Nothing is allocated or freed, by the library or by any routine it
 *   calls.
 * - The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 * - All calls on a device share the one array.  Its contents on entry do not
 *   matter (every value read is first written by the same call), but two
 *   calls that overlap on the GPU (different streams, no ordering) race on
 *   it: order them, or use k3da_attn_qknorm with separate workspaces.
 */
int k3da_attn_qknorm_noalloc(void *out, const void *qkv, const void *kv_pool, int64_t num_pages,
                             const int32_t *page_table, int page_stride, const int32_t *ctx_lens,
                             int num_requests, int block_len, int num_q_heads,
                             int num_kv_heads, int head_dim, float softmax_scale,
                             const void *positions, int pos_dtype, const void *q_norm_w,
                             const void *k_norm_w, float eps, float rope_base, int32_t *status,
                             void *stream);

/* Bytes of the fixed scratch array k3da_attn_qknorm_noalloc uses. */
size_t k3da_noalloc_scratch_bytes(void);

/*
 * CTAs the split pass launches on `device` (-1 = current): SM count times
 * the CTAs per SM its resources allow.  Configures the device like a first
 * call does.  Returns 0 when the device cannot be configured.
 */
int k3da_split_grid(int device);

/*
 * YaRN RoPE scaling (next to "YaRN 4.0", the drafter's setting on the page
 * cited above; the method is the "NTK-by-parts" interpolation of "YaRN:
 * Efficient Context Window Extension of Large Language Models", Peng et al.
 * 2023).  Pair j of the plain table turns at theta_j = rope_base^(-2j/64);
 * with r_j = original_max_position * theta_j / (2 pi) (its wavelengths in the
 * original context) and the ramp g = clamp((r_j - beta_slow) / (beta_fast -
 * beta_slow), 0, 1), it turns at g * theta_j + (1 - g) * theta_j / factor.
 * Both rotated outputs are multiplied by mscale (the YaRN paper's sqrt(1/t),
 * applied to q and k; pass 1 when the model folds it elsewhere, or 0 to have
 * the library use the paper's 0.1 * ln(factor) + 1, formed in fp64 and
 * rounded once to fp32).  factor 1 with mscale 1 is plain NeoX RoPE.  Host
 * memory; read during the call only.
 */
typedef struct {
    float factor;                /* >= 1 */
    float original_max_position; /* > 0 */
    float beta_fast;             /* > beta_slow (32 in the YaRN paper) */
    float beta_slow;             /* > 0 (1 in the YaRN paper) */
    float mscale;                /* > 0, or 0 for 0.1 * ln(factor) + 1 */
} k3da_yarn;

/*
 * k3da_attn_qknorm_yarn -- k3da_attn_qknorm with the block's q and k rotated
 * by YaRN RoPE (`yarn`, see k3da_yarn) instead of plain NeoX RoPE; every
 * other argument, the workspace contract and the errors are those of
 * k3da_attn_qknorm.  K3DA_EINVAL when `yarn` is NULL or out of range.
 */
int k3da_attn_qknorm_yarn(void *out, const void *qkv, const void *kv_pool, int64_t num_pages,
                          const int32_t *page_table, int page_stride, const int32_t *ctx_lens,
                          int num_requests, int block_len, int num_q_heads, int num_kv_heads,
                          int head_dim, float softmax_scale, const void *positions, int pos_dtype,
                          const void *q_norm_w, const void *k_norm_w, float eps, float rope_base,
                          const k3da_yarn *yarn, void *workspace, size_t workspace_bytes,
                          int32_t *status, void *stream);

/*
 * k3da_qk_norm_rope -- the drafter's fused q/k RMSNorm + NeoX RoPE cell on
 * its own (fused_qk_norm_rope in the commit adding the ops' contracts on the
 * page "[None][feat] Share Kimi K3 FP4 modeling and add NVFP4 support on
 * SM103"), in place: for every token t, each query head row of qkv becomes
 * rope(rmsnorm(q, q_norm_w), positions[t]) and each key head row
 * rope(rmsnorm(k, k_norm_w), positions[t]), rounded to bf16; value head rows
 * are not touched.  RMSNorm is x * (mean(x^2) + eps)^(-1/2) * w over the 64
 * dims of a head; RoPE turns the pairs (j, j+32) by positions[t] *
 * rope_base^(-2j/64).  It is the transform k3da_attn_qknorm applies to the
 * block's q and k before attending, exported for the step that writes new
 * K into the pool.  It rounds exactly as k3da_attn_qknorm does, so this call
 * followed by k3da_attn gives k3da_attn_qknorm's output bit for bit.
 *
 *   qkv          [T, (Hq + 2*Hkv)*64] bf16, read and written.  16-byte aligned.
 *   num_tokens   T >= 1 (the drafter runs 1..64).
 *   num_q_heads, num_kv_heads   (6, 1) or (24, 4);  head_dim 64.
 *   positions    [T] int32 or int64 (pos_dtype), aligned to its type.
 *   q_norm_w, k_norm_w  [64] bf16, 2-byte aligned.
 *   eps          finite, >= 0;  rope_base finite, > 1.
 *   stream       cudaStream_t (NULL = legacy default stream).
 *
 * Returns K3DA_OK once the kernel is enqueued, else a k3da_error; nothing
 * is written on a refusal.  Allocates nothing; graph-capturable.
 */
int k3da_qk_norm_rope(void *qkv, int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                      const void *positions, int pos_dtype, const void *q_norm_w,
                      const void *k_norm_w, float eps, float rope_base, void *stream);

/* k3da_qk_norm_rope with YaRN RoPE (`yarn`, see k3da_yarn). */
int k3da_qk_norm_rope_yarn(void *qkv, int num_tokens, int num_q_heads, int num_kv_heads,
                           int head_dim, const void *positions, int pos_dtype,
                           const void *q_norm_w, const void *k_norm_w, float eps, float rope_base,
                           const k3da_yarn *yarn, void *stream);

/* Static description of a k3da_error or K3DA_STATUS_* bit set. */
const char *k3da_error_string(int code);

/*
 * k3da_selftest_wait_timeout -- diagnostic of the failure path: launches one
 * CTA that waits, through the same bounded wait every kernel here uses, on a
 * barrier nothing completes.  Warp 0 gives up after limit_ns (1 ns .. 2 s)
 * and raises the abort flag; the other warps must leave on the flag.  The
 * kernel ORs K3DA_STATUS_TIMEOUT into *status (a device int32 the caller
 * clears), and 0x100 if a wait that can never complete did.  The context
 * stays usable.  K3DA_EINVAL on a NULL/misaligned status or a limit out of
 * range.
 */
int k3da_selftest_wait_timeout(int32_t *status, unsigned long long limit_ns, void *stream);

/* Library version, major*10000 + minor*100 + patch. */
int k3da_version(void);

#ifdef __cplusplus
}
#endif
#endif /* K3DA_H */
