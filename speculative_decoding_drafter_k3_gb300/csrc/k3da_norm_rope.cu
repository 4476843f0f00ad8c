// k3da_norm_rope.cu -- the drafter's fused q/k RMSNorm + NeoX RoPE cell as a
// call of its own (sm_103a).
//
// The cell is the fused_qk_norm_rope step of the commit adding the ops'
// contracts on the page "[None][feat] Share Kimi K3 FP4 modeling and add
// NVFP4 support on SM103" (NVIDIA/TensorRT-LLM PR #20532): per token, per
// head, RMSNorm over the 64 dims (eps 1e-5, one weight vector for q and one
// for k) followed by NeoX RoPE (pairs (j, j+32), base 10000), in place on the
// q and k heads of qkv; v heads are left alone.  k3da_qk_norm_rope_yarn
// turns the pairs by the YaRN frequencies of k3da_yarn instead and scales
// the rotated values by its mscale.
//
// Design: the work is a few KB per token, so the call is launch- and
// latency-bound.  A CTA of 64 threads takes one token (24/4 heads) or four
// (6/1), so that a call spreads over many SMs.  First its threads bring the
// norm weights into shared memory and form the tokens' (cos, sin) pairs
// there, one angle at a time: the angle is
// reduced exactly in integer arithmetic (position times a 64-bit fixed-point
// turn rate, wrapping), then turned by an accurate sincospif.  Then two
// threads per (token, q-or-k head) row, as in the fused attention's
// prologue: thread hp of a row holds pairs 16 hp .. 16 hp + 15, loaded with
// 16-byte loads.  The arithmetic is the prologue's, operation for operation
// (a sum of squares chained over the thread's 16 pairs, then one shuffle;
// x * inv * w; the same rotation), so this call followed by k3da_attn gives
// the bits of k3da_attn_qknorm.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <cstring>

#include "k3da.h"
#include "rope_table.h"

namespace {

constexpr int kD = 64;
constexpr int kThreads = 64;
constexpr int kMaxTokensPerCta = kThreads / (2 * 7);  // 7 = the fewest q + k heads a token has
constexpr unsigned kFull = 0xffffffffu;

struct NormRopeParams {
    __nv_bfloat16 *qkv;
    const void *positions;
    const __nv_bfloat16 *q_w;
    const __nv_bfloat16 *k_w;
    int T;
    int Hq, Hkv;
    int tokens_per_cta;  // max(1, floor(kThreads / (2 (Hq + Hkv))))
    int pos_i64;
    float eps;
    float mscale;  // multiplier of the rotated q and k (YaRN), 1 for plain RoPE
    unsigned long long turn_rate[kD / 2];  // RoPE frequency of pair j in turns per position, 2^64 = one turn
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(kThreads) k3da_norm_rope_kernel(const __grid_constant__ NormRopeParams p) {
    __shared__ float2 trig[kMaxTokensPerCta * (kD / 2)];  // [local token][pair]: (cos, sin) * mscale
    __shared__ float wsm[2 * kD];                         // q weights, then k weights
    const int lane = threadIdx.x & 31;
    const int qk_heads = p.Hq + p.Hkv;
    const int t0 = blockIdx.x * p.tokens_per_cta;
    const int ntok = p.T - t0 < p.tokens_per_cta ? p.T - t0 : p.tokens_per_cta;

    // This thread's half row, loaded first.
    const int rl = threadIdx.x >> 1, hp = threadIdx.x & 1;
    const bool valid = rl < ntok * qk_heads;
    const int tl = valid ? rl / qk_heads : 0;
    const int h = valid ? rl - tl * qk_heads : 0;
    __nv_bfloat16 *x = p.qkv + (static_cast<long long>(t0 + tl) * (qk_heads + p.Hkv) + h) * kD;
    uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0, b0 = a0, b1 = a0;
    if (valid) {
        const uint4 *xs = reinterpret_cast<const uint4 *>(x);
        a0 = xs[2 * hp];
        a1 = xs[2 * hp + 1];
        b0 = xs[4 + 2 * hp];
        b1 = xs[4 + 2 * hp + 1];
    }

    // Every global read is issued before any of them is used: the norm
    // weights (two per thread), and the positions of this thread's angles
    // (entry e = local token e / 32, pair e % 32 = lane; at most two per
    // thread).
    static_assert(2 * kD == 2 * kThreads && kMaxTokensPerCta * (kD / 2) <= 2 * kThreads, "two of each per thread");
    const __nv_bfloat16 w_a = p.q_w[threadIdx.x], w_b = p.k_w[threadIdx.x];
    long long pos[2] = {0, 0};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int e = threadIdx.x + k * kThreads;
        if (e < ntok * (kD / 2)) {
            const int t = t0 + (e >> 5);
            pos[k] = p.pos_i64 ? reinterpret_cast<const long long *>(p.positions)[t]
                               : reinterpret_cast<const int *>(p.positions)[t];
        }
    }
    // The rate is read with constant indices (a lane-dependent index into
    // the parameters would serialize the warp).
    unsigned long long rate = 0;
#pragma unroll
    for (int j = 0; j < kD / 2; ++j)
        if (lane == j) rate = p.turn_rate[j];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int e = threadIdx.x + k * kThreads;
        if (e < ntok * (kD / 2)) {
            // The angle's fraction of a turn, exactly (integer arithmetic
            // wraps whole turns away); its top 32 bits are the signed
            // fraction in [-1/2, 1/2).
            const unsigned long long turns = static_cast<unsigned long long>(pos[k]) * rate;
            const float half_turns = static_cast<float>(static_cast<int>(turns >> 32)) * 0x1p-31f;
            float sn, cs;
            sincospif(half_turns, &sn, &cs);
            trig[e] = make_float2(__fmul_rn(cs, p.mscale), __fmul_rn(sn, p.mscale));
        }
    }
    wsm[threadIdx.x] = __bfloat162float(w_a);
    wsm[kD + threadIdx.x] = __bfloat162float(w_b);
    __syncthreads();

    float lo[16], hi[16];
    {
        const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            lo[2 * e] = bf16_lo(av[e]);
            lo[2 * e + 1] = bf16_hi(av[e]);
            hi[2 * e] = bf16_lo(bv[e]);
            hi[2 * e + 1] = bf16_hi(bv[e]);
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) ss = __fmaf_rn(lo[e], lo[e], __fmaf_rn(hi[e], hi[e], ss));
    ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 1));  // every thread takes part, valid or not
    if (!valid) return;
    const float inv = rsqrtf(__fmaf_rn(ss, 1.0f / kD, p.eps));
    const float *w = wsm + (h < p.Hq ? 0 : kD);
    const float2 *tr = trig + tl * (kD / 2);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const int jp = 16 * hp + e;
        const float n_lo = __fmul_rn(__fmul_rn(lo[e], inv), w[jp]);
        const float n_hi = __fmul_rn(__fmul_rn(hi[e], inv), w[jp + 32]);
        const float2 cs = tr[jp];
        lo[e] = __fmaf_rn(n_lo, cs.x, -__fmul_rn(n_hi, cs.y));
        hi[e] = __fmaf_rn(n_hi, cs.x, __fmul_rn(n_lo, cs.y));
    }
    uint4 *xd = reinterpret_cast<uint4 *>(x);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        xd[2 * hp + c] = make_uint4(pack2(lo[8 * c], lo[8 * c + 1]), pack2(lo[8 * c + 2], lo[8 * c + 3]),
                                    pack2(lo[8 * c + 4], lo[8 * c + 5]), pack2(lo[8 * c + 6], lo[8 * c + 7]));
        xd[4 + 2 * hp + c] = make_uint4(pack2(hi[8 * c], hi[8 * c + 1]), pack2(hi[8 * c + 2], hi[8 * c + 3]),
                                        pack2(hi[8 * c + 4], hi[8 * c + 5]), pack2(hi[8 * c + 6], hi[8 * c + 7]));
    }
}

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int launch_norm_rope(void *qkv, int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                     const void *positions, int pos_dtype, const void *q_norm_w, const void *k_norm_w, float eps,
                     float rope_base, const k3da_yarn *yarn, void *stream) {
    if (!qkv || !positions || !q_norm_w || !k_norm_w) return K3DA_EINVAL;
    if (num_tokens < 1) return K3DA_EINVAL;
    if (head_dim != kD) return K3DA_EUNSUPPORTED;
    if (!((num_q_heads == 6 && num_kv_heads == 1) || (num_q_heads == 24 && num_kv_heads == 4)))
        return K3DA_EUNSUPPORTED;
    if (pos_dtype != K3DA_POS_I32 && pos_dtype != K3DA_POS_I64) return K3DA_EINVAL;
    if (!aligned_to(qkv, 16) || !aligned_to(q_norm_w, 2) || !aligned_to(k_norm_w, 2) ||
        !aligned_to(positions, pos_dtype == K3DA_POS_I64 ? 8 : 4))
        return K3DA_EINVAL;
    if (!(eps >= 0.f) || !std::isfinite(eps) || !(rope_base > 1.f) || !std::isfinite(rope_base))
        return K3DA_EINVAL;
    NormRopeParams prm;
    std::memset(&prm, 0, sizeof prm);
    prm.qkv = static_cast<__nv_bfloat16 *>(qkv);
    prm.positions = positions;
    prm.q_w = static_cast<const __nv_bfloat16 *>(q_norm_w);
    prm.k_w = static_cast<const __nv_bfloat16 *>(k_norm_w);
    prm.T = num_tokens;
    prm.tokens_per_cta = kThreads / (2 * (num_q_heads + num_kv_heads));
    if (prm.tokens_per_cta < 1) prm.tokens_per_cta = 1;
    prm.Hq = num_q_heads;
    prm.Hkv = num_kv_heads;
    prm.pos_i64 = pos_dtype == K3DA_POS_I64;
    prm.eps = eps;
    {
        double inv_freq[kD / 2];
        k3da_host::rope_frequencies(inv_freq, kD / 2, rope_base, yarn);
        for (int j = 0; j < kD / 2; ++j) prm.turn_rate[j] = k3da_host::turn_rate_fixed64(inv_freq[j]);
    }
    prm.mscale = yarn != nullptr ? k3da_host::yarn_mscale(yarn) : 1.0f;
    const long long ctas = (static_cast<long long>(num_tokens) + prm.tokens_per_cta - 1) / prm.tokens_per_cta;
    k3da_norm_rope_kernel<<<static_cast<unsigned>(ctas), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(prm);
    return cudaGetLastError() == cudaSuccess ? K3DA_OK : K3DA_ECUDA;
}

}  // namespace

extern "C" int k3da_qk_norm_rope(void *qkv, int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                                 const void *positions, int pos_dtype, const void *q_norm_w,
                                 const void *k_norm_w, float eps, float rope_base, void *stream) {
    return launch_norm_rope(qkv, num_tokens, num_q_heads, num_kv_heads, head_dim, positions, pos_dtype, q_norm_w,
                            k_norm_w, eps, rope_base, nullptr, stream);
}

extern "C" int k3da_qk_norm_rope_yarn(void *qkv, int num_tokens, int num_q_heads, int num_kv_heads,
                                      int head_dim, const void *positions, int pos_dtype, const void *q_norm_w,
                                      const void *k_norm_w, float eps, float rope_base, const k3da_yarn *yarn,
                                      void *stream) {
    if (!k3da_host::yarn_valid(yarn)) return K3DA_EINVAL;
    return launch_norm_rope(qkv, num_tokens, num_q_heads, num_kv_heads, head_dim, positions, pos_dtype, q_norm_w,
                            k_norm_w, eps, rope_base, yarn, stream);
}
