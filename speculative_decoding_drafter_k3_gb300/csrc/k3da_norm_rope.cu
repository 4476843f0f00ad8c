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
// latency-bound.  One warp per (token, q-or-k head) row; lane j holds the
// pair (j, j+32): two coalesced 64-byte loads per row, one shuffle reduction
// for the sum of squares, the angle pos * inv_freq[j] reduced to [-pi, pi]
// in fp64 (positions reach 2^20 and beyond, where an fp32 angle is off by
// radians' worth of ulps), then an accurate fp32 sincos, and two coalesced
// stores.  inv_freq is a host fp64 table passed with the launch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <cstring>

#include "k3da.h"
#include "rope_table.h"

namespace {

constexpr int kD = 64;
constexpr int kRowsPerCta = 8;  // warps per CTA
constexpr unsigned kFull = 0xffffffffu;

struct NormRopeParams {
    __nv_bfloat16 *qkv;
    const void *positions;
    const __nv_bfloat16 *q_w;
    const __nv_bfloat16 *k_w;
    long long rows;  // T * (Hq + Hkv)
    int Hq, Hkv;
    int pos_i64;
    float eps;
    float mscale;  // multiplier of the rotated q and k (YaRN), 1 for plain RoPE
    double inv_freq[kD / 2];
};

__global__ void __launch_bounds__(32 * kRowsPerCta) k3da_norm_rope_kernel(const __grid_constant__ NormRopeParams p) {
    const int lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5);
    if (row >= p.rows) return;  // whole warp
    const int qk_heads = p.Hq + p.Hkv;
    const long long t = row / qk_heads;
    const int h = static_cast<int>(row - t * qk_heads);
    __nv_bfloat16 *x = p.qkv + (t * (qk_heads + p.Hkv) + h) * kD;
    const float lo = __bfloat162float(x[lane]);
    const float hi = __bfloat162float(x[lane + 32]);
    float ss = fmaf(lo, lo, hi * hi);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(kFull, ss, off);
    const float inv = rsqrtf(ss * (1.0f / kD) + p.eps);
    const __nv_bfloat16 *w = h < p.Hq ? p.q_w : p.k_w;
    const float n_lo = lo * inv * __bfloat162float(w[lane]);
    const float n_hi = hi * inv * __bfloat162float(w[lane + 32]);
    const long long pos = p.pos_i64 ? reinterpret_cast<const long long *>(p.positions)[t]
                                    : reinterpret_cast<const int *>(p.positions)[t];
    const double theta = static_cast<double>(pos) * p.inv_freq[lane];
    const double turns = rint(theta * 0.15915494309189535);  // 1 / (2 pi)
    double red = fma(-turns, 6.283185307179586, theta);        // 2 pi, high part
    red = fma(-turns, 2.4492935982947064e-16, red);            // 2 pi, low part
    float sn, cs;
    sincosf(static_cast<float>(red), &sn, &cs);
    cs *= p.mscale;
    sn *= p.mscale;
    x[lane] = __float2bfloat16_rn(n_lo * cs - n_hi * sn);
    x[lane + 32] = __float2bfloat16_rn(n_hi * cs + n_lo * sn);
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
    if (!aligned_to(qkv, 2) || !aligned_to(q_norm_w, 2) || !aligned_to(k_norm_w, 2) ||
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
    prm.rows = static_cast<long long>(num_tokens) * (num_q_heads + num_kv_heads);
    prm.Hq = num_q_heads;
    prm.Hkv = num_kv_heads;
    prm.pos_i64 = pos_dtype == K3DA_POS_I64;
    prm.eps = eps;
    k3da_host::rope_frequencies(prm.inv_freq, kD / 2, rope_base, yarn);
    prm.mscale = yarn != nullptr ? k3da_host::yarn_mscale(yarn) : 1.0f;
    const long long ctas = (prm.rows + kRowsPerCta - 1) / kRowsPerCta;
    if (ctas > 0x7fffffffLL) return K3DA_EINVAL;
    k3da_norm_rope_kernel<<<static_cast<unsigned>(ctas), 32 * kRowsPerCta, 0, static_cast<cudaStream_t>(stream)>>>(
        prm);
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
