"""Pins of the fp64 oracle against what the mathematics fixes (CPU only).

Each test ties the oracle to something other than itself: textbook values,
closed forms, invariants, a library routine on a special case, or an
independently written brute force.  The op is defined on the page "[None]
[feat] Share Kimi K3 FP4 modeling and add NVFP4 support on SM103"
(NVIDIA/TensorRT-LLM PR #20532): the commit adding k3_drafter_attn /
k3_drafter_attn_qknorm (dense non-causal attention of each draft token to its
request's paged context plus its own block, block K/V from qkv, GQA 6:1,
head_dim 64, HND pages of 64, per-head q/k RMSNorm and NeoX RoPE in the fused
variant) and the commit adding the contracts and the fused_qk_norm_rope cell
(eps 1e-5, base 10000, NeoX; head layouts 6/1 and 24/4).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")
D = 64
P = 64


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def bf16(a):
    """Round to bf16 and return the uint16 bit pattern plus the exact value."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return oracle.bf16_bits(t), t.to(torch.float64).numpy()


# ----------------------------------------------------------------- RoPE ----

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(0).standard_normal(D)
    np.testing.assert_array_equal(oracle.rope_neox(x, 0.0), x)


def test_rope_unit_vectors_match_textbook_angles():
    g = golden()
    trig = {1: (g["cos_1"], g["sin_1"]), 2: (g["cos_2"], g["sin_2"])}
    for case in g["rope_cases"]["cases"]:
        j, pos = case["j"], case["pos"]
        c, s = trig[case["theta"]]
        e = np.zeros(D)
        e[j] = 1.0
        y = oracle.rope_neox(e, pos)
        expect = np.zeros(D)
        expect[j], expect[j + 32] = c, s
        np.testing.assert_allclose(y, expect, atol=1e-13, rtol=0)
        e = np.zeros(D)
        e[j + 32] = 1.0
        y = oracle.rope_neox(e, pos)
        expect = np.zeros(D)
        expect[j], expect[j + 32] = -s, c
        np.testing.assert_allclose(y, expect, atol=1e-13, rtol=0)


def test_rope_matches_complex_rotation():
    # Independent formulation: (x_j + i x_{j+32}) * exp(i pos f_j), f_j = 1e4^(-j/32).
    rng = np.random.default_rng(1)
    for pos in [0, 1, 7, 2041, 131079]:
        x = rng.standard_normal(D)
        z = (x[:32] + 1j * x[32:]) * np.exp(1j * pos * np.power(1e4, -np.arange(32) / 32.0))
        y = oracle.rope_neox(x, pos)
        np.testing.assert_allclose(y[:32], z.real, atol=1e-9, rtol=0)
        np.testing.assert_allclose(y[32:], z.imag, atol=1e-9, rtol=0)


def test_rope_preserves_pair_norms_and_depends_on_relative_position():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    for p in [3, 100, 5000]:
        y = oracle.rope_neox(q, p)
        np.testing.assert_allclose(y[:32] ** 2 + y[32:] ** 2, q[:32] ** 2 + q[32:] ** 2, rtol=1e-12)
    d0 = oracle.rope_neox(q, 17) @ oracle.rope_neox(k, 5)
    for shift in [1, 40, 1000]:
        d1 = oracle.rope_neox(q, 17 + shift) @ oracle.rope_neox(k, 5 + shift)
        assert abs(d1 - d0) < 1e-9 * max(1.0, abs(d0))


# -------------------------------------------------------------- RMSNorm ----

def test_rmsnorm_unit_weight_gives_unit_rms_up_to_eps():
    rng = np.random.default_rng(3)
    for scale in [1e-2, 1.0, 30.0]:
        x = scale * rng.standard_normal(D)
        y = oracle.rmsnorm(x, np.ones(D), eps=1e-5)
        ms = np.mean(x * x)
        assert abs(np.mean(y * y) - ms / (ms + 1e-5)) < 1e-12


def test_rmsnorm_constant_row_closed_form():
    w = np.linspace(0.5, 1.5, D)
    for c in [2.0, -0.25]:
        y = oracle.rmsnorm(np.full(D, c), w, eps=1e-5)
        np.testing.assert_allclose(y, c / math.sqrt(c * c + 1e-5) * w, rtol=1e-14)


def test_rmsnorm_matches_torch_rms_norm_fp64():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, D))
    w = 1 + 0.1 * rng.standard_normal(D)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (D,), torch.tensor(w), eps=1e-5).numpy()
    for i in range(5):
        np.testing.assert_allclose(oracle.rmsnorm(x[i], w, 1e-5), ref[i], rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------ attention ----

def make_problem(R, B, Hq, Hkv, lens, page_stride, num_pages, seed, qknorm=False):
    rng = np.random.default_rng(seed)
    T = R * B
    qkv_bits, qkv = bf16(rng.standard_normal((T, (Hq + 2 * Hkv) * D)))
    pool_bits, pool = bf16(rng.standard_normal((num_pages, 2, Hkv, P, D)))
    perm = rng.permutation(num_pages).astype(np.int32)
    pt = np.full((R, page_stride), -1, np.int32)
    used = num_pages // R
    for r in range(R):
        n = min(page_stride, used)
        pt[r, :n] = perm[r * used:r * used + n]
    prob = dict(qkv_bits=qkv_bits, qkv=qkv, pool_bits=pool_bits, pool=pool, pt=pt,
                lens=np.array(lens, np.int32), R=R, B=B, Hq=Hq, Hkv=Hkv, qknorm=qknorm)
    if qknorm:
        prob["pos"] = np.array([lens[r] + i for r in range(R) for i in range(B)], np.int64)
        prob["qw_bits"], prob["qw"] = bf16(1 + 0.1 * rng.standard_normal(D))
        prob["kw_bits"], prob["kw"] = bf16(1 + 0.1 * rng.standard_normal(D))
    return prob


def run_oracle(p, **over):
    kw = dict(num_requests=p["R"], block_len=p["B"], num_q_heads=p["Hq"], num_kv_heads=p["Hkv"],
              qknorm=p["qknorm"])
    if p["qknorm"]:
        kw.update(positions=p["pos"], q_norm_w=p["qw_bits"], k_norm_w=p["kw_bits"])
    kw.update(over)
    return oracle.attn(p["qkv_bits"], p["pool_bits"], p["pt"], p["lens"], **kw)


def rope_complex(x, pos):
    z = (x[:32] + 1j * x[32:]) * np.exp(1j * pos * np.power(1e4, -np.arange(32) / 32.0))
    return np.concatenate([z.real, z.imag])


def reference_by_sdpa(p):
    """Independent route: numpy fancy-index gather, torch rms_norm, complex
    RoPE and torch scaled_dot_product_attention in fp64 (no mask, GQA by
    repeating KV heads)."""
    R, B, Hq, Hkv = p["R"], p["B"], p["Hq"], p["Hkv"]
    G = Hq // Hkv
    out = np.zeros((R * B, Hq * D))
    for r in range(R):
        L = int(p["lens"][r])
        rows = p["qkv"][r * B:(r + 1) * B]
        q = rows[:, :Hq * D].reshape(B, Hq, D)
        kb = rows[:, Hq * D:(Hq + Hkv) * D].reshape(B, Hkv, D)
        vb = rows[:, (Hq + Hkv) * D:].reshape(B, Hkv, D)
        if p["qknorm"]:
            qn = torch.nn.functional.rms_norm(torch.tensor(q), (D,), torch.tensor(p["qw"]), eps=1e-5).numpy()
            kn = torch.nn.functional.rms_norm(torch.tensor(kb), (D,), torch.tensor(p["kw"]), eps=1e-5).numpy()
            pos = p["pos"][r * B:(r + 1) * B]
            q = np.stack([[rope_complex(qn[i, h], pos[i]) for h in range(Hq)] for i in range(B)])
            kb = np.stack([[rope_complex(kn[i, h], pos[i]) for h in range(Hkv)] for i in range(B)])
        tok = np.arange(L)
        pages = p["pt"][r, tok // P]
        kc = p["pool"][pages, 0, :, tok % P, :]  # [L, Hkv, D]
        vc = p["pool"][pages, 1, :, tok % P, :]
        K = np.concatenate([kc, kb], 0).transpose(1, 0, 2)  # [Hkv, L+B, D]
        V = np.concatenate([vc, vb], 0).transpose(1, 0, 2)
        Q = torch.tensor(q.transpose(1, 0, 2))  # [Hq, B, D]
        Kt = torch.tensor(K).repeat_interleave(G, 0)
        Vt = torch.tensor(V).repeat_interleave(G, 0)
        o = torch.nn.functional.scaled_dot_product_attention(Q, Kt, Vt, scale=0.125).numpy()
        out[r * B:(r + 1) * B] = o.transpose(1, 0, 2).reshape(B, Hq * D)
    return out


def brute_force(p):
    """Pure-Python loops: walk the page table token by token, explicit exp
    and sums; no vectorised library call."""
    R, B, Hq, Hkv = p["R"], p["B"], p["Hq"], p["Hkv"]
    G = Hq // Hkv
    W = (Hq + 2 * Hkv) * D
    qkv = p["qkv"].reshape(-1).tolist()
    pool = p["pool"]
    out = np.zeros((R * B, Hq * D))
    for r in range(R):
        L = int(p["lens"][r])
        for g in range(Hkv):
            keys, vals = [], []
            for c in range(L):
                page = int(p["pt"][r][c // P])
                keys.append([float(pool[page, 0, g, c % P, j]) for j in range(D)])
                vals.append([float(pool[page, 1, g, c % P, j]) for j in range(D)])
            for jb in range(B):
                t = r * B + jb
                keys.append([qkv[t * W + (Hq + g) * D + j] for j in range(D)])
                vals.append([qkv[t * W + (Hq + Hkv + g) * D + j] for j in range(D)])
            for hl in range(G):
                h = g * G + hl
                for i in range(B):
                    t = r * B + i
                    q = [qkv[t * W + h * D + j] for j in range(D)]
                    scores = [0.125 * sum(q[j] * k[j] for j in range(D)) for k in keys]
                    mx = max(scores)
                    wts = [math.exp(s - mx) for s in scores]
                    tot = sum(wts)
                    for j in range(D):
                        out[t, h * D + j] = sum(wts[k] * vals[k][j] for k in range(len(keys))) / tot
    return out


@pytest.mark.parametrize("R,B,lens", [(1, 1, [0]), (1, 2, [65]), (2, 2, [130, 1]), (2, 1, [64, 0])])
def test_attention_matches_python_brute_force(R, B, lens):
    p = make_problem(R, B, 6, 1, lens, page_stride=3, num_pages=6, seed=10 + R * 3 + B)
    np.testing.assert_allclose(run_oracle(p), brute_force(p), atol=1e-12, rtol=0)


@pytest.mark.parametrize("Hq,Hkv,qknorm", [(6, 1, False), (6, 1, True), (24, 4, True), (24, 4, False)])
def test_attention_matches_torch_sdpa_fp64(Hq, Hkv, qknorm):
    p = make_problem(3, 5, Hq, Hkv, [0, 70, 191], page_stride=4, num_pages=12, seed=20 + Hq,
                     qknorm=qknorm)
    np.testing.assert_allclose(run_oracle(p), reference_by_sdpa(p), atol=1e-10, rtol=1e-10)


def test_single_key_returns_its_value():
    p = make_problem(1, 1, 6, 1, [0], page_stride=1, num_pages=1, seed=30)
    p["pt"][:] = -1  # context is empty: no page id may be read
    out = run_oracle(p)
    v = p["qkv"][0, 7 * D:8 * D]
    for h in range(6):
        np.testing.assert_array_equal(out[0, h * D:(h + 1) * D], v)


def test_identical_keys_return_mean_of_values():
    p = make_problem(1, 3, 6, 1, [100], page_stride=2, num_pages=2, seed=31)
    key = p["pool_bits"][0, 0, 0, 5].copy()
    p["pool_bits"][:, 0] = key
    p["qkv_bits"][:, 6 * D:7 * D] = key
    vals = [p["pool"][p["pt"][0, c // P], 1, 0, c % P] for c in range(100)]
    vals += [p["qkv"][i, 7 * D:8 * D] for i in range(3)]
    np.testing.assert_allclose(run_oracle(p), np.tile(np.mean(vals, 0), (3, 6)), atol=1e-12)


def test_zero_query_returns_mean_of_values():
    p = make_problem(1, 2, 6, 1, [77], page_stride=2, num_pages=2, seed=32)
    p["qkv_bits"][:, :6 * D] = 0
    vals = [p["pool"][p["pt"][0, c // P], 1, 0, c % P] for c in range(77)]
    vals += [p["qkv"][i, 7 * D:8 * D] for i in range(2)]
    np.testing.assert_allclose(run_oracle(p), np.tile(np.mean(vals, 0), (2, 6)), atol=1e-12)


def test_two_keys_give_the_logistic_weight():
    # q = 8 e_0, context key e_0, block key 0: scores 0.125*8 = 1 and 0.
    p = make_problem(1, 1, 6, 1, [1], page_stride=1, num_pages=1, seed=33)
    one = oracle.bf16_bits(torch.tensor([1.0], dtype=torch.bfloat16))[0]
    eight = oracle.bf16_bits(torch.tensor([8.0], dtype=torch.bfloat16))[0]
    p["qkv_bits"][:] = 0
    p["qkv_bits"][0, 0:6 * D:D] = eight
    p["pool_bits"][:] = 0
    p["pool_bits"][0, 0, 0, 0, 0] = one
    p["pool_bits"][0, 1, 0, 0, 3] = one      # context value e_3
    p["qkv_bits"][0, 7 * D + 5] = one         # block value e_5
    out = run_oracle(p)
    s1 = golden()["sigmoid_1"]
    for h in range(6):
        np.testing.assert_allclose(out[0, h * D + 3], s1, atol=1e-15)
        np.testing.assert_allclose(out[0, h * D + 5], 1 - s1, atol=1e-15)


def test_context_slot_mapping_through_page_table():
    # Token 70 of a 100-token context lives in page pt[1], slot 6.  Give it a
    # dominant key and read its value back.
    p = make_problem(1, 1, 6, 1, [100], page_stride=2, num_pages=2, seed=34)
    p["pt"][0] = [1, 0]
    p["qkv_bits"][:, :6 * D] = 0
    p["qkv_bits"][0, 0:6 * D:D] = oracle.bf16_bits(torch.tensor([8.0], dtype=torch.bfloat16))[0]
    p["pool_bits"][:, 0] = 0
    p["qkv_bits"][0, 6 * D:7 * D] = 0
    p["pool_bits"][0, 0, 0, 6, 0] = oracle.bf16_bits(torch.tensor([100.0], dtype=torch.bfloat16))[0]
    out = run_oracle(p)
    v = p["pool"][0, 1, 0, 6]
    for h in range(6):
        np.testing.assert_allclose(out[0, h * D:(h + 1) * D], v, atol=1e-12)


def test_gqa_maps_query_head_to_kv_head_by_division():
    p = make_problem(2, 2, 24, 4, [90, 3], page_stride=2, num_pages=4, seed=35)
    for g in range(4):
        c = oracle.bf16_bits(torch.tensor([float(g + 1)], dtype=torch.bfloat16))[0]
        p["pool_bits"][:, 1, g] = c
        p["qkv_bits"][:, (24 + 4 + g) * D:(24 + 4 + g + 1) * D] = c
    out = run_oracle(p)
    for h in range(24):
        np.testing.assert_allclose(out[:, h * D:(h + 1) * D], h // 6 + 1, atol=1e-12)


def test_block_is_non_causal():
    # Token 0 must see the block key of the last token.
    p = make_problem(1, 4, 6, 1, [0], page_stride=1, num_pages=1, seed=36)
    p["qkv_bits"][:, :7 * D] = 0
    p["qkv_bits"][0, 0:6 * D:D] = oracle.bf16_bits(torch.tensor([8.0], dtype=torch.bfloat16))[0]
    p["qkv_bits"][3, 6 * D] = oracle.bf16_bits(torch.tensor([100.0], dtype=torch.bfloat16))[0]
    out = run_oracle(p)
    v_last = p["qkv"][3, 7 * D:8 * D]
    np.testing.assert_allclose(out[0, :D], v_last, atol=1e-12)


def test_empty_context_is_block_only_attention():
    p = make_problem(2, 3, 6, 1, [0, 0], page_stride=2, num_pages=4, seed=37, qknorm=True)
    p["pt"][:] = -1  # never read
    out = run_oracle(p)
    np.testing.assert_allclose(out, reference_by_sdpa(p), atol=1e-10)


def test_block_only_attention_depends_on_relative_positions():
    p = make_problem(1, 5, 6, 1, [0], page_stride=1, num_pages=1, seed=38, qknorm=True)
    a = run_oracle(p)
    p["pos"] = p["pos"] + 12345
    b = run_oracle(p)
    np.testing.assert_allclose(a, b, atol=1e-9)


def test_page_permutation_invariance():
    p = make_problem(2, 4, 24, 4, [200, 129], page_stride=4, num_pages=8, seed=39, qknorm=True)
    a = run_oracle(p)
    perm = np.random.default_rng(0).permutation(8)
    moved = np.empty_like(p["pool_bits"])
    moved[perm] = p["pool_bits"]        # page k moves to slot perm[k]
    pt = np.where(p["pt"] >= 0, perm[np.maximum(p["pt"], 0)], -1).astype(np.int32)
    b = oracle.attn(p["qkv_bits"], moved, pt, p["lens"], num_requests=2, block_len=4,
                    num_q_heads=24, num_kv_heads=4, qknorm=True, positions=p["pos"],
                    q_norm_w=p["qw_bits"], k_norm_w=p["kw_bits"])
    np.testing.assert_array_equal(a, b)


def test_requests_are_independent():
    p = make_problem(3, 2, 6, 1, [10, 150, 64], page_stride=3, num_pages=9, seed=40, qknorm=True)
    full = run_oracle(p)
    for r in range(3):
        sub = oracle.attn(p["qkv_bits"][r * 2:(r + 1) * 2], p["pool_bits"], p["pt"][r:r + 1],
                          p["lens"][r:r + 1], num_requests=1, block_len=2, num_q_heads=6,
                          num_kv_heads=1, qknorm=True, positions=p["pos"][r * 2:(r + 1) * 2],
                          q_norm_w=p["qw_bits"], k_norm_w=p["kw_bits"])
        np.testing.assert_array_equal(full[r * 2:(r + 1) * 2], sub)


def test_out_of_range_inputs_are_refused():
    p = make_problem(1, 1, 6, 1, [65], page_stride=2, num_pages=2, seed=41)
    p["pt"][0, 1] = 2
    _, st = run_oracle(p, check=False)
    assert st == oracle.BAD_PAGE
    p["pt"][0, 1] = 1
    p["lens"][0] = 129
    _, st = run_oracle(p, check=False)
    assert st == oracle.BAD_LENGTH


def test_oracle_matches_its_stored_regression_fixture():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "make_oracle_golden", os.path.join(os.path.dirname(__file__), "golden", "make_oracle_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(os.path.dirname(__file__), "golden", "oracle_small.json")) as f:
        stored = json.load(f)
    p = mod.problem()
    for key, qk in [("plain", False), ("qknorm", True)]:
        np.testing.assert_allclose(mod.compute(p, qk).reshape(-1), np.array(stored[key]),
                                   atol=1e-12, rtol=1e-12)


# ------------------------------------- standalone q/k norm + RoPE cell ----

def _norm_rope_case(T, Hq, Hkv, seed):
    g = torch.Generator().manual_seed(seed)
    qkv = torch.randn(T, (Hq + 2 * Hkv) * D, generator=g).to(torch.bfloat16)
    qw = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    pos = torch.randint(0, 1 << 20, (T,), generator=g, dtype=torch.int64)
    return qkv, qw, kw, pos


def _rotate(x, pos):
    """NeoX rotation as a complex product: (x_j + i x_{j+32}) e^{i pos 10000^(-2j/64)}."""
    j = np.arange(D // 2)
    z = (x[..., :D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * pos * 10000.0 ** (-2.0 * j / D))
    return np.concatenate([z.real, z.imag], axis=-1)


@pytest.mark.parametrize("Hq,Hkv", [(6, 1), (24, 4)])
def test_norm_rope_cell_matches_rms_norm_and_complex_rotation(Hq, Hkv):
    T = 5
    qkv, qw, kw, pos = _norm_rope_case(T, Hq, Hkv, 40 + Hq)
    out = oracle.qk_norm_rope(qkv, pos, qw, kw, num_q_heads=Hq, num_kv_heads=Hkv)
    x = qkv.double().view(T, Hq + 2 * Hkv, D)
    for h in range(Hq + 2 * Hkv):
        got = out[:, h * D:(h + 1) * D]
        if h < Hq + Hkv:
            w = (qw if h < Hq else kw).double()
            n = torch.nn.functional.rms_norm(x[:, h], (D,), weight=w, eps=1e-5).numpy()
            want = np.stack([_rotate(n[t], float(pos[t])) for t in range(T)])
            # Angles reach 2^20 rad: fp64 rounding of pos * inv_freq alone
            # moves sin/cos by ~2^20 * 2^-53.
            np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-9)
        else:  # value heads pass through exactly
            assert np.array_equal(got, x[:, h].numpy())


def test_norm_rope_cell_at_position_zero_is_the_norm_alone():
    qkv, qw, kw, _ = _norm_rope_case(3, 6, 1, 7)
    out = oracle.qk_norm_rope(qkv, torch.zeros(3, dtype=torch.int64), qw, kw, num_q_heads=6, num_kv_heads=1)
    x = qkv.double().view(3, 8, D)
    for h in range(7):
        w = (qw if h < 6 else kw).double()
        want = torch.nn.functional.rms_norm(x[:, h], (D,), weight=w, eps=1e-5).numpy()
        np.testing.assert_allclose(out[:, h * D:(h + 1) * D], want, rtol=1e-13, atol=1e-13)


def test_norm_rope_cell_scores_depend_on_relative_position():
    # q of token 0 against k of token 1: shifting both positions by the same
    # amount leaves the dot product unchanged (RoPE is a relative encoding).
    qkv, qw, kw, _ = _norm_rope_case(2, 6, 1, 11)
    dots = []
    for shift in (0, 977, 123456):
        out = oracle.qk_norm_rope(qkv, torch.tensor([5 + shift, 12 + shift]), qw, kw,
                                  num_q_heads=6, num_kv_heads=1)
        dots.append(float(out[0, 2 * D:3 * D] @ out[1, 6 * D:7 * D]))
    assert max(dots) - min(dots) < 1e-9 * max(1.0, abs(dots[0]))


# ----------------------------------------------------------------- YaRN ----
# The pages name YaRN with factor 4.0 for the drafter; the method is the
# "NTK-by-parts" interpolation of the YaRN paper (Peng et al. 2023): pairs
# with many wavelengths in the original context keep their frequency, pairs
# with less than one are slowed by the factor, a linear ramp in between, and
# q and k are scaled by mscale.

def _plain_inv(D=64, base=10000.0):
    return base ** (-2.0 * np.arange(D // 2) / D)


def test_yarn_factor_one_is_the_plain_table():
    np.testing.assert_allclose(oracle.yarn_inv_freq(64, 10000.0, 1.0, 4096.0), _plain_inv(), rtol=1e-15)


def test_yarn_keeps_fast_pairs_and_slows_slow_pairs_by_the_factor():
    inv0 = _plain_inv()
    r = 4096.0 * inv0 / (2 * math.pi)  # wavelengths of each pair inside 4096 positions
    inv = oracle.yarn_inv_freq(64, 10000.0, 4.0, 4096.0, beta_fast=32.0, beta_slow=1.0)
    fast, slow = r > 32.0, r < 1.0
    assert fast.any() and slow.any() and (~fast & ~slow).any()
    np.testing.assert_allclose(inv[fast], inv0[fast], rtol=1e-15)
    np.testing.assert_allclose(inv[slow], inv0[slow] / 4.0, rtol=1e-15)
    mid = ~fast & ~slow
    assert (inv[mid] < inv0[mid]).all() and (inv[mid] > inv0[mid] / 4.0).all()
    # Frequencies stay in decreasing order through the ramp.
    assert (np.diff(inv) < 0).all()


def test_yarn_ramp_midpoint_closed_form():
    # Put pair 10 exactly halfway up the ramp (r = (1 + 32) / 2): it turns at
    # theta * ((1 - 1/2) / 4 + 1/2) = 0.625 theta.
    theta = 10000.0 ** (-20.0 / 64)
    orig = 16.5 * 2 * math.pi / theta
    inv = oracle.yarn_inv_freq(64, 10000.0, 4.0, orig, beta_fast=32.0, beta_slow=1.0)
    assert abs(inv[10] / theta - 0.625) < 1e-13


def test_yarn_with_every_pair_slowed_is_rope_at_a_scaled_position():
    g = np.random.default_rng(3)
    x = g.standard_normal(64)
    inv = oracle.yarn_inv_freq(64, 10000.0, 4.0, 1e-3)  # no pair completes a wavelength: all slowed
    np.testing.assert_allclose(inv, _plain_inv() / 4.0, rtol=1e-15)
    for pos in (0, 4, 4 * 977, 4 * 123457):
        np.testing.assert_allclose(oracle.rope_table(x, pos, inv), oracle.rope_neox(x, pos // 4), rtol=1e-12,
                                   atol=1e-12)


def test_rope_table_scales_every_pair_norm_by_mscale():
    g = np.random.default_rng(4)
    x = g.standard_normal(64)
    y = oracle.rope_table(x, 12345.0, _plain_inv(), mscale=1.3862943611198906)
    n_in = np.hypot(x[:32], x[32:])
    n_out = np.hypot(y[:32], y[32:])
    np.testing.assert_allclose(n_out, 1.3862943611198906 * n_in, rtol=1e-13)


def _attn_case(seed):
    g = torch.Generator().manual_seed(seed)
    R, B, Hq, Hkv, S = 2, 3, 6, 1, 3
    qkv = torch.randn(R * B, (Hq + 2 * Hkv) * D, generator=g).to(torch.bfloat16)
    pool = torch.randn(6, 2, Hkv, P, D, generator=g).to(torch.bfloat16)
    pt = torch.tensor([[4, 1, 0], [2, 5, 3]], dtype=torch.int32)
    lens = torch.tensor([130, 70], dtype=torch.int32)
    qw = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    return dict(qkv=qkv, pool=pool, page_table=pt, ctx_lens=lens, num_requests=R, block_len=B,
                num_q_heads=Hq, num_kv_heads=Hkv, qknorm=True, q_norm_w=qw, k_norm_w=kw)


def test_attention_with_yarn_factor_one_is_the_fused_variant():
    c = _attn_case(21)
    pos = torch.tensor([130, 131, 132, 70, 71, 72])
    plain = oracle.attn(positions=pos, **c)
    yarn = oracle.attn(positions=pos, yarn=dict(factor=1.0, original_max_position=4096.0, beta_fast=32.0,
                                                beta_slow=1.0, mscale=1.0), **c)
    np.testing.assert_allclose(yarn, plain, rtol=1e-14, atol=1e-14)


def test_attention_with_every_pair_slowed_and_mscale_closed_form():
    # All pairs slowed by 4 and q, k scaled by m: with block keys only (the
    # pool's context keys are used as stored, unscaled) the scores are those
    # of the plain fused variant at positions / 4 with the scale times m^2.
    c = _attn_case(22)
    c["ctx_lens"] = torch.zeros(2, dtype=torch.int32)
    pos = torch.tensor([4 * 130, 4 * 131, 4 * 132, 4 * 70, 4 * 71, 4 * 72])
    m = 0.1 * math.log(4.0) + 1.0
    yarn = oracle.attn(positions=pos, yarn=dict(factor=4.0, original_max_position=1e-3, beta_fast=32.0,
                                                beta_slow=1.0, mscale=m), **c)
    plain = oracle.attn(positions=pos // 4, scale=0.125 * m * m, **c)
    np.testing.assert_allclose(yarn, plain, rtol=1e-11, atol=1e-12)


def test_norm_rope_cell_with_yarn_factor_one_is_the_plain_cell():
    qkv, qw, kw, pos = _norm_rope_case(4, 24, 4, 13)
    plain = oracle.qk_norm_rope(qkv, pos, qw, kw, num_q_heads=24, num_kv_heads=4)
    yarn = oracle.qk_norm_rope(qkv, pos, qw, kw, num_q_heads=24, num_kv_heads=4,
                               yarn=dict(factor=1.0, original_max_position=4096.0, beta_fast=32.0,
                                         beta_slow=1.0, mscale=1.0))
    np.testing.assert_allclose(yarn, plain, rtol=1e-14, atol=1e-14)


def test_norm_rope_cell_with_every_pair_slowed_closed_form():
    qkv, qw, kw, pos = _norm_rope_case(4, 6, 1, 14)
    m = 1.1386294361119891
    yarn = oracle.qk_norm_rope(qkv, 4 * pos, qw, kw, num_q_heads=6, num_kv_heads=1,
                               yarn=dict(factor=4.0, original_max_position=1e-3, beta_fast=32.0,
                                         beta_slow=1.0, mscale=m))
    plain = oracle.qk_norm_rope(qkv, pos, qw, kw, num_q_heads=6, num_kv_heads=1)
    qk = 7 * D  # q and k heads scale by m; v heads pass through
    np.testing.assert_allclose(yarn[:, :qk], m * plain[:, :qk], rtol=1e-11, atol=1e-11)
    assert np.array_equal(yarn[:, qk:], plain[:, qk:])
