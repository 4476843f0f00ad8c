"""The oracle's pins have teeth: plant one plausible mistake at a time in a
copy of the oracle's C source (on the CPU, in a temporary directory), rebuild
it, and check that the pin suite fails on every mutant."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# name -> (text in the oracle, the planted mistake)
MUTANTS = {
    "rope_frequency_exponent": ("double inv_freq = pow(base, -2.0 * (double)j / (double)D);",
                                "double inv_freq = pow(base, -1.0 * (double)j / (double)D);"),
    "rope_rotation_sign": ("tmp[j] = lo * c - hi * s;", "tmp[j] = lo * c + hi * s;"),
    "rope_interleaved_pairs": ("double lo = x[j], hi = x[j + half];\n        tmp[j] = lo * c - hi * s;",
                               "double lo = x[j], hi = x[(j + 1) % D];\n        tmp[j] = lo * c - hi * s;"),
    "gqa_head_modulo": ("const int h = g * G + hl;", "const int h = hl * Hkv + g;"),
    "softmax_scale_dropped": ("s[k] = scale * dot;", "s[k] = dot;"),
    "page_slot_off_by_one": ("int64_t slot = c % page_size;", "int64_t slot = (c + 1) % page_size;"),
    "pool_k_v_swapped": ("pool + (((page * 2 + 0) * Hkv + g)", "pool + (((page * 2 + 1) * Hkv + g)"),
    "rmsnorm_eps_dropped": ("1.0 / sqrt(mean_sq + eps)", "1.0 / sqrt(mean_sq)"),
    "rmsnorm_wrong_mean": ("double mean_sq = sum_sq / (double)D;", "double mean_sq = sum_sq / (double)(D - 1);"),
    "block_v_from_k_region": ("(int64_t)(Hq + Hkv + g) * D;", "(int64_t)(Hq + g) * D;"),
    "causal_block_mask": ("for (int64_t k = 0; k < nkeys; ++k) {\n                        double dot",
                          "for (int64_t k = 0; k < L + i + 1; ++k) {\n                        double dot"),
    "block_k_position_of_first_token": ("k3o_rope_neox(tmp, D, (double)positions[t], base, kdst);",
                                        "k3o_rope_neox(tmp, D, (double)positions[(int64_t)r * B], base, kdst);"),
    "k_normed_with_q_weight": ("k3o_rmsnorm(raw, wk, D, eps, tmp);", "k3o_rmsnorm(raw, wq, D, eps, tmp);"),
    "cell_k_heads_with_q_weight": ("k3o_rmsnorm(raw, h < Hq ? wq : wk, D, eps, tmp);",
                                   "k3o_rmsnorm(raw, wq, D, eps, tmp);"),
    "cell_v_heads_normalised": ("if (h < Hq + Hkv) {", "if (h < Hq + 2 * Hkv) {"),
    "cell_position_of_first_token": ("(double)positions[t], base, dst);", "(double)positions[0], base, dst);"),
    "yarn_ramp_inverted": ("inv_freq[j] = (1.0 - gamma) * theta / factor + gamma * theta;",
                           "inv_freq[j] = gamma * theta / factor + (1.0 - gamma) * theta;"),
    "yarn_wavelength_without_two_pi": ("double wavelength = two_pi / theta;", "double wavelength = 1.0 / theta;"),
    "yarn_mscale_on_one_output": ("tmp[j + half] = (hi * c + lo * s) * mscale;",
                                  "tmp[j + half] = (hi * c + lo * s);"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pin_suite_rejects_planted_mistake(name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "k3da_oracle.c")).read()
    before, after = MUTANTS[name]
    assert src.count(before) == 1, name
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    (pkg / "k3da_oracle.c").write_text(src.replace(before, after))
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), pkg / "__init__.py")
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("test_oracle_mutants.py", "__pycache__"))
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
