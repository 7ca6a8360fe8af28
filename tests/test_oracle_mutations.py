"""Mutation check of the oracle's pins: plant plausible mistakes in a copy of
the oracle's C source (on the CPU), rebuild it, and require the pin suite to
fail for every one of them.  A pin set that lets one of these through is too
weak to trust the oracle with.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attn_oracle.c")
PINS = ["tests/test_oracle_full.py", "tests/test_oracle_na3d.py",
        "tests/test_oracle_decode_rope.py"]

MUTATIONS = {
    "drop_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "no_max_subtraction": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "clamp_with_requested_kernel": ("if (st > n - keff) st = n - keff;",
                                    "if (st > n - k) st = n - k;"),
    "rope_freq_over_head_dim": ("pow(theta, -2.0 * (double)i / (double)na)",
                                "pow(theta, -2.0 * (double)i / (double)D)"),
    "rope_sign": ("xr[c + 2 * i] = x0 * cs - x1 * sn;", "xr[c + 2 * i] = x0 * cs + x1 * sn;"),
    "rope_half_split_pairs": (
        "const double x0 = xr[c + 2 * i], x1 = xr[c + 2 * i + 1];\n"
        "                xr[c + 2 * i] = x0 * cs - x1 * sn;\n"
        "                xr[c + 2 * i + 1] = x0 * sn + x1 * cs;",
        "const double x0 = xr[c + i], x1 = xr[c + i + na / 2];\n"
        "                xr[c + i] = x0 * cs - x1 * sn;\n"
        "                xr[c + i + na / 2] = x0 * sn + x1 * cs;"),
    "rope_axis_block_offset": ("c += na;", "c += na / 2;"),
    "gqa_interleaved_groups": ("const int64_t kvh = hq / group;", "const int64_t kvh = hq % Hkv;"),
    "na_grid_transposed": ("keys[n++] = ((int64_t)a * Hg + b) * W + c;",
                           "keys[n++] = ((int64_t)a * W + b) * Hg + c;"),
    "wrong_head_base": ("const int64_t bh = row / Nq;", "const int64_t bh = row / Nkv;"),
    "unnormalised_p": ("for (int d = 0; d < D; ++d) o[d] += pj * vj[d];",
                       "for (int d = 0; d < D; ++d) o[d] += s[j] * vj[d];"),
    "decode_drops_last_row": ("const int64_t L = seq_len[b];",
                              "const int64_t L = seq_len[b] > 1 ? seq_len[b] - 1 : 1;"),
    "causal_sees_one_future_key": ("attend_row(q + row * D, k + kvbase, v + kvbase, keys, i + 1,",
                                   "attend_row(q + row * D, k + kvbase, v + kvbase, keys, i + (i + 1 < N ? 2 : 1),"),
    "causal_gqa_interleaved": ("(b * Hkv + hq / group)", "(b * Hkv + hq % Hkv)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(before) >= 1, f"mutation site for {name} not found"
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src.replace(before, after))
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(so), str(c), "-lm"], check=True)
    env = dict(os.environ, ATTN_ORACLE_LIB=str(so), OMP_NUM_THREADS="4")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu", *PINS], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"
