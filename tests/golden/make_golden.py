"""Writes the hand-worked golden fixtures in this folder.

Every value is a closed form of a rule stated on the attention pages (cited in
each file's "source" field), evaluated with Python's math module.  Nothing here
calls the oracle or the CUDA library.  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def _dump(name, obj):
    with open(os.path.join(HERE, name), "w") as f:
        json.dump(obj, f, indent=1)


def main():
    na = {
        "source": "candle PR #11 'perf(cuda): make the cuDNN convolution path usable, and 4.4x faster', "
                  "commit 'kernel exceeds grid extent': a window wider than its axis degrades to full "
                  "attention on that axis (start 0, width = extent); repro shapes grid [9,64,64] kernel "
                  "[11,11,11] and grid [1,4,4] kernel [3,7,7]. Window start per axis = clamp(i - k//2, 0, "
                  "extent - min(k, extent)) as stated for the clamp workloads. Values below are worked by "
                  "hand from that rule.",
        "cases": [
            {"grid": [1, 4, 4], "kernel": [3, 7, 7], "k_eff": [1, 4, 4], "window_size": 16,
             "note": "every axis clamps (two even extents): every query attends to all 16 tokens"},
            {"grid": [9, 64, 64], "kernel": [11, 11, 11], "k_eff": [9, 11, 11], "window_size": 1089,
             "t_window_all_queries": [0, 9],
             "hw_starts": {"0": 0, "5": 0, "6": 1, "32": 27, "53": 48, "58": 53, "63": 53},
             "note": "time axis clamps to 9 (full); h/w windows of 11 shifted at the borders: "
                     "start = clamp(i-5, 0, 53)"},
        ],
    }
    _dump("na_clamp_cases.json", na)

    cases = []
    for axis, pair, pos in [(1, 8, 100), (3, 4, 7), (2, 0, 3), (3, 12, 511)]:
        phi = pos * 10000.0 ** (-2.0 * pair / 32)
        cases.append({"axis": axis, "pair": pair, "pos": pos, "phi": phi,
                      "unit_first": [math.cos(phi), math.sin(phi)],
                      "unit_second": [-math.sin(phi), math.cos(phi)]})
    rope = {
        "source": "iris.c issue #15 'CUDA codepath !', GGML lessons item 3 (FLUX's custom RoPE: 4 axes "
                  "[32,32,32,32], separate text/image positions, repeat_interleave); FLUX joint workload "
                  "statement: theta 10000 on adjacent (2i,2i+1) pairs, image positions (0,row,col,0), text "
                  "positions (0,0,0,j). Angles worked by hand: phi = pos * theta^(-2i/32) for pair i of an "
                  "axis block.",
        "theta": 10000.0, "axes_dim": [32, 32, 32, 32],
        "freq": {"0": 1.0, "4": 0.1, "8": 0.01, "12": 0.001},
        "cases": cases,
    }
    _dump("rope_angles.json", rope)

    e = math.e
    sm = {
        "source": "closed form of scaled-dot-product attention with two keys (S = QK^T*scale, row "
                  "softmax, O = PV as named by the attention pages): p1 = 1/(1+exp(s2-s1)).",
        "q": [[1.0, 0.0]], "k": [[1.0, 0.0], [0.0, 0.0]], "v": [[2.0, -1.0], [0.0, 3.0]],
        "scale": 1.0,
        "p": [e / (1 + e), 1 / (1 + e)],
        "o": [2 * e / (1 + e), (-e + 3) / (1 + e)],
    }
    _dump("two_key_closed_form.json", sm)


if __name__ == "__main__":
    main()
