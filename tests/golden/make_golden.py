"""Writes q4k_handbuilt.txt: hand-built Q4_K blocks (inputs only).

The blocks are packed from chosen fields by the test-side packer; the file
stores the fields, the packed bytes and, for each block, the closed form of its
weights.  No expected number is computed here: the test evaluates the closed
form from the fields.  Format reference: the GGUF Q4_K super-block, the format
of the "UD-Q4_K_XL" distribution named in "Layer Package Repository Spec",
section "Repository Identity".
Run: python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
from _q4k_fields import pack_block  # noqa: E402

BLOCKS = [
    # name, d bits, dmin bits, sc, m, quant rule, closed form
    ("ramp", 0x3C00, 0x3800, [1, 2, 3, 4, 5, 6, 7, 8], [0, 2, 4, 6, 8, 10, 12, 14],
     "i%16", "w_i = (j+1)*(i%16) - j, j = i//32  (d = 1, dmin = 1/2)"),
    ("max_scales", 0x2C00, 0x2800, [63] * 8, [63] * 8,
     "15-i%16", "w_i = 63/16*(15 - i%16) - 63/32  (d = 2^-4, dmin = 2^-5)"),
    ("high_bits_only", 0x3C00, 0x3C00, [0, 0, 0, 0, 48, 48, 48, 48], [0, 0, 0, 0, 48, 48, 48, 48],
     "7*i%16", "w_i = 0 for j < 4; 48*((7*i)%16) - 48 for j >= 4"),
    ("low_bits_only", 0x3C00, 0x4000, [1, 2, 3, 4, 15, 14, 13, 12], [5, 6, 7, 8, 9, 10, 11, 15],
     "3", "w_i = 3*sc_j - 2*m_j with the listed sc, m  (d = 1, dmin = 2)"),
    ("subnormal_d", 0x0001, 0x03FF, [1, 2, 3, 4, 5, 6, 7, 8], [8, 7, 6, 5, 4, 3, 2, 1],
     "i%16", "w_i = 2^-24*(j+1)*(i%16) - 1023*2^-24*(8-j)"),
    ("zero", 0x0000, 0x0000, [0] * 8, [0] * 8, "0", "w_i = 0"),
    ("negative_d", 0xBC00, 0xB800, [1, 1, 1, 1, 1, 1, 1, 1], [1, 1, 1, 1, 1, 1, 1, 1],
     "i%16", "w_i = -(i%16) + 1/2  (d = -1, dmin = -1/2)"),
]


def quants(rule):
    out = []
    for i in range(256):
        out.append(eval(rule, {}, {"i": i}) % 16)
    return out


def main():
    lines = [
        "# Hand-built Q4_K super-blocks (inputs) with the closed form of their weights.",
        "# Written by tests/golden/make_golden.py from chosen fields with the test-side packer.",
        "# Format: the GGUF Q4_K super-block of the UD-Q4_K_XL distribution",
        "# ('Layer Package Repository Spec', section 'Repository Identity').",
        "# Columns: name | d bits | dmin bits | sc_0..7 | m_0..7 | quant rule (python, in i) | hex bytes | closed form",
    ]
    for name, d, dm, sc, m, rule, form in BLOCKS:
        blk = pack_block(d, dm, sc, m, quants(rule))
        lines.append(" | ".join([name, f"{d:04x}", f"{dm:04x}", ",".join(map(str, sc)),
                                 ",".join(map(str, m)), rule, blk.hex(), form]))
    with open(os.path.join(HERE, "q4k_handbuilt.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
