"""The kernels' IQ4_NL decode constants, checked on the CPU.

The library stores 4-bit labels (table index i relabelled as
(i >> 1) + 8 * (i & 1)) and decodes four labels with two PTX prmt byte
permutes whose sign-replicate mode supplies the missing table half.  This
test emulates prmt as the PTX ISA defines it and checks, for every label,
that the constants in device_utils.cuh give the IQ4_NL table value, and that
the CUDA-core kernels' float table agrees.
"""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "quantized_moe_expert_sigmoid_gb300", "csrc")
# IQ4_NL table, index order (HelloSun/xing4_0-29b-IQ4_NL_EPQ model card,
# "16-entry nonlinear table"; values as given with the synthetic workloads)
CODEBOOK = [-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113]


def prmt(a, b, c):
    """PTX prmt.b32 default mode."""
    src = (a & 0xFFFFFFFF) | ((b & 0xFFFFFFFF) << 32)
    r = 0
    for i in range(4):
        sel = (c >> (4 * i)) & 0xF
        byte = (src >> (8 * (sel & 7))) & 0xFF
        if sel & 8:
            byte = 0xFF if byte & 0x80 else 0x00
        r |= byte << (8 * i)
    return r


def _consts():
    src = open(os.path.join(CSRC, "device_utils.cuh")).read()
    vals = dict(re.findall(r"(kT[LH][01]) = (0x[0-9A-Fa-f]+)u", src))
    return {k: int(v, 16) for k, v in vals.items()}


def _label(i):
    return (i >> 1) + 8 * (i & 1)


def _decode4(q):
    k = _consts()
    qx = q ^ 0x8888
    return prmt(k["kTL0"], k["kTL1"], q) ^ prmt(k["kTH0"], k["kTH1"], qx)


def test_every_label_decodes_to_its_table_value():
    label_table = [0] * 16
    for i, v in enumerate(CODEBOOK):
        label_table[_label(i)] = v
    for lab in range(16):
        for pos in range(4):
            q = lab << (4 * pos)
            byte = (_decode4(q) >> (8 * pos)) & 0xFF
            assert np.int8(np.uint8(byte)) == label_table[lab], (lab, pos)


def test_mixed_words_decode_bytewise():
    rng = np.random.default_rng(0)
    for q in rng.integers(0, 1 << 16, 200):
        out = _decode4(int(q))
        for pos in range(4):
            lab = (int(q) >> (4 * pos)) & 15
            idx = [i for i in range(16) if _label(i) == lab][0]
            assert np.int8(np.uint8((out >> (8 * pos)) & 0xFF)) == CODEBOOK[idx]


def test_relabel_pairs_share_a_sign():
    for j in range(8):
        a, b = CODEBOOK[2 * j], CODEBOOK[2 * j + 1]
        assert (a < 0) == (b < 0)
