"""Build the hand-made blocks described in tests/golden/*.json (byte assembly only)."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f16(bits):
    return [bits & 0xFF, bits >> 8]


def _hexbits(s):
    return int(s.split()[0], 16)


def q4_k():
    g = load("q4_k_block.json")
    f = g["fields"]
    b = np.zeros(144, np.uint8)
    b[0:2] = _f16(_hexbits(f["d_f16_bits"]))
    b[2:4] = _f16(_hexbits(f["dmin_f16_bits"]))
    b[4:16] = f["scales"]
    for i, v in f["qs_nonzero"].items():
        b[16 + int(i)] = v
    return b, {int(k): v for k, v in g["expected"].items()}


def q5_k():
    g = load("q5_k_block.json")
    f = g["fields"]
    b = np.zeros(176, np.uint8)
    b[0:2] = _f16(_hexbits(f["d_f16_bits"]))
    b[2:4] = _f16(_hexbits(f["dmin_f16_bits"]))
    b[4:16] = f["scales"]
    for i, v in f["qh_nonzero"].items():
        b[16 + int(i)] = v
    for i, v in f["qs_nonzero"].items():
        b[48 + int(i)] = v
    return b, {int(k): v for k, v in g["expected"].items()}


def q6_k():
    g = load("q6_k_block.json")
    f = g["fields"]
    b = np.zeros(210, np.uint8)
    for i, v in f["ql_nonzero"].items():
        b[int(i)] = v
    for i, v in f["qh_nonzero"].items():
        b[128 + int(i)] = v
    b[192:208] = np.array(f["scales_i8"], np.int8).view(np.uint8)
    b[208:210] = _f16(_hexbits(f["d_f16_bits"]))
    return b, {int(k): v for k, v in g["expected"].items()}


def q8_0():
    g = load("q8_0_block.json")
    out = []
    b0 = np.zeros(34, np.uint8)
    b0[0:2] = _f16(_hexbits(g["blocks"][0]["d_f16_bits"]))
    q = np.arange(32, dtype=np.int64) - 16
    q[0] = -128
    b0[2:34] = q.astype(np.int8).view(np.uint8)
    out.append((b0, {int(k): v for k, v in g["blocks"][0]["expected"].items()}))
    b1 = np.zeros(34, np.uint8)
    b1[0:2] = _f16(_hexbits(g["blocks"][1]["d_f16_bits"]))
    b1[2:34] = 3
    out.append((b1, {int(k): v for k, v in g["blocks"][1]["expected"].items()}))
    return out


def _b32(name, size, q_off, qh_off=None, m=False):
    g = load(name)
    f = g["fields"]
    b = np.zeros(size, np.uint8)
    b[0:2] = _f16(_hexbits(f["d_f16_bits"]))
    if m:
        b[2:4] = _f16(_hexbits(f["m_f16_bits"]))
    if qh_off is not None:
        b[qh_off:qh_off + 4] = f["qh"]
    for i, v in f["qs_nonzero"].items():
        b[q_off + int(i)] = v
    return b, {int(k): v for k, v in g["expected"].items()}


def q4_0():
    return _b32("q4_0_block.json", 18, 2)


def q4_1():
    return _b32("q4_1_block.json", 20, 4, m=True)


def q5_0():
    return _b32("q5_0_block.json", 22, 6, qh_off=2)


def q5_1():
    return _b32("q5_1_block.json", 24, 8, qh_off=4, m=True)


def q2_k():
    g = load("q2_k_block.json")
    f = g["fields"]
    b = np.zeros(84, np.uint8)
    b[0:16] = f["scales"]
    for i, v in f["qs_nonzero"].items():
        b[16 + int(i)] = v
    b[80:82] = _f16(_hexbits(f["d_f16_bits"]))
    b[82:84] = _f16(_hexbits(f["dmin_f16_bits"]))
    return b, {int(k): v for k, v in g["expected"].items()}


def q3_k():
    g = load("q3_k_block.json")
    f = g["fields"]
    b = np.zeros(110, np.uint8)
    for i, v in f["hmask_nonzero"].items():
        b[int(i)] = v
    for i, v in f["qs_nonzero"].items():
        b[32 + int(i)] = v
    b[96:108] = f["scales"]
    b[108:110] = _f16(_hexbits(f["d_f16_bits"]))
    return b, {int(k): v for k, v in g["expected"].items()}
