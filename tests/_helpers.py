"""Shared helpers for the tests: golden-file parsing, exact brute force, tolerances.

Nothing here is on the product path; the exact brute force uses Python
fractions and decodes scale bytes through torch's float8 dtypes (a library
routine), so it shares no arithmetic with the C oracle.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def e2m1_golden() -> dict[int, float]:
    """code -> value from tests/golden/e2m1_values.txt."""
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            table[int(c)] = float(v)
    return table


def torch_scale_values(fmt: str) -> np.ndarray:
    """All 256 scale bytes decoded by torch (float8_e4m3fn or float8_e8m0fnu) as float64."""
    import torch
    codes = torch.arange(256, dtype=torch.uint8)
    dt = torch.float8_e4m3fn if fmt == "nvfp4" else torch.float8_e8m0fnu
    return codes.view(dt).to(torch.float64).numpy()


def parse_worked_examples():
    """List of dicts: fmt, M, N, K, alpha, A, sfA, B, sfB (numpy uint8), D (list)."""
    out = []
    cur = None
    with open(os.path.join(GOLDEN, "worked_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            key = tok[0]
            if key == "example":
                cur = {"name": tok[1], "rows": {}}
            elif key == "fmt":
                cur["fmt"] = tok[1]
            elif key == "shape":
                cur["M"], cur["N"], cur["K"] = map(int, tok[1:4])
            elif key == "alpha":
                cur["alpha"] = float(tok[1])
            elif key == "D":
                cur["D"] = [float(t) for t in tok[1:]]
            elif key == "end":
                out.append(_materialise(cur))
                cur = None
            else:
                cur["rows"][key] = tok[1:]
    return out


def _materialise(ex):
    M, N, K = ex["M"], ex["N"], ex["K"]
    vec = 16 if ex["fmt"] == "nvfp4" else 32
    A = np.zeros((M, K // 2), np.uint8)
    B = np.zeros((N, K // 2), np.uint8)
    sfA = np.zeros((M, K // vec), np.uint8)
    sfB = np.zeros((N, K // vec), np.uint8)

    def fill(dst, spec):
        for t in spec:
            if t.startswith("fill="):
                dst[:] = int(t[5:], 16)
            else:
                i, v = t.split(":")
                dst[int(i)] = int(v, 16)

    for key, spec in ex["rows"].items():
        if key.startswith("sfA"):
            sfA[int(key[3:])] = [int(t, 16) for t in spec]
        elif key.startswith("sfB"):
            sfB[int(key[3:])] = [int(t, 16) for t in spec]
        elif key.startswith("A"):
            fill(A[int(key[1:])], spec)
        elif key.startswith("B"):
            fill(B[int(key[1:])], spec)
    from workloads import GemmInputs
    inp = GemmInputs(ex["fmt"], M, N, K, A, sfA, B, sfB, ex["alpha"], "f32", ex["name"])
    return inp, np.array(ex["D"], dtype=np.float64).reshape(M, N)


def unpack_codes(packed: np.ndarray, K: int) -> np.ndarray:
    """[rows][K/2] bytes -> [rows][K] codes; element 2j is the low nibble of byte j."""
    packed = np.asarray(packed, dtype=np.uint8).reshape(-1, K // 2)
    codes = np.empty((packed.shape[0], K), np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    return codes


def exact_gemm(inp):
    """Exact rational D and |alpha|*sum|a b| by brute force (pure Python; tiny shapes only)."""
    table = e2m1_golden()
    sv = torch_scale_values(inp.fmt)
    vec = inp.vec
    ca = unpack_codes(inp.A, inp.K)
    cb = unpack_codes(inp.B, inp.K)
    sfA = np.asarray(inp.sfA).reshape(inp.M, -1)
    sfB = np.asarray(inp.sfB).reshape(inp.N, -1)
    alpha = Fraction(inp.alpha)
    D, ABS = [], []
    for i in range(inp.M):
        row, arow = [], []
        for j in range(inp.N):
            acc = Fraction(0)
            aacc = Fraction(0)
            for k in range(inp.K):
                a = Fraction(table[int(ca[i, k])]) * Fraction(float(sv[sfA[i, k // vec]]))
                b = Fraction(table[int(cb[j, k])]) * Fraction(float(sv[sfB[j, k // vec]]))
                acc += a * b
                aacc += abs(a * b)
            row.append(alpha * acc)
            arow.append(abs(alpha) * aacc)
        D.append(row)
        ABS.append(arow)
    return D, ABS


# ---- tolerances used by every parity test ---------------------------------------

def f32_tol(absdot: np.ndarray) -> np.ndarray:
    """fp32 output: |D - ref| <= 1e-5 * |alpha| * sum_k |a_k b_k| + 1e-6."""
    return 1e-5 * absdot + 1e-6


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    """ulp of a bf16 value: 2^(floor(log2|x|) - 7), at least the subnormal quantum 2^-133."""
    v = np.abs(bf16_bits_to_f64(bits))
    out = np.full(v.shape, 2.0 ** -133)
    nz = v > 0
    e = np.floor(np.log2(v[nz]))
    out[nz] = np.maximum(2.0 ** (e - 7), 2.0 ** -133)
    return out
