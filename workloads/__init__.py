"""Seeded synthetic inputs for the block-scaled FP4 GEMM.

Shared by the tests, the benchmark and the smoke check; used by both the CUDA
path and the CPU oracle, so it holds none of the GEMM's arithmetic: it draws
random values and *encodes* them into E2M1 codes and per-block scale bytes.
Nothing here decodes an E2M1 code or computes a product.

Recipes (the workloads these shapes and distributions stand for):

* ``nvfp4_128x128x256_f32`` -- M=N=128, K=256, codes uniform over all 16 E2M1
  codes, E4M3 scales 2^u with u uniform in [-3, 3], alpha = 1, fp32 output.
* ``nvfp4_4096_bf16`` -- M=N=K=4096, N(0,1) values quantised per 16-element K
  block (E4M3 scale = absmax/6 rounded to E4M3), alpha = 1/(448*6)^2, bf16 out.
* ``mxfp4_8192_f32`` -- M=N=K=8192, N(0,1) values, E8M0 scale per 32 elements
  = 2^(floor(log2 absmax) - 2), fp32 output.
* ``nvfp4_proj_m{16,128,1024,8192}_n14336_k4096`` and ``..._n4096_k14336`` --
  LLM projection shapes: weights B ~ N(0, 0.02), activations A ~ N(0, 1),
  E4M3 per-16 scales from absmax/6, alpha = 1, bf16 output.
* ``nvfp4_8191x3000x5120_f32`` and ``nvfp4_1x28672x4096_f32`` -- Student-t(3)
  values, per-16 E4M3 scales, alpha = 1, fp32 output (partial tiles, tails).

Quantisation rules (the generator's, not the GEMM's): a value x in a block
with decoded scale s becomes the E2M1 code nearest to x/s, ties to the even
code, saturating at +-6, sign kept (so tiny negatives give code 8, -0). A zero
scale gives all-zero codes. The NVFP4 scale is absmax/6 clamped to 448 and
rounded to E4M3 (torch's float8_e4m3fn cast, round to nearest even). The
MXFP4 scale exponent is floor(log2 absmax) - 2 clamped to [-127, 127]; an
all-zero block gets the E8M0 byte 0 (2^-127).

Random numbers come from numpy's PCG64 (``default_rng``): the A side draws
from seed ``2*seed``, the B side from ``2*seed + 1``. PCG64 with the standard
normal / Student-t samplers is bit-reproducible across x86_64 and aarch64.
"""
from __future__ import annotations

import dataclasses

import numpy as np

NV_VEC = 16
MX_VEC = 32

# Boundaries between adjacent E2M1 magnitudes (code c | code c+1) and whether
# an exact tie goes up (the upper code is the even one).
_E2M1_BOUNDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float64)
_E2M1_TIE_UP = np.array([False, True, False, True, False, True, False])


@dataclasses.dataclass
class GemmInputs:
    """One problem: packed codes, row-major scale bytes and the call's scalars."""
    fmt: str            # "nvfp4" (vec 16, E4M3 scales) or "mxfp4" (vec 32, E8M0 scales)
    M: int
    N: int
    K: int
    A: np.ndarray       # uint8 [M][K/2], low nibble = even k
    sfA: np.ndarray     # uint8 [M][K/vec]
    B: np.ndarray       # uint8 [N][K/2]
    sfB: np.ndarray     # uint8 [N][K/vec]
    alpha: float
    out: str            # "f32" or "bf16"
    name: str = ""

    @property
    def vec(self) -> int:
        return NV_VEC if self.fmt == "nvfp4" else MX_VEC

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


# ---- encoders --------------------------------------------------------------

def encode_e2m1(x: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code (ties to the even code, saturate at +-6, sign kept)."""
    x = np.asarray(x)
    ax = np.abs(x)
    code = np.zeros(x.shape, dtype=np.uint8)
    for b, up in zip(_E2M1_BOUNDS, _E2M1_TIE_UP):
        step = (ax > b) | ((ax == b) if up else False)
        code += step.astype(np.uint8)
    code |= (np.signbit(x).astype(np.uint8) << 3)
    return code


def encode_e4m3(s: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Non-negative values -> (E4M3 bytes, the values those bytes stand for), RN-even."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(np.minimum(s, 448.0), dtype=np.float32))
    q = t.to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy().copy(), q.to(torch.float32).numpy().astype(np.float32)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """[rows][K] codes -> [rows][K/2] bytes, low nibble = even k."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape[-1] % 2 == 0
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def quantize_nvfp4(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """[rows][K] float values -> (packed codes [rows][K/2], E4M3 scales [rows][K/16])."""
    rows, K = x.shape
    blk = x.reshape(rows, K // NV_VEC, NV_VEC)
    amax = np.abs(blk).max(axis=2)
    sf, s_dec = encode_e4m3(amax.astype(np.float32) / np.float32(6.0))
    s = s_dec[:, :, None]
    safe = np.where(s > 0, s, np.float32(1.0))
    codes = np.where(s > 0, encode_e2m1(blk / safe), np.uint8(0)).astype(np.uint8)
    return pack_codes(codes.reshape(rows, K)), sf


def quantize_mxfp4(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """[rows][K] float values -> (packed codes [rows][K/2], E8M0 scales [rows][K/32])."""
    rows, K = x.shape
    blk = x.reshape(rows, K // MX_VEC, MX_VEC).astype(np.float32)
    amax = np.abs(blk).max(axis=2)
    _, e = np.frexp(amax)                        # amax = f * 2^e, f in [0.5, 1)
    exp = np.where(amax > 0, e.astype(np.int64) - 1 - 2, -127)
    exp = np.clip(exp, -127, 127)
    sf = (exp + 127).astype(np.uint8)
    scale = np.ldexp(np.float32(1.0), exp.astype(np.int32)).astype(np.float32)[:, :, None]
    codes = np.where(amax[:, :, None] > 0, encode_e2m1(blk / scale), np.uint8(0)).astype(np.uint8)
    return pack_codes(codes.reshape(rows, K)), sf


# ---- value samplers ---------------------------------------------------------

def _quantize_rows(draw, rows: int, K: int, fmt: str, chunk_rows: int = 1024):
    """Draw rows x K values chunk by chunk (bounded memory) and quantise them."""
    q = quantize_nvfp4 if fmt == "nvfp4" else quantize_mxfp4
    vec = NV_VEC if fmt == "nvfp4" else MX_VEC
    packed = np.empty((rows, K // 2), dtype=np.uint8)
    sf = np.empty((rows, K // vec), dtype=np.uint8)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        p, s = q(draw((r1 - r0, K)))
        packed[r0:r1] = p
        sf[r0:r1] = s
    return packed, sf


def _normal(rng, std):
    return lambda shape: (rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def _student_t3(rng):
    return lambda shape: rng.standard_t(3, shape).astype(np.float32)


def make_random(fmt: str, M: int, N: int, K: int, *, dist: str = "normal", a_std: float = 1.0,
                b_std: float = 1.0, alpha: float = 1.0, out: str = "f32", seed: int = 0,
                name: str = "") -> GemmInputs:
    """Values drawn from ``dist`` ("normal" or "t3"), quantised blockwise into ``fmt``."""
    ra = np.random.default_rng(2 * seed)
    rb = np.random.default_rng(2 * seed + 1)
    if dist == "normal":
        da, db = _normal(ra, a_std), _normal(rb, b_std)
    elif dist == "t3":
        da, db = _student_t3(ra), _student_t3(rb)
    else:
        raise ValueError(dist)
    A, sfA = _quantize_rows(da, M, K, fmt)
    B, sfB = _quantize_rows(db, N, K, fmt)
    return GemmInputs(fmt, M, N, K, A, sfA, B, sfB, float(alpha), out, name)


def make_uniform_codes(fmt: str, M: int, N: int, K: int, *, alpha: float = 1.0, out: str = "f32",
                       seed: int = 0, u_range=(-3, 3), name: str = "") -> GemmInputs:
    """Codes uniform over all 16 E2M1 codes; scales 2^u with u uniform in u_range."""
    ra = np.random.default_rng(2 * seed)
    rb = np.random.default_rng(2 * seed + 1)
    vec = NV_VEC if fmt == "nvfp4" else MX_VEC

    def side(rng, rows):
        codes = rng.integers(0, 16, size=(rows, K), dtype=np.uint8)
        u = rng.integers(u_range[0], u_range[1] + 1, size=(rows, K // vec))
        # 2^u as a scale byte: E4M3 exponent field u + 7 (mantissa 0), E8M0 byte u + 127.
        sf = ((u + 7) << 3) if fmt == "nvfp4" else (u + 127)
        return pack_codes(codes), sf.astype(np.uint8)

    A, sfA = side(ra, M)
    B, sfB = side(rb, N)
    return GemmInputs(fmt, M, N, K, A, sfA, B, sfB, float(alpha), out, name)


# ---- the named workloads ------------------------------------------------------

PROJ_MS = (16, 128, 1024, 8192)


def config_names() -> list[str]:
    names = ["nvfp4_128x128x256_f32", "nvfp4_4096_bf16", "mxfp4_8192_f32"]
    for m in PROJ_MS:
        names.append("nvfp4_proj_m%d_n14336_k4096" % m)
        names.append("nvfp4_proj_m%d_n4096_k14336" % m)
    names += ["nvfp4_8191x3000x5120_f32", "nvfp4_1x28672x4096_f32", "nvfp4_8192_f32"]
    return names


def config_shape(name: str) -> dict:
    """fmt, M, N, K, out, alpha of a named workload (no data drawn)."""
    if name == "nvfp4_128x128x256_f32":
        return dict(fmt="nvfp4", M=128, N=128, K=256, out="f32", alpha=1.0)
    if name == "nvfp4_4096_bf16":
        return dict(fmt="nvfp4", M=4096, N=4096, K=4096, out="bf16", alpha=1.0 / (448.0 * 6.0) ** 2)
    if name == "mxfp4_8192_f32":
        return dict(fmt="mxfp4", M=8192, N=8192, K=8192, out="f32", alpha=1.0)
    if name.startswith("nvfp4_proj_"):
        parts = name.split("_")
        m, n, k = int(parts[2][1:]), int(parts[3][1:]), int(parts[4][1:])
        return dict(fmt="nvfp4", M=m, N=n, K=k, out="bf16", alpha=1.0)
    if name == "nvfp4_8191x3000x5120_f32":
        return dict(fmt="nvfp4", M=8191, N=3000, K=5120, out="f32", alpha=1.0)
    if name == "nvfp4_1x28672x4096_f32":
        return dict(fmt="nvfp4", M=1, N=28672, K=4096, out="f32", alpha=1.0)
    if name == "nvfp4_8192_f32":
        # the 8192^3 GEMM in the NVFP4 format (the MXFP4 workload's values, per-16 E4M3 scales)
        return dict(fmt="nvfp4", M=8192, N=8192, K=8192, out="f32", alpha=1.0)
    raise KeyError(name)


def make_config(name: str, seed: int = 0) -> GemmInputs:
    s = config_shape(name)
    fmt, M, N, K, out, alpha = s["fmt"], s["M"], s["N"], s["K"], s["out"], s["alpha"]
    if name == "nvfp4_128x128x256_f32":
        return make_uniform_codes(fmt, M, N, K, alpha=alpha, out=out, seed=seed, name=name)
    if name.startswith("nvfp4_proj_"):
        return make_random(fmt, M, N, K, dist="normal", a_std=1.0, b_std=0.02, alpha=alpha,
                           out=out, seed=seed, name=name)
    if name in ("nvfp4_8191x3000x5120_f32", "nvfp4_1x28672x4096_f32"):
        return make_random(fmt, M, N, K, dist="t3", alpha=alpha, out=out, seed=seed, name=name)
    return make_random(fmt, M, N, K, dist="normal", alpha=alpha, out=out, seed=seed, name=name)


# ---- GEMMs with a fused epilogue ------------------------------------------------
#
# FFN projections whose epilogue is fused into the GEMM: the gate/up projection
# of a SwiGLU FFN (d_model 4096 -> 2 x 14336, gate and up weight rows
# interleaved, so D is 8192 x 14336) and a squared-ReLU up projection with a
# bias. Operands as the nvfp4_proj_* workloads (activations N(0, 1), weights
# N(0, 0.02^2), quantised blockwise); the bias is N(0, 0.5^2) in fp32.

FUSED_WORKLOADS = {
    "ffn_swiglu_nvfp4_m8192_n28672_k4096": dict(fmt="nvfp4", M=8192, N=28672, K=4096, out="bf16",
                                                act="swiglu", bias=False),
    "ffn_relu2_bias_nvfp4_m8192_n14336_k4096": dict(fmt="nvfp4", M=8192, N=14336, K=4096, out="bf16",
                                                    act="relu2", bias=True),
}


def make_bias(N: int, *, std: float = 0.5, seed: int = 0) -> np.ndarray:
    """N fp32 bias values, N(0, std^2)."""
    rng = np.random.default_rng(1000 + seed)
    return (rng.standard_normal(N) * std).astype(np.float32)


def make_fused(name: str, seed: int = 0):
    """(GemmInputs, act, bias or None) of a named fused-epilogue workload."""
    w = FUSED_WORKLOADS[name]
    inp = make_random(w["fmt"], w["M"], w["N"], w["K"], dist="normal", a_std=1.0, b_std=0.02, alpha=1.0,
                      out=w["out"], seed=seed, name=name)
    bias = make_bias(w["N"], seed=seed) if w["bias"] else None
    return inp, w["act"], bias


# ---- grouped (mixture-of-experts) GEMMs -----------------------------------------
#
# A grouped GEMM is one GEMM per expert: expert g applies its weights B_g
# (N x K) to the rows routed to it, which sit at rows offsets[g] ..
# offsets[g+1]-1 of A and D. The routed workloads below draw, for T tokens,
# `top` distinct experts per token with probability proportional to
# (rank + 1)^-0.8 over a seeded random ranking of the experts (a skewed load,
# some experts empty at small T), and sort the routed rows by expert.


@dataclasses.dataclass
class GroupedInputs:
    fmt: str
    offsets: np.ndarray      # int64 [G + 1]: group g = rows offsets[g] .. offsets[g+1]-1
    N: int
    K: int
    A: np.ndarray            # uint8 [M_total][K/2]
    sfA: np.ndarray          # uint8 [M_total][K/vec]
    B: np.ndarray            # uint8 [G*N][K/2]: B_g = rows g*N .. g*N+N-1
    sfB: np.ndarray          # uint8 [G*N][K/vec]
    alpha: float
    out: str
    name: str = ""

    @property
    def G(self) -> int:
        return len(self.offsets) - 1

    @property
    def M(self) -> int:
        return int(self.offsets[-1])

    @property
    def vec(self) -> int:
        return NV_VEC if self.fmt == "nvfp4" else MX_VEC

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


def make_grouped(fmt: str, sizes, N: int, K: int, *, a_std: float = 1.0, b_std: float = 1.0, alpha: float = 1.0,
                 out: str = "f32", seed: int = 0, name: str = "") -> GroupedInputs:
    """Group g has sizes[g] rows; values N(0, a_std^2) / N(0, b_std^2), quantised blockwise."""
    sizes = np.asarray(sizes, dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    ra = np.random.default_rng(2 * seed)
    rb = np.random.default_rng(2 * seed + 1)
    A, sfA = _quantize_rows(_normal(ra, a_std), int(offsets[-1]), K, fmt)
    B, sfB = _quantize_rows(_normal(rb, b_std), len(sizes) * N, K, fmt)
    return GroupedInputs(fmt, offsets, N, K, A, sfA, B, sfB, float(alpha), out, name)


def route_tokens(tokens: int, experts: int, top: int, seed: int = 0) -> np.ndarray:
    """Rows per expert after routing `tokens` tokens to `top` distinct experts each."""
    rng = np.random.default_rng(500 + seed)
    rank = rng.permutation(experts)
    p = (rank + 1.0) ** -0.8
    p /= p.sum()
    counts = np.zeros(experts, dtype=np.int64)
    for _ in range(tokens):
        counts[rng.choice(experts, size=top, replace=False, p=p)] += 1
    return counts


GROUPED_WORKLOADS = {
    # an expert up-projection of a squared-ReLU MoE: 64 experts, d_model 4096,
    # expert width 2048, top-8 routing; prefill (4096 tokens) and decode (64)
    "moe_nvfp4_e64_t4096_top8_n2048_k4096": dict(fmt="nvfp4", experts=64, tokens=4096, top=8, N=2048, K=4096,
                                                 out="bf16", act="relu2"),
    "moe_nvfp4_e64_t64_top8_n2048_k4096": dict(fmt="nvfp4", experts=64, tokens=64, top=8, N=2048, K=4096,
                                               out="bf16", act="relu2"),
}


def make_grouped_workload(name: str, seed: int = 0):
    """(GroupedInputs, act) of a named MoE workload."""
    w = GROUPED_WORKLOADS[name]
    sizes = route_tokens(w["tokens"], w["experts"], w["top"], seed)
    gin = make_grouped(w["fmt"], sizes, w["N"], w["K"], a_std=1.0, b_std=0.02, out=w["out"], seed=seed, name=name)
    return gin, w["act"]


# ---- raw values for the quantisation step -------------------------------------
#
# The quantiser's inputs are plain activations: seeded draws rounded to the
# input dtype (bf16 through torch's float32 -> bfloat16 cast, round to nearest
# even). Nothing here quantises them.

QUANT_WORKLOADS = {
    # the A-side activations of the 8192 x 14336 x 4096 and 8192 x 4096 x 14336
    # projections, and of the 8192^3 MXFP4 GEMM
    "quant_nvfp4_8192x4096_bf16": dict(fmt="nvfp4", rows=8192, K=4096, dtype="bf16"),
    "quant_nvfp4_8192x14336_bf16": dict(fmt="nvfp4", rows=8192, K=14336, dtype="bf16"),
    "quant_mxfp4_8192x8192_bf16": dict(fmt="mxfp4", rows=8192, K=8192, dtype="bf16"),
    "quant_nvfp4_8192x4096_f32": dict(fmt="nvfp4", rows=8192, K=4096, dtype="f32"),
}


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (torch's cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def make_values(rows: int, K: int, *, dist: str = "normal", std: float = 1.0, dtype: str = "bf16",
                seed: int = 0) -> np.ndarray:
    """rows x K activations: float32 values, or uint16 bf16 bit patterns for dtype "bf16"."""
    rng = np.random.default_rng(2 * seed)
    if dist == "normal":
        x = rng.standard_normal((rows, K), dtype=np.float32) * np.float32(std)
    elif dist == "t3":
        x = (rng.standard_t(3, (rows, K)) * std).astype(np.float32)
    else:
        raise ValueError(dist)
    return x if dtype == "f32" else to_bf16_bits(x)


def make_quant_workload(name: str, seed: int = 0):
    """(fmt, X) of a named quantisation workload."""
    w = QUANT_WORKLOADS[name]
    return w["fmt"], make_values(w["rows"], w["K"], dtype=w["dtype"], seed=seed)
