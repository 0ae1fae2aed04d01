"""Seeded synthetic inputs for the routed-MoE layer (weights, router, tokens).

Every array here is a pure function of (seed, identifiers) through the
counter-based SplitMix64 streams of ``gen.c``. The module holds the input
recipe only -- distributions, storage formats and shapes -- and none of the
method's arithmetic: the oracle and the CUDA library each read these bytes
with their own code.

Input recipe (shapes and distributions of the workloads):
  * 4-bit expert matrices, affine, group 64 along the input dimension:
    code ~ U{0..15}; scale = fp16(U(0.002, 0.02)) rounded to nearest even;
    bias = -8 * scale (exact in fp16), so the weight is (code - 8) * scale.
  * Router weights: fp32 N(0, sd = 0.02) [E][H]; for the 8-bit router the same
    fp32 draw is encoded affine group-64 (min/max per group, fp16 scale/bias).
  * Router bias (skewed popularity): p_e proportional to r_e ** -1.1 with r a
    seeded permutation of 1..E, normalised; bias_e = ln p_e (fp32).
  * Activations: fp32 N(0, 1), then rounded to bfloat16 for bf16 I/O.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libseeded_inputs.so")
_lock = threading.Lock()
_lib = None

# stream tags
TAG_ROUTER = 1
TAG_EXPERT_CODES = 2
TAG_EXPERT_SCALE = 3
TAG_TOKENS = 4
TAG_BIAS_PERM = 5
TAG_SCORE_BIAS = 6
TAG_OUTLIER_POS = 7

MAT_GATE, MAT_UP, MAT_DOWN = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile gen.c into a shared library (gcc, OpenMP when available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.si_key.restype = u64
            lib.si_key.argtypes = [u64, u64, u64, u64, u64]
            lib.si_fill_u64.argtypes = [u64, u64, u64, vp]
            lib.si_fill_bytes.argtypes = [u64, u64, vp]
            lib.si_fill_f16_uniform.argtypes = [u64, u64, dbl, dbl, vp]
            lib.si_fill_normal_f32.argtypes = [u64, u64, dbl, vp]
            lib.si_fill_normal_bf16.argtypes = [u64, u64, dbl, vp]
            lib.si_permutation.argtypes = [u64, i64, vp]
            lib.si_fill_normal_outliers.argtypes = [u64, u64, u64, u64, dbl, vp, vp]
            lib.si_encode_q8g64.argtypes = [vp, i64, i64, vp, vp, vp]
            lib.si_f64_to_f16.restype = ctypes.c_uint16
            lib.si_f64_to_f16.argtypes = [dbl]
            lib.si_f32_to_bf16.restype = ctypes.c_uint16
            lib.si_f32_to_bf16.argtypes = [ctypes.c_float]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def key(seed: int, tag: int, a: int = 0, b: int = 0, c: int = 0) -> int:
    m = (1 << 64) - 1
    return int(_load().si_key(seed & m, tag & m, a & m, b & m, c & m))


def stream_u64(k: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _load().si_fill_u64(k, start, n, _ptr(out))
    return out


def stream_bytes(k: int, n: int, out: np.ndarray | None = None) -> np.ndarray:
    if out is None:
        out = np.empty(n, np.uint8)
    assert out.dtype == np.uint8 and out.size == n
    _load().si_fill_bytes(k, n, _ptr(out))
    return out


def f16_uniform(k: int, n: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, np.uint16)
    _load().si_fill_f16_uniform(k, n, lo, hi, _ptr(out))
    return out


def normal_f32(k: int, n: int, sd: float = 1.0) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load().si_fill_normal_f32(k, n, sd, _ptr(out))
    return out


def normal_bf16(k: int, n: int, sd: float = 1.0) -> np.ndarray:
    """bfloat16 bit patterns (uint16) of N(0, sd) draws rounded to nearest even."""
    out = np.empty(n, np.uint16)
    _load().si_fill_normal_bf16(k, n, sd, _ptr(out))
    return out


def permutation(k: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int64)
    _load().si_permutation(k, n, _ptr(out))
    return out


def f64_to_f16_bits(v: float) -> int:
    return int(_load().si_f64_to_f16(float(v)))


def f32_to_bf16_bits(v: float) -> int:
    return int(_load().si_f32_to_bf16(float(v)))


def encode_q8g64(w: np.ndarray):
    """Affine group-64 8-bit encoding of a float32 [N][K] matrix -> (codes, scale, bias)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % 64 == 0
    codes = np.empty((N, K), np.uint8)
    scale = np.empty((N, K // 64), np.uint16)
    bias = np.empty((N, K // 64), np.uint16)
    _load().si_encode_q8g64(_ptr(w), N, K, _ptr(codes), _ptr(scale), _ptr(bias))
    return codes, scale, bias


# ---------------------------------------------------------------------------
# canonical containers
# ---------------------------------------------------------------------------

@dataclass
class QMat:
    """Affine group-64 matrix [N][K] in canonical storage.

    codes: uint8 [N][K/2] (4-bit, low nibble = even k), [N][K/4] (2-bit,
    element k at bits 2 (k % 4) of byte k/4) or [N][K] (8-bit);
    scale, bias: uint16 binary16 bit patterns [N][K/64].
    """
    codes: np.ndarray
    scale: np.ndarray
    bias: np.ndarray
    bits: int
    N: int
    K: int

    @property
    def nbytes(self) -> int:
        return self.codes.nbytes + self.scale.nbytes + self.bias.nbytes


@dataclass
class Expert:
    gate: QMat
    up: QMat
    down: QMat

    @property
    def nbytes(self) -> int:
        return self.gate.nbytes + self.up.nbytes + self.down.nbytes


@dataclass
class Router:
    """fp32 [E][H] (``w``) or 8-bit affine group-64 (``q``)."""
    fmt: str                      # "f32" or "q8g64"
    w: np.ndarray | None = None   # float32 [E][H]
    q: QMat | None = None

    @property
    def nbytes(self) -> int:
        return self.w.nbytes if self.fmt == "f32" else self.q.nbytes


@dataclass(frozen=True)
class LayerSpec:
    hidden: int
    inter: int
    n_experts: int
    top_k: int = 8
    n_shared: int = 1
    router_fmt: str = "f32"       # "f32" | "q8g64"
    act: str = "bf16"             # "bf16" | "f32"
    zipf_alpha: float | None = None   # router bias from skewed popularity
    router_sd: float = 0.02
    router_score: str = "softmax"     # "softmax" | "sigmoid"
    routed_scaling: float = 1.0       # sigmoid scoring: multiplies the routing weights
    score_bias_sd: float | None = None   # sigmoid scoring: selection bias N(0, sd) per expert
    expert_bits: int = 4              # 4 (q4g64) or 2 (q2g64) expert codes

    def expert_bytes(self) -> int:
        """Canonical bytes of one group-64 expert: 3*H*I*(bits/8 + 4/64)."""
        w = 3 * self.hidden * self.inter
        return w * self.expert_bits // 8 + 2 * 2 * (w // 64)


def gen_qmat4(seed: int, layer: int, expert: int, mat: int, N: int, K: int) -> QMat:
    assert K % 64 == 0 and N > 0
    codes = stream_bytes(key(seed, TAG_EXPERT_CODES, layer, expert, mat), N * K // 2).reshape(N, K // 2)
    scale = f16_uniform(key(seed, TAG_EXPERT_SCALE, layer, expert, mat), N * K // 64, 0.002, 0.02)
    # bias = -8 * scale is exact in binary16 for these magnitudes: flip the sign
    # bit and add 3 to the exponent field (all scales are normal numbers).
    assert np.all(((scale >> 10) & 0x1F) >= 1) and np.all(((scale >> 10) & 0x1F) <= 27)
    bias = (scale + np.uint16(3 << 10)) | np.uint16(0x8000)
    return QMat(codes, scale.reshape(N, K // 64), bias.reshape(N, K // 64), 4, N, K)


def gen_qmat2(seed: int, layer: int, expert: int, mat: int, N: int, K: int) -> QMat:
    """2-bit codes uniform on 0..3 (four per seeded byte), scales as for 4 bits,
    bias = -2 * scale (exact in binary16: sign flip, exponent + 1)."""
    assert K % 64 == 0 and N > 0
    codes = stream_bytes(key(seed, TAG_EXPERT_CODES, layer, expert, mat), N * K // 4).reshape(N, K // 4)
    scale = f16_uniform(key(seed, TAG_EXPERT_SCALE, layer, expert, mat), N * K // 64, 0.002, 0.02)
    assert np.all(((scale >> 10) & 0x1F) >= 1) and np.all(((scale >> 10) & 0x1F) <= 29)
    bias = (scale + np.uint16(1 << 10)) | np.uint16(0x8000)
    return QMat(codes, scale.reshape(N, K // 64), bias.reshape(N, K // 64), 2, N, K)


def gen_expert(seed: int, layer: int, expert: int, spec: LayerSpec) -> Expert:
    """Expert ``expert`` of layer ``layer``; index ``n_experts`` is the shared expert."""
    H, I = spec.hidden, spec.inter
    gen = gen_qmat2 if spec.expert_bits == 2 else gen_qmat4
    return Expert(gate=gen(seed, layer, expert, MAT_GATE, I, H),
                  up=gen(seed, layer, expert, MAT_UP, I, H),
                  down=gen(seed, layer, expert, MAT_DOWN, H, I))


def gen_router(seed: int, layer: int, spec: LayerSpec) -> Router:
    E, H = spec.n_experts, spec.hidden
    w = normal_f32(key(seed, TAG_ROUTER, layer), E * H, spec.router_sd).reshape(E, H)
    if spec.router_fmt == "f32":
        return Router("f32", w=w)
    if spec.router_fmt == "q8g64":
        c, s, b = encode_q8g64(w)
        return Router("q8g64", q=QMat(c, s, b, 8, E, H))
    raise ValueError(spec.router_fmt)


def gen_router_bias(seed: int, layer: int, spec: LayerSpec) -> np.ndarray | None:
    """ln p_e with p_e proportional to rank_e ** -alpha (rank a seeded permutation of 1..E);
    with sigmoid scoring and score_bias_sd, a seeded N(0, sd) bias per expert instead."""
    if spec.router_score == "sigmoid" and spec.score_bias_sd is not None:
        return normal_f32(key(seed, TAG_SCORE_BIAS, layer), spec.n_experts, spec.score_bias_sd)
    if spec.zipf_alpha is None:
        return None
    E = spec.n_experts
    rank = permutation(key(seed, TAG_BIAS_PERM, layer), E) + 1
    p = rank.astype(np.float64) ** (-spec.zipf_alpha)
    p /= p.sum()
    return np.log(p).astype(np.float32)


def gen_tokens(seed: int, t0: int, T: int, spec: LayerSpec) -> np.ndarray:
    """Activations for tokens t0..t0+T-1: float32 [T][H] (f32 I/O) or
    bfloat16 bit patterns uint16 [T][H] (bf16 I/O). Token t uses stream (seed, x, t)."""
    H = spec.hidden
    if spec.act == "f32":
        return np.stack([normal_f32(key(seed, TAG_TOKENS, t), H, 1.0) for t in range(t0, t0 + T)])
    return np.stack([normal_bf16(key(seed, TAG_TOKENS, t), H, 1.0) for t in range(t0, t0 + T)])


def gen_tokens_scaled(seed: int, t0: int, T: int, spec: LayerSpec, sd: float) -> np.ndarray:
    """Like gen_tokens, with N(0, sd) activations (the same streams times sd,
    rounded once): sd far from 1 gives tokens of tiny or huge magnitude."""
    H = spec.hidden
    if spec.act == "f32":
        return np.stack([normal_f32(key(seed, TAG_TOKENS, t), H, sd) for t in range(t0, t0 + T)])
    return np.stack([normal_bf16(key(seed, TAG_TOKENS, t), H, sd) for t in range(t0, t0 + T)])


def gen_tokens_outliers(seed: int, t0: int, T: int, spec: LayerSpec, factor: float,
                        group: int = 32) -> np.ndarray:
    """Like gen_tokens, with one outlier channel in every run of `group`
    activations (a seeded position per run, value times `factor`): the wide
    dynamic range within a run that real activations show."""
    H = spec.hidden
    rows = []
    for t in range(t0, t0 + T):
        f32 = np.empty(H, np.float32)
        b16 = np.empty(H, np.uint16)
        _load().si_fill_normal_outliers(key(seed, TAG_TOKENS, t), key(seed, TAG_OUTLIER_POS, t), H, group,
                                        float(factor), _ptr(f32), _ptr(b16))
        rows.append(f32 if spec.act == "f32" else b16)
    return np.stack(rows)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Layer:
    spec: LayerSpec
    router: Router
    experts: list            # n_experts routed Expert objects
    shared: Expert | None
    router_bias: np.ndarray | None = None
    seed: int = 0
    layer: int = 0


def gen_layer(seed: int, layer: int, spec: LayerSpec) -> Layer:
    experts = [gen_expert(seed, layer, e, spec) for e in range(spec.n_experts)]
    shared = gen_expert(seed, layer, spec.n_experts, spec) if spec.n_shared else None
    return Layer(spec, gen_router(seed, layer, spec), experts, shared,
                 gen_router_bias(seed, layer, spec), seed, layer)


# ---------------------------------------------------------------------------
# named workloads
# ---------------------------------------------------------------------------

CONFIGS = {
    # tiny layer for the oracle: H512 I256 E32, fp32 router and fp32 I/O
    "tiny": LayerSpec(hidden=512, inter=256, n_experts=32, act="f32"),
    # GLM-scale single-layer decode: H6144 I2048 E256, bf16 activations
    "glm_decode": LayerSpec(hidden=6144, inter=2048, n_experts=256),
    # the same shape with 2-bit experts
    "glm_decode_q2": LayerSpec(hidden=6144, inter=2048, n_experts=256, expert_bits=2),
    # Gemma-style decode: H2816 I704 E128, 8-bit group-64 router
    "gemma_decode": LayerSpec(hidden=2816, inter=704, n_experts=128, router_fmt="q8g64"),
    # 128-token prefill chunk on the GLM-scale layer with skewed popularity bias
    "glm_prefill": LayerSpec(hidden=6144, inter=2048, n_experts=256, zipf_alpha=1.1),
}
