"""Seeded synthetic inputs for the fused (add +) RMSNorm + group-quant path.

This module is shared by the CPU oracle's tests, the CUDA path's tests and the
benchmark, and therefore holds none of the method's arithmetic: it only draws
numbers and rounds them once to bf16 (through torch's own cast) to make the
inputs.

Generator (stated here so that it can be re-implemented anywhere):

* counter-based splitmix64: the k-th 64-bit word of stream ``key`` is
  ``mix(key + (k + 1) * 0x9E3779B97F4A7C15)`` with the splitmix64 finaliser
  ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
  z ^= z >> 31`` (all mod 2**64);
* a stream's key is ``mix(seed * 0x100000001B3 + tensor_id)``;
* a uniform in (0, 1] is ``((word >> 11) + 1) * 2**-53``;
* a standard normal is Box-Muller's cosine branch on words 2i and 2i+1:
  ``sqrt(-2 ln u1) * cos(2 pi u2)``, evaluated in float64;
* N(mu, v) is read with v the VARIANCE (so "N(0,4)" has sigma 2), uniformly
  for every tensor;
* Student-t with nu = 3 is ``Z / sqrt((Z1^2 + Z2^2 + Z3^2) / 3)`` from four
  independent normal streams;
* outlier channels: 1 % of the H channels (72 of 7168), chosen per seed as
  the indices of the smallest keys of a uniform stream, are multiplied by 20
  before the bf16 rounding.

The workloads mirror the DeepSeek-V3/R1 activations the pages fuse: hidden
size 7168 with 1x128 FP8 groups for the input RMSNorm (page "fused rmsnorm
quant fp8 work", Motivation), MLA q_a / kv_a latents of 1536 / 512 for the
q/k latent norm (same page, Modifications, "q, k_"; ATOM PR "Support
input_rmsnorm_quant & qknorm_quant fused", Technical Details), decode batch
sizes up to 256 and chunked prefill up to 16384 tokens (sglang PR "[AMD] Add
fused all-reduce RMSNorm per-group quant", server command).
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20

# Stable tensor identifiers: each tensor of a workload draws its own stream.
TENSOR_IDS = {
    "x": 1, "residual": 2, "gamma": 3, "outlier": 4,
    "q_a": 5, "kv_a": 6, "gamma_q": 7, "gamma_kv": 8,
    "chi1": 9, "chi2": 10, "chi3": 11,
    "w_codes": 12, "w_scales": 13,
}


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor: str) -> np.uint64:
    base = np.array([(seed * 0x100000001B3 + TENSOR_IDS[tensor]) % (1 << 64)],
                    dtype=np.uint64)
    return _mix(base)[0]


def words(key: np.uint64, start: int, count: int) -> np.ndarray:
    """64-bit words ``start .. start+count-1`` of the stream ``key``."""
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + k * _GOLDEN)


def uniforms(key: np.uint64, start: int, count: int) -> np.ndarray:
    w = words(key, start, count)
    return ((w >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)


def normals(seed: int, tensor: str, n: int) -> np.ndarray:
    """``n`` standard normals (float64) of stream (seed, tensor)."""
    key = stream_key(seed, tensor)
    out = np.empty(n, dtype=np.float64)

    def fill(s: int) -> None:
        c = min(_CHUNK, n - s)
        u = uniforms(key, 2 * s, 2 * c)
        u1, u2 = u[0::2], u[1::2]
        out[s:s + c] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)

    starts = range(0, n, _CHUNK)
    if n <= _CHUNK:
        for s in starts:
            fill(s)
    else:
        # numpy ufuncs release the GIL, so chunks fill in parallel threads;
        # each chunk's values depend only on its counters.
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, starts))
    return out


def to_bf16(a: np.ndarray, shape) -> torch.Tensor:
    """Round float values to bf16 with torch's cast (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).reshape(shape).to(torch.bfloat16)


def gaussian_bf16(seed: int, tensor: str, shape, mean=0.0, var=1.0) -> torch.Tensor:
    n = int(np.prod(shape))
    v = normals(seed, tensor, n) * math.sqrt(var) + mean
    return to_bf16(v, shape)


def student_t3_bf16(seed: int, tensor: str, shape) -> torch.Tensor:
    n = int(np.prod(shape))
    z = normals(seed, tensor, n)
    chi = normals(seed, "chi1", n) ** 2 + normals(seed, "chi2", n) ** 2 + normals(seed, "chi3", n) ** 2
    return to_bf16(z / np.sqrt(chi / 3.0), shape)


def outlier_channels(seed: int, H: int, frac: float = 0.01) -> np.ndarray:
    n_out = max(1, int(round(H * frac)))
    keys = uniforms(stream_key(seed, "outlier"), 0, H)
    return np.sort(np.argsort(keys, kind="stable")[:n_out])


def hidden_with_outliers_bf16(seed: int, shape, scale: float = 20.0) -> torch.Tensor:
    M, H = shape
    v = normals(seed, "x", M * H).reshape(M, H)
    v[:, outlier_channels(seed, H)] *= scale
    return to_bf16(v, shape)


def mxfp4_weights(seed: int, N: int, K: int, scale_lo: int = 118, scale_hi: int = 122):
    """Synthetic MXFP4 weights of a linear layer [N, K]: packed codes
    (uint8 [N, K/2], every nibble uniform over the 16 E2M1 codes: byte j of
    the stream is word j // 8's byte j % 8) and E8M0 scale bytes (uint8
    [N, K/32], uniform in [scale_lo, scale_hi), i.e. 2^-9 .. 2^-6 by default,
    the size of trained weights' block scales). The values are drawn, not
    quantised from anything: the GEMM consumes codes and scales as given."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    nb = N * K // 2
    w = words(stream_key(seed, "w_codes"), 0, (nb + 7) // 8)
    codes = w.astype("<u8").view(np.uint8)[:nb].reshape(N, K // 2).copy()
    ns = N * K // 32
    sw = words(stream_key(seed, "w_scales"), 0, ns)
    scales = (scale_lo + (sw % np.uint64(scale_hi - scale_lo))).astype(np.uint8).reshape(N, K // 32)
    return torch.from_numpy(codes), torch.from_numpy(scales)


@dataclass
class Workload:
    """One named workload: its sizes, and how its tensors are drawn."""
    name: str
    kind: str                  # "fp8", "qknorm", "mxfp4"
    M: int
    H: int = 0
    Hq: int = 0
    Hkv: int = 0
    seed: int = 0
    group: int = 128
    eps: float = 1e-6
    residual: bool = True
    keep_bf16: bool = False
    scale_layout: str = "row"  # "row": [M, H/G]; "col": [H/G, M]
    x_dist: str = "normal"     # "normal", "outliers", "student_t3"
    res_var: float = 1.0
    kv_var: float = 1.0
    notes: dict = field(default_factory=dict)


# The five workloads, 0..4: tiny, decode, prefill (the headline), MLA latent
# norm, MXFP4.
WORKLOADS = {
    "tiny": Workload("tiny", "fp8", M=4, H=256, seed=0, x_dist="normal", res_var=1.0),
    "decode": Workload("decode", "fp8", M=64, H=7168, seed=1, x_dist="outliers",
                       res_var=4.0, scale_layout="col"),
    "prefill": Workload("prefill", "fp8", M=16384, H=7168, seed=2, x_dist="outliers",
                        res_var=4.0, keep_bf16=True),
    "qknorm": Workload("qknorm", "qknorm", M=8192, Hq=1536, Hkv=512, seed=3,
                       residual=False, kv_var=2.0),
    "mxfp4": Workload("mxfp4", "mxfp4", M=8192, H=7168, seed=4, group=32,
                      x_dist="student_t3", res_var=1.0),
}
WORKLOAD_ORDER = ["tiny", "decode", "prefill", "qknorm", "mxfp4"]


def make_inputs(w: Workload, M: int | None = None) -> dict:
    """CPU bf16 tensors for workload ``w``; ``M`` overrides the row count.

    Element (m, h) is word ``m*H + h`` of its stream, so ``M`` smaller than
    the workload's row count gives exactly the first ``M`` rows of the full
    draw, and a larger ``M`` extends it.
    """
    M = w.M if M is None else M
    out = {}
    if w.kind == "qknorm":
        out["q_a"] = gaussian_bf16(w.seed, "q_a", (M, w.Hq))
        out["kv_a"] = gaussian_bf16(w.seed, "kv_a", (M, w.Hkv), var=w.kv_var)
        out["gamma_q"] = gaussian_bf16(w.seed, "gamma_q", (w.Hq,), mean=1.0, var=0.1)
        out["gamma_kv"] = gaussian_bf16(w.seed, "gamma_kv", (w.Hkv,), mean=1.0, var=0.1)
        return out
    if w.x_dist == "outliers":
        out["x"] = hidden_with_outliers_bf16(w.seed, (M, w.H))
    elif w.x_dist == "student_t3":
        out["x"] = student_t3_bf16(w.seed, "x", (M, w.H))
    else:
        out["x"] = gaussian_bf16(w.seed, "x", (M, w.H))
    if w.residual:
        out["residual"] = gaussian_bf16(w.seed, "residual", (M, w.H), var=w.res_var)
    out["gamma"] = gaussian_bf16(w.seed, "gamma", (w.H,), mean=1.0, var=0.1)
    return out


def random_bf16(seed: int, shape, var: float = 1.0, tensor: str = "x") -> torch.Tensor:
    """Plain N(0, var) bf16 tensor for ad-hoc shapes (edge-case tests)."""
    return gaussian_bf16(seed, tensor, shape, var=var)
