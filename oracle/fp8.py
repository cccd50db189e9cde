"""FP8 (E4M3) block quantization, incoherent processing, and the reference
result of the FP8 forward -- TEST INFRASTRUCTURE ONLY.

Like the rest of ``oracle/``, only the test suite, the smoke check and the
benchmark's CPU legs use this module; the library never does, and nothing here
is shared with the CUDA path.

The method ("FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화 분석",
youngju.dev, section 9.2, item 3, FP8 low-precision support) names two steps:

* block quantization -- every block of the input keeps its own scale factor,
  so that each block's dynamic range survives the 8-bit format;
* incoherent processing -- the inputs are multiplied by a random orthogonal
  matrix before quantization, which spreads outlier values over all
  coordinates.

Readings taken where the page is silent.  The quantization readings fix the
codes and scales, which are compared bit for bit; the bound on the forward's
result follows from the E4M3 format alone:

* the format is E4M3 (sign, 4 exponent bits with bias 7, 3 mantissa bits, no
  infinities; normal values 2^-6 .. 448, subnormals k * 2^-9);
* a block is 128 consecutive rows of one head for Q and K, and the whole head
  for V; s = amax / 448 in fp32 (IEEE division), s = 1 for an all-zero block;
* a value x is coded as E4M3(x * fp32(1 / s)): the reciprocal and the product
  are fp32 operations rounded to nearest even, the conversion rounds to
  nearest even and saturates at +-448;
* the random orthogonal matrix is M = diag(sigma) H / sqrt(d), with sigma a
  vector of d random signs (an input, drawn by the seeded generators) and H
  the Sylvester-Hadamard matrix; it is applied to the rows of Q and of K only,
  which leaves Q K^T unchanged because M M^T = I.  The product with H is taken
  as the fast Walsh-Hadamard butterfly in fp32 (stages h = 1, 2, 4, ..., d/2,
  each pair (a, b) becoming (a + b, a - b)), without the 1/sqrt(d); that
  factor, fp32(1/sqrt(d)), multiplies the block's scale instead (an fp32
  product), so that codes times scales stand for the rows of Q M and K M;
* the FP8 path aims at exact attention on the dequantized inputs (codes times
  scales), with the softmax weights P V multiplies also held in FP8.  The
  plainest reading is that each weight p in [0, 1] (relative to its row's
  maximum) is replaced by an E4M3 value.  The format alone then bounds the
  change of a weight: at or above the smallest normal 2^-6 the three mantissa
  bits give a relative error <= 2^-4; below it the subnormal step 2^-9 gives
  an absolute error <= 2^-10.  An implementation that rounds p * 2^e for some
  0 <= e <= 8 (any such scaling keeps the largest weight below 448) and
  divides by 2^e again only shrinks the absolute part, so the bound holds for
  every such choice.  `forward_fp8_reference` turns it into a bound per output
  element.
"""
from __future__ import annotations

import numpy as np

import oracle

E4M3_MAX = 448.0
BLOCK_ROWS = 128


def e4m3_round(v) -> np.ndarray:
    """Nearest E4M3 value (ties to even, saturating at +-448) of each value,
    returned exactly as float64."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                       # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)                # binade exponent; subnormals share -6
    quantum = np.ldexp(1.0, (e - 3).astype(np.int64))   # 3 mantissa bits
    r = np.round(a / quantum) * quantum       # np.round: half to even
    r = np.minimum(r, E4M3_MAX)
    r = np.where(a == 0, 0.0, r)
    return np.copysign(r, v)


def hadamard_rows(x, signs) -> np.ndarray:
    """(x * signs) H along the last axis, as the fp32 butterfly: stages
    h = 1, 2, ..., d/2, each pair (x[i], x[i+h]) with i & h == 0 replaced by
    (x[i] + x[i+h], x[i] - x[i+h]).  No normalisation."""
    y = _f32(x) * _f32(signs)
    d = y.shape[-1]
    lead = y.shape[:-1]
    h = 1
    while h < d:
        z = y.reshape(*lead, d // (2 * h), 2, h)
        a, b = z[..., 0, :], z[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(*lead, d)
        h *= 2
    return y


def _f32(x) -> np.ndarray:
    """fp32 numpy copy of an array or CPU tensor (bf16 and fp16 widen exactly)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float32)


def _scale_of(amax) -> np.ndarray:
    amax = np.asarray(amax, dtype=np.float32)
    s = amax / np.float32(E4M3_MAX)
    return np.where(amax == 0, np.float32(1.0), s).astype(np.float32)


def _codes(x32, s) -> np.ndarray:
    inv = (np.float32(1.0) / s).astype(np.float32)
    return e4m3_round((x32 * inv).astype(np.float32))


def _rotation_factor(d: int) -> np.float32:
    return np.float32(1.0 / np.sqrt(float(d)))


def quantize_rows(x, signs=None):
    """Q or K [B,H,N,d] -> (codes as float64 [B,H,N,d], dequantization scales
    fp32 [B,H,ceil(N/128)]), one scale per 128-row block; with ``signs`` the
    rows are first multiplied by the random orthogonal matrix."""
    x32 = _f32(x)
    if signs is not None:
        x32 = hadamard_rows(x32, signs)
    B, H, N, d = x32.shape
    nb = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    scales = np.empty((B, H, nb), dtype=np.float32)
    codes = np.empty(x32.shape, dtype=np.float64)
    for blk in range(nb):
        sl = slice(blk * BLOCK_ROWS, min(N, (blk + 1) * BLOCK_ROWS))
        s = _scale_of(np.abs(x32[:, :, sl]).max(axis=(2, 3)))
        codes[:, :, sl] = _codes(x32[:, :, sl], s[:, :, None, None])
        scales[:, :, blk] = (s * _rotation_factor(d)).astype(np.float32) if signs is not None else s
    return codes, scales


def quantize_heads(x):
    """V [B,H,N,d] -> (codes [B,H,N,d], scales fp32 [B,H]): one scale per head."""
    x32 = _f32(x)
    s = _scale_of(np.abs(x32).max(axis=(2, 3)))
    return _codes(x32, s[:, :, None, None]), s


def dequantize_rows(codes, scales) -> np.ndarray:
    N = codes.shape[2]
    rows = np.arange(N) // BLOCK_ROWS
    return codes * scales[:, :, rows][..., None].astype(np.float64)


def dequantized(q, k, v, signs=None):
    """The FP8 path's inputs as float64: Q M, K M (M = I without ``signs``) and
    V, each as codes times block scales."""
    qc, qs = quantize_rows(q, signs)
    kc, ks = quantize_rows(k, signs)
    vc, vs = quantize_heads(v)
    return dequantize_rows(qc, qs), dequantize_rows(kc, ks), vc * vs[:, :, None, None].astype(np.float64)


# Change of one softmax weight p in [0, 1] when it is held as an E4M3 value,
# from the format alone: relative 2^-4 (half the step of 3 mantissa bits) for
# normal values, absolute 2^-10 (half the subnormal step 2^-9) below 2^-6.
P_REL = 2.0 ** -4
P_ABS = 2.0 ** -10
OUT_REL = 2.0 ** -8      # bf16 output: half an ulp is 2^-9 relative; doubled


def forward_fp8_reference(q, k, v, scale: float, causal: bool, signs=None, rows=None,
                          p_rel: float = P_REL, p_abs: float = P_ABS):
    """(O, LSE, bound, sigma) for the FP8 forward.

    O and LSE are exact attention (float64) on the dequantized inputs.  For each
    output element, ``bound`` is
        sum_j max(p_rel p_j, p_abs) |v_j| / l + OUT_REL |O|  (+ 1e-5),
    with p_j = exp(s_j - max_j s_j) and l = sum_j p_j: what E4M3 weights and a
    bf16 output can move the result at most (by default the format's own
    limits, P_REL and P_ABS).  ``sigma`` is the standard deviation of that
    error if each weight's rounding error is an independent, zero-mean value
    no larger than the bound allows (uniform: bound / sqrt 3), for a
    statistical check of the typical error.  ``rows`` restricts all four to
    the given query rows."""
    qd, kd, vd = dequantized(q, k, v, signs)
    B, H, N, d = qd.shape
    rows = np.arange(N) if rows is None else np.asarray(rows)
    o, lse = oracle.attention_forward_rows(qd, kd, vd, rows, scale, causal)
    bound = np.zeros((B, H, len(rows), d))
    var = np.zeros((B, H, len(rows), d))
    key = np.arange(N)
    for b in range(B):
        for h in range(H):
            s = scale * (qd[b, h, rows] @ kd[b, h].T)
            if causal:
                s = np.where(key[None, :] <= rows[:, None], s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            l = p.sum(axis=1, keepdims=True)
            w = np.where(np.isfinite(s), np.maximum(p_rel * p, p_abs), 0.0)
            bound[b, h] = (w @ np.abs(vd[b, h])) / l
            var[b, h] = ((w * w / 3.0) @ (vd[b, h] ** 2)) / (l * l)
    bound += OUT_REL * np.abs(o) + 1e-5
    sigma = np.sqrt(var + (OUT_REL * o) ** 2 / 3.0) + 1e-6
    return o, lse, bound, sigma
