"""Seeded synthetic inputs for the block-quantized matvec workloads.

This module only draws random bytes and values and writes them into the
byte positions the three block formats reserve for them.  It holds none of
the method's arithmetic (no unpacking, no dequantization, no dot product),
so both the CPU oracle and the CUDA library can be fed from it.

Formats (GGUF-style, little-endian):
  Q4_K  144 B / 256 weights: fp16 d @0, fp16 dmin @2, 12 B packed 6-bit
        scales/mins @4, 128 B of 4-bit quants @16.
  Q6_K  210 B / 256 weights: 128 B low nibbles @0, 64 B high 2-bit @128,
        16 int8 scales @192, fp16 d @208.
  Q8_0   34 B /  32 weights: fp16 d @0, 32 int8 quants @2.

Value distributions follow the workload descriptions of the larql
architecture-shader map (Gemma-3 4B, Llama, Mixtral tables):
  * Q4_K quants and the 12 scale/min bytes uniform random bytes (the 6-bit
    scales and mins are then uniform on 0..63, because the 12 bytes are a
    bijective packing of sixteen 6-bit fields); d, dmin fp16 of U[1e-4, 2e-3].
  * Q6_K quant bytes uniform; int8 scales uniform on [-63, 63]; d as above.
  * Q8_0 int8 quants uniform on [-127, 127]; d as above.
  * activations fp32 N(0, 1); router fp32 N(0, 0.02).
"""
from __future__ import annotations

import numpy as np

Q4_K, Q6_K, Q8_0 = 1, 2, 3
FMT_NAMES = {Q4_K: "Q4_K", Q6_K: "Q6_K", Q8_0: "Q8_0"}
BLOCK_BYTES = {Q4_K: 144, Q6_K: 210, Q8_0: 34}
BLOCK_ELEMS = {Q4_K: 256, Q6_K: 256, Q8_0: 32}

D_LO, D_HI = 1e-4, 2e-3


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def row_bytes(fmt: int, cols: int) -> int:
    assert cols % BLOCK_ELEMS[fmt] == 0
    return cols // BLOCK_ELEMS[fmt] * BLOCK_BYTES[fmt]


def _fp16_field(g: np.random.Generator, shape) -> np.ndarray:
    """uniform draws rounded to fp16 by numpy, returned as their two LE bytes."""
    v = g.uniform(D_LO, D_HI, size=shape).astype(np.float16)
    return v.view(np.uint8).reshape(*shape, 2)


def q4k(g: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    nb = cols // 256
    blk = g.integers(0, 256, size=(rows, nb, 144), dtype=np.uint8)
    blk[..., 0:2] = _fp16_field(g, (rows, nb))
    blk[..., 2:4] = _fp16_field(g, (rows, nb))
    return blk.reshape(rows, nb * 144)


def q6k(g: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    nb = cols // 256
    blk = g.integers(0, 256, size=(rows, nb, 210), dtype=np.uint8)
    sc = g.integers(-63, 64, size=(rows, nb, 16), dtype=np.int16).astype(np.int8)
    blk[..., 192:208] = sc.view(np.uint8)
    blk[..., 208:210] = _fp16_field(g, (rows, nb))
    return blk.reshape(rows, nb * 210)


def q8_0(g: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    nb = cols // 32
    blk = np.empty((rows, nb, 34), dtype=np.uint8)
    blk[..., 0:2] = _fp16_field(g, (rows, nb))
    q = g.integers(-127, 128, size=(rows, nb, 32), dtype=np.int16).astype(np.int8)
    blk[..., 2:34] = q.view(np.uint8)
    return blk.reshape(rows, nb * 34)


def weights(g: np.random.Generator, fmt: int, rows: int, cols: int) -> np.ndarray:
    return {Q4_K: q4k, Q6_K: q6k, Q8_0: q8_0}[fmt](g, rows, cols)


def activations(g: np.random.Generator, batch: int, cols: int) -> np.ndarray:
    return g.standard_normal((batch, cols), dtype=np.float32)


def rms_normed(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """unit-gain RMS normalisation of generated activations (input preparation
    for the lm_head workload; not a step of the quantized path)."""
    x64 = x.astype(np.float64)
    return (x64 / np.sqrt(np.mean(x64 * x64, axis=-1, keepdims=True) + eps)).astype(np.float32)


def router(g: np.random.Generator, n_experts: int, hidden: int, std: float = 0.02) -> np.ndarray:
    return (g.standard_normal((n_experts, hidden), dtype=np.float32) * np.float32(std)).astype(np.float32)


# ---------------------------------------------------------------------------
# Named workloads (shapes of the pages' models; every byte drawn from `seed`).
# ---------------------------------------------------------------------------

def matvec_small(seed: int = 0):
    """single Q4_K matvec, batch 1: 256 x 2560."""
    g = rng(seed)
    W = q4k(g, 256, 2560)
    x = activations(g, 1, 2560)
    return W, x


GEMMA3_HIDDEN, GEMMA3_INTER = 2560, 10240
GEMMA3_NQ, GEMMA3_NKV = 2048, 1024


def gemma3_layer(seed: int = 0):
    """one Gemma-3-4B-shaped decode layer's quantized weights and input x."""
    g = rng(seed)
    H, I = GEMMA3_HIDDEN, GEMMA3_INTER
    L = {
        "wq": q4k(g, GEMMA3_NQ, H),
        "wk": q4k(g, GEMMA3_NKV, H),
        "wv": q6k(g, GEMMA3_NKV, H),
        "wo": q4k(g, H, GEMMA3_NQ),
        "wg": q4k(g, I, H),
        "wu": q4k(g, I, H),
        "wd": q6k(g, H, I),
    }
    x = activations(g, 1, H)
    return L, x


LLAMA_HIDDEN, LLAMA_INTER = 4096, 14336


def llama_ffn(fmt: int, batch: int, seed: int = 0):
    g = rng(seed)
    H, I = LLAMA_HIDDEN, LLAMA_INTER
    W = {"wg": weights(g, fmt, I, H), "wu": weights(g, fmt, I, H), "wd": weights(g, fmt, H, I)}
    X = activations(g, batch, H)
    return W, X


LM_HEAD_VOCAB = 262144


def lm_head(seed: int = 0, vocab: int = LM_HEAD_VOCAB, hidden: int = GEMMA3_HIDDEN):
    g = rng(seed)
    W = q4k(g, vocab, hidden)
    x = rms_normed(activations(g, 1, hidden))
    return W, x


MIXTRAL_E, MIXTRAL_TOPK, MIXTRAL_HIDDEN, MIXTRAL_INTER, MIXTRAL_NTOK = 8, 2, 4096, 14336, 16


def mixtral_moe(seed: int = 0, n_experts=MIXTRAL_E, hidden=MIXTRAL_HIDDEN, inter=MIXTRAL_INTER,
                ntok=MIXTRAL_NTOK, fmt=Q4_K):
    g = rng(seed)
    R = router(g, n_experts, hidden)
    W1 = [weights(g, fmt, inter, hidden) for _ in range(n_experts)]
    W3 = [weights(g, fmt, inter, hidden) for _ in range(n_experts)]
    W2 = [weights(g, fmt, hidden, inter) for _ in range(n_experts)]
    X = activations(g, ntok, hidden)
    return R, W1, W3, W2, X
