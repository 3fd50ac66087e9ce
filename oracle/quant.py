"""Affine group-quantized weights and the 16-bit float formats, written out plainly.

Weight format (mlx-dspark wiki page, "Key techniques": the verify kernel works
per "weight group"; the group size, code widths and fp16 scale/bias come from
the affine format of the quantized targets the pages run, 2-bit ones included
(PyPI page, "Models")):

* ``wq``     uint32 [N, K * bits / 32].  Weight (n, k) is the code stored in word
  ``k // (32 // bits)`` of row n, at bit offset ``(k % (32 // bits)) * bits``
  (least significant field first).
* ``scales`` fp16 [N, K / group], ``biases`` fp16 [N, K / group].
* dequantized weight ``w_hat[n, k] = scale[n, k // group] * code[n, k] + bias[n, k // group]``
  evaluated in fp32 as one multiply, rounded, then one add, rounded.

16-bit floats are carried as uint16 bit patterns so that nothing here depends on
a library's bf16 support.
"""

import numpy as np

GROUP = 64


def unpack_codes(wq, K, bits):
    """Codes uint8 [N, K] from packed words uint32 [N, K*bits/32] (layout above)."""
    if bits not in (2, 4, 8):
        raise ValueError("bits must be 2, 4 or 8")
    wq = np.asarray(wq, dtype=np.uint32)
    per_word = 32 // bits
    N = wq.shape[0]
    if wq.shape[1] * per_word != K:
        raise ValueError("packed width does not match K")
    mask = np.uint32((1 << bits) - 1)
    codes = np.empty((N, K), dtype=np.uint8)
    for j in range(per_word):
        # field j of every word holds element k = word_index * per_word + j
        codes[:, j::per_word] = ((wq >> np.uint32(j * bits)) & mask).astype(np.uint8)
    return codes


def pack_codes(codes, bits):
    """Inverse of ``unpack_codes``: uint8 codes [N, K] -> uint32 words."""
    codes = np.asarray(codes, dtype=np.uint32)
    per_word = 32 // bits
    N, K = codes.shape
    if K % per_word:
        raise ValueError("K must fill whole words")
    if codes.max(initial=0) >= (1 << bits):
        raise ValueError("code does not fit in the field")
    wq = np.zeros((N, K // per_word), dtype=np.uint32)
    for j in range(per_word):
        wq |= codes[:, j::per_word] << np.uint32(j * bits)
    return wq


def fp16_bits_to_f32(u16):
    return np.asarray(u16, dtype=np.uint16).view(np.float16).astype(np.float32)


def bf16_bits_to_f32(u16):
    """bf16 bit pattern -> fp32 (exact: bf16 is the top half of an fp32)."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_bits(x):
    """fp32 -> bf16 bit pattern, round to nearest, ties to even; NaN stays NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        rounded = rounded.copy()
        rounded[nan] = ((u[nan] >> np.uint64(16)).astype(np.uint16)) | np.uint16(0x0040)
    return rounded


def dequantize(wq, scales, biases, K, bits, group=GROUP):
    """w_hat fp32 [N, K] = scale * code + bias, one rounding after each operation."""
    if group != GROUP:
        raise ValueError("group size must be 64")
    codes = unpack_codes(wq, K, bits).astype(np.float32)
    s = fp16_bits_to_f32(scales)
    b = fp16_bits_to_f32(biases)
    if s.shape != (codes.shape[0], K // group) or b.shape != s.shape:
        raise ValueError("scales/biases must be [N, K/group]")
    g = np.arange(K) // group          # group index of every column k
    prod = (s[:, g] * codes).astype(np.float32)   # rounded fp32 product
    return (prod + b[:, g]).astype(np.float32)     # rounded fp32 sum
