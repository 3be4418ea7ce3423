"""Counter-based, device-independent synthetic value generator.

Used by both the tests' oracle side and the library side, so it holds no
arithmetic of the attention method: it only turns (seed, element index) into a
bfloat16 number.  Every element is a pure function of its flat index, so any
subset of a tensor (a few rows of a multi-gigabyte Q) can be regenerated on the
CPU bit-identically to the full tensor generated on the GPU.

Definition
----------
* ``mix(x)`` is SplitMix64's output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014): add the
  golden-ratio increment, then two xor-shift-multiply rounds and a final
  xor-shift, all modulo 2**64.
* Stream key ``k = mix(seed)``.  Element n takes two words
  ``h0 = mix(k + 2n)`` and ``h1 = mix(k + 2n + 1)``, i.e. eight 16-bit lanes
  u_0..u_7.
* ``x = (2*sum(u) - 8*65535) * c`` in float32 with ``c = 1 / (65536*sqrt(8/3))``
  (unit variance, an 8-term Irwin-Hall approximation of N(0,1) bounded in
  about [-4.9, 4.9]); then rounded to bfloat16 (round to nearest even).
  The integer numerator is exact in float32 and the one float32 multiply and
  the bf16 rounding are correctly rounded on every device, so CPU and GPU give
  the same bits.

Implemented with torch int64 tensors, whose additions and multiplications wrap
modulo 2**64 on CPU and CUDA alike; right shifts are made logical by masking.
"""
import math

import torch

_GOLDEN = 0x9E3779B97F4A7C15 - (1 << 64)
_M1 = 0xBF58476D1CE4E5B9 - (1 << 64)
_M2 = 0x94D049BB133111EB - (1 << 64)
_SCALE = float(torch.tensor(1.0 / (65536.0 * math.sqrt(8.0 / 3.0)), dtype=torch.float32))


def _lsr(z, k):
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix(x):
    z = x + _GOLDEN
    z = (z ^ _lsr(z, 30)) * _M1
    z = (z ^ _lsr(z, 27)) * _M2
    return z ^ _lsr(z, 31)


def _key(seed):
    return int(_mix(torch.tensor([int(seed)], dtype=torch.int64))[0])


def normal_bf16_at(seed, index):
    """bf16 values for the int64 element indices ``index`` (any shape/device)."""
    index = index.to(torch.int64)
    k = _key(seed)
    acc = torch.zeros_like(index)
    for w in range(2):
        h = _mix(index * 2 + (k + w))
        for lane in range(4):
            acc += _lsr(h, 16 * lane) & 0xFFFF
    num = (acc * 2 - 8 * 65535).to(torch.float32)
    return (num * _SCALE).to(torch.bfloat16)


def normal_bf16(seed, shape, device="cpu", chunk=1 << 26):
    """Full tensor of the given shape: element n (row-major flat index) is
    ``normal_bf16_at(seed, n)``.  Generated in chunks to bound temporaries."""
    numel = 1
    for s in shape:
        numel *= int(s)
    out = torch.empty(numel, dtype=torch.bfloat16, device=device)
    for lo in range(0, numel, chunk):
        hi = min(numel, lo + chunk)
        idx = torch.arange(lo, hi, dtype=torch.int64, device=device)
        out[lo:hi] = normal_bf16_at(seed, idx)
    return out.view(*shape)


def rows_bf16(seed, rows, row_elems):
    """Rows ``rows`` (int sequence) of a [N, row_elems] tensor, on the CPU."""
    rows = torch.as_tensor(rows, dtype=torch.int64)
    idx = rows[:, None] * row_elems + torch.arange(row_elems, dtype=torch.int64)[None, :]
    return normal_bf16_at(seed, idx)


def gdn_inputs(seed, F, C, H, W, device="cpu"):
    """Synthetic inputs of the GDN token mixer on F forwarded positions:
    x [F, C] bf16 (the q|k|v projections, N(0,1)), w [C, W] fp32 conv
    weights (N(0,1) / W), g [F, H] fp32 log decays in (-0.5, 0] and
    beta [F, H] fp32 write strengths in (0.05, 0.95).  g and beta are made
    from generator values z by -0.1|z| and 0.05 + 0.9 |z| / (1 + |z|):
    float32 operations that round correctly on every device, so the CPU and
    the GPU get the same bits."""
    x = normal_bf16(seed, (F, C), device)
    w = normal_bf16(seed + 1, (C, W), device).to(torch.float32) / float(W)
    zg = normal_bf16(seed + 2, (F, H), device).to(torch.float32).abs()
    zb = normal_bf16(seed + 3, (F, H), device).to(torch.float32).abs()
    return x, w, zg * -0.1, 0.05 + 0.9 * (zb / (1.0 + zb))


def gdn_rows(seed, rows, C, H):
    """Rows ``rows`` of gdn_inputs' x, g and beta, on the CPU (same bits)."""
    x = rows_bf16(seed, rows, C)
    zg = rows_bf16(seed + 2, rows, H).to(torch.float32).abs()
    zb = rows_bf16(seed + 3, rows, H).to(torch.float32).abs()
    return x, zg * -0.1, 0.05 + 0.9 * (zb / (1.0 + zb))
