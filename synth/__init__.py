"""Seeded synthetic inputs shared by the oracle side and the GPU side.

This module holds the workload shapes and the random draws only: it computes none of the
products.  Weight generators emit the source block formats, whose byte layout is:

* ``Q1_0``: 18-byte blocks of 128 weights -- fp16 scale (little-endian) then 16 sign bytes,
  weight ``i`` in bit ``i % 8`` of byte ``i // 8`` (bit 1 = +1).
* ``Q2_0_g64``: 18-byte blocks of 64 weights -- fp16 scale then 16 code bytes, weight ``4k + r``
  in bits ``2r..2r+1`` of byte ``k`` (code c means weight c - 1).
* planar ternary: per row and per 64 columns one 16-byte beat ``{u64 pos, u64 neg}``, column
  ``64g + c`` in bit ``c`` of beat ``g``.
* bf16 head: row-major ``[N][K]`` bfloat16 bit patterns.

Value distributions follow the workloads the pages measure: sign bits Bernoulli(0.5); ternary
codes at 31/38/31 % for -1/0/+1 (the split the pages report for a real ternary file) and no +2;
block scales fp16(|N(0, 0.02)|); activations N(0, 1).
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------------------------
# workload shapes (rows N x columns K of each projection)
# ---------------------------------------------------------------------------------------------
QWEN3_8B_PROJ = [  # per decoder layer; hidden 4096, ffn 12288, 36 layers
    ("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
    ("gate", 12288, 4096), ("up", 12288, 4096), ("down", 4096, 12288),
]
QWEN3_8B_LAYERS = 36
BITNET_2B4T_PROJ = [  # per decoder layer; hidden 2560, ffn 6912, 30 layers
    ("q", 2560, 2560), ("k", 640, 2560), ("v", 640, 2560), ("o", 2560, 2560),
    ("gate", 6912, 2560), ("up", 6912, 2560), ("down", 2560, 6912),
]
BITNET_2B4T_LAYERS = 30
BITNET_HEAD = (128256, 2560)
PREFILL_M = 512

TERNARY_PROBS = (0.31, 0.38, 0.31, 0.0)   # codes 0, 1, 2, 3  ->  weights -1, 0, +1, +2
SCALE_SIGMA = 0.02


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _fp16_scales(g: np.random.Generator, shape, sigma=SCALE_SIGMA) -> np.ndarray:
    return np.abs(g.normal(0.0, sigma, size=shape)).astype(np.float16).view(np.uint16)


def _draw_codes(g: np.random.Generator, shape, probs) -> np.ndarray:
    u = g.random(size=shape, dtype=np.float64)
    edges = np.cumsum(np.asarray(probs, dtype=np.float64))[:-1]
    return np.searchsorted(edges, u, side="right").astype(np.uint8)


def q1_0_blocks(N: int, K: int, seed: int, scales=None) -> np.ndarray:
    """[N][K/128][18] uint8 Q1_0 blocks; sign bits Bernoulli(0.5), scales fp16 |N(0,0.02)|."""
    assert K % 128 == 0
    g = rng(seed)
    nb = K // 128
    out = np.empty((N, nb, 18), dtype=np.uint8)
    sc = _fp16_scales(g, (N, nb)) if scales is None else np.asarray(scales, np.uint16)
    out[:, :, 0] = (sc & 0xFF).astype(np.uint8)
    out[:, :, 1] = (sc >> 8).astype(np.uint8)
    out[:, :, 2:] = g.integers(0, 256, size=(N, nb, 16), dtype=np.uint8)
    return out


def pack_q2_codes(codes: np.ndarray) -> np.ndarray:
    """codes [..., 64] in 0..3  ->  [..., 16] bytes, weight 4k+r at bits 2r of byte k."""
    c = codes.reshape(codes.shape[:-1] + (16, 4)).astype(np.uint8)
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def q2_0_blocks(N: int, K: int, seed: int, probs=TERNARY_PROBS, codes=None,
                scales=None) -> np.ndarray:
    """[N][K/64][18] uint8 Q2_0_g64 blocks; codes drawn with ``probs``; scales fp16 |N(0,0.02)|."""
    assert K % 64 == 0
    g = rng(seed)
    nb = K // 64
    sc = _fp16_scales(g, (N, nb)) if scales is None else np.asarray(scales, np.uint16)
    if codes is None:
        codes = _draw_codes(g, (N, nb, 64), probs)
    out = np.empty((N, nb, 18), dtype=np.uint8)
    out[:, :, 0] = (sc & 0xFF).astype(np.uint8)
    out[:, :, 1] = (sc >> 8).astype(np.uint8)
    out[:, :, 2:] = pack_q2_codes(np.asarray(codes).reshape(N, nb, 64))
    return out


def trits_to_planes(trits: np.ndarray) -> np.ndarray:
    """trits [N][K] in {-1,0,+1}  ->  planes [N][K/64][2] uint64 {pos, neg}."""
    N, K = trits.shape
    t = trits.reshape(N, K // 64, 64)
    weights = (np.uint64(1) << np.arange(64, dtype=np.uint64))
    pos = ((t == 1).astype(np.uint64) * weights).sum(axis=-1, dtype=np.uint64)
    neg = ((t == -1).astype(np.uint64) * weights).sum(axis=-1, dtype=np.uint64)
    return np.stack([pos, neg], axis=-1).astype(np.uint64)


def trit_planes(N: int, K: int, seed: int, probs=TERNARY_PROBS[:3]):
    """Random ternary matrix as planar beats; returns (planes [N][K/64][2] u64, trits int8)."""
    assert K % 64 == 0
    g = rng(seed)
    trits = (_draw_codes(g, (N, K), probs).astype(np.int8) - 1)
    return trits_to_planes(trits), trits


def w_scale(seed: int) -> float:
    return float(np.float32(abs(rng(seed).normal(0.0, SCALE_SIGMA))))


def activations(B: int, K: int, seed: int) -> np.ndarray:
    """fp32 [B][K] activations N(0, 1)."""
    return rng(seed).standard_normal(size=(B, K), dtype=np.float32)


def int8_codes(B: int, K: int, seed: int, extremes: bool = False) -> np.ndarray:
    """int8 [B][K] uniform over the full int8 range (includes -128); ``extremes`` draws only
    from {-128, -127, 127}."""
    g = rng(seed)
    if extremes:
        return g.choice(np.array([-128, -127, 127], dtype=np.int8), size=(B, K))
    return g.integers(-128, 128, size=(B, K), dtype=np.int16).astype(np.int8)


def q8_scales(B: int, K: int, seed: int) -> np.ndarray:
    """fp16 [B][K/32] positive activation block scales (as a q8_0 quantizer of N(0,1) emits)."""
    g = rng(seed)
    return (np.abs(g.normal(0.0, 1.0, size=(B, K // 32))) * (3.0 / 127.0) + 1e-3).astype(
        np.float16).view(np.uint16)


def bf16_weights(N: int, K: int, seed: int, sigma: float = SCALE_SIGMA) -> np.ndarray:
    """[N][K] bf16 bit patterns of N(0, sigma) (round to nearest even from fp32)."""
    f = rng(seed).normal(0.0, sigma, size=(N, K)).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def proj_seed(base: int, layer: int, proj: int) -> int:
    """Per-projection seed: base + layer*16 + proj."""
    return base + layer * 16 + proj


# ---------------------------------------------------------------------------------------------
# device-side generation for the large timed workloads (torch only moves and draws bytes here)
# ---------------------------------------------------------------------------------------------
def device_bytes(nbytes: int, seed: int, device="cuda"):
    """Uniform random bytes on the device (seeded torch generator)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=device, generator=gen)


def device_q2_codes_packed(nbytes: int, seed: int, probs=TERNARY_PROBS, device="cuda"):
    """``nbytes`` code bytes whose 2-bit fields are i.i.d. with ``probs`` (seeded, on device)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    u = torch.rand((nbytes, 4), device=device, generator=gen)
    edges = torch.tensor(np.cumsum(probs)[:-1], device=device, dtype=torch.float32)
    c = torch.bucketize(u, edges, right=True).to(torch.uint8)
    return c[:, 0] | (c[:, 1] << 2) | (c[:, 2] << 4) | (c[:, 3] << 6)


def device_trit_planes(N: int, K: int, seed: int, probs=TERNARY_PROBS[:3], device="cuda"):
    """Planar beats as uint8 bytes [N*K/64*16] on the device (seeded)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    u = torch.rand((N, K // 64, 64), device=device, generator=gen)
    edges = torch.tensor(np.cumsum(probs)[:-1], device=device, dtype=torch.float32)
    t = torch.bucketize(u, edges, right=True).to(torch.int8) - 1
    bitw = (torch.ones(64, dtype=torch.int64, device=device) << torch.arange(64, device=device))
    pos = ((t == 1).to(torch.int64) * bitw).sum(-1)
    neg = ((t == -1).to(torch.int64) * bitw).sum(-1)
    beats = torch.stack([pos, neg], dim=-1).contiguous()
    return beats.view(torch.uint8).reshape(-1)


def device_fp16_scales(count: int, seed: int, sigma=SCALE_SIGMA, device="cuda"):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return (torch.randn(count, device=device, generator=gen) * sigma).abs().to(torch.float16)
