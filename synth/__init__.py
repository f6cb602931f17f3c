"""Seeded synthetic inputs for the routed expert-FFN layer.

This module is shared by the CPU oracle tests and by the CUDA path's tests and
benchmark. It only draws random numbers and lays them out in the storage
format; it holds none of the layer's arithmetic (no routing, no activation
quantisation, no expert matmul).

Shapes follow the model the Strata pages describe: 48 layers of 512 experts,
10 active per token ("Strata - the details", section "Which model?"; the
upstream Strata README, "How does it work?").  The pages give neither the
hidden sizes nor the bit layout of Q2_0, so the recipe here is this library's:

* activations  x ~ N(0, 1) fp32, [T, H]
* router       Wr ~ N(0, 0.02) fp32, [E, H]; bias zero unless skewed
* experts      gate/up [I, H] and down [H, I] drawn N(0, 0.02) in fp32 and
               stored as symmetric blocks of 32 along the input dimension with
               one fp16 scale per block:
                 2-bit: s = fp16(amax / 2), code = clamp(rint(w / s), -2, 1) + 2
                 3-bit: s = fp16(amax / 4), code = clamp(rint(w / s), -4, 3) + 4
               (the weight quantiser is part of the input recipe only; the
               layer itself never quantises weights)

Storage layout of one [N rows, K in] matrix of expert e (block-column-major):
  codes [E][K/32][N][bytes_per_block]   bytes_per_block = 8 (2-bit), 12 (3-bit)
  scales[E][K/32][N]                    fp16
2-bit element i of a block sits in byte i/4 at bit 2*(i%4); 3-bit element i
occupies bits 3i..3i+2 of the block's 96-bit little-endian word.
"""
from __future__ import annotations

import dataclasses
import math

import torch

MATS = ("gate", "up", "down")

# Zipf-skewed router bias: b_e = -ZIPF_GAMMA * ZIPF_S * ln(rank_e) for a seeded
# ranking of the experts, and ZIPF_DEAD_BIAS for the lowest ZIPF_DEAD_FRAC of the
# ranks (so that some experts receive no token).  ZIPF_GAMMA was chosen so that,
# with x ~ N(0,1) and Wr ~ N(0, 0.02) at H=2048, E=512, k=10, the realised
# per-expert token counts of a 4,096-token chunk fall off with a log-log slope
# close to -ZIPF_S over the live ranks.
ZIPF_S = 1.1
ZIPF_GAMMA = 0.5
ZIPF_DEAD_FRAC = 0.05
ZIPF_DEAD_BIAS = -30.0


@dataclasses.dataclass(frozen=True)
class LayerShape:
    H: int
    I: int
    E: int
    k: int
    bits: int = 2

    @property
    def bytes_per_block(self) -> int:
        return 4 * self.bits

    def validate(self) -> None:
        if self.H % 32 or self.I % 32:
            raise ValueError("H and I must be multiples of 32")
        if self.bits not in (2, 3):
            raise ValueError("bits must be 2 or 3")
        if not 1 <= self.k <= self.E:
            raise ValueError("need 1 <= k <= E")


# The workloads the pages' model implies (see the module docstring).
TINY = LayerShape(H=256, I=128, E=16, k=2)
FULL = LayerShape(H=2048, I=512, E=512, k=10)
FULL3 = LayerShape(H=2048, I=512, E=512, k=10, bits=3)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919) % (2**63 - 1))
    return g


def _stream(layer: int, tensor: int, chunk: int = 0) -> int:
    return layer * 100_000 + tensor * 1_000 + chunk


def _quantise_weights(w: torch.Tensor, bits: int):
    """w fp32 [e, N, K] -> (codes uint8 [e, K/32, N, 4*bits], scales fp16 [e, K/32, N])."""
    e, N, K = w.shape
    wb = w.view(e, N, K // 32, 32)
    amax = wb.abs().amax(-1)
    lo, hi = (-2, 1) if bits == 2 else (-4, 3)
    s16 = (amax / float(-lo)).to(torch.float16)
    sf = s16.float().unsqueeze(-1)
    q = torch.where(sf > 0, torch.round(wb / torch.where(sf > 0, sf, torch.ones_like(sf))), torch.zeros_like(wb))
    c = (q.clamp(lo, hi) - lo).to(torch.uint8)            # [e, N, KB, 32]
    c = c.permute(0, 2, 1, 3).contiguous()                   # [e, KB, N, 32]
    if bits == 2:
        packed = c[..., 0::4] | (c[..., 1::4] << 2) | (c[..., 2::4] << 4) | (c[..., 3::4] << 6)
    else:
        bitpos = torch.arange(96, device=w.device)
        elem = bitpos // 3
        shift = bitpos % 3
        bitv = (c[..., elem] >> shift.to(torch.uint8)) & 1    # [e, KB, N, 96]
        bitv = bitv.view(*bitv.shape[:-1], 12, 8).to(torch.int32)
        weights = (1 << torch.arange(8, device=w.device, dtype=torch.int32))
        packed = (bitv * weights).sum(-1).to(torch.uint8)
    scales = s16.permute(0, 2, 1).contiguous()
    return packed.contiguous(), scales


@dataclasses.dataclass
class Layer:
    shape: LayerShape
    Wr: torch.Tensor                 # fp32 [E, H]
    bias: torch.Tensor | None        # fp32 [E] or None
    codes: list                      # 3 x uint8 tensors
    scales: list                     # 3 x fp16 tensors

    def to(self, device) -> "Layer":
        return Layer(self.shape, self.Wr.to(device),
                     None if self.bias is None else self.bias.to(device),
                     [c.to(device) for c in self.codes], [s.to(device) for s in self.scales])

    def numpy(self):
        """Host copies as numpy arrays (scales as raw uint16 fp16 bits)."""
        c = [t.cpu().contiguous().numpy() for t in self.codes]
        s = [t.cpu().contiguous().view(torch.int16).numpy().view("uint16") for t in self.scales]
        b = None if self.bias is None else self.bias.cpu().numpy()
        return self.Wr.cpu().numpy(), b, c, s


def make_router(shape: LayerShape, seed: int = 0, layer: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed, _stream(layer, 0), device)
    return torch.randn(shape.E, shape.H, generator=g, device=device) * 0.02


def make_zipf_bias(shape: LayerShape, seed: int = 0, layer: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed, _stream(layer, 4), "cpu")
    perm = torch.randperm(shape.E, generator=g)
    rank = torch.empty(shape.E, dtype=torch.float64)
    rank[perm] = torch.arange(1, shape.E + 1, dtype=torch.float64)
    b = -ZIPF_GAMMA * ZIPF_S * torch.log(rank)
    dead = rank > math.ceil((1.0 - ZIPF_DEAD_FRAC) * shape.E)
    b[dead] = ZIPF_DEAD_BIAS
    return b.to(torch.float32).to(device)


def make_experts(shape: LayerShape, seed: int = 0, layer: int = 0, device="cpu", chunk_experts: int = 32):
    """Quantised gate, up and down matrices of every expert of one layer."""
    shape.validate()
    dims = {"gate": (shape.I, shape.H), "up": (shape.I, shape.H), "down": (shape.H, shape.I)}
    codes, scales = [], []
    for m, name in enumerate(MATS):
        N, K = dims[name]
        cs, ss = [], []
        for c0 in range(0, shape.E, chunk_experts):
            ne = min(chunk_experts, shape.E - c0)
            g = _gen(seed, _stream(layer, 1 + m, c0 // chunk_experts), device)
            w = torch.randn(ne, N, K, generator=g, device=device) * 0.02
            c, s = _quantise_weights(w, shape.bits)
            cs.append(c)
            ss.append(s)
            del w
        codes.append(torch.cat(cs))
        scales.append(torch.cat(ss))
    return codes, scales


def make_layer(shape: LayerShape, seed: int = 0, layer: int = 0, device="cpu", skew: bool = False) -> Layer:
    shape.validate()
    Wr = make_router(shape, seed, layer, device)
    bias = make_zipf_bias(shape, seed, layer, device) if skew else None
    codes, scales = make_experts(shape, seed, layer, device)
    return Layer(shape, Wr, bias, codes, scales)


def make_x(T: int, H: int, seed: int = 0, stream: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed, _stream(999, 5, stream), device)
    return torch.randn(T, H, generator=g, device=device)


def redraw_rows(x: torch.Tensor, rows, seed: int, attempt: int) -> torch.Tensor:
    """Replace the given rows of x with fresh N(0,1) draws from a seeded side stream."""
    rows = torch.as_tensor(rows, dtype=torch.long)
    if rows.numel() == 0:
        return x
    g = _gen(seed, _stream(998, 6, attempt), "cpu")
    fresh = torch.randn(rows.numel(), x.shape[1], generator=g)
    x = x.clone()
    x[rows.to(x.device)] = fresh.to(x.device)
    return x
