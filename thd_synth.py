"""Seeded synthetic THD packs for the CSA/HCA compressor pooling.

This module only draws inputs. It holds none of the pooling arithmetic, and it is
the one piece of code that both the oracle-side tests and the CUDA-side tests and
bench share.

Generator (counter based, so any slice of any tensor can be reproduced alone):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014). Draw ``i`` (0-based) of a stream with key ``k`` is
  ``mix64(k + (i + 1) * GOLDEN)``, with ``GOLDEN = 0x9E3779B97F4A7C15`` and
  ``mix64`` the published SplitMix64 finaliser.
* A uniform in [0, 1) is ``(draw >> 11) * 2**-53``.
* Normals come from the Box-Muller transform on consecutive uniform pairs
  ``(u0, u1)``: ``sqrt(-2 ln(1 - u0)) * (cos, sin)(2 pi u1)``, in float64.
* A bf16 value is the round-to-nearest-even of the float32 rounding of the
  float64 normal, stored as its 16-bit pattern (``uint16``).
* Each tensor has its own stream: key = ``mix64(seed * GOLDEN + tag)`` with tags
  kv=1, score=2, ape=3, dout=4, lengths=5, and for the KPool packs key=6, gate=7,
  lead=8.

The workloads follow the shapes and distributions of the pages' THD packs
(ratio=4 / coff=2 packs of 8192-token sequences at head dims 128 and 512), plus a
tiny ragged pack, a ragged ratio=2 pack and a long-window ratio=128 pack. No
dataset is involved: the pages measure synthetic packs only.

KPool packs (the DSA indexer's key pooling) hold indexer keys and gates [tokens, d]
(both N(0,1) bf16), THD segments, and optionally each segment's lead (the offset of
its first valid key, drawn uniformly in [0, max_lead]); the pools are P keys wide.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TAG_KV, TAG_SCORE, TAG_APE, TAG_DOUT, TAG_LENGTHS = 1, 2, 3, 4, 5
TAG_KEY, TAG_GATE, TAG_LEAD = 6, 7, 8


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, tag: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.uint64(seed) * GOLDEN + np.uint64(tag)
    return _mix64(np.array([base], dtype=np.uint64))[0]


def draws(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Raw 64-bit draws ``start .. start+count-1`` of the stream with ``key``."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * GOLDEN)


def uniforms(key: np.uint64, start: int, count: int) -> np.ndarray:
    return (draws(key, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normals(key: np.uint64, count: int, chunk: int = 1 << 22) -> np.ndarray:
    """``count`` standard normals (float64) by Box-Muller on uniform pairs."""
    out = np.empty(count, dtype=np.float64)
    npairs = (count + 1) // 2
    for p0 in range(0, npairs, chunk):
        p1 = min(npairs, p0 + chunk)
        u = uniforms(key, 2 * p0, 2 * (p1 - p0))
        rad = np.sqrt(-2.0 * np.log1p(-u[0::2]))
        ang = (2.0 * np.pi) * u[1::2]
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = rad * np.cos(ang)
        z[1::2] = rad * np.sin(ang)
        n = min(count, 2 * p1) - 2 * p0
        out[2 * p0:2 * p0 + n] = z[:n]
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values (finite) to bf16, ties to even; returns uint16 patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Pack:
    """One synthetic THD pack, host side (numpy)."""
    name: str
    ratio: int
    coff: int
    d: int
    capacity: int
    cu_seqlens: np.ndarray  # int32 [S+1]
    kv: np.ndarray          # uint16 (bf16 bits) [capacity, coff*d]
    score: np.ndarray       # uint16 (bf16 bits) [capacity, coff*d]
    ape: np.ndarray         # float32 [ratio, coff*d]
    dout: np.ndarray        # uint16 (bf16 bits) [total_comp, d]

    @property
    def S(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def C(self) -> int:
        return self.coff * self.d

    @property
    def total_comp(self) -> int:
        lens = np.diff(self.cu_seqlens.astype(np.int64))
        return int(np.sum(lens // self.ratio))


@dataclasses.dataclass(frozen=True)
class PackSpec:
    name: str
    lengths: Optional[List[int]]  # None: drawn (ragged ratio=2 pack)
    ratio: int
    coff: int
    d: int
    pad_rows: int = 0            # capacity = sum(lengths) + pad_rows
    score_scale: float = 1.0     # exact power-of-two scale applied to bf16 scores
    seed: int = 0
    length_seed: int = 7
    n_drawn_segments: int = 16
    max_drawn_length: int = 4096


# The five packs: a tiny ragged oracle pack, the pages' 1x8192 d128 and 3x8192 d512
# ratio=4 coff=2 shapes, a ragged ratio=2 pack with capacity padding, and a
# long-window ratio=128 coff=1 pack with sharpened scores.
SPECS: Dict[str, PackSpec] = {
    "tiny": PackSpec("tiny", [37, 12, 3], ratio=4, coff=2, d=8, pad_rows=64 - 52),
    "1x8192_d128": PackSpec("1x8192_d128", [8192], ratio=4, coff=2, d=128),
    "3x8192_d512": PackSpec("3x8192_d512", [8192] * 3, ratio=4, coff=2, d=512),
    "ragged_r2_d512": PackSpec("ragged_r2_d512", None, ratio=2, coff=2, d=512, pad_rows=1024),
    "long_r128_d512": PackSpec("long_r128_d512", [16384] * 4, ratio=128, coff=1, d=512,
                               score_scale=4.0),
    # The pages' two other ratio=4 coff=2 shapes, kept as context rows for the bench.
    "3x8192_d128": PackSpec("3x8192_d128", [8192] * 3, ratio=4, coff=2, d=128),
    "1x8192_d512": PackSpec("1x8192_d512", [8192], ratio=4, coff=2, d=512),
    # The pages' ratio=128 coff=2 d=128 example (65k tokens), as eight 8192-token
    # sequences, kept as a context row for the long-window kernel's 256-position windows.
    "r128c2_d128": PackSpec("r128c2_d128", [8192] * 8, ratio=128, coff=2, d=128),
}

HEADLINE = "3x8192_d512"


def drawn_lengths(spec: PackSpec) -> List[int]:
    key = stream_key(spec.length_seed, TAG_LENGTHS)
    u = uniforms(key, 0, spec.n_drawn_segments)
    return [int(1 + np.floor(x * spec.max_drawn_length)) for x in u]


def make_pack(spec: PackSpec | str, *, lengths: Optional[List[int]] = None,
              pad_rows: Optional[int] = None, seed: Optional[int] = None) -> Pack:
    """Draw a pack. ``lengths``/``pad_rows``/``seed`` override the spec (for tests)."""
    if isinstance(spec, str):
        spec = SPECS[spec]
    if lengths is None:
        lengths = spec.lengths if spec.lengths is not None else drawn_lengths(spec)
    pad = spec.pad_rows if pad_rows is None else pad_rows
    seed = spec.seed if seed is None else seed
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    T = int(cu[-1])
    capacity = T + pad
    C = spec.coff * spec.d
    total_comp = int(sum(L // spec.ratio for L in lengths))
    kv = f32_to_bf16_bits(normals(stream_key(seed, TAG_KV), capacity * C).astype(np.float32))
    sc = normals(stream_key(seed, TAG_SCORE), capacity * C).astype(np.float32)
    score = f32_to_bf16_bits(sc)
    if spec.score_scale != 1.0:
        score = f32_to_bf16_bits(bf16_bits_to_f32(score) * np.float32(spec.score_scale))
    ape = (0.02 * normals(stream_key(seed, TAG_APE), spec.ratio * C)).astype(np.float32)
    dout = f32_to_bf16_bits(normals(stream_key(seed, TAG_DOUT), total_comp * spec.d)
                            .astype(np.float32))
    return Pack(spec.name, spec.ratio, spec.coff, spec.d, capacity, cu,
                kv.reshape(capacity, C), score.reshape(capacity, C),
                ape.reshape(spec.ratio, C), dout.reshape(total_comp, spec.d))


def make_custom(lengths: List[int], ratio: int, coff: int, d: int, *, pad_rows: int = 0,
                seed: int = 0, score_scale: float = 1.0) -> Pack:
    """A pack with explicit segment lengths (tests: ragged, short and empty segments)."""
    spec = PackSpec("custom", list(lengths), ratio=ratio, coff=coff, d=d, pad_rows=pad_rows,
                    score_scale=score_scale, seed=seed)
    return make_pack(spec)


def to_torch(pack: Pack, device="cuda") -> Dict[str, "object"]:
    """Uploads a pack to torch tensors on ``device`` (bf16 tensors keep their bits)."""
    import torch
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return {
        "kv": bf(pack.kv).to(device),
        "score": bf(pack.score).to(device),
        "ape": torch.from_numpy(np.ascontiguousarray(pack.ape)).to(device),
        "cu_seqlens": torch.from_numpy(np.ascontiguousarray(pack.cu_seqlens)).to(device),
        "dout": bf(pack.dout).to(device),
    }


def bf16_tensor_bits(t) -> np.ndarray:
    """uint16 bit patterns of a torch bf16 tensor (copied to the host)."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# ----------------------------------------------------------------------------------
# KPool packs
# ----------------------------------------------------------------------------------

@dataclasses.dataclass
class KPoolPack:
    """One synthetic KPool input, host side (numpy)."""
    name: str
    pool: int
    d: int
    capacity: int
    cu_seqlens: np.ndarray        # int32 [S+1]
    lead: Optional[np.ndarray]    # int32 [S] (first valid key of segment s: cu[s] + lead[s]) or None
    key: np.ndarray               # uint16 (bf16 bits) [capacity, d]
    gate: np.ndarray              # uint16 (bf16 bits) [capacity, d]

    @property
    def S(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def total_pools(self) -> int:
        lens = np.diff(self.cu_seqlens.astype(np.int64))
        lead = np.zeros_like(lens) if self.lead is None else self.lead.astype(np.int64)
        return int(np.sum(np.maximum(lens - lead, 0) // self.pool))


@dataclasses.dataclass(frozen=True)
class KPoolSpec:
    name: str
    lengths: Optional[List[int]]  # None: drawn like the ragged compressor pack
    pool: int
    d: int
    pad_rows: int = 0
    max_lead: int = 0             # > 0: leads drawn uniformly in [0, max_lead]
    leads: Optional[List[int]] = None  # explicit leads (instead of drawn ones)
    gate_scale: float = 1.0       # exact power-of-two scale applied to bf16 gates
    seed: int = 0
    length_seed: int = 7
    n_drawn_segments: int = 16
    max_drawn_length: int = 4096


# Indexer keys of head dim 128 pooled four at a time (the pages' grid [0:4], [4:8], ...):
# a tiny ragged pack with leads, a 16-sequence pack of 8192 tokens, a ragged pack with
# leads and padding, and the 64-sequence bench pack (512k keys, larger than L2).
KPOOL_SPECS: Dict[str, KPoolSpec] = {
    "kpool_tiny": KPoolSpec("kpool_tiny", [13, 4, 0, 9, 2, 11], pool=4, d=8, pad_rows=5,
                            leads=[1, 3, 0, 2, 5, 0]),
    "kpool_16x8192_d128_p4": KPoolSpec("kpool_16x8192_d128_p4", [8192] * 16, pool=4, d=128),
    "kpool_ragged_d128_p4": KPoolSpec("kpool_ragged_d128_p4", None, pool=4, d=128,
                                      pad_rows=1024, max_lead=7),
    "kpool_64x8192_d128_p4": KPoolSpec("kpool_64x8192_d128_p4", [8192] * 64, pool=4, d=128),
}


def make_kpool(spec: KPoolSpec | str, *, lengths: Optional[List[int]] = None,
               leads: Optional[List[int]] = None, pool: Optional[int] = None,
               d: Optional[int] = None, pad_rows: Optional[int] = None,
               seed: Optional[int] = None, gate_scale: Optional[float] = None) -> KPoolPack:
    """Draw a KPool pack; the keyword arguments override the spec (for tests)."""
    if isinstance(spec, str):
        spec = KPOOL_SPECS[spec]
    if lengths is None:
        if spec.lengths is not None:
            lengths = spec.lengths
        else:
            u = uniforms(stream_key(spec.length_seed, TAG_LENGTHS), 0, spec.n_drawn_segments)
            lengths = [int(1 + np.floor(x * spec.max_drawn_length)) for x in u]
    P = spec.pool if pool is None else pool
    d = spec.d if d is None else d
    pad = spec.pad_rows if pad_rows is None else pad_rows
    seed = spec.seed if seed is None else seed
    gscale = spec.gate_scale if gate_scale is None else gate_scale
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    capacity = int(cu[-1]) + pad
    lead = None
    if leads is None:
        leads = spec.leads
    if leads is not None:
        lead = np.asarray(leads, dtype=np.int32)
    elif spec.max_lead > 0:
        u = uniforms(stream_key(seed, TAG_LEAD), 0, len(lengths))
        lead = np.floor(u * (spec.max_lead + 1)).astype(np.int32)
    key = f32_to_bf16_bits(normals(stream_key(seed, TAG_KEY), capacity * d).astype(np.float32))
    gate = f32_to_bf16_bits(normals(stream_key(seed, TAG_GATE), capacity * d).astype(np.float32))
    if gscale != 1.0:
        gate = f32_to_bf16_bits(bf16_bits_to_f32(gate) * np.float32(gscale))
    return KPoolPack(spec.name, P, d, capacity, cu, lead, key.reshape(capacity, d),
                     gate.reshape(capacity, d))


def make_kpool_custom(lengths: List[int], pool: int, d: int, *, leads: Optional[List[int]] = None,
                      pad_rows: int = 0, seed: int = 0, gate_scale: float = 1.0) -> KPoolPack:
    """A KPool pack with explicit segment lengths (and leads)."""
    spec = KPoolSpec("kpool_custom", list(lengths), pool=pool, d=d, pad_rows=pad_rows,
                     gate_scale=gate_scale, seed=seed)
    return make_kpool(spec, leads=leads)


def kpool_to_torch(pack: KPoolPack, device="cuda") -> Dict[str, "object"]:
    """Uploads a KPool pack to torch tensors on ``device``."""
    import torch
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    t = {"key": bf(pack.key).to(device), "gate": bf(pack.gate).to(device),
         "cu_seqlens": torch.from_numpy(np.ascontiguousarray(pack.cu_seqlens)).to(device)}
    if pack.lead is not None:
        t["lead"] = torch.from_numpy(np.ascontiguousarray(pack.lead)).to(device)
    return t

