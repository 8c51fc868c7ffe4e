"""Counter-based random inputs and cache quantizers.

Random numbers: splitmix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) evaluated at a counter, so any
slice of a stream can be regenerated on its own; normals by the Box-Muller
transform.  Every tensor of a problem draws from its own stream.

Quantizers (input generation only; the decoders live on each side):
  q8_0  -- 32 values per block; the block scale d = amax/127 is stored as
           IEEE binary16 followed by 32 int8 codes round(x/d) (ties away
           from zero, clamped to +-127).  34 bytes per block.
  q4_0  -- 32 values per block; d = m/(-8) where m is the signed value of
           largest magnitude, stored as binary16, then 16 bytes: byte b
           holds code(b) in its low nibble and code(b+16) in its high
           nibble, code = min(15, trunc(x/d + 8.5)).  18 bytes per block.
           A code c decodes to (c - 8) * d.
  f16   -- IEEE binary16, 2 bytes per value.
  f32   -- IEEE binary32, 4 bytes per value.
A cache row (one key, one KV head) is the concatenation of its blocks; the
cache is laid out [M][Hkv][row].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

TYPE_F32, TYPE_F16, TYPE_Q8_0, TYPE_Q4_0 = 0, 1, 2, 3
TYPE_NAMES = {TYPE_F32: "f32", TYPE_F16: "f16", TYPE_Q8_0: "q8_0", TYPE_Q4_0: "q4_0"}
_TYPE_BY_NAME = {v: k for k, v in TYPE_NAMES.items()}

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

# stream ids, one per tensor of a problem
S_Q, S_K, S_V, S_DO, S_MASK, S_ROWS, S_SAMPLE = 1, 2, 3, 4, 5, 6, 7


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        a = _mix(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
        b = _mix(np.array([(int(a) ^ (stream * 0xD1B54A32D192ED03)) & 0xFFFFFFFFFFFFFFFF],
                          dtype=np.uint64))[0]
    return b


def u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit outputs number start .. start+count-1 of one stream."""
    base = _stream_base(seed, stream)
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + k * _GOLDEN)


def uniform(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    return (u64(seed, stream, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """count standard normals (float64) by Box-Muller, generated in chunks."""
    out = np.empty(count, dtype=np.float64)
    npairs = (count + 1) // 2
    pos = 0
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        x = u64(seed, stream, 2 * p0, 2 * (p1 - p0))
        u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
        u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)          # [0, 1)
        r = np.sqrt(-2.0 * np.log(u1))
        t = (2.0 * math.pi) * u2
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        n = min(count - pos, z.size)
        out[pos:pos + n] = z[:n]
        pos += n
    return out


def normal_f32(seed: int, stream: int, shape, scale: float = 1.0, offset: float = 0.0) -> np.ndarray:
    n = int(np.prod(shape))
    return (offset + scale * normal(seed, stream, n)).astype(np.float32).reshape(shape)


def sample_indices(seed: int, stream: int, n: int, k: int) -> np.ndarray:
    """k distinct indices from range(n), sorted (seeded, without replacement)."""
    keys = u64(seed, stream, 0, n)
    return np.sort(np.argsort(keys, kind="stable")[:k]).astype(np.int64)


# ----------------------------------------------------------------------------------------------
# quantizers (produce raw cache bytes)

def row_bytes(t: int, D: int) -> int:
    if t == TYPE_F32:
        return 4 * D
    if t == TYPE_F16:
        return 2 * D
    if t == TYPE_Q8_0:
        return (D // 32) * 34
    if t == TYPE_Q4_0:
        return (D // 32) * 18
    raise ValueError(t)


def _quant_q8_0(x: np.ndarray) -> np.ndarray:
    b = x.reshape(-1, 32).astype(np.float32)
    amax = np.max(np.abs(b), axis=1)
    d = (amax / np.float32(127.0)).astype(np.float32)
    inv = np.where(d != 0, np.float32(1.0) / np.where(d != 0, d, np.float32(1.0)), np.float32(0.0)).astype(np.float32)
    y = b * inv[:, None]
    q = np.trunc(y + np.copysign(np.float32(0.5), y))  # ties away from zero
    q = np.clip(q, -127, 127).astype(np.int8)
    out = np.empty((b.shape[0], 34), dtype=np.uint8)
    out[:, 0:2] = d.astype(np.float16).view(np.uint8).reshape(-1, 2)
    out[:, 2:34] = q.view(np.uint8)
    return out


def _quant_q4_0(x: np.ndarray) -> np.ndarray:
    b = x.reshape(-1, 32).astype(np.float32)
    idx = np.argmax(np.abs(b), axis=1)
    m = b[np.arange(b.shape[0]), idx]
    d = (m / np.float32(-8.0)).astype(np.float32)
    inv = np.where(d != 0, np.float32(1.0) / np.where(d != 0, d, np.float32(1.0)), np.float32(0.0)).astype(np.float32)
    c = np.trunc(b * inv[:, None] + np.float32(8.5))
    c = np.clip(c, 0, 15).astype(np.uint8)
    out = np.empty((b.shape[0], 18), dtype=np.uint8)
    out[:, 0:2] = d.astype(np.float16).view(np.uint8).reshape(-1, 2)
    out[:, 2:18] = c[:, 0:16] | (c[:, 16:32] << np.uint8(4))
    return out


def quantize_rows(x: np.ndarray, t: int) -> np.ndarray:
    """x: float32 [..., D] -> uint8 [..., row_bytes(t, D)] raw rows."""
    D = x.shape[-1]
    lead = x.shape[:-1]
    if t == TYPE_F32:
        return np.ascontiguousarray(x.astype(np.float32)).view(np.uint8).reshape(*lead, 4 * D)
    if t == TYPE_F16:
        return np.ascontiguousarray(x.astype(np.float16)).view(np.uint8).reshape(*lead, 2 * D)
    if D % 32:
        raise ValueError("quantized rows need D % 32 == 0")
    rows = []
    flat = x.reshape(-1, D)
    if flat.shape[0] == 0:
        return np.zeros((*lead, row_bytes(t, D)), dtype=np.uint8)
    step = max(1, _CHUNK // D)
    for r0 in range(0, flat.shape[0], step):
        part = flat[r0:r0 + step]
        qb = _quant_q8_0(part) if t == TYPE_Q8_0 else _quant_q4_0(part)
        rows.append(qb.reshape(part.shape[0], -1))
    return np.concatenate(rows, axis=0).reshape(*lead, row_bytes(t, D))


# ----------------------------------------------------------------------------------------------
# problems

F16_NEG_INF = np.uint16(0xFC00)


@dataclass
class Problem:
    """One backward problem in the library's layouts.

    q   float32 [N][H][D]          dO  float32 [N][H][Dv]
    k   uint8   [M][Hkv][row]      v   uint8   [M][Hkv][row_v]
    mask uint16 (binary16 bits) [Hm][N][M] or None (element (j, i, hm) at (hm*N + i)*M + j)
    """
    name: str
    N: int
    M: int
    H: int
    Hkv: int
    D: int
    Dv: int
    k_type: int
    v_type: int
    causal: bool
    scale: float
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    dO: np.ndarray
    mask: Optional[np.ndarray] = None
    mask_heads: int = 0
    meta: dict = field(default_factory=dict)
    # optional extensions (none by default): ALiBi slopes [H], soft-cap c (0 = none), sink logits [H]
    alibi: Optional[np.ndarray] = None
    softcap: float = 0.0
    sinks: Optional[np.ndarray] = None

    @property
    def has_ext(self) -> bool:
        return self.alibi is not None or self.softcap > 0 or self.sinks is not None

    @property
    def G(self) -> int:
        return self.H // self.Hkv

    def visible_pairs(self) -> int:
        """(i, j) pairs the causal rule allows (the mask is not counted)."""
        if not self.causal:
            return self.N * self.M
        tot = 0
        for i in range(self.N):
            tot += max(0, min(self.M, self.M - self.N + i + 1))
        return tot

    def flops(self) -> float:
        """10 * D * H * visible pairs: five contractions of 2 flops per multiply-add."""
        return 10.0 * self.D * self.H * self.visible_pairs()

    def alg_bytes(self) -> int:
        """Each input read once plus each output written once."""
        b = self.q.nbytes + self.dO.nbytes + self.k.nbytes + self.v.nbytes
        if self.mask is not None:
            b += self.mask.nbytes
        b += 4 * (self.N * self.H * self.D + self.M * self.Hkv * (self.D + self.Dv) + 2 * self.N * self.H)
        return b


CONFIGS = {
    # tiny f32 sanity
    "0": dict(N=8, M=32, H=2, Hkv=1, D=64, Dv=64, k_type="f32", v_type="f32", causal=False, seed=1000),
    # q8_0 K/V, causal tail, short cache
    "1": dict(N=64, M=512, H=8, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0", causal=True, seed=1001),
    # cancellation variant of 1: V = 1 + 1e-3 N(0,1) before quantization
    "1c": dict(N=64, M=512, H=8, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0", causal=True, seed=1101,
               v_offset=1.0, v_sigma=1e-3),
    # tiny dO variant of 1
    "1t": dict(N=64, M=512, H=8, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0", causal=True, seed=1201,
               do_sigma=1e-6),
    # long cache, small N
    "2": dict(N=64, M=8192, H=8, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0", causal=True, seed=1002),
    # mixed types, additive mask with 10% -inf and 4 fully masked query rows
    "3": dict(N=128, M=4096, H=24, Hkv=4, D=256, Dv=256, k_type="q4_0", v_type="q8_0", causal=False, seed=1003,
              mask="random", mask_p=0.1, full_rows=4, mask_heads=24),
    # the long-context shape: q8_0, GQA 6, causal tail
    "4": dict(N=2048, M=75520, H=24, Hkv=4, D=256, Dv=256, k_type="q8_0", v_type="q8_0", causal=True, seed=1004),
}


def config(name: str, **over) -> dict:
    c = dict(CONFIGS[str(name)])
    c.update(over)
    c.setdefault("name", str(name))
    return c


def _type(t) -> int:
    return _TYPE_BY_NAME[t] if isinstance(t, str) else int(t)


def make_problem(name: str = "custom", *, N: int, M: int, H: int, Hkv: int, D: int, Dv: int,
                 k_type="f32", v_type="f32", causal: bool = False, seed: int = 1,
                 scale: Optional[float] = None, mask: Optional[str] = None, mask_p: float = 0.1,
                 full_rows: int = 0, mask_heads: int = 0, v_offset: float = 0.0, v_sigma: float = 1.0,
                 do_sigma: float = 1.0, q_sigma: float = 1.0, k_sigma: float = 1.0,
                 row_decades: float = 0.0, alibi: bool = False, softcap: float = 0.0,
                 sinks: Optional[float] = None) -> Problem:
    """Build a seeded problem.

    mask: None, "random" (entries -inf with probability mask_p, else 0, plus
    full_rows query rows set to -inf for every key and head) or "finite"
    (entries uniform in [-2, 0), plus the same -inf pattern).
    row_decades: when > 0, every (i, h) row of Q and of dO is multiplied by its own
    10**u, u uniform in [-row_decades, row_decades] (per-row dynamic range).
    alibi: ALiBi slopes 2^(-8 (h+1) / H) per query head; softcap: the soft-cap c (0 = none);
    sinks: when given, sink logits sinks * N(0,1) + 1 per query head.
    """
    kt, vt = _type(k_type), _type(v_type)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    q = normal_f32(seed, S_Q, (N, H, D), q_sigma)
    dO = normal_f32(seed, S_DO, (N, H, Dv), do_sigma)
    if row_decades > 0:
        fq = 10.0 ** (row_decades * (2.0 * uniform(seed, S_ROWS + 10, N * H) - 1.0))
        fo = 10.0 ** (row_decades * (2.0 * uniform(seed, S_ROWS + 11, N * H) - 1.0))
        q = (q * fq.reshape(N, H, 1)).astype(np.float32)
        dO = (dO * fo.reshape(N, H, 1)).astype(np.float32)
    kf = normal_f32(seed, S_K, (M, Hkv, D), k_sigma)
    vf = normal_f32(seed, S_V, (M, Hkv, Dv), v_sigma, v_offset)
    k = quantize_rows(kf, kt)
    del kf
    v = quantize_rows(vf, vt)
    del vf
    m = None
    hm = 0
    meta = {}
    if mask is not None:
        hm = mask_heads if mask_heads else H
        n = hm * N * M
        u = uniform(seed, S_MASK, n)
        m = np.zeros(n, dtype=np.uint16)
        if mask == "finite":
            m[:] = (-2.0 + 2.0 * uniform(seed, S_MASK + 100, n)).astype(np.float16).view(np.uint16)
        m[u < mask_p] = F16_NEG_INF
        m = m.reshape(hm, N, M)
        if full_rows:
            rows = sample_indices(seed, S_ROWS, N, full_rows)
            m[:, rows, :] = F16_NEG_INF
            meta["full_rows"] = rows
    slopes = (2.0 ** (-8.0 * (np.arange(H) + 1) / H)).astype(np.float32) if alibi else None
    sink = (1.0 + sinks * normal(seed, S_ROWS + 12, H)).astype(np.float32) if sinks is not None else None
    return Problem(name=name, N=N, M=M, H=H, Hkv=Hkv, D=D, Dv=Dv, k_type=kt, v_type=vt, causal=bool(causal),
                   scale=float(scale), q=q, k=k, v=v, dO=dO, mask=m, mask_heads=hm, meta=meta, alibi=slopes,
                   softcap=float(softcap), sinks=sink)


def from_config(name: str, **over) -> Problem:
    c = config(name, **over)
    return make_problem(**c)
