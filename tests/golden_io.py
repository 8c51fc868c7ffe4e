"""Reader for the text fixtures under tests/golden/ and the problems they describe."""
import math
import os
import re

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_NAMES = {"__builtins__": {}, "log": math.log, "inf": math.inf}


def value(expr: str) -> float:
    """One number written as an expression in log(), inf, fractions and powers."""
    if not re.fullmatch(r"[0-9a-z.+\-*/() ]+", expr.strip()):
        raise ValueError(f"unexpected characters in {expr!r}")
    return float(eval(expr, _NAMES, {}))  # noqa: S307 - fixed fixture text, restricted names


def load(name: str) -> dict:
    """{section: {key: text}} of one fixture; '#' lines are comments."""
    out, cur = {}, None
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("[") and line.endswith("]"):
            cur = out.setdefault(line[1:-1], {})
            continue
        key, _, rhs = line.partition("=")
        cur[key.strip()] = rhs.strip()
    return out


def vector(text: str) -> list:
    return [value(x) for x in text.split(",")]


def indexed(section: dict, name: str, shape: tuple, width: int) -> np.ndarray:
    """Array name[a][b] = vector (or scalar when width is 0) from 'name[a][b] = ...' entries;
    every entry of the shape must be given."""
    out = np.zeros(shape + ((width,) if width else ()), dtype=np.float64)
    seen = set()
    for key, text in section.items():
        m = re.fullmatch(rf"{name}\[(\d+)\]\[(\d+)\]", key)
        if m:
            a, b = int(m.group(1)), int(m.group(2))
            out[a, b] = vector(text) if width else value(text)
            seen.add((a, b))
    assert seen == {(a, b) for a in range(shape[0]) for b in range(shape[1])}, (name, sorted(seen))
    return out


def worked_problem(fix: dict, D_pad: int = 0):
    """The fixture's inputs as an f32-cache problem; D_pad > D embeds every vector in D_pad
    components with zeros after the given ones (no dot product changes)."""
    inp = fix["inputs"]
    N, M, H, Hkv = (int(inp[k]) for k in ("N", "M", "H", "Hkv"))
    D, Dv = int(inp["D"]), int(inp["Dv"])
    Hm = int(inp["mask_heads"])
    Dp, Dvp = max(D, D_pad), max(Dv, D_pad)

    def pad(a, width):
        out = np.zeros(a.shape[:-1] + (width,), dtype=np.float64)
        out[..., :a.shape[-1]] = a
        return out

    q = pad(indexed(inp, "q", (N, H), D), Dp).astype(np.float32)
    dO = pad(indexed(inp, "dO", (N, H), Dv), Dvp).astype(np.float32)
    k = pad(indexed(inp, "k", (M, Hkv), D), Dp).astype(np.float32)
    v = pad(indexed(inp, "v", (M, Hkv), Dv), Dvp).astype(np.float32)
    mask = None
    if Hm > 0:
        mask = np.ascontiguousarray(indexed(inp, "mask", (Hm, N), M).astype(np.float16).view(np.uint16))
    return synth.Problem(name="golden", N=N, M=M, H=H, Hkv=Hkv, D=Dp, Dv=Dvp, k_type=synth.TYPE_F32,
                         v_type=synth.TYPE_F32, causal=bool(int(inp["causal"])), scale=value(inp["scale"]),
                         q=q, k=np.ascontiguousarray(k).view(np.uint8), v=np.ascontiguousarray(v).view(np.uint8),
                         dO=dO, mask=mask, mask_heads=Hm)


def worked_expected(fix: dict, D_pad: int = 0) -> dict:
    inp, exp = fix["inputs"], fix["expected"]
    N, M, H, Hkv = (int(inp[k]) for k in ("N", "M", "H", "Hkv"))
    D, Dv = int(inp["D"]), int(inp["Dv"])
    Dp, Dvp = max(D, D_pad), max(Dv, D_pad)
    out = {"lse": indexed(exp, "lse", (N, H), 0), "delta": indexed(exp, "delta", (N, H), 0)}
    for name, shape, w, wp in (("dQ", (N, H), D, Dp), ("dK", (M, Hkv), D, Dp), ("dV", (M, Hkv), Dv, Dvp),
                               ("O", (N, H), Dv, Dvp)):
        a = indexed(exp, name, shape, w)
        full = np.zeros(shape + (wp,), dtype=np.float64)
        full[..., :w] = a
        out[name] = full
    return out
