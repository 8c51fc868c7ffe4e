"""PyTorch-facing wrapper: allocation with torch, one call of fa_back on the current stream."""
from __future__ import annotations

from typing import Optional

import torch

from . import _native as nat


class FaBackError(RuntimeError):
    pass


def _check(rc: int):
    if rc != 0:
        raise FaBackError(f"fa_back failed: {nat.STATUS.get(rc, rc)} ({nat.fa_back_status_string(rc)})")


class Workspace:
    """Reusable device workspace (grown on demand, owned by PyTorch's allocator)."""

    def __init__(self, device="cuda"):
        self.device = torch.device(device)
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def backward(q: torch.Tensor, k: torch.Tensor, k_type: int, v: torch.Tensor, v_type: int, dO: torch.Tensor,
             *, H: int, Hkv: int, D: int, Dv: int, M: int, scale: float, causal: bool = False,
             mask: Optional[torch.Tensor] = None, mask_heads: int = 0, out: Optional[dict] = None,
             workspace: Optional[Workspace] = None, stream: Optional[torch.cuda.Stream] = None,
             workspace_bytes: Optional[int] = None, lse: Optional[torch.Tensor] = None,
             delta: Optional[torch.Tensor] = None, alibi_slopes: Optional[torch.Tensor] = None,
             softcap: float = 0.0, sinks: Optional[torch.Tensor] = None, nocopy: bool = False) -> dict:
    """Run the backward on device tensors.

    q [N][H][D] f32, dO [N][H][Dv] f32, k/v uint8 raw cache rows [M][Hkv][row], mask int16/uint16
    binary16 bits [Hm][N][M] or None.  Returns {"dQ", "dK", "dV", "lse", "delta"} (f32 tensors).
    workspace_bytes (default fa_back_workspace_size) is the workspace given to fa_back, which
    runs the fastest plan that fits it (at least fa_back_workspace_size_min).  Given the forward's
    row statistics lse and delta ([N][H] f32), fa_back_with_stats runs instead and the result
    holds dQ, dK and dV only.  With ALiBi slopes ([H] f32), a soft cap c > 0 or sink logits ([H]
    f32), fa_back_ext runs; with sinks the result also holds "dsinks" ([H] f32).  nocopy runs
    fa_back_nocopy (plans without a decoded copy of the cache; default workspace
    fa_back_workspace_size_nocopy).
    """
    N = q.shape[0]
    dev = q.device
    if out is None:
        out = {
            "dQ": torch.empty((N, H, D), dtype=torch.float32, device=dev),
            "dK": torch.empty((M, Hkv, D), dtype=torch.float32, device=dev),
            "dV": torch.empty((M, Hkv, Dv), dtype=torch.float32, device=dev),
            "lse": torch.empty((N, H), dtype=torch.float32, device=dev),
            "delta": torch.empty((N, H), dtype=torch.float32, device=dev),
        }
    given = lse is not None or delta is not None
    if given and (lse is None or delta is None):
        raise FaBackError("lse and delta are given together")
    ext = alibi_slopes is not None or softcap != 0.0 or sinks is not None
    if ext and given:
        raise FaBackError("the score extensions need the backward's own lse/delta pass")
    if nocopy and (ext or given):
        raise FaBackError("nocopy runs the plain backward")
    if sinks is not None and "dsinks" not in out:
        out["dsinks"] = torch.empty((H,), dtype=torch.float32, device=dev)
    if given:
        out.pop("lse", None)
        out.pop("delta", None)
    for t in (q, k, v, dO, mask, lse, delta, alibi_slopes, sinks, *out.values()):
        if t is not None and not t.is_contiguous():
            raise FaBackError("tensors must be contiguous")
    size_fn = nat.fa_back_workspace_size_nocopy if nocopy else nat.fa_back_workspace_size
    ws_bytes = size_fn(N, M, H, Hkv, D, Dv) if workspace_bytes is None else int(workspace_bytes)
    ws = (workspace or Workspace(dev)).get(ws_bytes)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    nbytes = ws.numel() if workspace_bytes is None else ws_bytes
    if given:
        rc = nat.fa_back_with_stats(_ptr(q), _ptr(k), k_type, _ptr(v), v_type, _ptr(mask), mask_heads, _ptr(dO),
                                    _ptr(lse), _ptr(delta), scale, N, M, H, Hkv, D, Dv, causal, _ptr(out["dQ"]),
                                    _ptr(out["dK"]), _ptr(out["dV"]), ws.data_ptr(), nbytes, s.cuda_stream)
    elif nocopy:
        rc = nat.fa_back_nocopy(_ptr(q), _ptr(k), k_type, _ptr(v), v_type, _ptr(mask), mask_heads, _ptr(dO), scale,
                                N, M, H, Hkv, D, Dv, causal, _ptr(out["dQ"]), _ptr(out["dK"]), _ptr(out["dV"]),
                                _ptr(out["lse"]), _ptr(out["delta"]), ws.data_ptr(), nbytes, s.cuda_stream)
    elif ext:
        rc = nat.fa_back_ext(_ptr(q), _ptr(k), k_type, _ptr(v), v_type, _ptr(mask), mask_heads, _ptr(dO), scale,
                             N, M, H, Hkv, D, Dv, causal, _ptr(alibi_slopes), softcap, _ptr(sinks),
                             _ptr(out.get("dsinks")), _ptr(out["dQ"]), _ptr(out["dK"]), _ptr(out["dV"]),
                             _ptr(out["lse"]), _ptr(out["delta"]), ws.data_ptr(), nbytes, s.cuda_stream)
    else:
        rc = nat.fa_back(_ptr(q), _ptr(k), k_type, _ptr(v), v_type, _ptr(mask), mask_heads, _ptr(dO), scale,
                         N, M, H, Hkv, D, Dv, causal, _ptr(out["dQ"]), _ptr(out["dK"]), _ptr(out["dV"]),
                         _ptr(out["lse"]), _ptr(out["delta"]), ws.data_ptr(), nbytes, s.cuda_stream)
    _check(rc)
    return out


def forward(q: torch.Tensor, k: torch.Tensor, k_type: int, v: torch.Tensor, v_type: int, *, H: int, Hkv: int,
            D: int, Dv: int, M: int, scale: float, causal: bool = False, mask: Optional[torch.Tensor] = None,
            mask_heads: int = 0, workspace: Optional[Workspace] = None,
            stream: Optional[torch.cuda.Stream] = None) -> dict:
    """The forward over the raw cache: {"O": [N][H][Dv], "lse": [N][H]} (f32 tensors)."""
    N = q.shape[0]
    dev = q.device
    out = {"O": torch.empty((N, H, Dv), dtype=torch.float32, device=dev),
           "lse": torch.empty((N, H), dtype=torch.float32, device=dev)}
    for t in (q, k, v, mask):
        if t is not None and not t.is_contiguous():
            raise FaBackError("tensors must be contiguous")
    ws = (workspace or Workspace(dev)).get(nat.fa_forward_workspace_size(N, M, H, Hkv, D, Dv))
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    rc = nat.fa_forward(_ptr(q), _ptr(k), k_type, _ptr(v), v_type, _ptr(mask), mask_heads, scale, N, M, H, Hkv, D,
                        Dv, causal, _ptr(out["O"]), _ptr(out["lse"]), ws.data_ptr(), ws.numel(), s.cuda_stream)
    _check(rc)
    return out


def backward_strided(q: torch.Tensor, k: torch.Tensor, k_type: int, v: torch.Tensor, v_type: int, dO: torch.Tensor,
                     *, H: int, Hkv: int, D: int, Dv: int, M: int, scale: float, causal: bool = False,
                     mask: Optional[torch.Tensor] = None, mask_heads: int = 0, mask_bits: bool = False,
                     out: Optional[dict] = None, workspace: Optional[Workspace] = None,
                     stream: Optional[torch.cuda.Stream] = None, workspace_bytes: Optional[int] = None) -> dict:
    """fa_back_strided on device tensors that may be views.

    q [N][H][D] and dO [N][H][Dv] f32 with any non-negative strides; k, v uint8 [M][Hkv][row] with
    each row contiguous (last stride 1, the other two even); mask [Hm][N][M] binary16 bits
    (int16/uint16/float16) with the keys contiguous, or, with mask_bits, int32 words
    [Hm][N][ceil(M/32)] whose bit j % 32 of word j / 32 is set where key j is allowed.  The
    outputs are contiguous, as for backward().
    """
    N = q.shape[0]
    dev = q.device
    if out is None:
        out = {
            "dQ": torch.empty((N, H, D), dtype=torch.float32, device=dev),
            "dK": torch.empty((M, Hkv, D), dtype=torch.float32, device=dev),
            "dV": torch.empty((M, Hkv, Dv), dtype=torch.float32, device=dev),
            "lse": torch.empty((N, H), dtype=torch.float32, device=dev),
            "delta": torch.empty((N, H), dtype=torch.float32, device=dev),
        }
    for t in out.values():
        if not t.is_contiguous():
            raise FaBackError("outputs must be contiguous")
    for name, t in (("k", k), ("v", v)):
        if t.dim() != 3 or t.stride(2) != 1 or t.element_size() != 1:
            raise FaBackError(f"{name}: uint8 [M][Hkv][row] with contiguous rows expected")
    if mask is not None and (mask.dim() != 3 or mask.stride(2) != 1):
        raise FaBackError("mask: [Hm][N][keys or words] with the last dimension contiguous expected")
    for name, t in (("q", q), ("dO", dO)):
        if t.dim() != 3:
            raise FaBackError(f"{name}: [N][H][D] expected")
    st = nat.fa_strides(q_row=q.stride(0), q_head=q.stride(1), q_comp=q.stride(2),
                        do_row=dO.stride(0), do_head=dO.stride(1), do_comp=dO.stride(2),
                        k_cell=k.stride(0), k_head=k.stride(1), v_cell=v.stride(0), v_head=v.stride(1),
                        mask_head=0 if mask is None else mask.stride(0), mask_row=0 if mask is None else mask.stride(1))
    Hm = mask_heads if mask is not None else 0
    need = nat.fa_back_strided_workspace_size(N, M, H, Hkv, D, Dv, k_type, v_type, Hm)
    ws_bytes = need if workspace_bytes is None else int(workspace_bytes)
    ws = (workspace or Workspace(dev)).get(ws_bytes)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    fmt = nat.FA_MASK_BITS if mask_bits else nat.FA_MASK_F16
    rc = nat.fa_back_strided(_ptr(q), _ptr(k), k_type, _ptr(v), v_type, _ptr(mask), fmt, mask_heads, _ptr(dO), st,
                             scale, N, M, H, Hkv, D, Dv, causal, _ptr(out["dQ"]), _ptr(out["dK"]), _ptr(out["dV"]),
                             _ptr(out["lse"]), _ptr(out["delta"]), ws.data_ptr(), ws_bytes, s.cuda_stream)
    _check(rc)
    return out
