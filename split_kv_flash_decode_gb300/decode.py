"""Convenience layer over the C ABI: a Decoder owns a plan and its workspace.

Shapes and dtypes are checked here (the C ABI sees only pointers); every byte
of compute happens in fd_decode's kernel.
"""
from __future__ import annotations

import torch

from . import _binding as B

# q / out type and K / V storage type of each plan dtype.
_TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "f16_e4m3kv": torch.float16}
_KV_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "f16_e4m3kv": torch.uint8}


class Decoder:
    """Plan + zeroed workspace for one decode shape on one device."""

    def __init__(self, Hq, Hkv, d, seqlens, W, dtype="f16", flags=0, chunks=0, device=None,
                 num_sms=0, page_size=0):
        dev = torch.device(device if device is not None else "cuda")
        if dev.type != "cuda":
            raise ValueError("Decoder needs a CUDA device")
        self.device = torch.device("cuda", dev.index if dev.index is not None
                                   else torch.cuda.current_device())
        self.seqlens = [int(x) for x in seqlens]
        self.Bsz = len(self.seqlens)
        self.Hq, self.Hkv, self.d, self.dtype = int(Hq), int(Hkv), int(d), dtype
        self.n_tokens = sum(self.seqlens)
        self.page_size = int(page_size)
        with torch.cuda.device(self.device):
            if self.page_size:
                self.plan = B.fd_plan_paged(self.Bsz, Hq, Hkv, d, self.seqlens, W, self.page_size,
                                            dtype, flags, chunks, num_sms)
            else:
                self.plan = B.fd_plan(self.Bsz, Hq, Hkv, d, self.seqlens, W, dtype, flags, chunks,
                                      num_sms)
            self.workspace = torch.zeros(max(1, self.plan.workspace_bytes), dtype=torch.uint8,
                                         device=self.device)

    @property
    def info(self) -> dict:
        return self.plan.info

    def _check(self, name, t, shape):
        if t.device != self.device:
            raise ValueError(f"{name} is on {t.device}, expected {self.device}")
        want = (_KV_DTYPE if name in ("k", "v", "k_pages", "v_pages") else _TORCH_DTYPE)[self.dtype]
        if t.dtype != want:
            raise ValueError(f"{name} has dtype {t.dtype}, expected {want}")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")

    def __call__(self, q, k, v, out=None, lse=None, stream=None):
        self._check("q", q, (self.Bsz, self.Hq, self.d))
        self._check("k", k, (self.n_tokens, self.Hkv, self.d))
        self._check("v", v, (self.n_tokens, self.Hkv, self.d))
        if out is None:
            out = torch.empty_like(q)
        else:
            self._check("out", out, (self.Bsz, self.Hq, self.d))
        if lse is None:
            lse = torch.empty((self.Bsz, self.Hq), dtype=torch.float32, device=self.device)
        elif lse.dtype != torch.float32 or tuple(lse.shape) != (self.Bsz, self.Hq):
            raise ValueError("lse must be float32 [B, Hq]")
        with torch.cuda.device(self.device):
            B.fd_decode(self.plan, q, k, v, out, lse, self.workspace, stream)
        return out, lse

    def decode_paged(self, q, k_pages, v_pages, block_table, out=None, lse=None, stream=None):
        """Decode over a paged cache: pools [num_pages, page_size, Hkv, d], int32 block_table [B, stride]."""
        if not self.page_size:
            raise ValueError("this Decoder was planned for contiguous K/V")
        self._check("q", q, (self.Bsz, self.Hq, self.d))
        num_pages = k_pages.shape[0]
        for name, t in (("k_pages", k_pages), ("v_pages", v_pages)):
            self._check(name, t, (num_pages, self.page_size, self.Hkv, self.d))
        if block_table.dtype != torch.int32 or block_table.dim() != 2 or \
                block_table.shape[0] != self.Bsz or not block_table.is_contiguous() or \
                block_table.device != self.device:
            raise ValueError("block_table must be a contiguous int32 [B, stride] tensor on the device")
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((self.Bsz, self.Hq), dtype=torch.float32, device=self.device)
        with torch.cuda.device(self.device):
            B.fd_decode_paged(self.plan, q, k_pages, v_pages, num_pages, block_table,
                              block_table.shape[1], out, lse, self.workspace, stream)
        return out, lse

    def status(self, stream=None) -> int:
        with torch.cuda.device(self.device):
            return B.fd_workspace_status(self.plan, self.workspace, stream)


def flash_decode(q, k, v, seqlens, W, flags=0, chunks=0):
    """One-shot decode: plan, allocate, run.  Returns (out, lse)."""
    dtype = {torch.float16: "f16", torch.bfloat16: "bf16"}[q.dtype]
    if k.dtype == torch.uint8:
        dtype = "f16_e4m3kv"
    dec = Decoder(q.shape[1], k.shape[1], q.shape[2], seqlens, W, dtype, flags, chunks,
                  device=q.device)
    return dec(q, k, v)
