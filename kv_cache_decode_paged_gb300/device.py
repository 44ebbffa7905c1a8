"""Put a synthetic workload on the device through the C ABI.

Uploads the seeded inputs with torch and fills the paged pools with
kvattn_append; decode calls go through the binding.  Used by the tests, the
benchmark and the smoke check.
"""
from __future__ import annotations

import numpy as np

from . import (KVATTN_BF16, KVATTN_FP8_E4M3, KVATTN_GQA, KVATTN_MLA, PagedCache,
               kvattn_append, kvattn_decode_gqa, kvattn_decode_mla, workspace_for)
from . import inputs


def dev_bits(a: np.ndarray, device="cuda"):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device)
    if a.dtype == np.uint8:
        return torch.from_numpy(a).to(device)
    return torch.from_numpy(a).to(device)


class GpuWorkload:
    """A workload resident on the device: pools filled by kvattn_append."""

    def __init__(self, wl: inputs.Workload, poison: bool = True, device="cuda"):
        import torch
        self.wl = wl
        self.device = device
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.bt = torch.from_numpy(wl.block_table).to(device)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(device)
        self.q = dev_bits(wl.q, device)
        seq_idx, pos = wl.append_indices()
        self.seq_idx = torch.from_numpy(seq_idx).to(device)
        self.pos = torch.from_numpy(pos).to(device)
        if wl.kind == "gqa":
            fp8 = wl.kv_dtype == "fp8"
            dt = KVATTN_FP8_E4M3 if fp8 else KVATTN_BF16
            fill = (inputs.E4M3_NAN if fp8 else inputs.BF16_NAN) if poison else None
            self.cache = PagedCache.allocate_gqa(wl.num_blocks, wl.block_size, wl.h_kv, wl.d,
                                                    dtype=dt, k_scale=wl.k_scale,
                                                    v_scale=wl.v_scale, device=device,
                                                    fill_bits=fill)
            self.k_tok = dev_bits(wl.k, device)
            self.v_tok = dev_bits(wl.v, device)
            self.append(self.k_tok, self.v_tok, self.seq_idx, self.pos)
        else:
            fp8 = wl.kv_dtype == "fp8"
            fill = (inputs.E4M3_NAN if fp8 else inputs.BF16_NAN) if poison else None
            self.cache = PagedCache.allocate_mla(wl.num_blocks, wl.block_size, wl.d_c, wl.d_rope,
                                                    dtype=KVATTN_FP8_E4M3 if fp8 else KVATTN_BF16,
                                                    k_scale=wl.k_scale, v_scale=wl.v_scale,
                                                    device=device, fill_bits=fill)
            self.k_tok = dev_bits(wl.c_kv, device)
            self.v_tok = dev_bits(wl.k_r, device)
            self.append(self.k_tok, self.v_tok, self.seq_idx, self.pos)
        self.desc = self.cache.descriptor()
        self.out = None
        self.lse = None

    def append(self, k, v, seq_idx, pos):
        kvattn_append(self.cache.descriptor(), k, v, seq_idx, pos, self.bt, err=self.err)

    def workspace(self, num_ctas=0):
        wl = self.wl
        if wl.kind == "gqa":
            return workspace_for(KVATTN_GQA, wl.B, wl.h, wl.h_kv, wl.d, num_ctas, self.device)
        return workspace_for(KVATTN_MLA, wl.B, wl.h, 1, wl.d_c, num_ctas, self.device)

    def decode(self, num_ctas=0, ws=None, block_table=None):
        import torch
        wl = self.wl
        ws = self.workspace(num_ctas) if ws is None else ws
        bt = self.bt if block_table is None else block_table
        if wl.kind == "gqa":
            out = torch.empty((wl.B, wl.h, wl.d), dtype=torch.float32, device=self.device)
            lse = torch.empty((wl.B, wl.h), dtype=torch.float32, device=self.device)
            kvattn_decode_gqa(self.q, self.cache.descriptor(), bt, self.seq_lens, wl.h,
                                 wl.h_kv, wl.d, wl.scale, out, lse, ws, num_ctas=num_ctas,
                                 err=self.err)
        else:
            out = torch.empty((wl.B, wl.h, wl.d_c), dtype=torch.float32, device=self.device)
            lse = torch.empty((wl.B, wl.h), dtype=torch.float32, device=self.device)
            kvattn_decode_mla(self.q, self.cache.descriptor(), bt, self.seq_lens, wl.h,
                                 wl.d_c, wl.d_rope, wl.scale, out, lse, ws, num_ctas=num_ctas,
                                 err=self.err)
        torch.cuda.synchronize()
        return out.cpu().numpy(), lse.cpu().numpy()

    def decode_multi(self, q_multi, num_ctas=0, ws=None):
        """Multi-token decode of q_multi [B][q_len][h][d] (bf16 bits or a device
        tensor): returns out [B][q_len][h][d], lse [B][q_len][h]."""
        import torch
        from . import kvattn_decode_gqa_multi
        wl = self.wl
        q = q_multi if isinstance(q_multi, torch.Tensor) else dev_bits(q_multi, self.device)
        q_len = int(q.shape[1])
        if ws is None:
            ws = workspace_for(KVATTN_GQA, wl.B, wl.h * q_len, wl.h_kv, wl.d, num_ctas, self.device)
        out = torch.empty((wl.B, q_len, wl.h, wl.d), dtype=torch.float32, device=self.device)
        lse = torch.empty((wl.B, q_len, wl.h), dtype=torch.float32, device=self.device)
        kvattn_decode_gqa_multi(q, self.cache.descriptor(), self.bt, self.seq_lens, q_len, wl.h,
                                wl.h_kv, wl.d, wl.scale, out, lse, ws, num_ctas=num_ctas,
                                err=self.err)
        torch.cuda.synchronize()
        return out.cpu().numpy(), lse.cpu().numpy()

    def err_bits(self) -> int:
        return int(self.err.item())


