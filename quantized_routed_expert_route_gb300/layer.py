"""A resident MoE layer on top of the C ABI, with torch used only for device
memory and streams.

    layer = MoeLayer(geom_tuple, gate_up_rows, down_rows, scale_bank, device="cuda")
    out = layer.decode(x_bf16, topk_ids, topk_w)          # all on the device

``decode`` enqueues the library's kernels on torch's current stream and
returns without synchronizing, so it can be captured in a CUDA graph.
"""
from __future__ import annotations

import torch

from . import capi


class MoeLayer:
    def __init__(self, H: int, I: int, E: int, top_k: int, gate_up_type: int, down_type: int,
                 gate_up, down, scale_bank=None, borrow: bool = False, max_tokens: int = capi.MOE_DECODE_T_CHUNK,
                 glu: int = capi.MOE_GLU_SILU):
        """gate_up / down: uint8 tensors (host or CUDA) holding the compact rows;
        scale_bank: fp32 [E, 4] tensor on the same device, or None (ones).
        borrow=True keeps the CUDA tensors as the bank (no copy).  glu:
        MOE_GLU_SILU or MOE_GLU_GELU_TANH."""
        self.geom = capi.moe_layer_geom(H, I, E, top_k, gate_up_type, down_type, glu)
        self.H, self.I, self.E, self.top_k = H, I, E, top_k
        on_dev = gate_up.is_cuda
        if borrow and not on_dev:
            raise ValueError("borrow needs CUDA tensors")
        src = capi.MOE_SRC_DEVICE_BORROW if borrow else (capi.MOE_SRC_DEVICE if on_dev else capi.MOE_SRC_HOST)
        gate_up = gate_up.contiguous()
        down = down.contiguous()
        if scale_bank is not None:
            scale_bank = scale_bank.to(torch.float32).contiguous()
            if scale_bank.is_cuda != on_dev:
                raise ValueError("scale_bank must live with the rows")
        self._keep = (gate_up, down, scale_bank) if borrow else (scale_bank,)
        stream = torch.cuda.current_stream().cuda_stream
        self.bank = capi.moe_bank_create(self.geom, gate_up.data_ptr(), gate_up.numel(), down.data_ptr(),
                                         down.numel(), scale_bank.data_ptr() if scale_bank is not None else 0,
                                         src, stream)
        self.ws_bytes = capi.moe_workspace_bytes(self.bank, max_tokens)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        capi.moe_workspace_init(self.ws.data_ptr(), self.ws_bytes, stream)

    def decode(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor,
               out: torch.Tensor | None = None) -> torch.Tensor:
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        capi.moe_decode(self.bank, x.data_ptr(), T, topk_ids.data_ptr(), topk_w.data_ptr(), out.data_ptr(),
                        self.ws.data_ptr(), self.ws_bytes, torch.cuda.current_stream().cuda_stream)
        return out

    def error_bits(self) -> int:
        return capi.moe_get_error(self.ws.data_ptr(), self.ws_bytes, torch.cuda.current_stream().cuda_stream)

    def close(self) -> None:
        if getattr(self, "bank", None):
            capi.moe_bank_destroy(self.bank)
            self.bank = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
