"""A paged K/V cache held in torch device memory, driven through libpa.

``PagedKVCache`` owns the allocator state (``Pool``), the device K and V
pools, a device error word and a reusable decode workspace.  Every operation is
one libpa call on the current CUDA stream; this module only allocates torch
buffers and passes pointers.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (PA_OK, PaError, Pool, load, pa_append_rows, pa_append_rows_f16, pa_decode, pa_decode_workspace_size,
               pa_get_error)


class PagedKVCache:
    def __init__(self, n_blocks: int, page_size: int, k_type: int, v_type: int | None = None,
                 n_kv_heads: int = 4, head_dim: int = 256, device: torch.device | str = "cuda"):
        load()
        self.device = torch.device(device)
        self.pool = Pool(n_blocks, page_size, n_kv_heads, head_dim, k_type, v_type)
        self.page_size = page_size
        self.n_blocks = n_blocks
        self.n_kv_heads = n_kv_heads
        self.head_dim = head_dim
        self.k_type = k_type
        self.v_type = k_type if v_type is None else v_type
        self.k_pool = torch.zeros(self.pool.bytes(0), dtype=torch.uint8, device=self.device)
        self.v_pool = torch.zeros(self.pool.bytes(1), dtype=torch.uint8, device=self.device)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._ws = None
        self._ws_key = None

    # ------------------------------------------------------------ append
    def append(self, k_rows: torch.Tensor, v_rows: torch.Tensor, row_seq: torch.Tensor, row_pos: torch.Tensor,
               block_table: torch.Tensor, stream=None) -> None:
        """Scatter packed rows [n][n_kv_heads][row_bytes] (device uint8) into the pools."""
        n = int(row_seq.shape[0])
        pa_append_rows(self.pool, self.k_pool, self.v_pool, k_rows, v_rows, row_seq, row_pos, n, block_table,
                       int(block_table.shape[1]), int(block_table.shape[0]), self.err, stream)

    def append_f16(self, k_rows: torch.Tensor, v_rows: torch.Tensor, row_seq: torch.Tensor, row_pos: torch.Tensor,
                   block_table: torch.Tensor, stream=None) -> None:
        """Quantise binary16 rows [n][n_kv_heads][head_dim] (device, float16 or their uint16
        bit patterns) into the pools' formats while scattering them."""
        n = int(row_seq.shape[0])
        pa_append_rows_f16(self.pool, self.k_pool, self.v_pool, k_rows, v_rows, row_seq, row_pos, n, block_table,
                           int(block_table.shape[1]), int(block_table.shape[0]), self.err, stream)

    # ------------------------------------------------------------ decode
    def workspace(self, n_seq: int, n_qtok: int) -> torch.Tensor:
        dev = self.device.index if self.device.index is not None else torch.cuda.current_device()
        key = (n_seq, n_qtok, dev)
        if self._ws is None or self._ws_key != key:
            nbytes = pa_decode_workspace_size(self.pool, n_seq, n_qtok, dev)
            if nbytes == 0:
                raise PaError(1, "pa_decode_workspace_size")
            self._ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            self._ws_key = key
        return self._ws

    def decode(self, q: torch.Tensor, block_table: torch.Tensor, seq_lens_dev: torch.Tensor,
               seq_lens_host: np.ndarray, n_qtok: int, scale: float = 1.0 / 16.0, out: torch.Tensor | None = None,
               lse: torch.Tensor | None = None, want_lse: bool = True, stream=None, passes: str = "all"):
        """q: device fp32 [n_seq][n_qtok][n_q_heads][head_dim]; returns (out, lse)."""
        n_seq, _, hq, d = q.shape
        if out is None:
            out = torch.empty((n_seq, n_qtok, hq, d), dtype=torch.float32, device=self.device)
        if lse is None and want_lse:
            lse = torch.empty((n_seq, n_qtok, hq), dtype=torch.float32, device=self.device)
        sl = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
        ws = self.workspace(n_seq, n_qtok)
        pa_decode(self.pool, q, self.k_pool, self.v_pool, block_table, int(block_table.shape[1]), seq_lens_dev, sl,
                  n_seq, n_qtok, hq, scale, out, lse, ws, ws.numel(), self.err, stream, passes=passes)
        return out, lse

    def check(self, stream=None) -> int:
        """Synchronise, read and reset the device error word."""
        return pa_get_error(self.err, stream)

    def raise_on_error(self, stream=None) -> None:
        rc = self.check(stream)
        if rc != PA_OK:
            raise PaError(rc, "device")
