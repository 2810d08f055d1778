"""One target-verify step on the GPU, through the C ABI, for a synthetic batch.

``DeviceBatch`` holds a workload's inputs resident in device memory together
with every output buffer and the workspace; ``run_step`` runs the whole hot
path in order:

  build_tree_mask -> write_window_kv -> tree_verify_attention
  -> verify_tree_greedy -> compact_window_rows -> compact_rows

by default as three calls: verify_prologue (the first two), the attention,
verify_epilogue (the last three).

(the caller's logits/argmax sit between the attention and the walk; the
synthetic batch provides target_argmax directly). All calls go to one CUDA
stream; nothing synchronises inside a step.
"""
from __future__ import annotations

from typing import List, Optional

import numpy as np

from . import synth
from . import (build_tree_mask, write_window_kv, tree_verify_attention, tree_verify_attention_workspace,
               verify_tree_greedy, compact_window_rows, compact_rows, make_kv_table, verify_prologue,
               verify_epilogue)


def _torch():
    import torch
    return torch


def bf16_tensor(bits: np.ndarray, device):
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


class DeviceBatch:
    """Device-resident inputs, outputs and scratch of one verify step."""

    KERNELS_PER_STEP = 5  # prologue, attention prep, tree attention, merge, epilogue

    def __init__(self, inp: synth.VerifyInputs, device="cuda", fp8_layers: Optional[int] = None,
                 compact_attention_kv: bool = True):
        torch = _torch()
        w = inp.w
        self.w = w
        self.inp = inp
        self.device = device
        B, N = w.B, w.N
        i32 = torch.int32
        dev = device
        self.B, self.N = B, N
        self.max_prefix = int(inp.vc.max()) if B else 0
        self.page_size = w.page_size
        self.parents = torch.from_numpy(inp.parents).to(dev)
        self.depth = torch.from_numpy(inp.depth).to(dev)
        self.vc = torch.from_numpy(inp.vc.astype(np.int32)).to(dev)
        self.prefix_len = self.vc
        self.page_table = torch.from_numpy(inp.layout.page_table).to(dev)
        self.draft = torch.from_numpy(inp.draft).to(dev)
        self.target_argmax = torch.from_numpy(inp.target_argmax).to(dev)
        self.q = bf16_tensor(inp.q, dev)
        self.k_new = bf16_tensor(inp.k_new, dev)
        self.v_new = bf16_tensor(inp.v_new, dev)
        self.k_cache = bf16_tensor(inp.k_cache, dev)
        self.v_cache = bf16_tensor(inp.v_cache, dev)
        self.hidden = bf16_tensor(inp.hidden, dev) if inp.hidden is not None else None
        # outputs
        self.mask = torch.zeros((B, N), dtype=torch.int64, device=dev)
        self.positions = torch.zeros((B, N), dtype=i32, device=dev)
        self.next_token = torch.zeros((B, N), dtype=i32, device=dev)
        self.next_sibling = torch.zeros((B, N), dtype=i32, device=dev)
        self.write_locations = torch.zeros(B * N, dtype=torch.int64, device=dev)
        self.out = torch.zeros((B * N, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
        self.lse2 = torch.zeros((B * N, w.Hq), dtype=torch.float32, device=dev)
        ws = tree_verify_attention_workspace(B, N, w.Hq, w.Hkv, w.d, self.max_prefix)
        self.workspace = torch.empty(max(ws, 16) // 16 * 16 + 16, dtype=torch.uint8, device=dev)
        self.accept_len = torch.zeros(B, dtype=i32, device=dev)
        self.accepted_path = torch.zeros((B, N), dtype=i32, device=dev)
        self.accepted_tokens = torch.zeros((B, N), dtype=i32, device=dev)
        self.err = torch.zeros(1, dtype=i32, device=dev)
        # compaction: the attention layer's K and V, plus fp8 K/V buffers of `fp8_layers` layers
        self.fp8_buffers: List = []
        entries = []
        row_kv = w.Hkv * w.d * 2
        if compact_attention_kv:
            entries += [(self.k_cache, row_kv, self.k_cache.shape[0], row_kv),
                        (self.v_cache, row_kv, self.v_cache.shape[0], row_kv)]
        nl = w.fp8_layers if fp8_layers is None else fp8_layers
        if nl:
            row8 = w.Hkv * w.d  # one fp8 byte per element
            rows = synth.fp8_window_rows(w, 2 * nl, row8)
            wl = torch.from_numpy(inp.layout.write_locations).to(dev)
            for k in range(2 * nl):
                buf = torch.zeros((inp.layout.num_slots, row8), dtype=torch.uint8, device=dev)
                buf[wl] = torch.from_numpy(rows[k]).to(dev)
                self.fp8_buffers.append(buf)
                entries.append((buf, row8, buf.shape[0], row8))
        self.kv_entries = entries
        self.kv_table = make_kv_table(entries, device=dev) if entries else None

    # the individual calls -------------------------------------------------
    def mask_step(self, stream=None):
        build_tree_mask(self.parents, self.depth, self.vc, self.mask, self.positions, self.next_token,
                        self.next_sibling, err=self.err, stream=stream)

    def window_kv_step(self, stream=None):
        write_window_kv(self.k_new, self.v_new, self.positions, self.page_table, self.page_size, self.prefix_len,
                        self.k_cache, self.v_cache, self.w.rope_theta, write_locations=self.write_locations,
                        err=self.err, stream=stream, N=self.N)

    def attention_step(self, stream=None):
        tree_verify_attention(self.q, self.k_cache, self.v_cache, self.page_table, self.page_size, self.prefix_len,
                              self.max_prefix, self.mask, self.positions, self.w.rope_theta, self.out, self.lse2,
                              self.workspace, err=self.err, stream=stream, N=self.N)

    def walk_step(self, stream=None):
        verify_tree_greedy(self.draft, self.target_argmax, self.accept_len, self.accepted_path,
                           self.accepted_tokens, next_token=self.next_token, next_sibling=self.next_sibling,
                           err=self.err, stream=stream)

    # the fused launches: mask + window K/V, and walk + both compactions
    def prologue_step(self, stream=None):
        verify_prologue(self.parents, self.depth, self.vc, self.k_new, self.v_new, self.page_table, self.page_size,
                        self.prefix_len, self.k_cache, self.v_cache, self.w.rope_theta, self.mask, self.positions,
                        self.next_token, self.next_sibling, write_locations=self.write_locations, err=self.err,
                        stream=stream)

    def epilogue_step(self, stream=None, target_argmax=None):
        verify_epilogue(self.draft, self.target_argmax if target_argmax is None else target_argmax, self.accept_len,
                        self.accepted_path, self.accepted_tokens, table=self.kv_table,
                        write_locations=self.write_locations, hidden=self.hidden, positions=self.positions,
                        vc=self.vc, next_token=self.next_token, next_sibling=self.next_sibling, err=self.err,
                        stream=stream)

    def compact_step(self, stream=None):
        if self.kv_table is not None:
            compact_window_rows(self.kv_table, self.write_locations, self.accepted_path, self.accept_len,
                                err=self.err, stream=stream)
        compact_rows(self.hidden, self.positions, self.vc, self.accepted_path, self.accept_len, err=self.err,
                     stream=stream)


def run_step(db: DeviceBatch, stream=None, compact: bool = True, fused: bool = True):
    """One pass of the whole hot path; returns nothing (outputs stay on the
    device). fused: the prologue (mask + window K/V) and epilogue (walk +
    compactions) launches; otherwise the separate calls."""
    if fused and compact:
        db.prologue_step(stream)
        db.attention_step(stream)
        db.epilogue_step(stream)
        return
    db.mask_step(stream)
    db.window_kv_step(stream)
    db.attention_step(stream)
    db.walk_step(stream)
    if compact:
        db.compact_step(stream)
