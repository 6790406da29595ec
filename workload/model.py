"""Synthetic MoE stacks in device (or pinned host) memory for tests and the benchmark.

The weights are drawn by the seeded generators of this package and packed with
the library's own packer (tf_pack_expert), i.e. exactly the way a user would
load real weights. Nothing here computes any part of the layer.
"""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import workload as W
import bit_expert_streaming_layer_b300 as B

DEFAULT = dict(H=2816, I=704, E=128, k=8, S=2112)


def _u16_to_bf16_tensor(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def expert_logical_concat(seed: int, layer: int, e: int, H: int, I: int):
    """Logical codes, scales and biases of one expert, concatenated gate, up, down (tf_pack_expert input)."""
    L = W.lib()
    n_gu, n_d = I * H, H * I
    g_gu, g_d = I * H // W.GROUP, H * I // W.GROUP
    q = np.empty(2 * n_gu + n_d, np.uint8)
    s = np.empty(2 * g_gu + g_d, np.uint16)
    b = np.empty(2 * g_gu + g_d, np.uint16)
    qo = (0, n_gu, 2 * n_gu)
    so = (0, g_gu, 2 * g_gu)
    sizes = ((n_gu, g_gu), (n_gu, g_gu), (n_d, g_d))
    for m in range(3):
        nq, ng = sizes[m]
        L.wl_codes(W.key(seed, W.T_Q, layer, e, m), nq,
                   ctypes.cast(q.ctypes.data + qo[m], ctypes.POINTER(ctypes.c_uint8)))
        L.wl_uniform_f16(W.key(seed, W.T_S, layer, e, m), ng, W.SCALE_LO, W.SCALE_HI,
                         ctypes.cast(s.ctypes.data + 2 * so[m], ctypes.POINTER(ctypes.c_uint16)))
        L.wl_uniform_f16(W.key(seed, W.T_B, layer, e, m), ng, W.BIAS_LO, W.BIAS_HI,
                         ctypes.cast(b.ctypes.data + 2 * so[m], ctypes.POINTER(ctypes.c_uint16)))
    return q, s, b


def pack_layer_experts(seed: int, layer: int, E: int, H: int, I: int, host: torch.Tensor, offset: int = 0,
                       workers: int | None = None) -> None:
    """Generate and pack experts 0..E-1 of `layer` into a host uint8 tensor at offset + e * slot_bytes."""
    slot = B.tf_expert_slot_bytes(H, I)
    base = host.data_ptr() + offset
    workers = workers or min(32, os.cpu_count() or 1)

    def one(e):
        q, s, b = expert_logical_concat(seed, layer, e, H, I)
        B.tf_pack_expert(q, s, b, H, I, base + e * slot)

    with ThreadPoolExecutor(workers) as ex:
        list(ex.map(one, range(E)))


class SyntheticStack:
    """L MoE layers with seeded weights.

    resident=True : all L*E experts live in one device array (stride slot_bytes).
    resident=False: experts live in a pinned host store (L*E slots) and the device
                    holds only a pool of n_slots per layer for the LFU cache.
    """

    def __init__(self, seed: int, L: int, H=2816, I=704, E=128, k=8, S=2112, resident=True, n_slots=16,
                 T_max: int = 1, device="cuda"):
        self.seed, self.L, self.H, self.I, self.E, self.k, self.S = seed, L, H, I, E, k, S
        self.resident, self.n_slots, self.T_max = resident, n_slots, T_max
        self.slot = B.tf_expert_slot_bytes(H, I)
        self.payload = B.tf_expert_payload_bytes(H, I)
        dev = torch.device(device)
        self.Wr, self.Wsg, self.Wsu, self.Wsd = [], [], [], []
        workers = min(32, os.cpu_count() or 1)

        def dense(l):
            wr = W.router_weights(seed, l, E, H)
            sh = W.shared_weights(seed, l, H, S) if S > 0 else None
            return wr, sh

        with ThreadPoolExecutor(workers) as ex:
            for wr, sh in ex.map(dense, range(L)):
                self.Wr.append(_u16_to_bf16_tensor(wr).to(dev))
                if sh is not None:
                    for lst, a in zip((self.Wsg, self.Wsu, self.Wsd), sh):
                        lst.append(_u16_to_bf16_tensor(a).to(dev))
        layer_bytes = E * self.slot
        if resident:
            self.experts = torch.empty(L * layer_bytes, dtype=torch.uint8, device=dev)
            stage = torch.empty(layer_bytes, dtype=torch.uint8, pin_memory=True)
            for l in range(L):
                pack_layer_experts(seed, l, E, H, I, stage)
                self.experts[l * layer_bytes:(l + 1) * layer_bytes].copy_(stage, non_blocking=False)
            self.store = None
            self.pool = None
        else:
            self.store = torch.empty(L * layer_bytes, dtype=torch.uint8, pin_memory=True)
            for l in range(L):
                pack_layer_experts(seed, l, E, H, I, self.store, l * layer_bytes)
            self.pool = torch.zeros(L * n_slots * self.slot, dtype=torch.uint8, device=dev)
            self.experts = None
        self.layers, self.workspaces = [], []
        for l in range(L):
            table = (B.expert_table(self.experts.data_ptr() + l * layer_bytes, self.slot) if resident
                     else B.ExpertTable(None, 0, None))
            desc = B.layer_desc(H, I, E, k, S, self.Wr[l], self.Wsg[l] if S else None, self.Wsu[l] if S else None,
                                self.Wsd[l] if S else None, table)
            nbytes = B.tf_layer_workspace_bytes(desc, T_max)
            ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
            self.workspaces.append(ws)
            self.layers.append(B.Layer(desc, T_max, ws))
        self.cache = None
        if not resident:
            self.cache = B.ExpertCache(L, n_slots, E, self.slot, self.pool)

    def layer_table(self, l: int) -> B.ExpertTable:
        return B.expert_table(self.experts.data_ptr() + l * self.E * self.slot, self.slot)

    def close(self):
        for ly in self.layers:
            ly.close()
        if self.cache is not None:
            self.cache.close()


def hidden_tensor(seed: int, step: int, T: int, H: int, device="cuda") -> torch.Tensor:
    return _u16_to_bf16_tensor(W.hidden(seed, step, T, H)).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
