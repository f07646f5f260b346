"""Device set-up of a synthetic workload and one step of the hot path.

Moves a :class:`workloads.Workload` onto the GPU, writes its history into
zeroed caches through the library (slot mapping + append), and runs the
timed step: slot mapping of this step's rows, their append, and attention of
every query row.  Used by the benchmark, the smoke check and the GPU tests.
"""
import numpy as np
import torch

from . import (pkv_append, pkv_attention, pkv_attention_plan, pkv_attention_run, pkv_attention_workspace_size,
               pkv_slot_mapping)
from .workloads import Workload

CACHE_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}


def to_torch(a: np.ndarray, fmt: str, device) -> torch.Tensor:
    """numpy rows (f32, or bf16 bit patterns) -> a device tensor."""
    if fmt == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return t.to(device)


def cache_to_numpy(c: torch.Tensor) -> np.ndarray:
    """A device cache -> numpy in the oracle's storage format."""
    if c.dtype == torch.bfloat16:
        return c.view(torch.int16).cpu().numpy().view(np.uint16)
    if c.dtype == torch.float8_e4m3fn:
        return c.view(torch.uint8).cpu().numpy()
    return c.cpu().numpy()


class DeviceStep:
    """One workload resident on the GPU.

    layers > 1 keeps that many independent caches (the same contents), so
    that consecutive steps can read different memory, as the layers of a
    model do.
    """

    def __init__(self, wl: Workload, device="cuda", out_dtype=torch.float32, layers: int = 1,
                 max_q_len: int = None, slot_dtype=torch.int32, history_batch: int = 1 << 21,
                 soft_cap: float = 0.0, window_left: int = -1):
        self.wl = wl
        self.soft_cap, self.window_left = soft_cap, window_left
        self.device = torch.device(device)
        dev = self.device
        self.bt = torch.from_numpy(np.ascontiguousarray(wl.block_tables, np.int32)).to(dev)
        self.seq_lens = torch.from_numpy(wl.seq_lens.astype(np.int32)).to(dev)
        self.cu_q = torch.from_numpy(wl.cu_seqlens_q).to(dev)
        self.q = to_torch(wl.q, wl.src, dev)
        kn, vn = wl.new_rows()
        self.k_new = to_torch(kn, wl.src, dev)
        self.v_new = to_torch(vn, wl.src, dev)
        self.T = wl.T
        self.max_q_len = int(wl.q_lens.max()) if max_q_len is None and wl.B else (max_q_len or 0)
        cdt = CACHE_DTYPE[wl.kv]
        self.caches = []
        for _ in range(layers):
            kc = torch.zeros(wl.cache_shape(), dtype=cdt, device=dev)
            vc = torch.zeros(wl.cache_shape(), dtype=cdt, device=dev)
            self.caches.append((kc, vc))
        for s0, s1, cu, sl, k, v in wl.history_batches(history_batch):
            if k.shape[0] == 0:
                continue
            cu_t = torch.from_numpy(cu).to(dev)
            sl_t = torch.from_numpy(sl.astype(np.int32)).to(dev)
            bt_t = self.bt[s0:s1]
            kt, vt = to_torch(k, wl.src, dev), to_torch(v, wl.src, dev)
            slots = pkv_slot_mapping(cu_t, sl_t, bt_t, wl.block_size, T=k.shape[0])
            for kc, vc in self.caches:
                pkv_append(kt, vt, slots, kc, vc, wl.k_scale, wl.v_scale)
        self.slots = torch.empty(self.T, dtype=slot_dtype, device=dev)
        self.out = torch.empty((self.T, wl.Hq, wl.D), dtype=out_dtype, device=dev)
        self.ws = torch.empty(max(1, pkv_attention_workspace_size(self.q, self.bt, self.caches[0][0])),
                              dtype=torch.uint8, device=dev)

    def step(self, layer: int = 0, out=None):
        """One pass of the hot path on one layer's caches."""
        wl = self.wl
        kc, vc = self.caches[layer]
        pkv_slot_mapping(self.cu_q, self.seq_lens, self.bt, wl.block_size, out=self.slots)
        pkv_append(self.k_new, self.v_new, self.slots, kc, vc, wl.k_scale, wl.v_scale)
        pkv_attention(self.q, self.cu_q, self.seq_lens, self.bt, kc, vc, wl.scale,
                      self.out if out is None else out, wl.k_scale, wl.v_scale, self.max_q_len, self.ws,
                      soft_cap=self.soft_cap, window_left=self.window_left)
        return self.out if out is None else out

    def attention_only(self, layer: int = 0, out=None):
        wl = self.wl
        kc, vc = self.caches[layer]
        pkv_attention(self.q, self.cu_q, self.seq_lens, self.bt, kc, vc, wl.scale,
                      self.out if out is None else out, wl.k_scale, wl.v_scale, self.max_q_len, self.ws,
                      soft_cap=self.soft_cap, window_left=self.window_left)
        return self.out if out is None else out

    # ---- one plan per model step, one run per layer
    def plan(self):
        """The work lists of this step's lengths, into the workspace."""
        pkv_attention_plan(self.q, self.cu_q, self.seq_lens, self.bt, self.caches[0][0], self.ws,
                           max_q_len=self.max_q_len, window_left=self.window_left)

    def run(self, layer: int = 0, out=None, q=None):
        """Attention of one layer over the plan in the workspace."""
        wl = self.wl
        kc, vc = self.caches[layer]
        out = self.out if out is None else out
        pkv_attention_run(self.q if q is None else q, self.cu_q, self.seq_lens, self.bt, kc, vc, wl.scale, out,
                          self.ws, wl.k_scale, wl.v_scale, self.max_q_len, soft_cap=self.soft_cap,
                          window_left=self.window_left)
        return out

    def layer_step(self, layer: int = 0, out=None):
        """The per-layer part of a model step whose slots and plan are
        already made: append of the layer's new rows, then attention."""
        wl = self.wl
        kc, vc = self.caches[layer]
        pkv_append(self.k_new, self.v_new, self.slots, kc, vc, wl.k_scale, wl.v_scale)
        return self.run(layer, out)

    def model_step_start(self):
        """The per-step part: slot mapping of the new rows and the plan."""
        pkv_slot_mapping(self.cu_q, self.seq_lens, self.bt, self.wl.block_size, out=self.slots)
        self.plan()
