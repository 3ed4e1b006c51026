"""Shared set-up for the GPU parity tests: the seeded inputs, the library's drafter with its
state, and the oracle on the same inputs, plus the tolerance checks of the parity bar."""
from __future__ import annotations

import numpy as np
import torch

from block_diffusion_drafter_kv_gb300 import binding as B
from block_diffusion_drafter_kv_gb300.build import build
from oracle.dflash_ref import Oracle
from synth import inputs as I

# Parity bar: layer outputs within 2e-2 max relative error (max |gpu - oracle| / max |oracle|);
# logits within 5e-2 of the oracle logits' standard deviation; drafted tokens equal unless the
# oracle's top-2 logit gap is below 1e-2; acceptance and committed ids bit-exact.
LAYER_RTOL = 2e-2
LOGIT_TOL = 5e-2
GAP_EXEMPT = 1e-2


def max_rel(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(gpu - ref)) / den) if den > 0 else float(np.max(np.abs(gpu)))


def to_np64(t: torch.Tensor) -> np.ndarray:
    """A bf16, fp16 or fp32 tensor as float64 (every value widened exactly)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


class Setup:
    """Drafter on cuda:0 and the oracle, both on the same seeded weights."""

    def __init__(self, workload, seed: int, max_batch: int = None, kv_capacity: int = None):
        build()
        self.w = workload
        s = workload.shape
        self.s = s
        self.seed = seed
        self.weights_cpu = I.make_weights(s, seed, std=workload.weight_std, gain_std=workload.gain_std)
        self.weights = self.weights_cpu.to("cuda")
        self.bits = self.weights_cpu.bits()
        self.cap = kv_capacity or workload.kv_capacity()
        self.max_batch = max_batch or workload.batch
        self.drafter = B.Drafter(s, self.weights, max_block=16, max_batch=self.max_batch, kv_capacity=self.cap)
        self.oracle = Oracle(s, self.bits)
        torch.cuda.synchronize()

    def gpu_inject(self, hidden_cpu: torch.Tensor, n_new, rows_per_seq: int, batch: int):
        """hidden_cpu [k, batch*rows_per_seq, Ht] bf16; n_new list of ints."""
        h = hidden_cpu.to("cuda").contiguous()
        nn = torch.tensor(list(n_new), dtype=torch.int32, device="cuda")
        self.drafter.inject(h, rows_per_seq, nn, batch)

    def gpu_cache(self, seq: int, upto: int):
        k = to_np64(self.drafter.k_cache[:, seq, :upto])
        v = to_np64(self.drafter.v_cache[:, seq, :upto])
        return k, v


def check_draft(ores, gpu_drafted, gpu_logits, gpu_trace):
    """Tolerance checks of one sequence's draft against the oracle's DraftResult.
    Returns the slots whose drafted token legitimately differs (oracle top-2 gap < 1e-2)."""
    tr = max_rel(gpu_trace, ores.x_trace)
    assert tr <= LAYER_RTOL, f"residual trace max rel err {tr:.3e}"
    for l in range(ores.x_trace.shape[0]):
        e = max_rel(gpu_trace[l], ores.x_trace[l])
        assert e <= LAYER_RTOL, f"layer {l} max rel err {e:.3e}"
    excused = []
    if ores.logits.shape[0]:
        dz = np.max(np.abs(np.asarray(gpu_logits, np.float64) - ores.logits))
        sd = np.std(ores.logits)
        assert dz <= LOGIT_TOL * sd, f"logits max err {dz:.3e} vs {LOGIT_TOL} * std {sd:.3e}"
        for i in range(len(ores.drafted)):
            if int(gpu_drafted[i]) != int(ores.drafted[i]):
                assert ores.top2_gap[i] < GAP_EXEMPT, f"slot {i + 1}: drafted {gpu_drafted[i]} vs {ores.drafted[i]}"
                excused.append(i)
    return excused
