"""Shared test helpers: workload -> oracle config, tensor conversion, error metric."""
import numpy as np
import torch

import oracle
from llama_family_decoder_gb300.synth import Workload

# Parity bounds on max|err| / RMS(oracle output)
TOL = {"f32": 1e-4, "bf16": 2e-2}


def cfg_of(wl: Workload) -> oracle.BlockConfig:
    return oracle.BlockConfig(wl.hidden_size, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.intermediate_size,
                              wl.hidden_act, wl.rms_norm_eps, wl.rope_theta, wl.qk_norm, wl.xielu_alpha_p,
                              wl.xielu_alpha_n,
                              rope_scaling=oracle.RopeScaling(*wl.rope_scaling) if wl.rope_scaling else None,
                              sliding_window=wl.sliding_window, use_rope=wl.use_rope, attn_gate=wl.attn_gate,
                              sandwich_norm=wl.sandwich_norm)


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def weights_np(w: dict) -> dict:
    return {k: np64(v) for k, v in w.items()}


def to_dev(w: dict, device="cuda") -> dict:
    return {k: v.to(device) for k, v in w.items()}


def rel_err(got, ref) -> float:
    """max |got - ref| / RMS(ref)."""
    g = np64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(g - ref)) / np.sqrt(np.mean(ref * ref)))


def bf16_floor(ref) -> float:
    """Error of storing the exact result in bf16 alone (the unavoidable floor)."""
    r = torch.from_numpy(np.asarray(ref, dtype=np.float64))
    return rel_err(r.to(torch.bfloat16), ref)
