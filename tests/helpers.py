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


def check_relu2_zeros(neurons, pre):
    """relu(u)^2 is exactly zero wherever the pre-activation is not positive ("arcee",
    "A neuron is relu(x)^2, exactly zero below zero"). The GPU's pre-activation u differs
    from the oracle's by its GEMM's rounding: with bf16 operands (unit roundoff 2^-8)
    about 0.003 RMS(u) per element over a K-term product, under 0.015 RMS(u) at the 5-sigma
    tail of these sizes. So delta = 0.05 RMS(u): every neuron whose oracle pre-activation
    is <= -delta must be exactly 0.0, every one at >= +delta must be > 0, none negative.
    Where the GPU neuron is positive, sqrt of it is the GPU's own u: its distance from the
    oracle's u must stay below delta / 2, which checks that delta sits above the measured
    error rather than hiding it. Returns (fraction of exact zeros, measured max |du|/RMS)."""
    n = np64(neurons).reshape(-1)
    u = np.asarray(pre, dtype=np.float64).reshape(-1)
    rms = float(np.sqrt(np.mean(u * u)))
    delta = 0.05 * rms
    assert n.min() >= 0.0
    neg, pos = u <= -delta, u >= delta
    assert np.all(n[neg] == 0.0), int(np.sum(n[neg] != 0.0))
    assert np.all(n[pos] > 0.0), int(np.sum(n[pos] == 0.0))
    both = (n > 0) & (u > 0)
    du = float(np.max(np.abs(np.sqrt(n[both]) - u[both]))) / rms if both.any() else 0.0
    assert du <= 0.5 * delta / rms, du
    return float(np.mean(n == 0.0)), du
