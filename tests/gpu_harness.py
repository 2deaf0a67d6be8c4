"""Run the CUDA path on synthetic inputs (torch for device memory only)."""
from __future__ import annotations

import numpy as np


def bf16_tensor(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def upload(d: dict, device="cuda:0"):
    import torch
    x = {name: bf16_tensor(d[name], device) for name in ("q", "k", "v", "g", "beta")}
    x["A_log"] = torch.from_numpy(d["A_log"]).to(device)
    x["dt_bias"] = torch.from_numpy(d["dt_bias"]).to(device)
    s0 = d.get("initial_state")
    if s0 is None:
        x["initial_state"] = None
    elif s0.dtype == np.uint16:
        x["initial_state"] = bf16_tensor(s0, device)
    else:
        x["initial_state"] = torch.from_numpy(s0).to(device)
    cu = d.get("cu_seqlens")
    x["cu_seqlens"] = None if cu is None else torch.from_numpy(cu.astype(np.int32)).to(device)
    return x


def run_gpu(d: dict, final_dtype="f32", device="cuda:0", poison=True, x=None):
    """Run kda_fwd once; returns (out tensor bf16, final_state tensor or None)."""
    import torch
    import gated_delta_rule_39_gb300 as kda
    x = upload(d, device) if x is None else x
    B, T, H, K = d["q"].shape
    out = torch.empty((B, T, H, d["v"].shape[-1]), dtype=torch.bfloat16, device=device)
    if poison:
        out.fill_(float("nan"))
    N = d["N"]
    fs = None
    if final_dtype is not None:
        dt = torch.float32 if final_dtype == "f32" else torch.bfloat16
        fs = torch.full((N, H, K, d["v"].shape[-1]), float("nan"), dtype=dt, device=device)
    kda.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], out, x["A_log"],
                x["dt_bias"], d["lower_bound"], initial_state=x["initial_state"], final_state=fs,
                cu_seqlens=x["cu_seqlens"])
    torch.cuda.synchronize()
    return out, fs


def run_oracle(d: dict, heads=None, initial_state="from_inputs"):
    import oracle
    s0 = d.get("initial_state") if initial_state == "from_inputs" else initial_state
    return oracle.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"],
                          d["dt_bias"], d["lower_bound"], initial_state=s0,
                          cu_seqlens=d.get("cu_seqlens"), heads=heads)
