"""Host <-> device marshalling shared by the GPU tests (no arithmetic)."""
import numpy as np
import torch

import group_wise_affine_gb300 as gwa


def dev_bf16(a_u16: np.ndarray, device="cuda") -> torch.Tensor:
    a = np.ascontiguousarray(a_u16, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def dev_qweight(w, device="cuda") -> gwa.QWeight:
    """gwa_synth.QWeight (host numpy) -> gwa.QWeight (device tensors)."""
    wq = torch.from_numpy(np.ascontiguousarray(w.wq).view(np.int32)).to(device)
    return gwa.QWeight(wq, dev_bf16(w.scales, device), dev_bf16(w.biases, device),
                       w.N, w.K, w.bits, w.group)
