"""Shared helpers of the GPU tests: run the CUDA path and the oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import Inputs, bf16_bits_to_f32
from oracle.attention import bf16_bits_to_f64, mla_decode_ref
from oracle.quant import encode_with_scale, per_tensor_scale

# Tolerance of the decode output against the float64 oracle (elementwise
# |gpu - ref| <= ATOL + RTOL * |ref|): the pages' rtol with the stated atol.
RTOL, ATOL = 2e-2, 1e-2
# Diagnostic bound on the relative L2 error of a whole output.
REL_L2_MAX = 1e-2


def num_sms() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def bits_to_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


class DeviceCase:
    """Inputs on the GPU, the cache quantised there by the library."""

    def __init__(self, inp: Inputs, device="cuda"):
        self.inp = inp
        self.q = bits_to_bf16(inp.q_bits, device)
        kv_bf16 = bits_to_bf16(inp.kv_bits, device)
        n = max(1, kv_bf16.shape[0])
        self.kv_codes = torch.empty((n, 576), dtype=torch.uint8, device=device)
        self.kv_scale = torch.empty(1, dtype=torch.float32, device=device)
        tmp = torch.empty(16, dtype=torch.uint8, device=device)
        if kv_bf16.numel():
            binding.mla_fp8_quantize_per_tensor(kv_bf16, self.kv_codes, self.kv_scale, tmp)
        else:
            self.kv_codes.zero_()
            self.kv_scale.fill_(1.0)
        del kv_bf16
        self.qo_indptr = torch.from_numpy(inp.qo_indptr).to(device)
        self.kv_indptr = torch.from_numpy(inp.kv_indptr).to(device)
        self.kv_indices = (None if inp.kv_indices is None
                           else torch.from_numpy(inp.kv_indices).to(device))
        self.out = torch.empty((inp.batch * inp.qo_len, 16, 512), dtype=torch.bfloat16,
                               device=device)

    def run(self, sms: int | None = None, workspace=None, plan=None, persistent: bool = False):
        plan = plan or binding.mla_decode_plan(self.inp.batch, self.inp.max_kv_len,
                                               sms or num_sms(), qo_len=self.inp.qo_len,
                                               persistent=persistent)
        ws = workspace if workspace is not None else binding.new_workspace(plan)
        binding.mla_decode_fwd(self.q, self.kv_codes, self.kv_scale, self.qo_indptr,
                               self.kv_indptr, self.out, plan=plan, workspace=ws,
                               kv_indices=self.kv_indices)
        torch.cuda.synchronize()
        err = binding.mla_decode_read_error(ws)
        return self.out.float().cpu().numpy(), err, plan, ws


class OracleCase:
    """The oracle's own quantisation of the same bf16 cache, and its reference output."""

    def __init__(self, inp: Inputs):
        self.inp = inp
        self.kv_f32 = bf16_bits_to_f32(inp.kv_bits)
        self.scale = per_tensor_scale(self.kv_f32) if self.kv_f32.size else np.float32(1.0)
        self.q = bf16_bits_to_f64(inp.q_bits)

    def codes(self, rows=None):
        if rows is None:
            return encode_with_scale(self.kv_f32, self.scale)
        return encode_with_scale(self.kv_f32[rows], self.scale)

    def reference(self, rows=None):
        """float64 output; with ``rows`` only those batch rows are computed."""
        inp = self.inp
        if rows is None:
            return mla_decode_ref(self.q, self.codes(), self.scale, inp.qo_indptr, inp.kv_indptr,
                                  inp.kv_indices)
        # Encode only the cache rows the sampled batch rows read.
        n = inp.qo_len
        out = np.full((inp.batch * n, 16, 512), np.nan)
        for b in rows:
            j0, j1 = int(inp.kv_indptr[b]), int(inp.kv_indptr[b + 1])
            slots = (np.arange(j0, j1) if inp.kv_indices is None
                     else inp.kv_indices[j0:j1].astype(np.int64))
            codes = encode_with_scale(self.kv_f32[slots], self.scale) if slots.size else \
                np.zeros((0, 576), np.uint8)
            t0 = int(inp.qo_indptr[b])
            sub = mla_decode_ref(self.q[t0:t0 + n], codes, self.scale, np.array([0, n]),
                                 np.array([0, slots.size]))
            out[t0:t0 + n] = sub
        return out


def compare(gpu: np.ndarray, ref: np.ndarray, rows=None) -> dict:
    """Tolerance check plus diagnostics; returns the stats."""
    if rows is not None:
        gpu, ref = gpu[rows], ref[rows]
    diff = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    rel_l2 = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30))
    stats = {"max_abs": float(diff.max()) if diff.size else 0.0, "rel_l2": rel_l2,
             "violations": int((diff > bound).sum()), "finite": bool(np.isfinite(gpu).all())}
    return stats


def assert_close(gpu, ref, rows=None, rel_l2_max=REL_L2_MAX):
    st = compare(gpu, ref, rows)
    assert st["finite"], st
    assert st["violations"] == 0, st
    assert st["rel_l2"] <= rel_l2_max, st
    return st
